"""The multi-replica path of bench.py on the CPU: two gloo ranks.

With N GPUs the bench runs N independent replicas (the fused step has no
exchange between ranks: every rank updates its own layer), times each with a
barrier on both sides and reports the slowest rank's time; rank 0 alone prints
the JSON line.  These tests run that host logic with the gloo backend."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 1 + r ms in the timed region and 5 - r ms end to end
        t, e = bench.max_over_ranks([1.0 + rank, 5.0 - rank], torch.device("cpu"))
        dist.barrier()
        out[rank] = (t, e)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # every rank sees the slowest rank's time for each quantity
    assert res == {0: (2.0, 5.0), 1: (2.0, 5.0)}


def test_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas, each 1e12 FLOP in 0.5 s (the slowest rank): 4e12 FLOP/s
    assert bench.job_value(2, 1e12, 0.5) == pytest.approx(4e12)
    assert bench.job_value(1, 3.0, 1.5) == pytest.approx(2.0)


def test_reference_arm_under_torchrun_prints_once():
    # the reference arm (the CPU oracle) under a two-rank launch: rank 0 alone
    # runs and prints one JSON line; rank 1 exits 0 without work
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
           "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--reference-budget", "4"]
    env = dict(os.environ, OMP_NUM_THREADS="2", OPENBLAS_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_run_metadata_never_raises_and_serialises():
    # the bench line's `system` record: every field present, unreadable ones null
    import json

    import bench
    meta = bench.run_metadata()
    assert set(meta) == {"gpu", "driver", "cuda", "torch", "kernel_sources", "host_cores"}
    assert meta["kernel_sources"] == bench.source_digest()
    json.dumps(meta)


def test_bench_diagnostic_blocks_from_synthetic_timings():
    # the default line's diagnostic blocks are pure functions of the timings:
    # every key present, fractions consistent, JSON-serialisable
    import json

    import bench

    class FakeLayer:
        def params(self):
            return 218103808

        def h2d_bytes(self):
            return 83886080

    peaks = {"hbm_gbs": 6791.7, "bf16_tflops": 1891.5, "bf16_tflops_sustained": 1702.6}
    layer = FakeLayer()
    opt = bench.optimizers_block({i: 0.5 + 0.1 * i for i in range(7)}, 0, layer, peaks)
    assert opt["states"] == "fp32" and len([k for k in opt if isinstance(opt[k], dict)]) == 7
    nb = layer.params() * (4 + 2 * 4 * 2) + layer.h2d_bytes()     # NAdam: two fp32 states
    assert abs(opt["nadam"]["gbs"] - nb / (opt["nadam"]["ms_per_step"] * 1e-3) / 1e9) < 1e-6
    acc = bench.accumulate_block({1.0: 0.48, 0.0: 0.45}, layer, peaks)
    assert acc["beta_1"]["frac_hbm"] > acc["beta_0"]["frac_hbm"]
    flops = 2.0 * 512 * layer.params()
    bw = bench.backward_block(dict(dgrad_ms=0.25, cublas_dgrad_ms=0.15, linear_backward_ms=1.04,
                                   dgrad_config="tile=256x256 ctas=2 splits=2"),
                              flops, 0.70, peaks, "measured")
    assert abs(bw["dgrad"]["roofline"]["frac"] - flops / 0.25e-3 / 1e12 / 1891.5) < 1e-9
    assert abs(bw["dgrad"]["vs_cublas"] - 0.6) < 1e-9
    json.dumps([opt, acc, bw])


def test_roofline_uses_one_peak_for_the_bound_and_the_fraction():
    import bench
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    # tensor-bound: 223 TFLOP in 0.2 s against the burst peak, sustained reported beside it
    r = bench.roofline_of(223e12 * 0.2, 4e9, 0.2, peaks, "measured")
    assert r["bound"] == "tensor" and r["peak"] == 1900.0
    assert r["frac"] == pytest.approx(223.0 / 1900.0)
    assert r["frac_sustained"] == pytest.approx(223.0 / 1700.0)
    # HBM-bound: 4.45 GB in 0.7 ms
    r = bench.roofline_of(2 * 512 * 218e6, 4.45e9, 0.7e-3, peaks, "measured", traffic=4.4e9)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] == 4.4e9
    assert r["frac"] == pytest.approx(4.45e9 / 0.7e-3 / 1e9 / 6800.0)
    st = bench.launch_stats([1.0, 3.0, 2.0])
    assert st == {"launches": 3, "median_ms": 2.0, "min_ms": 1.0, "max_ms": 3.0, "mean_ms": 2.0}
