"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element
by element, on small and ragged shapes, plus the invariants of the FORGE page:
the fused step equals the unfused pair bit for bit (Appendix A,
"Floating-point characterization"), zero gradients give pure decay, BT = 0
has no special case (Remark 1), and the fused call allocates no gradient
memory (Eq. 5)."""
import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs

from .gpu_util import (DEV, gpu_fused, gpu_unfused, ref_inputs, require_gpu, same_moment,
                       hyper_kwargs, dev_state)
from .parity import check_step, tau_bound

pytestmark = pytest.mark.gpu

FMTS = [O.FMT_FP32, O.FMT_BF16, O.FMT_INT8]
TINY = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(params=[("stream", "128", "1"), ("mma", "128", "1"), ("balanced", "128", "1"),
                        ("stream", "256", "1"), ("mma", "256", "1"), ("stream", "256", "2"),
                        ("balanced", "256", "2"), ("mma", "256", "2"), ("deep", "128", "1"),
                        ("deep", "256", "2")],
                ids=lambda p: f"{p[0]}-bn{p[1]}-cta{p[2]}")
def profile(request, tune):
    """Every pipeline profile, tile width and CTA grouping of the tensor-core
    kernel (the library picks them by token count; FORGE_PROFILE, FORGE_BN and
    FORGE_CG force them; 1-CTA int8 moments always use 128-wide tiles)."""
    tune(profile=request.param[0], bn=int(request.param[1]), cg=int(request.param[2]))
    return request.param


def _trajectory(fmt, bt, d_in, d_out, steps, cfg, x_std=1.0, dy_std=0.01, spike=0.0,
                hyper=TINY, rows=None):
    """Run `steps` steps; at each step the GPU starts from the oracle's state
    and both results are compared."""
    inp0 = make_step_inputs(cfg, 0, 0, 0, d_in, d_out, with_w=True)
    w = bf16_bits(inp0.w)
    m = O.zero_moment(fmt, d_out, d_in)
    v = O.zero_moment(fmt, d_out, d_in)
    out = []
    for t in range(1, steps + 1):
        s = make_step_inputs(cfg, 0, t, bt, d_in, d_out, x_std=x_std, dy_std=dy_std,
                             spike_frac=spike)
        ref = ref_inputs(s.x, s.dy, w, m, v)
        gw, gm, gv = gpu_fused(s.x, s.dy, w, m, v, hyper, t)
        rep = check_step(gw, gm, gv, ref, hyper, t, fmt, bt, label=f"fmt{fmt} t{t}")
        out.append(rep)
        w, m, v = O.step(bf16_bits(s.x), bf16_bits(s.dy), w, m, v, hyper, t)
    return out


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_config_three_steps(fmt):
    # X [64, 256] ~ N(0,1), dY [64, 128] ~ N(0, 0.01), W ~ N(0, 0.02), 3 steps
    reps = _trajectory(fmt, 64, 256, 128, 3, cfg=0)
    print(reps)


@pytest.mark.parametrize("fmt,bt,d_in,d_out", [
    (O.FMT_FP32, 200, 264, 392),     # ragged along every axis, several tiles
    (O.FMT_BF16, 200, 264, 392),
    (O.FMT_INT8, 200, 384, 136),
    (O.FMT_FP32, 1, 136, 8),
    (O.FMT_FP32, 63, 512, 256),
    (O.FMT_BF16, 65, 256, 264),
    (O.FMT_INT8, 1000, 256, 256),
])
def test_ragged_shapes(fmt, bt, d_in, d_out, profile):
    _trajectory(fmt, bt, d_in, d_out, 2, cfg=7, dy_std=1e-3, spike=0.02)


@pytest.mark.parametrize("fmt", FMTS)
def test_no_tokens_is_decay_without_special_case(fmt):
    d_in, d_out, t = 256, 136, 4
    inp = make_step_inputs(8, 0, 0, 0, d_in, d_out, with_w=True)
    w = bf16_bits(inp.w)
    rng = np.random.default_rng(3)
    m = O.encode_moment(fmt, rng.normal(0, 1e-3, (d_out, d_in)), False)
    v = O.encode_moment(fmt, rng.uniform(1e-8, 1e-6, (d_out, d_in)), True)
    gw, gm, gv = gpu_fused(inp.x, inp.dy, w, m, v, TINY, t)
    ref = ref_inputs(inp.x, inp.dy, w, m, v)
    check_step(gw, gm, gv, ref, TINY, t, fmt, 0, label="bt0")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(200, 384, 392), (512, 4096, 1024)])
def test_fused_equals_unfused_bitwise(fmt, shape, profile):
    bt, d_in, d_out = shape
    if fmt == O.FMT_INT8 and d_in % 128:
        pytest.skip("int8 needs 128 | d_in")
    s = make_step_inputs(9, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True, spike_frac=0.01)
    w = bf16_bits(s.w)
    rng = np.random.default_rng(4)
    m = O.encode_moment(fmt, rng.normal(0, 1e-4, (d_out, d_in)), False)
    v = O.encode_moment(fmt, rng.uniform(1e-10, 1e-8, (d_out, d_in)), True)
    a = gpu_fused(s.x, s.dy, w, m, v, TINY, 7)
    b = gpu_unfused(s.x, s.dy, w, m, v, TINY, 7)
    assert np.array_equal(a[0], b[0])
    assert same_moment(a[1], b[1])
    assert same_moment(a[2], b[2])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(64, 256, 128), (200, 264, 392), (4096, 512, 256)])
def test_wgrad_against_oracle(dtype, shape, profile):
    bt, d_in, d_out = shape
    s = make_step_inputs(10, 0, 1, bt, d_in, d_out, dy_std=1e-3)
    dW = torch.full((d_out, d_in), float("nan"), dtype=dtype, device=DEV)
    F.wgrad(s.x.to(DEV), s.dy.to(DEV), dW)
    assert F.device_error() == 0
    xb, db = bf16_bits(s.x), bf16_bits(s.dy)
    G, S = O.wgrad(xb, db), O.wgrad_abs(xb, db)
    tau = tau_bound(S, bt)
    if dtype == torch.float32:
        got = dW.cpu().numpy().astype(np.float64)
        err = np.abs(got - G)
        ratio = float(np.max(err / np.maximum(S, 1e-300))) * 2 ** 23
        print(f"max |G_gpu - G| / (2^-23 S) = {ratio:.2f} (bt={bt})")
        assert np.all(err <= tau)
    else:
        from .parity import bf16_ordered
        got = bf16_ordered(bf16_bits(dW.cpu()))
        lo = bf16_ordered(O.f64_to_bf16(G - tau))
        hi = bf16_ordered(O.f64_to_bf16(G + tau))
        assert np.all((got >= lo - 1) & (got <= hi + 1))


def test_wgrad_no_tokens_writes_zeros():
    dW = torch.full((128, 256), 7.0, dtype=torch.float32, device=DEV)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    dy = torch.empty((0, 128), dtype=torch.bfloat16, device=DEV)
    F.wgrad(x, dy, dW)
    torch.cuda.synchronize()
    assert torch.all(dW == 0)


def test_zero_gradient_pure_decay_bit_exact():
    d_in, d_out, bt = 512, 256, 128
    s = make_step_inputs(11, 0, 1, bt, d_in, d_out, with_w=True)
    dy = torch.zeros_like(s.dy)
    w = bf16_bits(s.w)
    gw, gm, gv = gpu_fused(s.x, dy, w, O.zero_moment(0, d_out, d_in),
                           O.zero_moment(0, d_out, d_in), TINY, 1)
    lr, _, _, _, wd = TINY.as_f64()
    want = O.f64_to_bf16((1 - lr * wd) * O.bf16_to_f64(w))
    from .parity import bf16_ulp_diff
    d = bf16_ulp_diff(gw, want)
    assert d.max() <= 1 and np.mean(d == 0) > 0.999
    assert np.all(gm.data == 0) and np.all(gv.data == 0)


def test_deterministic_repeat():
    s = make_step_inputs(12, 0, 1, 777, 384, 392, dy_std=1e-3, with_w=True)
    w = bf16_bits(s.w)
    m = O.zero_moment(0, 392, 384)
    v = O.zero_moment(0, 392, 384)
    a = gpu_fused(s.x, s.dy, w, m, v, TINY, 1)
    b = gpu_fused(s.x, s.dy, w, m, v, TINY, 1)
    assert np.array_equal(a[0], b[0]) and same_moment(a[1], b[1]) and same_moment(a[2], b[2])


def test_fused_allocates_no_gradient_memory():
    d_in, d_out, bt = 4096, 4096, 512
    s = make_step_inputs(13, 0, 1, bt, d_in, d_out, with_w=True)
    X, dY, W = s.x.to(DEV), s.dy.to(DEV), s.w.to(DEV)
    m, v, _, _ = F.alloc_moments(d_out, d_in, F.MOM_FP32, DEV)
    F.wgrad_adamw(X, dY, W, m, v, step=1, **hyper_kwargs(TINY))   # warm-up (descriptors, attrs)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.max_memory_allocated()
    F.wgrad_adamw(X, dY, W, m, v, step=2, **hyper_kwargs(TINY))
    torch.cuda.synchronize()
    assert torch.cuda.max_memory_allocated() - before == 0


def test_guard_bands_untouched():
    # outputs written through TMA with ragged edges: the bytes around every
    # buffer must not change
    bt, d_in, d_out = 130, 264, 136
    s = make_step_inputs(14, 0, 1, bt, d_in, d_out, with_w=True)
    pad = 4096
    n = d_in * d_out

    def guarded(dtype, count, fill):
        buf = torch.full((count + 2 * pad,), fill, dtype=dtype, device=DEV)
        return buf, buf[pad:pad + count]

    wbuf, w = guarded(torch.bfloat16, n, 3.0)
    w.copy_(s.w.reshape(-1).to(DEV))
    mbuf, m = guarded(torch.float32, n, 5.0)
    vbuf, v = guarded(torch.float32, n, 6.0)
    m.zero_()
    v.zero_()
    F.wgrad_adamw(s.x.to(DEV), s.dy.to(DEV), w.view(d_out, d_in), m.view(d_out, d_in),
                  v.view(d_out, d_in), step=1, **hyper_kwargs(TINY))
    torch.cuda.synchronize()
    for buf, fill in ((wbuf, 3.0), (mbuf, 5.0), (vbuf, 6.0)):
        assert torch.all(buf[:pad] == fill) and torch.all(buf[pad + n:] == fill)
    gbuf, g = guarded(torch.float32, n, 9.0)
    F.wgrad(s.x.to(DEV), s.dy.to(DEV), g.view(d_out, d_in))
    torch.cuda.synchronize()
    assert torch.all(gbuf[:pad] == 9.0) and torch.all(gbuf[pad + n:] == 9.0)


def test_bounded_wait_reports_timeout_and_recovers():
    # the testing aid skips one operand arrival: the kernel's waits run out,
    # it records FORGE_ERR_DEVICE_TIMEOUT and returns; the context stays usable
    bt, d_in, d_out = 256, 256, 128
    s = make_step_inputs(15, 0, 1, bt, d_in, d_out, with_w=True)
    w = bf16_bits(s.w)
    W, md, vd, _, _ = dev_state(w, O.zero_moment(0, d_out, d_in), O.zero_moment(0, d_out, d_in))
    F.set_wait_limit_ns(50_000_000)
    try:
        F.debug_drop_first_arrival(True)
        F.wgrad_adamw(s.x.to(DEV), s.dy.to(DEV), W, md, vd, step=1, **hyper_kwargs(TINY))
        assert F.device_error() == 9
        assert F.device_error() == 0      # cleared
    finally:
        F.debug_drop_first_arrival(False)
        F.set_wait_limit_ns(2_000_000_000)
    # a normal call afterwards is correct
    m0, v0 = O.zero_moment(0, d_out, d_in), O.zero_moment(0, d_out, d_in)
    gw, gm, gv = gpu_fused(s.x, s.dy, w, m0, v0, TINY, 1)
    check_step(gw, gm, gv, ref_inputs(s.x, s.dy, w, m0, v0), TINY, 1, 0, bt, label="after")


def _group_case(fmt, shapes, bt, share_x, seed):
    """Host state for several layers; layers with the same d_in share X when
    share_x (as q, k, v do)."""
    layers = []
    xs = {}
    rng = np.random.default_rng(seed)
    for i, (d_out, d_in) in enumerate(shapes):
        s = make_step_inputs(20 + seed, i, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True,
                             spike_frac=0.01)
        x = xs.setdefault(d_in, s.x) if share_x else s.x
        m = O.encode_moment(fmt, rng.normal(0, 1e-4, (d_out, d_in)), False)
        v = O.encode_moment(fmt, rng.uniform(1e-10, 1e-8, (d_out, d_in)), True)
        layers.append(dict(x=x, dy=s.dy, w=bf16_bits(s.w), m=m, v=v))
    return layers


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("bt", [200, 2048])
def test_grouped_equals_separate_calls_bitwise(fmt, bt):
    shapes = [(392, 256), (1024, 512), (136, 256), (256, 384), (512, 512)]
    layers = _group_case(fmt, shapes, bt, share_x=True, seed=1)
    sep = [gpu_fused(l["x"], l["dy"], l["w"], l["m"], l["v"], TINY, 3) for l in layers]
    dev = []
    xdev = {}
    for l in layers:
        W, md, vd, ms, vs = dev_state(l["w"], l["m"], l["v"])
        X = xdev.setdefault(id(l["x"]), l["x"].to(DEV))
        dev.append(dict(X=X, dY=l["dy"].to(DEV), W=W, m=md, v=vd, m_scale=ms, v_scale=vs))
    F.wgrad_adamw_grouped(dev, step=3, **hyper_kwargs(TINY))
    assert F.device_error() == 0
    from .gpu_util import mom_from_dev
    for a, d in zip(sep, dev):
        assert np.array_equal(a[0], bf16_bits(d["W"].cpu()))
        assert same_moment(a[1], mom_from_dev(fmt, d["m"], d["m_scale"]))
        assert same_moment(a[2], mom_from_dev(fmt, d["v"], d["v_scale"]))


def test_grouped_against_oracle_all_profiles(profile):
    fmt = O.FMT_FP32
    shapes = [(264, 136), (128, 256), (392, 264)]
    bt = 130
    layers = _group_case(fmt, shapes, bt, share_x=False, seed=2)
    dev = []
    for l in layers:
        W, md, vd, ms, vs = dev_state(l["w"], l["m"], l["v"])
        dev.append(dict(X=l["x"].to(DEV), dY=l["dy"].to(DEV), W=W, m=md, v=vd))
    F.wgrad_adamw_grouped(dev, step=5, **hyper_kwargs(TINY))
    assert F.device_error() == 0
    from .gpu_util import mom_from_dev
    for l, d in zip(layers, dev):
        ref = ref_inputs(l["x"], l["dy"], l["w"], l["m"], l["v"])
        check_step(bf16_bits(d["W"].cpu()), mom_from_dev(fmt, d["m"], None),
                   mom_from_dev(fmt, d["v"], None), ref, TINY, 5, fmt, bt, label="grouped")


@pytest.mark.parametrize("group_m", [1, 3, 5])
@pytest.mark.parametrize("cg", ["1", "2"])
def test_raster_group_sizes(group_m, cg, tune):
    # tile orders whose last raster group is partial (1000 rows: 8 tiles of
    # 128 or 4 of 256; group sizes 3 and 5 leave remainders) give the same
    # step as the oracle, on one CTA and on CTA pairs
    tune(group_m=group_m, cg=int(cg), profile="balanced")
    fmt = O.FMT_FP32
    shapes = [(1000, 776), (264, 512)]
    bt = 96
    layers = _group_case(fmt, shapes, bt, share_x=False, seed=3)
    dev = []
    for l in layers:
        W, md, vd, ms, vs = dev_state(l["w"], l["m"], l["v"])
        dev.append(dict(X=l["x"].to(DEV), dY=l["dy"].to(DEV), W=W, m=md, v=vd))
    F.wgrad_adamw_grouped(dev, step=2, **hyper_kwargs(TINY))
    assert F.device_error() == 0
    from .gpu_util import mom_from_dev
    for l, d in zip(layers, dev):
        ref = ref_inputs(l["x"], l["dy"], l["w"], l["m"], l["v"])
        check_step(bf16_bits(d["W"].cpu()), mom_from_dev(fmt, d["m"], None),
                   mom_from_dev(fmt, d["v"], None), ref, TINY, 2, fmt, bt,
                   label=f"group_m={group_m} cg={cg}")


@pytest.mark.parametrize("fmt,bt,cfg", [
    (O.FMT_FP32, 4096, ("deep", 256, 2)),     # the configuration that prefetches by default
    (O.FMT_BF16, 1000, ("balanced", 256, 2)),
    (O.FMT_INT8, 300, ("balanced", 128, 1)),  # 8-bit slices: two W boxes per slot
], ids=["fp32-deep-pair", "bf16-balanced-pair", "int8-balanced-cta"])
def test_state_prefetch_changes_no_bits(fmt, bt, cfg, tune):
    # the state loader's L2 prefetch is a hint: with any distance the step is
    # bit for bit the step without it (which the other tests hold to the oracle)
    d_out, d_in = 520, 1024
    s = make_step_inputs(60, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
    tune(profile=cfg[0], bn=cfg[1], cg=cfg[2])
    outs = []
    for pf in (0, 3, 16):
        tune(state_prefetch=pf)
        m, v, ms, vs = F.alloc_moments(d_out, d_in, fmt, DEV)
        W = s.w.to(DEV)
        F.wgrad_adamw(s.x.to(DEV), s.dy.to(DEV), W, m, v, step=2, m_scale=ms, v_scale=vs,
                      **hyper_kwargs(TINY))
        assert F.device_error() == 0
        outs.append([t.contiguous().view(torch.uint8).cpu() for t in (W, m, v, ms, vs)
                     if t is not None])
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b)
