"""GPU parity of forge_wgrad_adamw_sr (the bf16 weight committed by
stochastic rounding, Philox4x64-10 random bits) against the SR oracle.

The kernel forms the update in fp32; the oracle rounds its fp64 update to
fp32 and then applies the same random bits.  Where the two fp32 updates
differ (by about one fp32 unit) the stochastic decision can differ, so the
weights must be within one bf16 ulp everywhere and equal nearly everywhere;
the moments follow the fused step's bars.  The method's defining property,
unbiasedness, is checked on the GPU over many seeds."""
import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import bf16_bits, bits_to_bf16, make_step_inputs

from .gpu_util import DEV, dev_state, hyper_kwargs, mom_from_dev, ref_inputs, require_gpu
from .parity import bf16_ordered, check_step

pytestmark = pytest.mark.gpu

H = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _state(fmt, d_out, d_in, seed):
    rng = np.random.default_rng(seed)
    m = O.encode_moment(fmt, rng.normal(0, 1e-4, (d_out, d_in)), False)
    v = O.encode_moment(fmt, rng.uniform(1e-10, 1e-8, (d_out, d_in)), True)
    return m, v


@pytest.fixture(params=[None, ("stream", "128", "1"), ("balanced", "128", "1"),
                        ("deep", "256", "2"), ("mma", "256", "2")],
                ids=lambda p: "auto" if p is None else f"{p[0]}-bn{p[1]}-cta{p[2]}")
def sr_cfg(request, tune):
    if request.param is not None:
        tune(profile=request.param[0], bn=int(request.param[1]), cg=int(request.param[2]))
    return request.param


def _compare(bt, d_in, d_out, t, fmt):
    s = make_step_inputs(900 + bt, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
    w_bits = bf16_bits(s.w)
    m, v = _state(fmt, d_out, d_in, bt + fmt)
    W, md, vd, ms, vs = dev_state(w_bits, m, v)
    seed = 0x1234_5678_9ABC_DEF0 + bt
    F.wgrad_adamw_sr(s.x.to(DEV), s.dy.to(DEV), W, md, vd, step=t, seed=seed, **hyper_kwargs(H))
    assert F.device_error() == 0
    gw = bf16_bits(W.cpu())
    ow, om, ov = O.step_sr(bf16_bits(s.x), bf16_bits(s.dy), w_bits, m, v, H, t, seed)
    d = np.abs(bf16_ordered(gw) - bf16_ordered(ow))
    print(f"bt={bt} max ulp {d.max()} exact {100 * np.mean(d == 0):.3f}%")
    assert d.max() <= 1 and np.mean(d == 0) >= 0.999
    # moments: the fused step's bars (W there is only checked to within 1 ulp
    # of the round-to-nearest range, which every stochastic result satisfies)
    check_step(gw, mom_from_dev(fmt, md, ms), mom_from_dev(fmt, vd, vs),
               ref_inputs(s.x, s.dy, w_bits, m, v), H, t, fmt, max(bt, 1), label="sr")


@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("bt,d_in,d_out,t", [(200, 264, 136, 3), (1000, 384, 264, 9)])
def test_sr_step_against_oracle(bt, d_in, d_out, t, fmt, sr_cfg):
    _compare(bt, d_in, d_out, t, fmt)


@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16], ids=["fp32", "bf16"])
def test_sr_step_without_tokens(fmt):
    # G = 0 (one CTA, the library's choice): decay and the moment-driven
    # update, still committed stochastically
    _compare(0, 256, 136, 2, fmt)


def test_sr_is_unbiased_and_not_round_to_nearest():
    # 64 seeds of the same step: the mean committed weight approaches the fp32
    # update (the oracle's), while round to nearest keeps its bias
    bt, d_in, d_out, t = 256, 256, 128, 1
    s = make_step_inputs(950, 0, 1, bt, d_in, d_out, dy_std=1e-2, with_w=True)
    w_bits = bf16_bits(s.w)
    m = O.zero_moment(O.FMT_FP32, d_out, d_in)
    v = O.zero_moment(O.FMT_FP32, d_out, d_in)
    h = O.Hyper(lr=3e-3, wd=0.0)
    _, _, _, (G, Wf, _, _) = O.step(bf16_bits(s.x), bf16_bits(s.dy), w_bits, m, v, h, t,
                                    return_f64=True)
    w32 = Wf.astype(np.float32).astype(np.float64)
    X, dY = s.x.to(DEV), s.dy.to(DEV)
    acc = np.zeros((d_out, d_in))
    n = 64
    for k in range(n):
        W = bits_to_bf16(w_bits).to(DEV)
        md = torch.zeros((d_out, d_in), device=DEV)
        vd = torch.zeros((d_out, d_in), device=DEV)
        F.wgrad_adamw_sr(X, dY, W, md, vd, step=t, seed=1000 + k, **hyper_kwargs(h))
        acc += O.bf16_to_f64(bf16_bits(W.cpu()))
    assert F.device_error() == 0
    mean = acc / n
    rne = O.bf16_to_f64(O.f64_to_bf16(w32))
    ulp = np.abs(O.bf16_to_f64(O.f64_to_bf16(w32) + 1) - rne)
    off = np.abs(w32 - rne) > 0.25 * ulp          # updates well off the bf16 grid
    err_sr = np.mean(np.abs(mean - w32)[off] / ulp[off])
    err_rne = np.mean(np.abs(rne - w32)[off] / ulp[off])
    print(f"mean |SR mean - fp32| {err_sr:.3f} ulp, |RNE - fp32| {err_rne:.3f} ulp")
    # 64 Bernoulli draws: the mean errs by about 0.5 / sqrt(64) = 0.06 ulp
    assert err_sr < 0.1 and err_rne > 0.3


def test_sr_is_deterministic_per_seed():
    s = make_step_inputs(960, 0, 1, 300, 512, 256, dy_std=1e-3, with_w=True)
    X, dY = s.x.to(DEV), s.dy.to(DEV)
    outs = []
    for seed in (5, 5, 6):
        W = s.w.to(DEV)
        m = torch.zeros((256, 512), device=DEV)
        v = torch.zeros((256, 512), device=DEV)
        F.wgrad_adamw_sr(X, dY, W, m, v, step=4, seed=seed, **hyper_kwargs(H))
        outs.append(W.view(torch.int16).clone())
    assert F.device_error() == 0
    assert torch.equal(outs[0], outs[1])
    assert not torch.equal(outs[0], outs[2])
