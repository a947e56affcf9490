"""GPU parity of forge_wgrad_accumulate (B' = beta B + dY^T X into fp32)
against the accumulate-mode oracle.

The GPU adds its fp32 accumulator G~ (within tau of the exact G, the bound of
``tests/parity.py``) to beta B with one fused multiply-add, so B' must lie in
the fp32 range the oracle gives over [G - tau, G + tau], widened by one fp32
unit; with integer inputs every step is exact and the results equal the
oracle bit for bit.

The step at the final micro-batch (forge_wgrad_adamw_acc, reading R28)
reads fp32(B + G): against the oracle through the parity checker with the
bound of that sum, and bit for bit against forge_wgrad_accumulate then
forge_adamw."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs

from .gpu_util import (DEV, dev_state, hyper_kwargs, mom_from_dev, require_gpu, same_moment)
from .parity import check_step, tau_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def f32_ordered(x):
    """Monotone integer image of float32 values (+0 and -0 both map to 0)."""
    b = np.asarray(x, np.float32).view(np.int32).astype(np.int64)
    return np.where(b < 0, -(b & 0x7FFFFFFF), b)


def check_accum(gpu, x_bits, dy_bits, B, beta, label=""):
    G = O.wgrad(x_bits, dy_bits)
    tau = tau_bound(O.wgrad_abs(x_bits, dy_bits), x_bits.shape[0])
    b = float(np.float32(beta))
    base = 0.0 if b == 0.0 else b * B.astype(np.float64)
    lo = f32_ordered(O.f64_to_f32(base + G - tau))
    hi = f32_ordered(O.f64_to_f32(base + G + tau))
    g = f32_ordered(gpu)
    bad = int(np.sum((g < lo - 1) | (g > hi + 1)))
    exact = float(np.mean(g == f32_ordered(O.accumulate(x_bits, dy_bits, B, beta))))
    print(label, f"n={g.size} outside={bad} exact={100 * exact:.2f}%")
    assert bad == 0, label


def _case(seed, bt, d_in, d_out):
    s = make_step_inputs(600 + seed, 0, 1, bt, d_in, d_out, dy_std=1e-3, spike_frac=0.01)
    return s.x, s.dy


@pytest.fixture(params=[None, ("stream", "128", "1"), ("balanced", "256", "1"),
                        ("mma", "256", "2")],
                ids=lambda p: "auto" if p is None else f"{p[0]}-bn{p[1]}-cta{p[2]}")
def acc_cfg(request, tune):
    if request.param is not None:
        tune(profile=request.param[0], bn=int(request.param[1]), cg=int(request.param[2]))
    return request.param


@pytest.mark.parametrize("beta", [0.0, 1.0, 0.95])
@pytest.mark.parametrize("bt,d_in,d_out", [(200, 264, 136), (1000, 384, 264)])
def test_accumulate_against_oracle(bt, d_in, d_out, beta, acc_cfg):
    x, dy = _case(1, bt, d_in, d_out)
    B0 = np.random.default_rng(3).normal(0, 1e-2, (d_out, d_in)).astype(np.float32)
    if beta == 0.0:
        B0[:] = np.nan                          # beta = 0 must not read the buffer
    Bd = torch.from_numpy(B0.copy()).to(DEV)
    F.wgrad_accumulate(x.to(DEV), dy.to(DEV), Bd, beta)
    assert F.device_error() == 0
    check_accum(Bd.cpu().numpy(), bf16_bits(x), bf16_bits(dy), B0, beta, label=f"beta={beta}")


def test_beta_zero_equals_the_stored_fp32_gradient():
    # the same main loop and tile choice as forge_wgrad with an fp32 dW
    x, dy = _case(2, 700, 512, 384)
    B = torch.full((384, 512), float("nan"), device=DEV)
    G = torch.empty((384, 512), device=DEV)
    F.wgrad_accumulate(x.to(DEV), dy.to(DEV), B, 0.0)
    F.wgrad(x.to(DEV), dy.to(DEV), G)
    assert F.device_error() == 0
    assert torch.equal(B.view(torch.int32), G.view(torch.int32))


def test_integer_micro_batches_are_exact():
    # small integers: every product and partial sum is exact in fp32, so
    # four micro-batches accumulate to the whole batch's gradient bit for bit
    rng = np.random.default_rng(4)
    bt, d_in, d_out = 512, 256, 136
    x = O.f64_to_bf16(rng.integers(-3, 4, (bt, d_in)).astype(np.float64))
    dy = O.f64_to_bf16(rng.integers(-3, 4, (bt, d_out)).astype(np.float64))
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(DEV)
    dyt = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16).to(DEV)
    B = torch.full((d_out, d_in), float("nan"), device=DEV)
    for i, sl in enumerate(np.array_split(np.arange(bt), 4)):
        F.wgrad_accumulate(xt[sl[0]:sl[-1] + 1], dyt[sl[0]:sl[-1] + 1], B, 0.0 if i == 0 else 1.0)
    assert F.device_error() == 0
    whole = O.bf16_to_f64(dy).T @ O.bf16_to_f64(x)
    np.testing.assert_array_equal(B.cpu().numpy().astype(np.float64), whole)


def test_muon_momentum_steps_and_no_tokens():
    # B <- 0.95 B + G over three fresh micro-batches, each compared from the
    # oracle's own previous B; then a call without tokens scales B exactly
    d_in, d_out = 384, 264
    B = np.random.default_rng(5).normal(0, 1e-2, (d_out, d_in)).astype(np.float32)
    for k in range(3):
        x, dy = _case(10 + k, 300, d_in, d_out)
        Bd = torch.from_numpy(B.copy()).to(DEV)
        F.wgrad_accumulate(x.to(DEV), dy.to(DEV), Bd, 0.95)
        assert F.device_error() == 0
        check_accum(Bd.cpu().numpy(), bf16_bits(x), bf16_bits(dy), B, 0.95, label=f"step {k}")
        B = O.accumulate(bf16_bits(x), bf16_bits(dy), B, 0.95)
    Bd = torch.from_numpy(B.copy()).to(DEV)
    F.wgrad_accumulate(torch.empty((0, d_in), dtype=torch.bfloat16, device=DEV),
                       torch.empty((0, d_out), dtype=torch.bfloat16, device=DEV), Bd, 0.95)
    assert F.device_error() == 0
    want = (np.float64(np.float32(0.95)) * B.astype(np.float64)).astype(np.float32)
    np.testing.assert_array_equal(Bd.cpu().numpy(), want)


def test_exact_accumulation_then_one_step_matches_the_whole_batch():
    # the page's exact-accumulation mode: accumulate k micro-batches in fp32,
    # then one AdamW step on the accumulator (forge_adamw); the result must
    # match the oracle's step on the whole batch within the bars of the
    # fused step, with tau taken over all the batch's tokens plus one fp32
    # rounding per micro-batch
    from .parity import check_step
    bt, d_in, d_out, k = 1024, 256, 136, 4
    s = make_step_inputs(700, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
    m0 = O.zero_moment(O.FMT_FP32, d_out, d_in)
    v0 = O.zero_moment(O.FMT_FP32, d_out, d_in)
    X, dY = s.x.to(DEV), s.dy.to(DEV)
    B = torch.empty((d_out, d_in), device=DEV)
    for i, sl in enumerate(np.array_split(np.arange(bt), k)):
        F.wgrad_accumulate(X[sl[0]:sl[-1] + 1], dY[sl[0]:sl[-1] + 1], B, 0.0 if i == 0 else 1.0)
    W = s.w.to(DEV)
    m = torch.zeros((d_out, d_in), device=DEV)
    v = torch.zeros((d_out, d_in), device=DEV)
    F.adamw(B, W, m, v, step=1, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    assert F.device_error() == 0
    xb, db = bf16_bits(s.x), bf16_bits(s.dy)
    # k micro-batch bounds (ceil(bt_i/16) + 8 each) and k fp32 roundings of the
    # running sum (2^-24 S each): scale S so that check_step's single-batch
    # tau, (ceil(bt/16) + 8) 2^-23 S, covers (ceil(bt/16) + 9k) 2^-23 S
    n16 = math.ceil(bt / 16)
    S = O.wgrad_abs(xb, db) * ((n16 + 9 * k) / (n16 + 8))
    ref = dict(G=O.wgrad(xb, db), S=S, W_bits=bf16_bits(s.w), m=m0, v=v0)
    check_step(bf16_bits(W.cpu()), O.Moment(O.FMT_FP32, m.cpu().numpy()),
               O.Moment(O.FMT_FP32, v.cpu().numpy()), ref, O.Hyper(), 1, O.FMT_FP32, bt,
               label="micro-batches")


# ---------------------------------------------------------------------------
# the step at the final micro-batch (forge_wgrad_adamw_acc): AdamW on
# fp32(B + dY^T X), reading R28
# ---------------------------------------------------------------------------

HYPER = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def _final_case(seed, bt, d_in, d_out, fmt):
    """Inputs of the last micro-batch, the accumulator of three earlier ones
    (formed by the oracle's accumulate), and a warmed state."""
    x, dy = _case(seed, bt, d_in, d_out)
    B = np.zeros((d_out, d_in), np.float32)
    for i in range(3):
        px, pdy = _case(seed + 10 + i, 256, d_in, d_out)
        B = O.accumulate(bf16_bits(px), bf16_bits(pdy), B, 0.0 if i == 0 else 1.0)
    rng = np.random.default_rng(seed)
    w = O.f64_to_bf16(rng.normal(0, 0.02, (d_out, d_in)))
    m = O.encode_moment(fmt, rng.normal(0, 1e-3, (d_out, d_in)), False)
    v = O.encode_moment(fmt, rng.normal(0, 1e-3, (d_out, d_in)) ** 2, True)
    return x, dy, B, w, m, v


def _final_ref(x, dy, B, w, m, v):
    """The parity checker's inputs for the final step: the gradient the step
    reads is fp32(B + G); the GPU's differs from it by the accumulator's
    bound tau plus the roundings of the two fp32 sums (one fp32 unit of
    |B| + |G| + tau, taken as 2^-22 of it)."""
    xb, db = bf16_bits(x), bf16_bits(dy)
    G = O.wgrad(xb, db)
    S = O.wgrad_abs(xb, db)
    tau = tau_bound(S, max(x.shape[0], 1))
    g = O.f64_to_f32(B.astype(np.float64) + G).astype(np.float64)
    tau_g = tau + 2.0 ** -22 * (np.abs(B.astype(np.float64)) + np.abs(G) + tau)
    return dict(G=g, S=S, tau=tau_g, W_bits=w, m=m, v=v)


def _gpu_final(x, dy, B, w, m, v, t):
    W, md, vd, _, _ = dev_state(w, m, v)
    Bd = torch.from_numpy(B.copy()).to(DEV)
    F.wgrad_adamw_acc(x.to(DEV), dy.to(DEV), W, md, vd, Bd, step=t, **hyper_kwargs(HYPER))
    assert F.device_error() == 0
    assert torch.equal(Bd.cpu(), torch.from_numpy(B))   # the accumulator is read only
    return bf16_bits(W.cpu()), mom_from_dev(m.fmt, md, None), mom_from_dev(v.fmt, vd, None)


@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16])
@pytest.mark.parametrize("bt,d_in,d_out", [(192, 384, 256), (1000, 264, 392), (0, 256, 136)])
def test_final_step_against_oracle(bt, d_in, d_out, fmt, acc_cfg):
    x, dy, B, w, m, v = _final_case(20, bt, d_in, d_out, fmt)
    gw, gm, gv = _gpu_final(x, dy, B, w, m, v, 5)
    rep = check_step(gw, gm, gv, _final_ref(x, dy, B, w, m, v), HYPER, 5, fmt, max(bt, 1),
                     label=f"final bt={bt} fmt={fmt}")
    print(rep)
    # the oracle's own function gives the checker's reference W on almost
    # every entry (the rest sit at a rounding boundary of the checked range)
    ow, _, _ = O.step_accumulated(bf16_bits(x), bf16_bits(dy), w, m, v, B, HYPER, 5)
    assert np.mean(ow == gw) > 0.99


@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16])
def test_final_step_equals_accumulate_then_adamw(fmt, acc_cfg):
    # bit for bit: the epilogue's fp32 sum is the accumulate mode's, and the
    # AdamW arithmetic is forge_adamw's
    x, dy, B, w, m, v = _final_case(30, 700, 512, 384, fmt)
    gw, gm, gv = _gpu_final(x, dy, B, w, m, v, 3)
    W, md, vd, _, _ = dev_state(w, m, v)
    Bd = torch.from_numpy(B.copy()).to(DEV)
    F.wgrad_accumulate(x.to(DEV), dy.to(DEV), Bd, 1.0)
    F.adamw(Bd, W, md, vd, step=3, **hyper_kwargs(HYPER))
    assert F.device_error() == 0
    assert np.array_equal(gw, bf16_bits(W.cpu()))
    assert same_moment(gm, mom_from_dev(fmt, md, None))
    assert same_moment(gv, mom_from_dev(fmt, vd, None))


def test_final_step_grouped_equals_separate_calls():
    # three layers of different shapes in one launch against one call each
    shapes = [(384, 256), (512, 128), (256, 384)]
    cases = [_final_case(40 + i, 320, d_in, d_out, O.FMT_BF16) for i, (d_in, d_out) in
             enumerate(shapes)]
    sep = [_gpu_final(*c, 2) for c in cases]
    layers = []
    for x, dy, B, w, m, v in cases:
        W, md, vd, _, _ = dev_state(w, m, v)
        layers.append(dict(X=x.to(DEV), dY=dy.to(DEV), W=W, m=md, v=vd,
                           B=torch.from_numpy(B.copy()).to(DEV)))
    F.wgrad_adamw_acc_grouped(layers, step=2, **hyper_kwargs(HYPER))
    assert F.device_error() == 0
    for ly, (gw, gm, gv) in zip(layers, sep):
        assert np.array_equal(bf16_bits(ly["W"].cpu()), gw)
        assert same_moment(mom_from_dev(O.FMT_BF16, ly["m"], None), gm)
        assert same_moment(mom_from_dev(O.FMT_BF16, ly["v"], None), gv)


def test_final_step_on_llama_gate_at_512_tokens():
    # the gate projection (14336 x 4096) at 512 tokens, fp32 moments: whole
    # tensors against accumulate + adamw, bit for bit
    d_out, d_in, bt = 14336, 4096, 512
    g = torch.Generator(device=DEV)
    g.manual_seed(9)
    X = torch.randn((bt, d_in), generator=g, device=DEV).to(torch.bfloat16)
    dY = (torch.randn((bt, d_out), generator=g, device=DEV) * 1e-3).to(torch.bfloat16)
    W = (torch.randn((d_out, d_in), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    Bacc = torch.randn((d_out, d_in), generator=g, device=DEV) * 1e-2
    m = torch.randn((d_out, d_in), generator=g, device=DEV) * 1e-4
    v = (torch.randn((d_out, d_in), generator=g, device=DEV) * 1e-4) ** 2
    c = [t.clone() for t in (W, m, v, Bacc)]
    F.wgrad_adamw_acc(X, dY, W, m, v, Bacc, step=7, **hyper_kwargs(HYPER))
    F.wgrad_accumulate(X, dY, c[3], 1.0)
    F.adamw(c[3], c[0], c[1], c[2], step=7, **hyper_kwargs(HYPER))
    assert F.device_error() == 0
    assert torch.equal(W.view(torch.int16), c[0].view(torch.int16))
    assert torch.equal(m.view(torch.int32), c[1].view(torch.int32))
    assert torch.equal(v.view(torch.int32), c[2].view(torch.int32))
