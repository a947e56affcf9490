"""GPU parity of fp8 moments with per-tensor delayed scaling
(FORGE_MOM_FP8_E4M3) against the oracle's step_fp8 (oracle/fp8.py, readings
R21-R24): the fused weight-gradient step, the unfused pair, grouped launches
and the scale roll.

Every compared step starts from the oracle's own state: W bits, e4m3 codes of
m and r = sqrt(v), and the read and write scales, which both sides receive
identically.  Bars (the stated tolerance of the 8-bit formats):

* W (bf16): tests/parity.py's check_w: the stated bar (within 1 ulp of the
  oracle's range over G +- tau on at least 99.99 % of entries, never beyond
  2 ulp), and the fp32 bound of the arithmetic for entries where the update
  cancels most of W;
* codes of m and r: within one e4m3 level of the codes the oracle gives over
  G +- tau (the GPU encodes x * (1 / scale) in fp32, the oracle x / scale in
  fp64, so a value near a rounding boundary may land on the neighbour);
* amax: the GPU's max |m'| (max r') lies between the largest of the oracle's
  smallest and the largest of its largest |m'| over G +- tau, widened by
  1e-5 relative (each GPU moment is an fp32 value within that of the exact
  one; the maximum of such values is bounded the same way).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import (LLAMA31_8B_SHAPES, bf16_bits, bits_to_bf16,
                                               make_step_inputs)

from .gpu_util import DEV, hyper_kwargs, require_gpu
from .parity import check_w, oracle_outs, tau_bound

pytestmark = pytest.mark.gpu

HYPER = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
HEADROOM = 2.0


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def e4m3_ordered(codes) -> np.ndarray:
    """Monotone integer image of e4m3 codes (+0 and -0 both map to 0)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


class Fp8State:
    """One moment pair's oracle-side state: codes and the four scale words."""

    def __init__(self, m_codes, r_codes, m_read, m_write, r_read, r_write):
        self.m_codes, self.r_codes = m_codes, r_codes
        self.m_read, self.m_write = np.float32(m_read), np.float32(m_write)
        self.r_read, self.r_write = np.float32(r_read), np.float32(r_write)

    def to_dev(self):
        m = torch.from_numpy(self.m_codes.copy()).view(torch.float8_e4m3fn).to(DEV)
        v = torch.from_numpy(self.r_codes.copy()).view(torch.float8_e4m3fn).to(DEV)
        sc = F.alloc_fp8_scales(2, device=DEV)
        sc[0, 0], sc[0, 1] = float(self.m_read), float(self.m_write)
        sc[1, 0], sc[1, 1] = float(self.r_read), float(self.r_write)
        return m, v, sc


def random_state(d_out, d_in, seed, m_std=1e-4, r_hi=1e-4):
    """A non-trivial moment state: m ~ N(0, m_std), r ~ U(0, r_hi), encoded
    at scales fitted to them; the write scales are the read ones x 1.5."""
    rng = np.random.default_rng(seed)
    m0 = rng.normal(0, m_std, (d_out, d_in))
    r0 = rng.uniform(0, r_hi, (d_out, d_in))
    ms = np.float32(np.max(np.abs(m0)) / 448)
    rs = np.float32(np.max(r0) / 448)
    return Fp8State(O.encode_fp8(m0, ms), O.encode_fp8(r0, rs), ms, ms * 1.5, rs, rs * 1.5)


def oracle_range(x_bits, dy_bits, w_bits, st: Fp8State, t, bt, rows=None):
    """The oracle's fp64 AdamW results over G +- tau for the state (at G
    first; tests/parity.py's oracle_outs)."""
    G = O.wgrad(x_bits, dy_bits, rows)
    tau = tau_bound(O.wgrad_abs(x_bits, dy_bits, rows), bt)
    W = O.bf16_to_f64(w_bits)
    sel = slice(None) if rows is None else rows
    m = O.decode_fp8(st.m_codes[sel], st.m_read)
    r = O.decode_fp8(st.r_codes[sel], st.r_read)
    return oracle_outs(G, tau, W, m, r * r, HYPER, t)


def check_fp8(gpu_w, gpu_m, gpu_r, outs, st: Fp8State, w0_bits, label, amax=None):
    """Compare one GPU step (W bits, m and r codes, optionally the amax pair)
    with the oracle's results over G +- tau (`outs` from oracle_range, at G
    first), W
    under tests/parity.py's check_w; w0_bits: W before the step."""
    rep = {"W": str(check_w(gpu_w, [o[0] for o in outs], O.bf16_to_f64(w0_bits), label))}
    for which, codes, scale in (("m", gpu_m, st.m_write), ("r", gpu_r, st.r_write)):
        vals = [o[1] if which == "m" else np.sqrt(o[2]) for o in outs]
        cs = [e4m3_ordered(O.encode_fp8(x, scale)) for x in vals]
        clo, chi = np.minimum.reduce(cs), np.maximum.reduce(cs)
        gc = e4m3_ordered(codes)
        bad = (gc < clo - 1) | (gc > chi + 1)
        rep[which] = (f"max code diff {int(np.max(np.abs(gc - cs[0])))}, "
                      f"exact {100.0 * np.mean(gc == cs[0]):.3f}%")
        assert not bad.any(), f"{label} {which} codes: {int(bad.sum())} beyond one level"
        if amax is not None:
            mags = np.stack([np.abs(x) for x in vals])
            lo = np.max(np.min(mags, axis=0)) * (1 - 1e-5)
            hi = np.max(np.max(mags, axis=0)) * (1 + 1e-5)
            a = float(amax[0 if which == "m" else 1])
            assert lo <= a <= hi, f"{label} amax {which}: {a} not in [{lo}, {hi}]"
    return rep


def gpu_step(x, dy, w_bits, st: Fp8State, t):
    """One fused fp8 step on the GPU from the oracle-side state.  Returns W
    bits, m and r codes and the (amax_m, amax_r) words, on the host."""
    W = bits_to_bf16(w_bits).to(DEV)
    m, v, sc = st.to_dev()
    F.wgrad_adamw(x.to(DEV), dy.to(DEV), W, m, v, step=t, m_scale=sc[0], v_scale=sc[1],
                  **hyper_kwargs(HYPER))
    s = F.device_error()
    assert s == 0, F.status_string(s)
    return (bf16_bits(W.cpu()), m.view(torch.uint8).cpu().numpy(),
            v.view(torch.uint8).cpu().numpy(), sc[:, 2].cpu().numpy())


def first_write_scales(x_bits, dy_bits, w_bits, d_out, d_in):
    """Write scales for a first step from zero moments: the oracle's own
    amaxes of that step (a just-in-time first scale; R23 leaves the first
    step's scale to the caller) with the test's headroom."""
    z = np.zeros((d_out, d_in), dtype=np.uint8)
    *_, am, ar = O.step_fp8(x_bits, dy_bits, w_bits, z, 1.0, z, 1.0, 1.0, 1.0, HYPER, 1)
    return (O.roll_fp8_scales(1.0, 1.0, am, HEADROOM)[1],
            O.roll_fp8_scales(1.0, 1.0, ar, HEADROOM)[1])


def test_fp8_tiny_three_steps_delayed_scaling():
    # the tiny configuration, three steps with fresh inputs; each step starts
    # from the oracle's state and its scales roll by R24 from the oracle's
    # amaxes (the same scales go to both sides)
    bt, d_in, d_out = 64, 256, 128
    s1 = make_step_inputs(1, 0, 1, bt, d_in, d_out, dy_std=0.01, with_w=True)
    w = bf16_bits(s1.w)
    z = np.zeros((d_out, d_in), dtype=np.uint8)
    mw, rw = first_write_scales(bf16_bits(s1.x), bf16_bits(s1.dy), w, d_out, d_in)
    st = Fp8State(z, z, 1.0, mw, 1.0, rw)
    for t in range(1, 4):
        s = s1 if t == 1 else make_step_inputs(1, 0, t, bt, d_in, d_out, dy_std=0.01)
        xb, db = bf16_bits(s.x), bf16_bits(s.dy)
        gw, gm, gr, ga = gpu_step(s.x, s.dy, w, st, t)
        rep = check_fp8(gw, gm, gr, oracle_range(xb, db, w, st, t, bt), st, w, f"tiny t={t}",
                        amax=ga)
        print("tiny", t, rep)
        w, mc, rc, am, ar = O.step_fp8(xb, db, w, st.m_codes, st.m_read, st.r_codes, st.r_read,
                                       st.m_write, st.r_write, HYPER, t)
        m_next = O.roll_fp8_scales(st.m_read, st.m_write, am, HEADROOM)
        r_next = O.roll_fp8_scales(st.r_read, st.r_write, ar, HEADROOM)
        st = Fp8State(mc, rc, m_next[0], m_next[1], r_next[0], r_next[1])


@pytest.fixture(params=[None, ("stream", 128, 1), ("balanced", 128, 1), ("mma", 256, 2),
                        ("balanced", 256, 2)],
                ids=lambda p: "auto" if p is None else f"{p[0]}-bn{p[1]}-cta{p[2]}")
def f8_cfg(request, tune):
    if request.param is not None:
        tune(profile=request.param[0], bn=request.param[1], cg=request.param[2])
    return request.param


@pytest.mark.parametrize("bt,d_in,d_out", [(65, 272, 136), (200, 400, 264), (1000, 512, 392)])
def test_fp8_ragged_shapes_every_profile(bt, d_in, d_out, f8_cfg):
    # widths that are multiples of 16 but not of the 128-column slice, rows
    # past a tile edge, token counts with a partial last stage
    s = make_step_inputs(31, 0, 3, bt, d_in, d_out, dy_std=1e-3, with_w=True, spike_frac=0.01)
    xb, db, w = bf16_bits(s.x), bf16_bits(s.dy), bf16_bits(s.w)
    st = random_state(d_out, d_in, seed=bt)
    gw, gm, gr, ga = gpu_step(s.x, s.dy, w, st, 3)
    rep = check_fp8(gw, gm, gr, oracle_range(xb, db, w, st, 3, bt), st, w,
                    f"ragged {bt}x{d_in}x{d_out} {f8_cfg}", amax=ga)
    print(bt, d_in, d_out, f8_cfg, rep)


@pytest.mark.parametrize("bt", [0, 96, 1500])
def test_fp8_fused_equals_unfused_pair(bt):
    # forge_wgrad (fp32) + forge_adamw give the fused call's bits: W, codes
    # and both amax words (Appendix A, "Floating-point characterization");
    # with no tokens the fused call itself is forge_adamw with a zero gradient
    d_in, d_out = 1040, 520
    s = make_step_inputs(32, 0, 2, bt, d_in, d_out, dy_std=1e-3, with_w=True)
    st = random_state(d_out, d_in, seed=7)
    outs = []
    for arm in ("fused", "unfused"):
        W = s.w.to(DEV)
        m, v, sc = st.to_dev()
        X, dY = s.x.to(DEV), s.dy.to(DEV)
        if arm == "fused":
            F.wgrad_adamw(X, dY, W, m, v, step=2, m_scale=sc[0], v_scale=sc[1],
                          **hyper_kwargs(HYPER))
        else:
            dW = torch.empty((d_out, d_in), dtype=torch.float32, device=DEV)
            F.wgrad(X, dY, dW)
            F.adamw(dW, W, m, v, step=2, m_scale=sc[0], v_scale=sc[1], **hyper_kwargs(HYPER))
        assert F.device_error() == 0
        outs.append((W.view(torch.int16).cpu(), m.view(torch.uint8).cpu(),
                     v.view(torch.uint8).cpu(), sc.view(torch.int32).cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    xb, db, w = bf16_bits(s.x), bf16_bits(s.dy), bf16_bits(s.w)
    check_fp8(outs[0][0].numpy().view(np.uint16), outs[0][1].numpy(), outs[0][2].numpy(),
              oracle_range(xb, db, w, st, 2, bt), st, w, f"fused bt={bt}",
              amax=outs[0][3].view(torch.float32)[:, 2].numpy())


def test_fp8_grouped_equals_separate_calls():
    # a grouped launch over layers of different shapes raises each layer's
    # own amax words, bit for bit as separate calls do
    bt = 256
    shapes = [(264, 512), (1024, 1040), (136, 272), (520, 2048)]
    runs = []
    for grouped in (True, False):
        layers = []
        for i, (d_out, d_in) in enumerate(shapes):
            s = make_step_inputs(33, i, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
            m, v, sc = random_state(d_out, d_in, seed=40 + i).to_dev()
            layers.append(dict(X=s.x.to(DEV), dY=s.dy.to(DEV), W=s.w.to(DEV), m=m, v=v,
                               m_scale=sc[0], v_scale=sc[1], sc=sc))
        if grouped:
            F.wgrad_adamw_grouped([{k: v for k, v in ly.items() if k != "sc"} for ly in layers],
                                  step=4, **hyper_kwargs(HYPER))
        else:
            for ly in layers:
                F.wgrad_adamw(ly["X"], ly["dY"], ly["W"], ly["m"], ly["v"], step=4,
                              m_scale=ly["m_scale"], v_scale=ly["v_scale"],
                              **hyper_kwargs(HYPER))
        assert F.device_error() == 0
        runs.append(layers)
    for a, b in zip(*runs):
        for k in ("W", "m", "v", "sc"):
            assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k


def test_fp8_roll_kernel_matches_the_oracle_roll():
    # read <- write, write <- amax * headroom / 448 (amax > 0), amax <- 0
    rng = np.random.default_rng(5)
    n = 300
    words = np.zeros((n, 4), dtype=np.float32)
    words[:, 0] = rng.uniform(1e-9, 1e-3, n)
    words[:, 1] = rng.uniform(1e-9, 1e-3, n)
    words[:, 2] = rng.uniform(0, 0.5, n).astype(np.float32)
    words[::7, 2] = 0.0
    for headroom in (1.0, 2.0, 1.37):
        d = torch.from_numpy(words.copy()).to(DEV)
        F.fp8_roll_scales(d, headroom)
        got = d.cpu().numpy()
        for i in range(n):
            r, w = O.roll_fp8_scales(words[i, 0], words[i, 1], words[i, 2], headroom)
            assert got[i, 0].view(np.uint32) == np.float32(r).view(np.uint32)
            assert got[i, 1].view(np.uint32) == np.float32(w).view(np.uint32), (i, headroom)
            assert got[i, 2] == 0.0
    with pytest.raises(F.ForgeError):
        F.fp8_roll_scales(torch.zeros((2, 4), device=DEV), 0.5)


def test_fp8_ten_step_trajectory():
    # ten steps of delayed scaling: each step starts from the oracle's state
    # with the scales its amax history gives (R24, headroom 2); after the
    # GPU's step, its own scale words roll on the device exactly as the
    # oracle's roll of the same words
    bt, d_in, d_out = 512, 512, 256
    s1 = make_step_inputs(34, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True, spike_frac=0.01)
    w = bf16_bits(s1.w)
    z = np.zeros((d_out, d_in), dtype=np.uint8)
    mw, rw = first_write_scales(bf16_bits(s1.x), bf16_bits(s1.dy), w, d_out, d_in)
    st = Fp8State(z, z, 1.0, mw, 1.0, rw)
    for t in range(1, 11):
        s = s1 if t == 1 else make_step_inputs(34, 0, t, bt, d_in, d_out, dy_std=1e-3,
                                               spike_frac=0.01)
        xb, db = bf16_bits(s.x), bf16_bits(s.dy)
        W = bits_to_bf16(w).to(DEV)
        m, v, sc = st.to_dev()
        F.wgrad_adamw(s.x.to(DEV), s.dy.to(DEV), W, m, v, step=t, m_scale=sc[0],
                      v_scale=sc[1], **hyper_kwargs(HYPER))
        assert F.device_error() == 0
        words = sc.cpu().numpy()
        check_fp8(bf16_bits(W.cpu()), m.view(torch.uint8).cpu().numpy(),
                  v.view(torch.uint8).cpu().numpy(), oracle_range(xb, db, w, st, t, bt), st, w,
                  f"trajectory t={t}", amax=words[:, 2])
        F.fp8_roll_scales(sc, HEADROOM)
        rolled = sc.cpu().numpy()
        for k in range(2):
            r_, w_ = O.roll_fp8_scales(words[k, 0], words[k, 1], words[k, 2], HEADROOM)
            assert rolled[k, 0] == r_ and rolled[k, 1] == w_ and rolled[k, 2] == 0.0
        w, mc, rc, am, ar = O.step_fp8(xb, db, w, st.m_codes, st.m_read, st.r_codes, st.r_read,
                                       st.m_write, st.r_write, HYPER, t)
        m_next = O.roll_fp8_scales(st.m_read, st.m_write, am, HEADROOM)
        r_next = O.roll_fp8_scales(st.r_read, st.r_write, ar, HEADROOM)
        st = Fp8State(mc, rc, m_next[0], m_next[1], r_next[0], r_next[1])


def test_fp8_llama_layer_bt512():
    # the seven Llama-3.1-8B projections at 512 tokens in one grouped launch,
    # the first step from zero moments, as the bench times it.  The oracle
    # forms every projection's whole gradient G (and sum |dY X| for tau):
    # with zero moments m' = (1 - beta1) g and r' = sqrt(1 - beta2) |g|, so
    # the amax bounds over G +- tau are closed forms of max |G| -+ tau.
    # Sampled rows are compared element by element; the whole tensors equal
    # the unfused pair's bit for bit.
    bt, t = 512, 1
    b1, b2 = HYPER.beta1, HYPER.beta2
    layers, copies, host = [], [], []
    for i, (name, d_out, d_in) in enumerate(LLAMA31_8B_SHAPES):
        s = make_step_inputs(4, i, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
        xb, db = bf16_bits(s.x), bf16_bits(s.dy)
        G = O.wgrad(xb, db)
        tau = tau_bound(O.wgrad_abs(xb, db), bt)
        gmax_lo = float(np.max(np.maximum(np.abs(G) - tau, 0.0)))
        gmax_hi = float(np.max(np.abs(G) + tau))
        del tau
        gmax = float(np.max(np.abs(G)))
        del G
        mw = O.roll_fp8_scales(1.0, 1.0, np.float32((1 - b1) * gmax), HEADROOM)[1]
        rw = O.roll_fp8_scales(1.0, 1.0, np.float32(math.sqrt(1 - b2) * gmax), HEADROOM)[1]
        z = np.zeros((d_out, d_in), dtype=np.uint8)
        st = Fp8State(z, z, 1.0, mw, 1.0, rw)
        for arm in (layers, copies):
            m, v, sc = st.to_dev()
            arm.append(dict(X=s.x.to(DEV), dY=s.dy.to(DEV), W=s.w.to(DEV), m=m, v=v,
                            m_scale=sc[0], v_scale=sc[1], sc=sc))
        host.append(dict(name=name, s=s, st=st, bounds=(gmax_lo, gmax_hi)))
    F.wgrad_adamw_grouped([{k: v for k, v in ly.items() if k != "sc"} for ly in layers],
                          step=t, **hyper_kwargs(HYPER))
    dw = torch.empty(14336 * 4096, dtype=torch.float32, device=DEV)
    for c in copies:
        g = dw[:c["W"].numel()].view(c["W"].shape)
        F.wgrad(c["X"], c["dY"], g)
        F.adamw(g, c["W"], c["m"], c["v"], step=t, m_scale=c["m_scale"], v_scale=c["v_scale"],
                **hyper_kwargs(HYPER))
    assert F.device_error() == 0
    for ly, c, h in zip(layers, copies, host):
        for k in ("W", "m", "v", "sc"):
            assert torch.equal(ly[k].view(torch.uint8), c[k].view(torch.uint8)), (h["name"], k)
        amax = ly["sc"][:, 2].cpu().numpy().astype(np.float64)
        lo, hi = h["bounds"]
        for k, f in enumerate((1 - b1, math.sqrt(1 - b2))):
            assert f * lo * (1 - 1e-5) <= amax[k] <= f * hi * (1 + 1e-5), (h["name"], k, amax[k])
        d_out = ly["W"].shape[0]
        rows = np.array(sorted({0, 127, 128, 255, 256, d_out // 2, d_out - 1}))
        st = h["st"]
        sub = Fp8State(st.m_codes[rows], st.r_codes[rows], st.m_read, st.m_write, st.r_read,
                       st.r_write)
        xb, db = bf16_bits(h["s"].x), bf16_bits(h["s"].dy)
        w = bf16_bits(h["s"].w)[rows]
        outs = oracle_range(xb, db, w, st, t, bt, rows=rows)
        rep = check_fp8(bf16_bits(ly["W"][rows].cpu()),
                        ly["m"].view(torch.uint8)[rows].cpu().numpy(),
                        ly["v"].view(torch.uint8)[rows].cpu().numpy(), outs, sub, w,
                        f"llama fp8 {h['name']}")
        print("llama fp8", h["name"], rep, amax)
