"""Pins for the CPU oracle: checks against what the FORGE pages and the
mathematics fix, none of which re-types the oracle's own formulas.

* number formats: exhaustive bf16 round trips, ties-to-even midpoints, and
  PyTorch's independent float32 -> bf16 conversion;
* the weight gradient (Eq. 3): exact rational brute force, a one-hot closed
  form that fails on any transposed or mis-indexed operand, and row subsets;
* AdamW (Algorithm 1): PyTorch's own ``torch.optim.AdamW`` in float64, the
  step-1 sign closed form, and the zero-gradient pure decay;
* int8 moments (Appendix B): exact round trips, the s/2 error bound, block
  locality along the row, the floor of the square-root second moment, and
  the accumulated-error bound s / (2 (1 - beta));
* the standard path's bf16 gradient truncation bias (section 3.1, App. B).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O


def rng(seed=0):
    return np.random.default_rng(seed)


def random_bf16_bits(r, shape, lo_exp=-5, hi_exp=5):
    """bf16 bit patterns with a random sign, exponent in [lo_exp, hi_exp] and
    random 7-bit mantissa."""
    sign = r.integers(0, 2, shape).astype(np.uint16) << 15
    exp = (r.integers(lo_exp, hi_exp + 1, shape) + 127).astype(np.uint16) << 7
    man = r.integers(0, 128, shape).astype(np.uint16)
    return (sign | exp | man).astype(np.uint16)


# ---------------------------------------------------------------------------
# bf16 / fp32 rounding
# ---------------------------------------------------------------------------

def test_bf16_roundtrip_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f64(bits)
    keep = ~np.isnan(vals)
    assert np.array_equal(O.f64_to_bf16(vals[keep]), bits[keep])
    assert np.all(O.f64_to_bf16(vals[~keep]) == 0x7FC0)


def test_bf16_midpoints_round_to_even():
    r = rng(1)
    b = r.integers(0x0001, 0x7F7F, 20000).astype(np.uint16)   # positive finite, not max
    lo, hi = O.bf16_to_f64(b), O.bf16_to_f64(b + 1)
    mid = (lo + hi) / 2                                       # exact in fp64
    even = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(O.f64_to_bf16(mid), even)
    assert np.array_equal(O.f64_to_bf16(-mid), even | np.uint16(0x8000))
    above = np.nextafter(mid, np.inf)
    below = np.nextafter(mid, -np.inf)
    assert np.array_equal(O.f64_to_bf16(above), (b + 1).astype(np.uint16))
    assert np.array_equal(O.f64_to_bf16(below), b)


def test_bf16_matches_torch_from_float32():
    # torch's float32 -> bf16 cast is round-to-nearest-even and independent of the
    # oracle; float32 -> fp64 is exact, so one rounding must give the same bits.
    r = rng(2)
    u = r.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_overflow_and_subnormals():
    maxf = O.bf16_to_f64(np.uint16(0x7F7F))
    assert O.f64_to_bf16(maxf) == 0x7F7F
    assert O.f64_to_bf16(2.0 ** 128) == 0x7F80
    assert O.f64_to_bf16((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80      # tie above max -> inf
    assert O.f64_to_bf16(np.nextafter((2 - 2 ** -8) * 2.0 ** 127, 0)) == 0x7F7F
    assert O.f64_to_bf16(2.0 ** -133) == 0x0001                      # smallest subnormal
    assert O.f64_to_bf16(2.0 ** -134) == 0x0000                      # tie -> even (zero)
    assert O.f64_to_bf16(1.5 * 2.0 ** -134) == 0x0001
    assert O.f64_to_bf16(-np.inf) == 0xFF80
    assert O.f64_to_bf16(-0.0) == 0x8000


def test_f32_rounding_is_nearest_even():
    x = 1.0 + 2.0 ** -24                  # midpoint between 1 and 1 + 2**-23
    assert O.f64_to_f32(x) == np.float32(1.0)
    assert O.f64_to_f32(1.0 + 3 * 2.0 ** -24) == np.float32(1.0 + 2 * 2.0 ** -23)


# ---------------------------------------------------------------------------
# Weight gradient (Eq. 3)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bt,dout,din", [(7, 3, 5), (1, 4, 2), (16, 5, 9)])
def test_wgrad_exact_rational_bruteforce(bt, dout, din):
    r = rng(bt * 100 + dout * 10 + din)
    xb = random_bf16_bits(r, (bt, din))
    db = random_bf16_bits(r, (bt, dout))
    X, dY = O.bf16_to_f64(xb), O.bf16_to_f64(db)
    G = O.wgrad(xb, db)
    assert G.shape == (dout, din)
    for p in range(dout):
        for q in range(din):
            exact = sum(Fraction(dY[t, p]) * Fraction(X[t, q]) for t in range(bt))
            # significands of 16 bits over a 20-bit exponent span: fp64 is exact
            assert Fraction(G[p, q]) == exact, (p, q)


def test_wgrad_one_hot_closed_form():
    # dY[t, p] = c_t when p == pi(t): row p of G is the c-weighted sum of the X
    # rows routed to p.  A transposed or swapped operand gives another shape or
    # other values.
    r = rng(3)
    bt, dout, din = 40, 6, 11
    xb = random_bf16_bits(r, (bt, din))
    X = O.bf16_to_f64(xb)
    pi = r.integers(0, dout, bt)
    c = np.array([1.0, 2.0, -0.5, 0.25])[r.integers(0, 4, bt)]
    dY = np.zeros((bt, dout))
    dY[np.arange(bt), pi] = c
    G = O.wgrad(xb, O.f64_to_bf16(dY))
    for p in range(dout):
        want = np.zeros(din)
        for t in range(bt):
            if pi[t] == p:
                want += c[t] * X[t]
        assert np.array_equal(G[p], want)


def test_wgrad_row_subset_is_exact():
    r = rng(4)
    xb = random_bf16_bits(r, (33, 24))
    db = random_bf16_bits(r, (33, 17))
    rows = np.array([16, 0, 5, 5, 11])
    assert np.array_equal(O.wgrad(xb, db, rows), O.wgrad(xb, db)[rows])
    assert np.array_equal(O.wgrad_abs(xb, db, rows), O.wgrad_abs(xb, db)[rows])


def test_wgrad_abs_bounds_gradient():
    r = rng(5)
    xb = random_bf16_bits(r, (20, 8))
    db = random_bf16_bits(r, (20, 6))
    G, S = O.wgrad(xb, db), O.wgrad_abs(xb, db)
    assert np.all(np.abs(G) <= S)
    pos_x = xb & np.uint16(0x7FFF)
    pos_d = db & np.uint16(0x7FFF)
    assert np.array_equal(O.wgrad(pos_x, pos_d), O.wgrad_abs(xb, db))


def test_wgrad_empty_tokens_is_zero():
    G = O.wgrad(np.zeros((0, 5), np.uint16), np.zeros((0, 3), np.uint16))
    assert G.shape == (3, 5) and np.all(G == 0)


# ---------------------------------------------------------------------------
# Input gradient dX = dY W (backward pass of Y = X W^T)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bt,dout,din", [(5, 3, 4), (1, 6, 2), (9, 7, 7)])
def test_dgrad_exact_rational_bruteforce(bt, dout, din):
    r = rng(bt * 1000 + dout * 10 + din)
    db = random_bf16_bits(r, (bt, dout))
    wb = random_bf16_bits(r, (dout, din))
    dY, W = O.bf16_to_f64(db), O.bf16_to_f64(wb)
    dX = O.dgrad(db, wb)
    assert dX.shape == (bt, din)
    for t in range(bt):
        for q in range(din):
            exact = sum(Fraction(dY[t, p]) * Fraction(W[p, q]) for p in range(dout))
            assert Fraction(dX[t, q]) == exact, (t, q)


@pytest.mark.parametrize("dout,din", [(6, 11), (7, 7)])
def test_dgrad_one_hot_closed_form(dout, din):
    # dY[t, p] = c_t when p == pi(t): row t of dX is c_t times row pi(t) of W.
    # W^T in place of W, reversed rows or a dropped output give other rows.
    r = rng(13 + din)
    bt = 30
    wb = random_bf16_bits(r, (dout, din))
    W = O.bf16_to_f64(wb)
    pi = r.integers(0, dout, bt)
    c = np.array([1.0, -2.0, 0.5, 0.25])[r.integers(0, 4, bt)]
    dY = np.zeros((bt, dout))
    dY[np.arange(bt), pi] = c
    dX = O.dgrad(O.f64_to_bf16(dY), wb)
    for t in range(bt):
        assert np.array_equal(dX[t], c[t] * W[pi[t]]), t


def test_dgrad_and_wgrad_are_adjoint_to_the_forward_pass():
    # For Y = X W^T and a loss gradient dY: <dX, X> = <dY, Y> = <G, W>, with
    # Y formed here from its own definition (section 2.1).  A transposed or
    # swapped operand in either gradient breaks the identity.
    r = rng(17)
    bt, dout, din = 12, 5, 9
    xb = random_bf16_bits(r, (bt, din))
    db = random_bf16_bits(r, (bt, dout))
    wb = random_bf16_bits(r, (dout, din))
    X, dY, W = O.bf16_to_f64(xb), O.bf16_to_f64(db), O.bf16_to_f64(wb)
    Y = np.array([[sum(Fraction(X[t, q]) * Fraction(W[p, q]) for q in range(din))
                   for p in range(dout)] for t in range(bt)], dtype=object)
    dy_y = sum(Fraction(dY[t, p]) * Y[t, p] for t in range(bt) for p in range(dout))
    dx_x = sum(Fraction(v) * Fraction(x) for v, x in zip(O.dgrad(db, wb).ravel(), X.ravel()))
    g_w = sum(Fraction(g) * Fraction(w) for g, w in zip(O.wgrad(xb, db).ravel(), W.ravel()))
    assert dx_x == dy_y and g_w == dy_y


def test_dgrad_row_subset_and_abs():
    r = rng(18)
    db = random_bf16_bits(r, (21, 8))
    wb = random_bf16_bits(r, (8, 13))
    rows = np.array([20, 0, 3, 3])
    assert np.array_equal(O.dgrad(db, wb, rows), O.dgrad(db, wb)[rows])
    dX, S = O.dgrad(db, wb), O.dgrad_abs(db, wb)
    assert np.all(np.abs(dX) <= S)
    assert np.array_equal(O.dgrad(db & np.uint16(0x7FFF), wb & np.uint16(0x7FFF)), S)


def test_linear_backward_reads_the_weight_before_the_update():
    # Algorithm 1 computes dX first: dX comes from W, not from W'
    r = rng(19)
    bt, dout, din = 16, 8, 12
    xb = random_bf16_bits(r, (bt, din))
    db = random_bf16_bits(r, (bt, dout))
    wb = random_bf16_bits(r, (dout, din))
    hyper = O.Hyper(lr=1e-1, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1)
    m = O.zero_moment(O.FMT_FP32, dout, din)
    v = O.zero_moment(O.FMT_FP32, dout, din)
    dx, w1, m1, v1 = O.linear_backward(xb, db, wb, m, v, hyper, 1)
    assert np.array_equal(dx, O.f64_to_bf16(O.dgrad(db, wb)))
    assert not np.array_equal(dx, O.f64_to_bf16(O.dgrad(db, w1)))
    w_only, m_only, _ = O.step(xb, db, wb, m, v, hyper, 1)
    assert np.array_equal(w1, w_only) and np.array_equal(m1.data, m_only.data)


# ---------------------------------------------------------------------------
# AdamW (Algorithm 1)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("t", [1, 2, 10, 1000])
def test_adamw_matches_torch_optim_adamw_f64(t):
    r = rng(10 + t)
    n = 4096
    hyper = O.Hyper(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-6, wd=0.1)
    lr, b1, b2, eps, wd = hyper.as_f64()
    W = r.normal(0, 0.02, n)
    G = r.normal(0, 1e-2, n)
    m = r.normal(0, 3e-3, n) if t > 1 else np.zeros(n)
    v = r.uniform(0, 1e-4, n) if t > 1 else np.zeros(n)
    W1, m1, v1 = O.adamw_f64(G, W, m, v, hyper, t)

    p = torch.nn.Parameter(torch.from_numpy(W.copy()))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                            foreach=False, fused=False)
    p.grad = torch.from_numpy(G.copy())
    if t > 1:
        opt.state[p]["step"] = torch.tensor(float(t - 1), dtype=torch.float64)
        opt.state[p]["exp_avg"] = torch.from_numpy(m.copy())
        opt.state[p]["exp_avg_sq"] = torch.from_numpy(v.copy())
    opt.step()
    st = opt.state[p]
    # atol: a few fp64 ulps of the 0.02-sized terms that cancel in W'
    np.testing.assert_allclose(W1, p.detach().numpy(), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(m1, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-18)
    np.testing.assert_allclose(v1, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-19)


def _bits_from_f64(a):
    return O.f64_to_bf16(a)


def test_step1_moves_each_weight_by_lr_times_sign():
    # t = 1, zero moments, eps = 0: mhat = g and vhat = g^2, so
    # W' = (1 - lr*wd) W - lr * sign(g).  Needs both bias corrections.
    r = rng(20)
    bt, dout, din = 32, 24, 40
    xb = _bits_from_f64(r.normal(0, 1, (bt, din)))
    db = _bits_from_f64(r.normal(0, 0.01, (bt, dout)))
    wb = _bits_from_f64(r.normal(0, 0.02, (dout, din)))
    G = O.wgrad(xb, db)
    assert np.all(G != 0)
    hyper = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=0.0, wd=0.01)
    lr, _, _, _, wd = hyper.as_f64()
    for fmt in (O.FMT_FP32, O.FMT_BF16):
        w1, m1, v1, (_, W1, _, _) = O.step(xb, db, wb, O.zero_moment(fmt, dout, din),
                                          O.zero_moment(fmt, dout, din), hyper, 1,
                                          return_f64=True)
        want = (1 - lr * wd) * O.bf16_to_f64(wb) - lr * np.sign(G)
        np.testing.assert_allclose(W1, want, rtol=0, atol=1e-17)
        assert np.array_equal(w1, O.f64_to_bf16(want))


def test_step1_with_eps_is_close_to_sign_step():
    r = rng(21)
    xb = _bits_from_f64(r.normal(0, 1, (64, 256)))
    db = _bits_from_f64(r.normal(0, 0.01, (64, 128)))
    wb = _bits_from_f64(r.normal(0, 0.02, (128, 256)))
    hyper = O.Hyper()
    lr, b1, b2, eps, wd = hyper.as_f64()
    G = O.wgrad(xb, db)
    _, _, _, (_, W1, m1, v1) = O.step(xb, db, wb, O.zero_moment(0, 128, 256),
                                      O.zero_moment(0, 128, 256), hyper, 1,
                                      return_f64=True)
    move = (1 - lr * wd) * O.bf16_to_f64(wb) - W1
    # |move - lr*sign(g)| = lr * eps / (|g| + eps)
    np.testing.assert_allclose(move, lr * np.sign(G) * np.abs(G) / (np.abs(G) + eps),
                               rtol=1e-12)
    # the float32 betas: 1 - beta1 = 0.1 and 1 - beta2 = 0.001 to within 1.3e-5
    np.testing.assert_allclose(m1, 0.1 * G, rtol=1e-6)
    np.testing.assert_allclose(v1, 0.001 * G * G, rtol=2e-5)
    np.testing.assert_allclose(v1, (1 - b2) * G * G, rtol=1e-14)


@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16, O.FMT_INT8])
def test_zero_gradient_is_pure_decay(fmt):
    r = rng(30)
    bt, dout, din = 16, 8, 256
    xb = _bits_from_f64(r.normal(0, 1, (bt, din)))
    db = np.zeros((bt, dout), np.uint16)
    wb = _bits_from_f64(r.normal(0, 0.02, (dout, din)))
    hyper = O.Hyper(lr=1e-2, wd=0.1)
    lr, _, _, _, wd = hyper.as_f64()
    w1, m1, v1 = O.step(xb, db, wb, O.zero_moment(fmt, dout, din),
                        O.zero_moment(fmt, dout, din), hyper, 1)
    assert np.array_equal(w1, O.f64_to_bf16((1 - lr * wd) * O.bf16_to_f64(wb)))
    assert np.all(O.decode_moment(m1, False) == 0)
    assert np.all(O.decode_moment(v1, True) == 0)


def test_no_tokens_decays_moments():
    # BT = 0 is G = 0 with no special case: m' = beta1 m, v' = beta2 v.
    r = rng(31)
    dout, din, t = 4, 128, 7
    hyper = O.Hyper()
    _, b1, b2, _, _ = hyper.as_f64()
    m = O.Moment(O.FMT_FP32, r.normal(0, 1e-3, (dout, din)).astype(np.float32))
    v = O.Moment(O.FMT_FP32, r.uniform(1e-8, 1e-6, (dout, din)).astype(np.float32))
    wb = _bits_from_f64(r.normal(0, 0.02, (dout, din)))
    _, _, _, (G, _, m1, v1) = O.step(np.zeros((0, din), np.uint16),
                                     np.zeros((0, dout), np.uint16), wb, m, v,
                                     hyper, t, return_f64=True)
    assert np.all(G == 0)
    np.testing.assert_allclose(m1 / m.data.astype(np.float64), b1, rtol=1e-15)
    np.testing.assert_allclose(v1 / v.data.astype(np.float64), b2, rtol=1e-15)


# ---------------------------------------------------------------------------
# int8 moments (Appendix B)
# ---------------------------------------------------------------------------

def test_int8_exactly_representable_block_round_trips():
    r = rng(40)
    s = 2.0 ** -10
    q = r.integers(-127, 128, (3, 256))
    q[:, 5] = 127
    q[:, 200] = -127
    codes, scale = O.quantize_int8_blocks(q * s, floor_one=False)
    assert np.array_equal(codes, q.astype(np.int8))
    assert np.all(scale == np.float32(s))


def test_int8_error_within_half_a_step():
    r = rng(41)
    x = r.normal(0, 1, (16, 512)) * np.exp(r.normal(0, 2, (16, 1)))
    codes, scale = O.quantize_int8_blocks(x, floor_one=False)
    s = np.repeat(scale.astype(np.float64), 128, axis=1)
    err = np.abs(codes * s - x)
    # s/2 plus the float32 rounding of the stored scale
    assert np.all(err <= s / 2 * (1 + 1e-6) + 127 * np.abs(s) * 2.0 ** -24)
    assert codes.min() >= -127 and codes.max() <= 127


def test_int8_blocks_are_128_wide_along_rows():
    x = np.full((2, 384), 1e-3)
    x[0, 130] = 5.0                      # outlier in row 0, block 1
    codes, scale = O.quantize_int8_blocks(x, floor_one=False)
    assert scale.shape == (2, 3)
    assert scale[0, 1] == np.float32(5.0 / 127)
    for (p, b) in [(0, 0), (0, 2), (1, 0), (1, 1), (1, 2)]:
        assert scale[p, b] == np.float32(1e-3 / 127)
        assert np.all(codes[p, 128 * b:128 * b + 128] == 127)


def test_int8_second_moment_floor():
    v = np.full((1, 128), 1e-12)
    v[0, 0] = 1.0
    mom = O.encode_moment(O.FMT_INT8, v, second=True)
    assert np.all(mom.data >= 1) and mom.data[0, 0] == 127
    assert np.all(O.decode_moment(mom, True) > 0)
    zero = O.encode_moment(O.FMT_INT8, np.zeros((1, 128)), second=True)
    assert np.all(zero.data == 0) and np.all(zero.scale == 0)


def test_int8_accumulated_error_bound():
    # Appendix B: with the same gradients, the stored first moment stays within
    # s / (2 (1 - beta1)) of the unquantized one, s the largest scale seen.
    r = rng(42)
    dout, din, steps = 8, 256, 10
    hyper = O.Hyper()
    _, b1, b2, _, _ = hyper.as_f64()
    mq = O.zero_moment(O.FMT_INT8, dout, din)
    vq = O.zero_moment(O.FMT_INT8, dout, din)
    m_exact = np.zeros((dout, din))
    r_exact = np.zeros((dout, din))
    v_exact = np.zeros((dout, din))
    smax_m = np.zeros((dout, din // 128))
    err_r_bound = np.zeros((dout, din))
    for t in range(1, steps + 1):
        G = r.normal(0, 1e-2, (dout, din))
        m1 = b1 * O.decode_moment(mq, False) + (1 - b1) * G
        v1 = b2 * O.decode_moment(vq, True) + (1 - b2) * G * G
        mq = O.encode_moment(O.FMT_INT8, m1, False)
        vq = O.encode_moment(O.FMT_INT8, v1, True)
        m_exact = b1 * m_exact + (1 - b1) * G
        v_exact = b2 * v_exact + (1 - b2) * G * G
        smax_m = np.maximum(smax_m, mq.scale)
        assert np.all(O.decode_moment(vq, True) > 0)
    bound_m = np.repeat(smax_m, 128, axis=1) / (2 * (1 - b1)) * (1 + 1e-5)
    assert np.all(np.abs(O.decode_moment(mq, False) - m_exact) <= bound_m)


# ---------------------------------------------------------------------------
# The standard path's bf16 gradient (section 3.1, Appendix B)
# ---------------------------------------------------------------------------

def test_bf16_gradient_bias_is_undamped():
    # Rounding G to bf16 before the update leaves a relative error in m of the
    # order of the rounding itself (not reduced by (1 - beta1)); the exact path
    # has none.
    r = rng(50)
    bt, dout, din, steps = 64, 32, 256, 20
    hyper = O.Hyper()
    wb = _bits_from_f64(r.normal(0, 0.02, (dout, din)))
    states = {}
    for arm in ("exact", "bf16"):
        states[arm] = [wb, O.zero_moment(0, dout, din), O.zero_moment(0, dout, din)]
    rel = []
    for t in range(1, steps + 1):
        xb = _bits_from_f64(r.normal(0, 1, (bt, din)))
        db = _bits_from_f64(r.normal(0, 1e-3, (bt, dout)))
        G = O.wgrad(xb, db)
        g_err = O.bf16_to_f64(O.f64_to_bf16(G)) - G
        for arm in ("exact", "bf16"):
            w, m, v = states[arm]
            states[arm] = list(O.step(xb, db, w, m, v, hyper, t,
                                      grad_bf16=(arm == "bf16")))
        me = states["exact"][1].data.astype(np.float64)
        mb = states["bf16"][1].data.astype(np.float64)
        rel.append(np.sqrt(np.mean((mb - me) ** 2) / np.mean(me ** 2)))
        grad_rel = np.sqrt(np.mean(g_err ** 2) / np.mean(G ** 2))
    # the exact arm differs from itself by nothing; the bf16 arm keeps an error
    # comparable to the gradient rounding at every step, never damped by 0.1
    assert min(rel) > 0.3 * grad_rel
    assert rel[-1] > 0.3 * grad_rel
    assert grad_rel > 2.0 ** -11
