"""Pins of the accumulate-mode oracle (``oracle/accum.py``) to things
other than itself: beta = 0 as the plain gradient (with the buffer's old
contents ignored), exactness of integer micro-batches against the whole
batch, closed forms of Muon's momentum accumulate on one-hot inputs, and the
one rounding per call.  The final micro-batch's fused step
(``step_accumulated``) is pinned to AdamW's first-step sign closed form with
an accumulator that flips the last micro-batch's signs, and to ``step`` when
the accumulator is zero and the gradient exact in fp32."""
import numpy as np
import pytest

import oracle as O
from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs


def _ints(rng, shape, lo=-3, hi=4):
    x = rng.integers(lo, hi, shape).astype(np.float32)
    return O.f64_to_bf16(x)          # small integers are exact in bf16


def test_beta_zero_is_the_gradient_and_ignores_the_buffer():
    s = make_step_inputs(500, 0, 1, 48, 40, 24, dy_std=1e-3)
    xb, db = bf16_bits(s.x), bf16_bits(s.dy)
    junk = np.full((24, 40), np.nan, np.float32)
    got = O.accumulate(xb, db, junk, 0.0)
    np.testing.assert_array_equal(got, O.wgrad(xb, db).astype(np.float32))


def test_integer_micro_batches_sum_to_the_whole_batch_exactly():
    # all partial sums are small integers, exact in fp32: accumulating four
    # micro-batches (beta 0, then 1) equals the gradient of the whole batch
    rng = np.random.default_rng(1)
    x = _ints(rng, (64, 40))
    dy = _ints(rng, (64, 24))
    B = np.zeros((24, 40), np.float32)
    for i, sl in enumerate(np.array_split(np.arange(64), 4)):
        B = O.accumulate(x[sl], dy[sl], B, 0.0 if i == 0 else 1.0)
    whole = O.bf16_to_f64(dy).T @ O.bf16_to_f64(x)
    np.testing.assert_array_equal(B.astype(np.float64), whole)


@pytest.mark.parametrize("p,q", [(0, 0), (3, 7), (5, 1)])
def test_muon_momentum_closed_form_on_one_hot_inputs(p, q):
    # one token with dY = 2 e_p and X = 3 e_q gives G = 6 e_p e_q^T:
    # B' = mu B + 6 at (p, q) and mu B elsewhere (mu = 0.5: every product exact)
    dout, din = 6, 8
    x = np.zeros((1, din), np.float32)
    x[0, q] = 3.0
    dy = np.zeros((1, dout), np.float32)
    dy[0, p] = 2.0
    B = np.arange(dout * din, dtype=np.float32).reshape(dout, din)
    got = O.accumulate(O.f64_to_bf16(x), O.f64_to_bf16(dy), B, 0.5)
    want = 0.5 * B
    want[p, q] += 6.0
    np.testing.assert_array_equal(got, want)


def test_no_tokens_scales_the_buffer_and_rounds_once():
    rng = np.random.default_rng(2)
    B = rng.normal(0, 1, (16, 24)).astype(np.float32)
    empty_x = np.zeros((0, 24), np.uint16)
    empty_dy = np.zeros((0, 16), np.uint16)
    got, exact = O.accumulate(empty_x, empty_dy, B, 0.95, return_f64=True)
    b = float(np.float32(0.95))
    np.testing.assert_array_equal(exact, b * B.astype(np.float64))
    np.testing.assert_array_equal(got, (b * B.astype(np.float64)).astype(np.float32))
    # one rounding of the fp64 value, not a rounding of beta B followed by a second one
    s = make_step_inputs(501, 0, 1, 32, 24, 16, dy_std=1e-3)
    xb, db = bf16_bits(s.x), bf16_bits(s.dy)
    got2, exact2 = O.accumulate(xb, db, B, 0.95, return_f64=True)
    np.testing.assert_array_equal(got2, O.f64_to_f32(exact2))
    np.testing.assert_array_equal(exact2, b * B.astype(np.float64) + O.wgrad(xb, db))


def test_final_step_moves_each_weight_against_the_sign_of_the_whole_sum():
    # step 1 from zero moments, no decay, eps far below |g|: every weight
    # moves by exactly lr against the sign of g = B + G_k (Algorithm 1 at t = 1:
    # m-hat = g, v-hat = g^2).  B = -2 G_k (exact: G_k is an integer) flips
    # every sign of the last micro-batch's gradient, so a step that read G_k
    # alone, or B alone with the wrong sign, moves the other way.
    rng = np.random.default_rng(7)
    x = _ints(rng, (16, 12))
    dy = _ints(rng, (16, 10))
    Gk = O.bf16_to_f64(dy).T @ O.bf16_to_f64(x)
    # where G_k = 0 the accumulator alone sets the sign (+1)
    B = np.where(Gk == 0, 1.0, -2.0 * Gk).astype(np.float32)
    w = O.f64_to_bf16(rng.normal(0, 1, (10, 12)))
    h = O.Hyper(lr=2.0 ** -6, beta1=0.9, beta2=0.999, eps=1e-20, wd=0.0)
    z = O.zero_moment(O.FMT_FP32, 10, 12)
    w1, m1, v1 = O.step_accumulated(x, dy, w, z, z, B, h, 1)
    g = B.astype(np.float64) + Gk
    want = O.f64_to_bf16(O.bf16_to_f64(w) - h.lr * np.sign(g))
    np.testing.assert_array_equal(w1, want)
    b1 = h.as_f64()[1]   # beta1 as the fp32 value received
    np.testing.assert_array_equal(m1.data.astype(np.float64),
                                  O.f64_to_f32((1.0 - b1) * g).astype(np.float64))


def test_final_step_with_a_zero_accumulator_is_the_plain_step():
    # integer inputs: G is exact in fp32, so adding a zero accumulator and
    # rounding to fp32 leaves the gradient the plain step reads
    rng = np.random.default_rng(8)
    x = _ints(rng, (24, 16))
    dy = _ints(rng, (24, 8))
    w = O.f64_to_bf16(rng.normal(0, 0.02, (8, 16)))
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
    for fmt in (O.FMT_FP32, O.FMT_BF16, O.FMT_INT8):
        cols = 128 if fmt == O.FMT_INT8 else 16
        xx = x if cols == 16 else _ints(rng, (24, cols))
        ww = w if cols == 16 else O.f64_to_bf16(rng.normal(0, 0.02, (8, cols)))
        m = O.encode_moment(fmt, rng.normal(0, 1e-3, (8, cols)), False)
        v = O.encode_moment(fmt, rng.normal(0, 1e-3, (8, cols)) ** 2, True)
        got = O.step_accumulated(xx, dy, ww, m, v, np.zeros((8, cols), np.float32), h, 3)
        want = O.step(xx, dy, ww, m, v, h, 3)
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_array_equal(got[1].data, want[1].data)
        np.testing.assert_array_equal(got[2].data, want[2].data)


def test_final_step_reads_the_gradient_rounded_to_fp32():
    # B = 1 and G_k = 2^-30 (one token, X = dY = 2^-15): B + G_k rounds to 1.0
    # in fp32, so with beta1 = 1/2 and m = -1 the new first moment is exactly
    # 0.5 (-1) + 0.5 (1) = 0; a step that read the unrounded sum would keep
    # 2^-31 of it (R16, R28: one rounding to fp32 before the optimizer)
    x = O.f64_to_bf16(np.full((1, 1), 2.0 ** -15))
    dy = O.f64_to_bf16(np.full((1, 1), 2.0 ** -15))
    B = np.ones((1, 1), np.float32)
    m = O.Moment(O.FMT_FP32, np.full((1, 1), -1.0, np.float32), None)
    v = O.Moment(O.FMT_FP32, np.ones((1, 1), np.float32), None)
    h = O.Hyper(lr=1e-3, beta1=0.5, beta2=0.5, eps=1e-8, wd=0.0)
    w = O.f64_to_bf16(np.zeros((1, 1)))
    _, m1, v1 = O.step_accumulated(x, dy, w, m, v, B, h, 2)
    assert m1.data[0, 0] == 0.0
    assert v1.data[0, 0] == 1.0      # 0.5 * 1 + 0.5 * 1^2
