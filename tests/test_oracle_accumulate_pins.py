"""Pins of the accumulate-mode oracle (``oracle/accum.py``) to things
other than itself: beta = 0 as the plain gradient (with the buffer's old
contents ignored), exactness of integer micro-batches against the whole
batch, closed forms of Muon's momentum accumulate on one-hot inputs, and the
one rounding per call."""
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
