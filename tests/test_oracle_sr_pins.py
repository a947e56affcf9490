"""Pins of the stochastic-rounding store oracle (``oracle/sr.py``):

* Philox4x64-10 against NumPy's own ``np.random.Philox`` bit generator
  (independent code; NumPy advances the 256-bit counter by one before each
  block, so its first block is the one at counter + 1);
* stochastic rounding: bf16 values and specials unchanged, the two extreme
  random draws give the two neighbours, and the mean over all 2^16 draws is
  the fp32 value exactly (the unbiasedness that defines the method);
* the SR step: every weight is one of the two bf16 neighbours of the fp32
  update, and with exactly representable updates it is the update itself.
"""
import numpy as np
import pytest

import oracle as O
from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs

MASK = (1 << 64) - 1


def _plus_one(c):
    c = [int(x) for x in c]
    for i in range(4):
        c[i] = (c[i] + 1) & MASK
        if c[i] != 0:
            break
    return c


@pytest.mark.parametrize("key,ctr", [
    ((0, 0), (0, 0, 0, 0)),
    ((0x0123456789ABCDEF, 0xFEDCBA9876543210), (5, 7, 11, 13)),
    ((MASK, MASK), (MASK, 3, MASK, MASK)),           # the increment carries into word 1
    ((42, 0), (MASK, MASK, 0, 9)),                  # ... and into word 2
])
def test_philox_matches_numpy(key, ctr):
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array(ctr, dtype=np.uint64))
    raw = [int(x) for x in bg.random_raw(8)]
    c1 = _plus_one(ctr)
    c2 = _plus_one(c1)
    assert list(O.philox4x64_10(c1, key)) == raw[:4]
    assert list(O.philox4x64_10(c2, key)) == raw[4:]


def test_sr_specials_and_extreme_draws():
    rng = np.random.default_rng(0)
    # bf16 values are unchanged whatever the draw
    b = O.f64_to_bf16(rng.normal(0, 1, 1000))
    x = O.bf16_to_f64(b).astype(np.float32)
    for r in (0, 1, 0x8000, 0xFFFF):
        np.testing.assert_array_equal(O.sr_to_bf16(x, np.full(x.shape, r)), b)
    # specials
    sp = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0], np.float32)
    got = O.sr_to_bf16(sp, np.full(5, 0xFFFF))
    assert list(got[:2]) == [0x7F80, 0xFF80] and got[2] & 0x7FFF > 0x7F80
    assert list(got[3:]) == [0x0000, 0x8000]
    # r = 0 truncates the magnitude, r = 0xFFFF rounds it up (values off the grid)
    y = rng.normal(0, 1, 1000).astype(np.float32)
    y = y[(y.view(np.uint32) & 0xFFFF) != 0]
    lo = O.sr_to_bf16(y, np.zeros(y.shape, np.uint32))
    hi = O.sr_to_bf16(y, np.full(y.shape, 0xFFFF))
    np.testing.assert_array_equal(np.abs(O.bf16_to_f64(lo)) < np.abs(y), True)
    np.testing.assert_array_equal(np.abs(O.bf16_to_f64(hi)) > np.abs(y), True)
    assert np.all((hi.astype(np.int64) & 0x7FFF) - (lo.astype(np.int64) & 0x7FFF) == 1)
    # the largest finite bf16 magnitude rounds up to infinity only when the draw says so
    big = np.array([3.3961e38, -3.3961e38], np.float32)
    assert list(O.sr_to_bf16(big, np.zeros(2, np.uint32))) == [0x7F7F, 0xFF7F]
    assert list(O.sr_to_bf16(big, np.full(2, 0xFFFF))) == [0x7F80, 0xFF80]


def test_sr_is_unbiased_exactly():
    # summed over all 2^16 draws, stochastic rounding returns 2^16 x exactly
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 1, 40), -np.abs(rng.normal(0, 1e-3, 40)),
                        rng.normal(0, 1e20, 4)]).astype(np.float32)
    r = np.arange(1 << 16, dtype=np.uint32)
    for v in x:
        got = O.bf16_to_f64(O.sr_to_bf16(np.full(r.shape, v, np.float32), r))
        assert got.sum() == np.float64(v) * (1 << 16)


def test_sr_bits_take_sixteen_bits_per_element_from_their_block():
    r = O.sr_bits([3, 1000], 40, seed=77, t=5)
    w = O.philox4x64_10((1000, 2, 5, 0), (77, 0))     # columns 32..47 of row 1000
    for q in (32, 33, 37, 39):
        e = q % 16
        assert r[1, q] == (w[e // 4] >> (16 * (e % 4))) & 0xFFFF
    assert r.max() < (1 << 16)
    assert len(np.unique(r)) > 70                      # 80 draws, nearly all distinct


def test_sr_step_lands_on_a_neighbour_of_the_update():
    s = make_step_inputs(800, 0, 1, 64, 48, 24, dy_std=1e-3, with_w=True)
    xb, db, wb = bf16_bits(s.x), bf16_bits(s.dy), bf16_bits(s.w)
    m = O.zero_moment(O.FMT_FP32, 24, 48)
    v = O.zero_moment(O.FMT_FP32, 24, 48)
    h = O.Hyper()
    W1, m1, v1, (G, Wf, mf, vf) = O.step(xb, db, wb, m, v, h, 1, return_f64=True)
    Ws, ms, vs = O.step_sr(xb, db, wb, m, v, h, 1, seed=9)
    w32 = Wf.astype(np.float32)
    lo = O.sr_to_bf16(w32, np.zeros(w32.shape, np.uint32))
    hi = O.sr_to_bf16(w32, np.full(w32.shape, 0xFFFF))
    assert np.all((Ws == lo) | (Ws == hi))
    np.testing.assert_array_equal(ms.data, m1.data)
    np.testing.assert_array_equal(vs.data, v1.data)
    # a different seed or step draws different bits for most off-grid weights
    Ws2, _, _ = O.step_sr(xb, db, wb, m, v, h, 1, seed=10)
    assert np.mean(Ws2 != Ws) > 0.1
