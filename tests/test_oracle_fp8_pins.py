"""Pins of the fp8-moment oracle (``oracle/fp8.py``):

* e4m3 encoding against PyTorch's own ``float8_e4m3fn`` cast (independent
  code) on in-range fp32 values, normal and subnormal, and decoding of all
  256 codes against PyTorch's;
* saturation at +-448 and the exact round trip of every code;
* per-tensor scaling: power-of-two scales move only the exponent;
* the step: decoded moments within half an e4m3 step of the fp64 AdamW
  moments, and the reported amaxes equal to those of the fp64 moments;
* the scale roll: an amax of exactly 448 / headroom gives a write scale of
  exactly 1, a moment at the old amax lands on the largest code after the
  roll, and a zero amax keeps the old scale.
"""
import warnings

import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs


def test_encoding_matches_torch_float8_e4m3fn():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 50, 4000), rng.uniform(-448, 448, 4000),
                        rng.normal(0, 1e-2, 4000), rng.normal(0, 1e-3, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.f64_to_e4m3(x.astype(np.float64)), ref)


def test_decoding_all_codes_matches_torch_and_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    dec = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = (dec == ref) | (np.isnan(dec) & np.isnan(ref))
    assert same.all()
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        back = O.f64_to_e4m3(dec)
    assert np.all((back == codes) | np.isnan(dec))
    assert np.nanmax(dec) == O.E4M3_MAX and np.nanmin(dec) == -O.E4M3_MAX


def test_saturation_and_power_of_two_scales():
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        sat = O.f64_to_e4m3(np.array([449.0, 463.9, 464.0, 500.0, 1e30, np.inf, -1e6, -np.inf]))
    assert list(sat) == [0x7E] * 6 + [0xFE] * 2
    rng = np.random.default_rng(1)
    x = rng.normal(0, 1e-4, 500)
    for k in (-20, -3, 0, 5):
        np.testing.assert_array_equal(O.encode_fp8(x * 2.0 ** k, 2.0 ** k), O.encode_fp8(x, 1.0))


def test_fp8_step_moments_and_amax():
    bt, d_in, d_out = 64, 48, 24
    s = make_step_inputs(1100, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
    xb, db, wb = bf16_bits(s.x), bf16_bits(s.dy), bf16_bits(s.w)
    rng = np.random.default_rng(2)
    m0, r0 = rng.normal(0, 1e-4, (d_out, d_in)), rng.uniform(1e-5, 1e-4, (d_out, d_in))
    ms, rs = np.max(np.abs(m0)) / 448, np.max(r0) / 448
    mc, rc = O.encode_fp8(m0, ms), O.encode_fp8(r0, rs)
    h = O.Hyper()
    G = O.wgrad(xb, db)
    W1, m1, v1 = O.adamw_f64(G, O.bf16_to_f64(wb), O.decode_fp8(mc, ms),
                             O.decode_fp8(rc, rs) ** 2, h, 3)
    new_ms, new_rs = np.max(np.abs(m1)) / 448, np.max(np.sqrt(v1)) / 448
    Wb, mc1, rc1, am, ar = O.step_fp8(xb, db, wb, mc, ms, rc, rs, new_ms, new_rs, h, 3)
    np.testing.assert_array_equal(Wb, O.f64_to_bf16(W1))
    assert am == np.float32(np.max(np.abs(m1))) and ar == np.float32(np.max(np.sqrt(v1)))
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normal codes
    # (plus the subnormal step near zero)
    for codes, scale, exact in ((mc1, new_ms, m1), (rc1, new_rs, np.sqrt(v1))):
        got = O.decode_fp8(codes, scale)
        bound = 2.0 ** -4 * np.abs(exact) + 2.0 ** -10 * float(np.float32(scale))
        assert np.all(np.abs(got - exact) <= bound)


def test_scale_roll_closed_forms():
    # the write scale becomes the read scale; amax * headroom / 448
    r, w = O.roll_fp8_scales(0.5, 0.25, 224.0, 2.0)
    assert r == np.float32(0.25) and w == np.float32(1.0)
    # a moment equal to the amax then encodes to the largest finite code
    amax = np.float32(3.7e-4)
    _, w = O.roll_fp8_scales(1.0, 1.0, amax, 1.0)
    assert O.encode_fp8(np.array([float(amax)]), w)[0] in (0x7E, 0x7D)
    assert abs(O.decode_fp8(O.encode_fp8(np.array([float(amax)]), w), w)[0] - amax) \
        <= 2.0 ** -4 * amax
    # headroom 2: the old amax sits one binade below saturation
    _, w2 = O.roll_fp8_scales(1.0, 1.0, amax, 2.0)
    assert w2 == np.float32(2.0) * w
    # no range to fit: keep the old write scale
    assert O.roll_fp8_scales(3.0, 5.0, 0.0, 2.0) == (np.float32(5.0), np.float32(5.0))
