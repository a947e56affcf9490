"""Plain CPU oracle for fp8 moments with per-tensor delayed scaling.

TEST INFRASTRUCTURE, like ``forge_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs import it; the library
never does, and the two share no code.

Source: "FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
LLM Training".  Its fp8 state mode stores the moments in fp8 with one scale
per tensor and delayed scaling; the page reports that mode's weight error
rather than bounding it (the weight-error table, Appendix B's discussion of
the quantized modes).  It does not fix the fp8 format, the scaling history or
the first step's scale.

Readings:

R21 Both moments are stored as e4m3 codes (the OCP "fn" variant: exponent
    bias 7, no infinities, largest finite value 448, NaN = 0x7F/0xFF) with one
    fp32 scale per tensor: value = decode(code) * scale.  The second moment is
    stored in the square-root domain, r = sqrt(v), as for int8 (R6).
R22 Encoding divides by the scale, rounds to nearest even and saturates at
    +-448 (a stored state must stay finite).
R23 Delayed scaling: a step reads its moments with the scales they were
    stored with and stores the new moments with scales the caller gives,
    formed from amaxes of earlier steps; the step reports the amax of the new
    fp64 moments (max |m'|, max sqrt(v')) for the caller's next scales, e.g.
    scale = amax / 448.
R24 The scale roll between steps (a history of one step): the scale the new
    moments were written with becomes the scale they are read with, and the
    next write scale is amax * headroom / 448 (headroom >= 1 leaves room for
    the moments to grow before they saturate), formed in fp32 as two
    rounded operations, product first; an amax of 0 keeps the old write
    scale (a tensor whose moments are all zero has no range to fit).
"""
from __future__ import annotations

import numpy as np

from .forge_oracle import adamw_f64, bf16_to_f64, f64_to_bf16, f64_to_f32, wgrad

__all__ = ["E4M3_MAX", "e4m3_to_f64", "f64_to_e4m3", "encode_fp8", "decode_fp8", "step_fp8",
           "roll_fp8_scales"]

E4M3_MAX = 448.0


def e4m3_to_f64(codes) -> np.ndarray:
    """Decode e4m3 (fn) codes: sign, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 is subnormal (m * 2^-9); 0x7F and 0xFF are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def f64_to_e4m3(x) -> np.ndarray:
    """Round fp64 values to e4m3 (fn) codes: nearest, ties to even, saturating
    at +-448 (R22); NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                       # a = f 2^e, 0.5 <= f < 1
    lead = e.astype(np.int64) - 1            # exponent of the leading bit
    qexp = np.where(lead >= -6, lead - 3, -9)   # spacing: 3 mantissa bits; subnormal step 2^-9
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.ldexp(np.rint(np.ldexp(a, -qexp)), qexp)
    r = np.minimum(r, E4M3_MAX)
    # encode the rounded magnitude
    _, e2 = np.frexp(r)
    lead2 = e2.astype(np.int64) - 1
    normal = r >= 2.0 ** -6
    with np.errstate(divide="ignore", invalid="ignore"):
        mant_n = np.rint((r / np.exp2(lead2) - 1.0) * 8.0)
    exp_bits = np.where(normal, lead2 + 7, 0)
    mant = np.where(normal, mant_n, np.rint(r / 2.0 ** -9))
    code = (exp_bits << 3) + mant.astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def encode_fp8(x, scale) -> np.ndarray:
    """fp64 values -> e4m3 codes at a per-tensor fp32 scale (R21, R22)."""
    s = float(np.float32(scale))
    return f64_to_e4m3(np.asarray(x, dtype=np.float64) / s)


def decode_fp8(codes, scale) -> np.ndarray:
    return e4m3_to_f64(codes) * float(np.float32(scale))


def step_fp8(x_bits, dy_bits, w_bits, m_codes, m_scale, r_codes, r_scale, m_scale_new,
             r_scale_new, hyper, t: int, rows=None):
    """One fused AdamW step with fp8 moments (R21-R23).  The moments are read
    with (m_scale, r_scale) and stored with (m_scale_new, r_scale_new).
    Returns (W' bits, m' codes, r' codes, amax of m', amax of r'), the amaxes
    as float32."""
    G = wgrad(x_bits, dy_bits, rows)
    W = bf16_to_f64(w_bits)
    m = decode_fp8(m_codes, m_scale)
    r = decode_fp8(r_codes, r_scale)
    W1, m1, v1 = adamw_f64(G, W, m, r * r, hyper, t)
    r1 = np.sqrt(v1)
    return (f64_to_bf16(W1), encode_fp8(m1, m_scale_new), encode_fp8(r1, r_scale_new),
            f64_to_f32(np.max(np.abs(m1))) if m1.size else np.float32(0),
            f64_to_f32(np.max(r1)) if r1.size else np.float32(0))


def roll_fp8_scales(read_scale, write_scale, amax, headroom):
    """R24: the scales of the next step, (read, write), as float32."""
    w = np.float32(write_scale)
    a = np.float32(amax)
    if a > 0:
        w = np.float32(np.float32(a * np.float32(headroom)) / np.float32(E4M3_MAX))
    return np.float32(write_scale), w
