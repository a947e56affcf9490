"""Plain CPU oracle for the stochastic-rounding store of the bf16 weight.

TEST INFRASTRUCTURE, like ``forge_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs import it; the library
never does, and the two share no code.

Source: "FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
LLM Training".  Its SR-store recipe keeps no fp32 master copy: the bf16 weight
is the only copy and is committed by stochastic rounding (Gupta et al. 2015),
which the page finds tracks the fp32-master trajectory about twice as closely
as plain bf16 storage (recipe classes; Appendix N, the stochastic-rounding
comparison).

Readings:

R18 Stochastic rounding of an fp32 value x to bf16 with a uniform 16-bit
    integer r: add r to the low 16 bits of x's magnitude and keep the upper
    16 bits, so |x| rounds up to the next bf16 value with probability
    (dropped bits) / 2^16, and the expected result is x exactly.  Values
    already in bf16, and NaN and infinity, are unchanged.
R19 The decision is taken in the kernel's precision: the updated weight is
    first rounded to fp32 (to nearest even), then stochastically to bf16.
R20 The random bits come from the counter-based generator Philox4x64-10
    (Salmon, Moraes, Dror, Shaw 2011, "Parallel random numbers: as easy as
    1, 2, 3"), implemented here and in the library from that definition.
    Weight element (p, q) at step t takes 16 bits of the block with counter
    (p, q // 16, t, 0) and key (seed, 0): bits 16 j .. 16 j + 15 of output
    word k, where q % 16 = 4 k + j.
"""
from __future__ import annotations

import numpy as np

from .forge_oracle import Moment, adamw_f64, bf16_to_f64, decode_moment, encode_moment, wgrad

__all__ = ["philox4x64_10", "sr_bits", "sr_to_bf16", "step_sr"]

_MASK = (1 << 64) - 1
# Philox4x64 multipliers and Weyl key increments (Salmon et al. 2011)
_M0, _M1 = 0xD2E7470EE14C6C93, 0xCA5A826395121157
_W0, _W1 = 0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B


def philox4x64_10(counter, key):
    """Philox4x64 with 10 rounds on one block: counter (c0, c1, c2, c3) and
    key (k0, k1), 64-bit words.  Each round multiplies c0 and c2 by the two
    multipliers into 128-bit products, mixes the high halves with c1, c3 and
    the key, permutes the words, and bumps the key by the Weyl constants."""
    c0, c1, c2, c3 = (int(x) & _MASK for x in counter)
    k0, k1 = (int(x) & _MASK for x in key)
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> 64, p0 & _MASK
        hi1, lo1 = p1 >> 64, p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def sr_bits(rows, cols, seed: int, t: int) -> np.ndarray:
    """The 16-bit random integers of the weight elements (rows x cols) at
    step t (R20); ``rows`` are the global row indices, ``cols`` the number of
    columns."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), cols), np.uint32)
    for i, p in enumerate(rows):
        for g in range((cols + 15) // 16):
            words = philox4x64_10((int(p), g, int(t), 0), (int(seed), 0))
            for e in range(16):
                q = 16 * g + e
                if q < cols:
                    out[i, q] = (words[e // 4] >> (16 * (e % 4))) & 0xFFFF
    return out


def sr_to_bf16(x32, r16) -> np.ndarray:
    """Stochastic rounding of float32 values to bf16 bit patterns (R18)."""
    x = np.asarray(x32, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    mag = b & 0x7FFFFFFF
    special = mag >= 0x7F800000                       # inf, nan: unchanged (nan quieted)
    up = (mag + np.asarray(r16, dtype=np.uint64)) >> 16
    up = np.minimum(up, np.uint64(0x7F80))           # past the largest finite value: inf
    sign = (b >> 16) & 0x8000
    nanv, infv = np.uint64(0x7FC0), np.uint64(0x7F80)
    res = np.where(special, np.where(mag > 0x7F800000, nanv, infv), up) | sign
    return res.astype(np.uint16)


def step_sr(x_bits, dy_bits, w_bits, m: Moment, v: Moment, hyper, t: int, seed: int,
            rows=None):
    """The fused AdamW step with the bf16 weight committed by stochastic
    rounding (R18-R20); moments round to nearest as in ``step``.  ``rows`` are
    the weight rows computed (global indices, which select the random bits).
    Returns (W' bits, m', v')."""
    G = wgrad(x_bits, dy_bits, rows)
    W = bf16_to_f64(w_bits)
    W1, m1, v1 = adamw_f64(G, W, decode_moment(m, False), decode_moment(v, True), hyper, t)
    rr = np.arange(G.shape[0]) if rows is None else np.asarray(rows)
    r16 = sr_bits(rr, G.shape[1], seed, t)
    w32 = W1.astype(np.float32)                       # R19: to fp32 first
    return (sr_to_bf16(w32, r16), encode_moment(m.fmt, m1, False),
            encode_moment(v.fmt, v1, True))
