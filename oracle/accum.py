"""Plain fp64 CPU oracle for the accumulate mode: B' = beta B + dY^T X.

TEST INFRASTRUCTURE, like ``forge_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs import it; the library
never does, and the two share no code.

Source: "FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
LLM Training".  Its optimizer regimes (section 2 and the table of regimes)
name Muon's state update B <- mu B + G as tile-local and affine, so the
weight-gradient multiply accumulates into the momentum buffer through the
GEMM's own beta and the gradient never exists.  Its exact-accumulation mode
(Appendix N.5, pipeline parallelism) holds an fp32 gradient-shaped
accumulator across micro-batches and steps once at the final one.  Both are
this one operation on an fp32 buffer B.

Readings:

R16 B' = beta B + G with beta the float32 value received (R9), G = dY^T X
    exact in fp64, rounded once to fp32 per call.  beta = 0 does not read B
    (the buffer may hold anything, as with a GEMM's beta = 0).
R17 Exact accumulation over micro-batches 1..k: the first accumulates with
    beta = 0, the others with beta = 1, each rounding once to fp32; then one
    optimizer step reads the fp32 accumulator as its gradient.
R28 The step at the final micro-batch may take the last accumulate into it:
    its gradient is the fp32 value B + G_k (the R17 accumulate with beta = 1,
    rounded once), which one AdamW step (Algorithm 1) then reads; the
    accumulator itself is read, not written.
"""
from __future__ import annotations

import numpy as np

from .forge_oracle import (Hyper, Moment, adamw_f64, bf16_to_f64, decode_moment, encode_moment,
                           f64_to_bf16, f64_to_f32, wgrad)

__all__ = ["accumulate", "step_accumulated"]


def accumulate(x_bits, dy_bits, B, beta: float, rows=None, return_f64: bool = False):
    """One accumulate call: B' = beta B + G in fp64, rounded once to fp32 (R16).

    ``B`` is the fp32 buffer [Dout, Din] (or the rows computed, with
    ``rows``); it is not read when beta is 0.  Returns float32 B', and with
    ``return_f64`` also the fp64 value before rounding."""
    G = wgrad(x_bits, dy_bits, rows)
    b = float(np.float32(beta))
    exact = G if b == 0.0 else b * np.asarray(B, dtype=np.float64) + G
    out = f64_to_f32(exact)
    return (out, exact) if return_f64 else out


def step_accumulated(x_bits, dy_bits, w_bits, m: Moment, v: Moment, B, hyper: Hyper, t: int,
                     rows=None, return_f64: bool = False):
    """The fused step at the final micro-batch of the exact-accumulation mode
    (Appendix N.5; R28): the last micro-batch's G = dY^T X is added to the
    fp32 accumulator B of the earlier ones and rounded once to fp32 (R16 with
    beta = 1), and one AdamW step reads that sum as its gradient, rounding
    W', m', v' once each like ``step``.

    ``B`` is fp32 [Dout, Din] (or the rows computed, with ``rows``).  Returns
    (W' bits, m', v') and, with ``return_f64``, also the fp64 (G, W', m', v')
    where G is the fp32 gradient the step read."""
    G = accumulate(x_bits, dy_bits, B, 1.0, rows).astype(np.float64)
    W = bf16_to_f64(w_bits)
    if W.shape != G.shape:
        raise ValueError(f"W rows {W.shape} do not match G {G.shape}")
    W1, m1, v1 = adamw_f64(G, W, decode_moment(m, False), decode_moment(v, True), hyper, t)
    out = (f64_to_bf16(W1), encode_moment(m.fmt, m1, False), encode_moment(v.fmt, v1, True))
    if return_f64:
        return out + ((G, W1, m1, v1),)
    return out
