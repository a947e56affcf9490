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
"""
from __future__ import annotations

import numpy as np

from .forge_oracle import f64_to_f32, wgrad

__all__ = ["accumulate"]


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
