"""Plain fp64 CPU oracle for one FORGE step on one linear layer.

TEST INFRASTRUCTURE.  This module is the definition the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` import it; the library never does,
and the two share no code.

Source: "FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
LLM Training" (arXiv 2606.22932).

What it computes:

* the weight gradient of a linear layer ``Y = X W^T`` (section 2.1, Eq. 2),
  ``G = dY^T X`` (Eq. 3; Appendix A "Setup": ``G_pq = sum_t dY_tp X_tq``);
* AdamW with decoupled weight decay and bias-corrected moments applied to
  that gradient (section 2.2, Algorithm 1: the two moment updates, the bias
  corrections and the weight update);
* one rounding per stored tensor: bf16 weights and fp32, bf16 or int8
  moments (section 1, Eq. 1: k = 8 / 4 / 2 bytes of state per parameter;
  Appendix B "INT8 states");
* the input gradient of the same layer, ``dX = dY W`` (the other half of the
  backward pass of ``Y = X W^T``, section 2.1), which Algorithm 1 computes
  from the weight before the update (its first line; Appendix A, Remark 2):
  ``linear_backward`` takes it from the pre-update W, then steps.

Proposition 1 (Appendix A.2) says the tile-fused schedule reaches exactly the
result of forming all of G and stepping once.  So the oracle is that plain
definition: one fp64 matrix product for G (products of bf16 values are exact
in fp64), the update in fp64, then one round-to-nearest-even per stored value.

Readings taken where the pages leave a step open:

R1  Weight decay is decoupled and multiplicative on the pre-update weight:
    ``W' = (1 - lr*wd) W - lr * mhat / (sqrt(vhat) + eps)`` (Algorithm 1,
    weight update).
R2  eps is added after the square root of the bias-corrected second moment.
R3  The step count t is 1-based and counts the step being taken.
R4  Every store rounds to nearest, ties to even.
R5  int8 moments use absmax blocks of 128 along each weight row (the pages use
    64), one fp32 scale per (row, block) and moment, codes in [-127, 127].
R6  The second moment is stored in the square-root domain, r = sqrt(v).  In a
    block whose absmax is non-zero every code is at least 1 (the pages floor v
    away from zero, Appendix B).
R7  The weight update reads this step's unrounded m' and v'; rounded values
    are read only at the next step (Appendix B: the update arithmetic stays in
    high precision).
R8  With no tokens (BT = 0), G = 0: the moments decay and W takes the decay and
    the m-driven update, with no special case (Appendix A, Remark 1).
R9  The hyperparameters are the float32 values the C interface receives,
    widened exactly to fp64.
R10 dX is stored in bf16, rounded once to nearest even from the exact fp64
    product (the layer's activations and their gradients are bf16).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

__all__ = [
    "FMT_FP32", "FMT_BF16", "FMT_INT8", "INT8_BLOCK",
    "Hyper", "Moment",
    "bf16_to_f64", "f64_to_bf16", "f64_to_f32",
    "wgrad", "wgrad_abs", "adamw_f64",
    "quantize_int8_blocks", "decode_moment", "encode_moment", "zero_moment",
    "step", "dgrad", "dgrad_abs", "linear_backward",
]

FMT_FP32, FMT_BF16, FMT_INT8 = 0, 1, 2
INT8_BLOCK = 128          # R5
INT8_QMAX = 127.0         # Appendix B: s = a / 127


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to fp64.  Exact: a bf16 value is the
    upper half of the float32 with the same bits."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round fp64 values to bf16 once, to nearest with ties to even (R4).

    bf16 has 8 significant bits and the float32 exponent range; below 2**-126
    the spacing is fixed at 2**-133 (subnormals).  The value is scaled by a
    power of two so that one spacing becomes 1, rounded with ``np.rint``
    (ties to even) and scaled back: both scalings are exact in fp64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                 # a = f * 2**e with 0.5 <= f < 1
    lead = e.astype(np.int64) - 1      # exponent of the leading bit
    qexp = np.where(lead >= -126, lead - 7, -133).astype(np.int32)
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.ldexp(np.rint(np.ldexp(a, -qexp)), qexp)
        overflow = ~(r < 2.0 ** 128)   # also true for inf and nan inputs
        r32 = np.where(overflow, 0.0, r).astype(np.float32)   # exact
    bits = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(overflow, np.uint16(0x7F80), bits)
    bits = np.where(np.signbit(x), bits | np.uint16(0x8000), bits)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def f64_to_f32(x) -> np.ndarray:
    """Round fp64 to float32 once, to nearest with ties to even (R4)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32)


# ---------------------------------------------------------------------------
# Hyperparameters and moment containers
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Hyper:
    """AdamW hyperparameters (Algorithm 1): learning rate eta, decays beta1 and
    beta2, stabiliser eps, weight decay lambda."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    wd: float = 0.01

    def as_f64(self):
        """R9: the float32 values the C interface receives, widened exactly."""
        return tuple(float(np.float32(v)) for v in
                     (self.lr, self.beta1, self.beta2, self.eps, self.wd))


@dataclass
class Moment:
    """One stored moment tensor [rows, cols].

    fmt FMT_FP32: ``data`` float32.  FMT_BF16: ``data`` uint16 bf16 bits.
    FMT_INT8: ``data`` int8 codes and ``scale`` float32 [rows, cols/128]."""
    fmt: int
    data: np.ndarray
    scale: Optional[np.ndarray] = None

    def rows(self, idx) -> "Moment":
        """The same moment restricted to the weight rows ``idx``."""
        return Moment(self.fmt, self.data[idx],
                      None if self.scale is None else self.scale[idx])


def zero_moment(fmt: int, rows: int, cols: int) -> Moment:
    if fmt == FMT_FP32:
        return Moment(fmt, np.zeros((rows, cols), np.float32))
    if fmt == FMT_BF16:
        return Moment(fmt, np.zeros((rows, cols), np.uint16))
    if fmt == FMT_INT8:
        if cols % INT8_BLOCK:
            raise ValueError("int8 moments need cols % 128 == 0")
        return Moment(fmt, np.zeros((rows, cols), np.int8),
                      np.zeros((rows, cols // INT8_BLOCK), np.float32))
    raise ValueError(f"unknown moment format {fmt}")


# ---------------------------------------------------------------------------
# The weight gradient (Eq. 3)
# ---------------------------------------------------------------------------

def wgrad(x_bits, dy_bits, rows=None) -> np.ndarray:
    """G = dY^T X in fp64 (Eq. 3), shape [Dout, Din] or [len(rows), Din].

    ``x_bits`` is X [BT, Din], ``dy_bits`` is dY [BT, Dout], both bf16 bits.
    Row p of G reads only column p of dY and all of X, so ``rows`` computes an
    exact subset of rows."""
    X = bf16_to_f64(x_bits)
    dY = bf16_to_f64(dy_bits)
    if rows is not None:
        dY = dY[:, rows]
    return dY.T @ X


def wgrad_abs(x_bits, dy_bits, rows=None) -> np.ndarray:
    """S = |dY|^T |X|, i.e. S_pq = sum_t |dY_tp X_tq|.  Any summation order of
    G_pq in a precision with unit roundoff u and n additions errs by at most
    about n*u*S_pq; the tests use S to bound what the GPU may differ by."""
    X = np.abs(bf16_to_f64(x_bits))
    dY = np.abs(bf16_to_f64(dy_bits))
    if rows is not None:
        dY = dY[:, rows]
    return dY.T @ X


# ---------------------------------------------------------------------------
# The input gradient (backward pass of Y = X W^T)
# ---------------------------------------------------------------------------

def dgrad(dy_bits, w_bits, rows=None) -> np.ndarray:
    """dX = dY W in fp64, shape [BT, Din] or [len(rows), Din].

    ``dy_bits`` is dY [BT, Dout], ``w_bits`` is W [Dout, Din], both bf16 bits:
    dX_tq = sum_p dY_tp W_pq.  Row t of dX reads only row t of dY and all of
    W, so ``rows`` (token rows) computes an exact subset of rows."""
    dY = bf16_to_f64(dy_bits)
    W = bf16_to_f64(w_bits)
    if rows is not None:
        dY = dY[rows]
    return dY @ W


def dgrad_abs(dy_bits, w_bits, rows=None) -> np.ndarray:
    """|dY| |W|: the bound on what any fp32 summation order of dX may differ
    by, as wgrad_abs is for G."""
    dY = np.abs(bf16_to_f64(dy_bits))
    W = np.abs(bf16_to_f64(w_bits))
    if rows is not None:
        dY = dY[rows]
    return dY @ W


# ---------------------------------------------------------------------------
# AdamW (Algorithm 1) in fp64
# ---------------------------------------------------------------------------

def adamw_f64(G, W, m, v, hyper: Hyper, t: int):
    """One AdamW step in fp64 with no rounding (Algorithm 1, moment updates,
    bias correction and weight update; readings R1-R3).

    G, W, m, v are fp64 arrays of one shape.  Returns (W', m', v')."""
    if t < 1:
        raise ValueError("step t is 1-based (R3)")
    lr, b1, b2, eps, wd = hyper.as_f64()
    m1 = b1 * m + (1.0 - b1) * G
    v1 = b2 * v + (1.0 - b2) * (G * G)
    mhat = m1 / (1.0 - b1 ** t)
    vhat = v1 / (1.0 - b2 ** t)
    with np.errstate(divide="ignore", invalid="ignore"):
        W1 = (1.0 - lr * wd) * W - lr * mhat / (np.sqrt(vhat) + eps)
    return W1, m1, v1


# ---------------------------------------------------------------------------
# Moment storage formats
# ---------------------------------------------------------------------------

def quantize_int8_blocks(x, floor_one: bool):
    """Blockwise absmax int8 (Appendix B "INT8 states", with R5/R6).

    Per row and per block of 128 columns: a = max |x|, s = a / 127,
    q = clamp(round(x / s), -127, 127) with ties to even; if a = 0 then s = 0
    and q = 0.  With ``floor_one`` every code of a block with a > 0 is at
    least 1 (the floor of the square-root-domain second moment, R6).
    Returns (int8 codes, float32 scales rounded once from fp64)."""
    x = np.asarray(x, dtype=np.float64)
    rows, cols = x.shape
    if cols % INT8_BLOCK:
        raise ValueError("int8 moments need cols % 128 == 0")
    xb = x.reshape(rows, cols // INT8_BLOCK, INT8_BLOCK)
    a = np.max(np.abs(xb), axis=2) if cols else np.zeros((rows, 0))
    s = a / INT8_QMAX
    nz = (a > 0)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(nz, np.rint(xb / np.where(nz, s[..., None], 1.0)), 0.0)
    q = np.clip(q, -INT8_QMAX, INT8_QMAX)
    if floor_one:
        q = np.where(nz, np.maximum(q, 1.0), q)
    return q.reshape(rows, cols).astype(np.int8), f64_to_f32(s)


def decode_moment(mom: Moment, second: bool) -> np.ndarray:
    """Stored moment -> fp64 value.  For int8 the value is code * scale; the
    second moment is stored as r = sqrt(v), so v = r * r (R6)."""
    if mom.fmt == FMT_FP32:
        return mom.data.astype(np.float64)
    if mom.fmt == FMT_BF16:
        return bf16_to_f64(mom.data)
    if mom.fmt == FMT_INT8:
        s = np.repeat(mom.scale.astype(np.float64), INT8_BLOCK, axis=1)
        r = mom.data.astype(np.float64) * s
        return r * r if second else r
    raise ValueError(f"unknown moment format {mom.fmt}")


def encode_moment(fmt: int, x, second: bool) -> Moment:
    """fp64 moment -> stored format, rounding once (R4-R6)."""
    if fmt == FMT_FP32:
        return Moment(fmt, f64_to_f32(x))
    if fmt == FMT_BF16:
        return Moment(fmt, f64_to_bf16(x))
    if fmt == FMT_INT8:
        q, s = quantize_int8_blocks(np.sqrt(x) if second else x, floor_one=second)
        return Moment(fmt, q, s)
    raise ValueError(f"unknown moment format {fmt}")


# ---------------------------------------------------------------------------
# One step
# ---------------------------------------------------------------------------

def step(x_bits, dy_bits, w_bits, m: Moment, v: Moment, hyper: Hyper, t: int,
         rows=None, grad_bf16: bool = False, return_f64: bool = False):
    """One fused step on one linear layer: G = dY^T X, AdamW, round once.

    x_bits   X  [BT, Din] bf16 bits      dy_bits  dY [BT, Dout] bf16 bits
    w_bits   W  bf16 bits, and m, v the stored moments, all for the weight rows
             computed: [Dout, Din], or [len(rows), Din] when ``rows`` is given.
    grad_bf16  round G to bf16 before the update: the standard path, which
             stores the gradient in bf16 before the optimizer reads it
             (section 3.1 and Appendix B "Undamped truncation bias").
    Returns (W' bits, m', v') and, with ``return_f64``, also the unrounded
    fp64 (G, W', m', v')."""
    G = wgrad(x_bits, dy_bits, rows)
    if grad_bf16:
        G = bf16_to_f64(f64_to_bf16(G))
    W = bf16_to_f64(w_bits)
    if W.shape != G.shape:
        raise ValueError(f"W rows {W.shape} do not match G {G.shape}")
    W1, m1, v1 = adamw_f64(G, W, decode_moment(m, False), decode_moment(v, True),
                           hyper, t)
    out = (f64_to_bf16(W1), encode_moment(m.fmt, m1, False),
           encode_moment(v.fmt, v1, True))
    if return_f64:
        return out + ((G, W1, m1, v1),)
    return out


def linear_backward(x_bits, dy_bits, w_bits, m: Moment, v: Moment, hyper: Hyper, t: int):
    """The layer's backward pass with the fused update: dX from the weight
    before the update (R10), then one step.  Returns (dX bits, W' bits, m', v')."""
    dx = f64_to_bf16(dgrad(dy_bits, w_bits))
    return (dx,) + step(x_bits, dy_bits, w_bits, m, v, hyper, t)
