"""Plain fp64 CPU oracle for the other coordinate-wise optimizers FORGE fuses.

TEST INFRASTRUCTURE, like ``forge_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs import it; the library
never does, and the two share no code.

Source: "FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
LLM Training".  Section 1 names the families whose state update enters one
coordinate at a time and so fuses entirely in the register epilogue (SGD, SGD
with momentum, Lion, RMSprop, Adagrad); section 2's definition of a tile-local
state update adds NAdam and RAdam; the appendix table of optimizer families
(regime 1) lists them with their shared hyperparameters (lr, wd, betas, eps).

What it computes, per optimizer, on one linear layer: G = dY^T X (Eq. 3), the
optimizer's state and weight update in fp64, then one round to nearest even
per stored value (W in bf16; states in fp32 or bf16).

Readings where the page leaves the update rule to the cited method (the page
checks each fused update against a reference PyTorch implementation, so the
plainest reading is PyTorch's published definition with default options):

R12 SGD, SGD with momentum, Adagrad, RMSprop, NAdam and RAdam follow the
    torch.optim definitions with default options: L2 weight decay added to the
    gradient before the state update, g = G + wd * W (W the weight before the
    update); SGD momentum with dampening 0 and no Nesterov term; Adagrad with
    lr_decay 0 and a zero initial accumulator; RMSprop plain (not centred, no
    momentum) with smoothing constant alpha; NAdam with momentum decay psi;
    RAdam with its variance rectification.
R13 Lion follows Chen et al. (2023): the update direction is the sign of
    c = beta1 m + (1 - beta1) G, the weight decay is decoupled,
    W' = (1 - lr wd) W - lr sign(c), and the state is m' = beta2 m + (1 - beta2) G.
    sign(0) = 0.
R14 States start at zero; step t is 1-based.  With a zero momentum buffer the
    first SGD-momentum step gives b = g, as PyTorch's first step does.
R15 Per-step scalars (NAdam's mu_t, mu_{t+1} and their running product,
    RAdam's rho_t and rectification, bias corrections) are functions of t and
    the hyperparameters, computed in fp64 from the float32 hyperparameters
    widened exactly (R9); NAdam's running product is prod_{i<=t} mu_i.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .forge_oracle import (Moment, bf16_to_f64, decode_moment, encode_moment, f64_to_bf16,
                           wgrad)

__all__ = [
    "OPT_SGD", "OPT_SGD_MOMENTUM", "OPT_ADAGRAD", "OPT_RMSPROP", "OPT_LION", "OPT_NADAM",
    "OPT_RADAM", "OPT_NAMES", "OPT_STATES", "OptHyper", "opt_f64", "opt_step",
    "nadam_scalars", "radam_scalars",
]

OPT_SGD, OPT_SGD_MOMENTUM, OPT_ADAGRAD, OPT_RMSPROP, OPT_LION, OPT_NADAM, OPT_RADAM = range(7)
OPT_NAMES = {OPT_SGD: "sgd", OPT_SGD_MOMENTUM: "sgd_momentum", OPT_ADAGRAD: "adagrad",
             OPT_RMSPROP: "rmsprop", OPT_LION: "lion", OPT_NADAM: "nadam", OPT_RADAM: "radam"}
# per-coordinate state tensors: SGD none; momentum buffer, Adagrad sum, RMSprop
# average, Lion m: one; NAdam and RAdam m and v: two
OPT_STATES = {OPT_SGD: 0, OPT_SGD_MOMENTUM: 1, OPT_ADAGRAD: 1, OPT_RMSPROP: 1, OPT_LION: 1,
              OPT_NADAM: 2, OPT_RADAM: 2}


@dataclass(frozen=True)
class OptHyper:
    """Hyperparameters of the regime-1 optimizers (the appendix table's
    columns, plus each method's own constant): learning rate, weight decay,
    betas (Lion, NAdam, RAdam), eps (Adagrad, RMSprop, NAdam, RAdam), momentum
    (SGD with momentum), alpha (RMSprop) and momentum_decay (NAdam's psi)."""
    lr: float = 1e-3
    weight_decay: float = 0.01
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    momentum: float = 0.9
    alpha: float = 0.99
    momentum_decay: float = 4e-3

    def as_f64(self):
        """R9/R15: the float32 values the C interface receives, widened exactly."""
        return {k: float(np.float32(getattr(self, k))) for k in
                ("lr", "weight_decay", "beta1", "beta2", "eps", "momentum", "alpha",
                 "momentum_decay")}


def nadam_scalars(h: dict, t: int):
    """NAdam's momentum schedule at step t (R15): mu_t, mu_{t+1} and the
    running product prod_{i<=t} mu_i, with mu_i = beta1 (1 - 0.5 * 0.96^(i psi))."""
    b1, psi = h["beta1"], h["momentum_decay"]

    def mu(i):
        return b1 * (1.0 - 0.5 * 0.96 ** (i * psi))
    prod = 1.0
    for i in range(1, t + 1):
        prod *= mu(i)
    return mu(t), mu(t + 1), prod


def radam_scalars(h: dict, t: int):
    """RAdam's rectification at step t (R15): (rho_t > 5, r_t), with
    rho_inf = 2 / (1 - beta2) - 1, rho_t = rho_inf - 2 t beta2^t / (1 - beta2^t)
    and r_t = sqrt((rho_t - 4)(rho_t - 2) rho_inf / ((rho_inf - 4)(rho_inf - 2) rho_t))."""
    b2 = h["beta2"]
    rho_inf = 2.0 / (1.0 - b2) - 1.0
    rho_t = rho_inf - 2.0 * t * b2 ** t / (1.0 - b2 ** t)
    if rho_t > 5.0:
        r = np.sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf /
                    ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t))
        return True, float(r)
    return False, 1.0


def opt_f64(opt: int, G, W, s1, s2, hyper: OptHyper, t: int):
    """One step of optimizer ``opt`` in fp64 with no rounding.

    G, W and the states s1, s2 (None where the optimizer has fewer) are fp64
    arrays of one shape.  Returns (W', s1', s2')."""
    if t < 1:
        raise ValueError("step t is 1-based (R14)")
    h = hyper.as_f64()
    lr, wd, eps = h["lr"], h["weight_decay"], h["eps"]
    b1, b2 = h["beta1"], h["beta2"]
    if opt == OPT_LION:                       # R13: decoupled decay, sign update
        c = b1 * s1 + (1.0 - b1) * G
        W1 = (1.0 - lr * wd) * W - lr * np.sign(c)
        return W1, b2 * s1 + (1.0 - b2) * G, None
    g = G + wd * W                            # R12: L2 decay through the gradient
    with np.errstate(divide="ignore", invalid="ignore"):
        if opt == OPT_SGD:
            return W - lr * g, None, None
        if opt == OPT_SGD_MOMENTUM:
            b = h["momentum"] * s1 + g
            return W - lr * b, b, None
        if opt == OPT_ADAGRAD:
            s = s1 + g * g
            return W - lr * g / (np.sqrt(s) + eps), s, None
        if opt == OPT_RMSPROP:
            a = h["alpha"]
            s = a * s1 + (1.0 - a) * (g * g)
            return W - lr * g / (np.sqrt(s) + eps), s, None
        m = b1 * s1 + (1.0 - b1) * g
        v = b2 * s2 + (1.0 - b2) * (g * g)
        if opt == OPT_NADAM:
            mu_t, mu_next, prod = nadam_scalars(h, t)
            denom = np.sqrt(v / (1.0 - b2 ** t)) + eps
            W1 = (W - lr * (1.0 - mu_t) / (1.0 - prod) * g / denom
                  - lr * mu_next / (1.0 - prod * mu_next) * m / denom)
            return W1, m, v
        if opt == OPT_RADAM:
            mhat = m / (1.0 - b1 ** t)
            rect, r = radam_scalars(h, t)
            if rect:
                W1 = W - lr * mhat * r * np.sqrt(1.0 - b2 ** t) / (np.sqrt(v) + eps)
            else:
                W1 = W - lr * mhat
            return W1, m, v
    raise ValueError(f"unknown optimizer {opt}")


def opt_step(opt: int, x_bits, dy_bits, w_bits, s1, s2, hyper: OptHyper, t: int, rows=None,
             return_f64: bool = False):
    """One fused step of optimizer ``opt`` on one linear layer: G = dY^T X, the
    update in fp64, one rounding per stored value.

    ``s1``, ``s2`` are stored states (``Moment``, fp32 or bf16) or None where
    the optimizer has fewer.  With ``rows`` the weight rows computed.
    Returns (W' bits, s1', s2') and, with ``return_f64``, also the fp64
    (G, W', s1', s2')."""
    G = wgrad(x_bits, dy_bits, rows)
    W = bf16_to_f64(w_bits)
    n = OPT_STATES[opt]
    d1 = decode_moment(s1, False) if n >= 1 else None
    d2 = decode_moment(s2, False) if n >= 2 else None
    W1, a1, a2 = opt_f64(opt, G, W, d1, d2, hyper, t)
    out = (f64_to_bf16(W1),
           encode_moment(s1.fmt, a1, False) if n >= 1 else None,
           encode_moment(s2.fmt, a2, False) if n >= 2 else None)
    if return_f64:
        return out + ((G, W1, a1, a2),)
    return out
