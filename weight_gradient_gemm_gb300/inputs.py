"""Seeded synthetic inputs for the fused weight-gradient + AdamW step.

This module draws the numbers both sides are fed: X, dY and the initial W.
It holds none of the method's arithmetic, so the CUDA path and the CPU oracle
can both take their inputs from it without sharing any computation.

Recipe (the workloads of "FORGE: Fused On-Register Gradient Elimination",
section 3 and Appendices D-E, replaced by Gaussian tensors of the same
shapes because no dataset or checkpoint is used):

* a CPU ``torch.Generator`` seeded with ``1000*config + 10*shape_idx + step``;
* draw order X, then dY, then W (W only when a layer is initialised);
* values drawn in float32 as ``std * N(0, 1)`` and cast to bf16 (round to
  nearest even);
* optional spikes: ``floor(frac * BT)`` token rows of dY, chosen by
  ``randperm(BT)`` from the same generator, scaled in float32 by ``scale``
  before the cast (a few tokens with much larger gradients, which stress the
  moments' range).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

# The seven projections of one Llama-3.1-8B decoder layer, W as [Dout, Din].
LLAMA31_8B_SHAPES = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
LLAMA31_8B_LAYERS = 32


def seed_of(config: int, shape_idx: int, step: int) -> int:
    return 1000 * config + 10 * shape_idx + step


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _normal_bf16(g: torch.Generator, shape, std: float) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


@dataclass
class StepInputs:
    """One step's activations X [BT, Din] and upstream gradient dY [BT, Dout]
    (bf16, CPU), and the layer's initial weight W [Dout, Din] when requested."""
    x: torch.Tensor
    dy: torch.Tensor
    w: torch.Tensor | None = None


def make_step_inputs(config: int, shape_idx: int, step: int, bt: int, d_in: int,
                     d_out: int, x_std: float = 1.0, dy_std: float = 1e-3,
                     w_std: float = 0.02, with_w: bool = False,
                     spike_frac: float = 0.0, spike_scale: float = 100.0) -> StepInputs:
    g = _gen(seed_of(config, shape_idx, step))
    x = _normal_bf16(g, (bt, d_in), x_std)
    dy32 = torch.randn((bt, d_out), generator=g, dtype=torch.float32) * dy_std
    w = _normal_bf16(g, (d_out, d_in), w_std) if with_w else None
    if spike_frac > 0 and bt > 0:
        n = int(math.floor(spike_frac * bt))
        if n:
            idx = torch.randperm(bt, generator=g)[:n]
            dy32[idx] *= spike_scale
    return StepInputs(x=x, dy=dy32.to(torch.bfloat16), w=w)


# Which activations each projection reads in the model: q, k, v share the
# attention input, gate and up the MLP input; o and down have their own.
LLAMA31_8B_X_GROUP = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp",
                      "up": "mlp", "down": "down"}
_X_GROUPS = ("attn", "o", "mlp", "down")


def make_layer_inputs(config: int, layer: int, step: int, bt: int, dy_std: float = 1e-3,
                      x_std: float = 1.0, w_std: float = 0.02, with_w: bool = False):
    """One decoder layer's step inputs with the model's sharing of X: a dict
    with ``x`` (group name -> X [BT, Din] bf16), ``dy`` (projection -> dY
    [BT, Dout] bf16) and, with ``with_w``, ``w`` (projection -> initial W).
    Every tensor has its own seed, ``seed_of(config, 20 * layer + j, step)``
    with j = 0..3 for the X groups and 4..10 for the projections (W: step 0
    of index 11..17)."""
    x, dy, w = {}, {}, {}
    for j, grp in enumerate(_X_GROUPS):
        d_in = 14336 if grp == "down" else 4096
        x[grp] = _normal_bf16(_gen(seed_of(config, 20 * layer + j, step)), (bt, d_in), x_std)
    for j, (name, d_out, d_in) in enumerate(LLAMA31_8B_SHAPES):
        g = _gen(seed_of(config, 20 * layer + 4 + j, step))
        dy[name] = _normal_bf16(g, (bt, d_out), dy_std)
        if with_w:
            gw = _gen(seed_of(config, 20 * layer + 11 + j, 0))
            w[name] = _normal_bf16(gw, (d_out, d_in), w_std)
    return dict(x=x, dy=dy, w=w)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a bf16 CPU tensor (what the oracle reads)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """A bf16 CPU tensor from uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
