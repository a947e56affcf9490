"""Grouped launches of the other modes: the other optimizers, the
stochastic-rounding store, the accumulate mode, the input gradient and the
layer's whole backward step, each over several linear layers in one launch.

A grouped launch walks one tile queue over all its layers; every layer's
result must be that of a separate call on the same inputs, bit for bit (the
separate calls are themselves checked against the oracle in their own
tests), and the grouped input gradient is also compared with the oracle on
sampled rows of the Llama-3.1-8B projections."""
import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import (LLAMA31_8B_SHAPES, bf16_bits, make_layer_inputs,
                                               make_step_inputs)

from .gpu_util import DEV, require_gpu
from .test_gpu_dgrad import check_dx

pytestmark = pytest.mark.gpu

SHAPES = [(264, 512), (1024, 1040), (136, 272), (520, 2048), (8, 128)]
ADAMW = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _layers(seed, bt, states, sdtype=torch.float32, shapes=SHAPES):
    out = []
    for i, (d_out, d_in) in enumerate(shapes):
        s = make_step_inputs(seed, i, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True,
                             spike_frac=0.01)
        ly = dict(X=s.x.to(DEV), dY=s.dy.to(DEV), W=s.w.to(DEV))
        g = torch.Generator().manual_seed(seed + i)
        for k in range(states):
            t = (torch.rand((d_out, d_in), generator=g) * 1e-4).to(sdtype)
            ly[f"s{k + 1}"] = t.to(DEV)
        out.append(ly)
    return out


def _clone(layers):
    mutable = ("W", "s1", "s2", "B", "m", "v", "m_scale", "v_scale", "dX")
    return [{k: (v.clone() if k in mutable and v is not None else v) for k, v in ly.items()}
            for ly in layers]


@pytest.mark.parametrize("bt", [200, 1000])
@pytest.mark.parametrize("opt", [F.OPT_SGD, F.OPT_SGD_MOMENTUM, F.OPT_LION, F.OPT_RADAM],
                         ids=["sgd", "momentum", "lion", "radam"])
@pytest.mark.parametrize("sdtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_opt_grouped_equals_separate_calls(bt, opt, sdtype):
    n_st = F.OPT_STATES[opt]
    hy = dict(lr=1e-3, weight_decay=0.01, beta1=0.9, beta2=0.99)
    a = _layers(10, bt, n_st, sdtype)
    b = _clone(a)
    F.wgrad_opt_grouped(a, opt, step=7, **hy)
    for ly in b:
        F.wgrad_opt(ly["X"], ly["dY"], ly["W"], opt, ly.get("s1"), ly.get("s2"), step=7, **hy)
    assert F.device_error() == 0
    for x, y in zip(a, b):
        for k in ("W", "s1", "s2"):
            if k in x:
                assert _same(x[k], y[k]), k


@pytest.mark.parametrize("bt", [200, 1000])
def test_sr_grouped_equals_separate_calls(bt):
    a = _layers(11, bt, 2)
    for ly in a:
        ly["m"], ly["v"] = ly.pop("s1"), ly.pop("s2")
    b = _clone(a)
    seeds = [100 + 17 * i for i in range(len(a))]
    F.wgrad_adamw_sr_grouped(a, seeds, step=3, **ADAMW)
    for ly, sd in zip(b, seeds):
        F.wgrad_adamw_sr(ly["X"], ly["dY"], ly["W"], ly["m"], ly["v"], step=3, seed=sd, **ADAMW)
    assert F.device_error() == 0
    for x, y in zip(a, b):
        for k in ("W", "m", "v"):
            assert _same(x[k], y[k]), k


@pytest.mark.parametrize("bt", [0, 200, 1000])
@pytest.mark.parametrize("beta", [0.0, 1.0, 0.9])
def test_accumulate_grouped_equals_separate_calls(bt, beta):
    a = _layers(12, bt, 0)
    for i, ly in enumerate(a):
        g = torch.Generator().manual_seed(i)
        ly["B"] = torch.randn(ly["W"].shape, generator=g).to(DEV)
    b = _clone(a)
    F.wgrad_accumulate_grouped(a, beta)
    for ly in b:
        F.wgrad_accumulate(ly["X"], ly["dY"], ly["B"], beta)
    assert F.device_error() == 0
    for x, y in zip(a, b):
        assert _same(x["B"], y["B"])


def _llama_dgrad_items(bt, seed=13):
    items, host = [], []
    inp = make_layer_inputs(seed, 0, 1, bt, with_w=True)
    for name, d_out, d_in in LLAMA31_8B_SHAPES:
        dy, w = inp["dy"][name], inp["w"][name]
        items.append(dict(dY=dy.to(DEV), W=w.to(DEV),
                          dX=torch.full((bt, d_in), float("nan"), dtype=torch.bfloat16,
                                        device=DEV)))
        host.append((name, dy, w))
    return items, host


@pytest.mark.parametrize("bt", [512, 1000])
def test_dgrad_grouped_unsplit_equals_dgrad_and_the_oracle(bt, tune):
    # the layer's seven projections in one launch without a workspace (no
    # split) against forge_dgrad with one split, and sampled rows against the
    # oracle
    items, host = _llama_dgrad_items(bt)
    F.dgrad_grouped(items)
    tune(splits=1)
    for it in items:
        ref = torch.empty_like(it["dX"])
        F.dgrad(it["dY"], it["W"], ref)
        assert F.device_error() == 0
        assert _same(it["dX"], ref)
    rows = np.array(sorted({0, 127, 128, 255, 256, bt // 2, bt - 1}))
    for it, (name, dy, w) in zip(items, host):
        check_dx(bf16_bits(it["dX"].cpu())[rows], bf16_bits(dy), bf16_bits(w), rows,
                 label=f"grouped dX {name}")


@pytest.mark.parametrize("splits,cap", [(2, None), (4, None), (4, "half")])
def test_dgrad_grouped_split_in_the_callers_workspace(splits, cap, tune):
    # forced splits with the partials in the caller's workspace: equal to
    # forge_dgrad at the same split count; a workspace of half the size runs
    # with fewer splits and equals forge_dgrad at that count
    bt = 256
    items, host = _llama_dgrad_items(bt, seed=14)
    items = [it for it, (name, _, _) in zip(items, host) if name in ("q", "gate", "down")]
    tune(splits=splits)
    need = F.dgrad_workspace_bytes(items)
    assert need > 0
    size = need if cap is None else need // 2
    ws = torch.empty(size // 4, dtype=torch.float32, device=DEV)
    F.dgrad_grouped(items, workspace=ws)
    # the split count that fits the workspace
    used = splits
    while used > 1 and need // splits * used > size:
        used -= 1
    tune(splits=used)
    for it in items:
        ref = torch.empty_like(it["dX"])
        F.dgrad(it["dY"], it["W"], ref)
        assert F.device_error() == 0
        assert _same(it["dX"], ref), (splits, used)


@pytest.mark.parametrize("fmt", [F.MOM_FP32, F.MOM_BF16, F.MOM_INT8_B128, F.MOM_FP8_E4M3])
def test_linear_backward_grouped_equals_per_layer_calls(fmt, tune):
    # one grouped dX launch and one grouped fused launch over the layer,
    # against forge_linear_backward per projection (one split on both sides);
    # fp8 moments include each tensor's amax words
    bt = 384
    tune(splits=1)
    inp = make_layer_inputs(15, 0, 1, bt, with_w=True)
    from weight_gradient_gemm_gb300.inputs import LLAMA31_8B_X_GROUP
    xs = {g: x.to(DEV) for g, x in inp["x"].items()}
    a = []
    for name, d_out, d_in in LLAMA31_8B_SHAPES:
        m, v, ms, vs = F.alloc_moments(d_out, d_in, fmt, DEV)
        if fmt == F.MOM_FP8_E4M3:   # write scales that keep the first moments representable
            ms[1], vs[1] = 1e-5, 1e-5
        a.append(dict(X=xs[LLAMA31_8B_X_GROUP[name]], dY=inp["dy"][name].to(DEV),
                      W=inp["w"][name].to(DEV), m=m, v=v, m_scale=ms, v_scale=vs,
                      dX=torch.empty((bt, d_in), dtype=torch.bfloat16, device=DEV)))
    b = _clone(a)
    F.linear_backward_grouped(a, step=1, **ADAMW)
    for ly in b:
        F.linear_backward(ly["X"], ly["dY"], ly["W"], ly["dX"], ly["m"], ly["v"], step=1,
                          m_scale=ly["m_scale"], v_scale=ly["v_scale"], **ADAMW)
    assert F.device_error() == 0
    for x, y in zip(a, b):
        for k in ("dX", "W", "m", "v", "m_scale", "v_scale"):
            if x[k] is not None:
                assert _same(x[k], y[k]), k


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_dgrad_grouped_ragged_against_the_oracle(splits, tune):
    # projections whose reductions over d_out differ and are not multiples of
    # the 64-deep k-step, widths off the 256-column tile, a token count off
    # the 256-row tile; split partials in a workspace the library sizes.  Every
    # element is compared with the oracle, and each dX equals forge_dgrad's at
    # the same split count bit for bit
    bt = 333
    shapes = [(136, 264), (1000, 520), (520, 1032), (2056, 128)]   # (d_out, d_in)
    tune(splits=splits)
    items, host = [], []
    for i, (d_out, d_in) in enumerate(shapes):
        s = make_step_inputs(16, i, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True,
                             spike_frac=0.01)
        items.append(dict(dY=s.dy.to(DEV), W=s.w.to(DEV),
                          dX=torch.full((bt, d_in), float("nan"), dtype=torch.bfloat16,
                                        device=DEV)))
        host.append(s)
    need = F.dgrad_workspace_bytes(items)
    ws = torch.empty(max(1, need // 4), dtype=torch.float32, device=DEV) if need else None
    F.dgrad_grouped(items, workspace=ws)
    assert F.device_error() == 0
    # the launch's split count: the forced one, capped by the longest
    # reduction's limit (at least 8 k-steps per split: 33 k-steps -> 4) and by
    # the shortest reduction's k-steps (3)
    grouped_splits = min(splits, 4, 3)
    for it, s, (d_out, d_in) in zip(items, host, shapes):
        check_dx(bf16_bits(it["dX"].cpu()), bf16_bits(s.dy), bf16_bits(s.w),
                 label=f"grouped ragged dX splits={splits}")
        single = int(F.describe_dgrad_config(bt, d_in, d_out).split("splits=")[1].split()[0])
        if single == grouped_splits:
            ref = torch.empty_like(it["dX"])
            F.dgrad(it["dY"], it["W"], ref)
            assert F.device_error() == 0
            assert _same(it["dX"], ref)
