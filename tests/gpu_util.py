"""Shared plumbing for the GPU tests: moving oracle states to the device and
back, and one call of the library per arm."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import bf16_bits, bits_to_bf16

DEV = torch.device("cuda:0")


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from weight_gradient_gemm_gb300 import _build
    _build.build()
    F.lib()
    torch.cuda.set_device(DEV)


def mom_to_dev(mom: O.Moment):
    if mom.fmt == O.FMT_FP32:
        return torch.from_numpy(mom.data.copy()).to(DEV), None
    if mom.fmt == O.FMT_BF16:
        return bits_to_bf16(mom.data).to(DEV), None
    return (torch.from_numpy(mom.data.copy()).to(DEV),
            torch.from_numpy(mom.scale.copy()).to(DEV))


def mom_from_dev(fmt: int, data: torch.Tensor, scale) -> O.Moment:
    if fmt == O.FMT_FP32:
        return O.Moment(fmt, data.cpu().numpy())
    if fmt == O.FMT_BF16:
        return O.Moment(fmt, bf16_bits(data.cpu()))
    return O.Moment(fmt, data.cpu().numpy(), scale.cpu().numpy())


def dev_state(w_bits, m: O.Moment, v: O.Moment):
    W = bits_to_bf16(w_bits).to(DEV)
    md, ms = mom_to_dev(m)
    vd, vs = mom_to_dev(v)
    return W, md, vd, ms, vs


def hyper_kwargs(h: O.Hyper):
    return dict(lr=h.lr, beta1=h.beta1, beta2=h.beta2, eps=h.eps, weight_decay=h.wd)


def gpu_fused(x, dy, w_bits, m, v, hyper, t):
    """One fused step on the GPU from the given (host) state.  Returns the new
    state as host objects (W bits, m, v)."""
    W, md, vd, ms, vs = dev_state(w_bits, m, v)
    X, dY = x.to(DEV), dy.to(DEV)
    F.wgrad_adamw(X, dY, W, md, vd, step=t, m_scale=ms, v_scale=vs, **hyper_kwargs(hyper))
    st = F.device_error()
    assert st == 0, F.status_string(st)
    return bf16_bits(W.cpu()), mom_from_dev(m.fmt, md, ms), mom_from_dev(v.fmt, vd, vs)


def gpu_unfused(x, dy, w_bits, m, v, hyper, t, dw_dtype=torch.float32):
    """forge_wgrad into a stored dW, then forge_adamw."""
    W, md, vd, ms, vs = dev_state(w_bits, m, v)
    X, dY = x.to(DEV), dy.to(DEV)
    dW = torch.empty((W.shape[0], W.shape[1]), dtype=dw_dtype, device=DEV)
    F.wgrad(X, dY, dW)
    F.adamw(dW, W, md, vd, step=t, m_scale=ms, v_scale=vs, **hyper_kwargs(hyper))
    st = F.device_error()
    assert st == 0, F.status_string(st)
    return bf16_bits(W.cpu()), mom_from_dev(m.fmt, md, ms), mom_from_dev(v.fmt, vd, vs)


def ref_inputs(x, dy, w_bits, m, v, rows=None):
    xb, db = bf16_bits(x), bf16_bits(dy)
    return dict(G=O.wgrad(xb, db, rows), S=O.wgrad_abs(xb, db, rows), W_bits=w_bits, m=m, v=v)


def same_moment(a: O.Moment, b: O.Moment) -> bool:
    ok = np.array_equal(a.data.view(np.uint8), b.data.view(np.uint8))
    if a.scale is not None:
        ok = ok and np.array_equal(a.scale.view(np.uint32), b.scale.view(np.uint32))
    return ok
