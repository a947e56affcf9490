"""Python binding for libforge (ctypes).  Argument marshalling only: every
step of the computation runs in the library's CUDA kernels.

PyTorch supplies device memory and the current CUDA stream.  There is no CPU
fallback: if ``libforge.so`` has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libforge.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "forge.h")

FORGE_OK = 0
STATUS_NAMES = {
    0: "FORGE_OK", 1: "FORGE_ERR_NULL", 2: "FORGE_ERR_ALIGN", 3: "FORGE_ERR_SHAPE",
    4: "FORGE_ERR_FORMAT", 5: "FORGE_ERR_HYPER", 6: "FORGE_ERR_ALIAS", 7: "FORGE_ERR_ARCH",
    8: "FORGE_ERR_LAUNCH", 9: "FORGE_ERR_DEVICE_TIMEOUT", 10: "FORGE_ERR_CUDA",
    11: "FORGE_ERR_DEVICE_CONFIG",
}
MOM_FP32, MOM_BF16, MOM_INT8_B128 = 0, 1, 2
DT_FP32, DT_BF16 = 0, 1


class ForgeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class ForgeMoment(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class ForgeOptHyper(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in ("lr", "weight_decay", "beta1", "beta2", "eps",
                                              "momentum", "alpha", "momentum_decay")]


# forge_optimizer values, and how many state tensors each keeps
OPT_SGD, OPT_SGD_MOMENTUM, OPT_ADAGRAD, OPT_RMSPROP, OPT_LION, OPT_NADAM, OPT_RADAM = range(7)
OPT_STATES = {OPT_SGD: 0, OPT_SGD_MOMENTUM: 1, OPT_ADAGRAD: 1, OPT_RMSPROP: 1, OPT_LION: 1,
              OPT_NADAM: 2, OPT_RADAM: 2}


class ForgeLinear(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("dY", ctypes.c_void_p), ("W", ctypes.c_void_p),
                ("m", ForgeMoment), ("v", ForgeMoment), ("d_in", ctypes.c_int64),
                ("d_out", ctypes.c_int64)]


MAX_GROUP = 8

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libforge.so (loaded once)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; "
                    f"g.build()\"` first")
            L = ctypes.CDLL(LIB_PATH)
            i64, f32, vp, st = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
            L.forge_wgrad_adamw.argtypes = [vp, vp, vp, ForgeMoment, ForgeMoment, i64, i64, i64,
                                            f32, f32, f32, f32, f32, i64, st, vp]
            L.forge_wgrad_adamw.restype = st
            L.forge_wgrad_opt.argtypes = [vp, vp, vp, ForgeMoment, ForgeMoment, i64, i64, i64,
                                          st, ctypes.POINTER(ForgeOptHyper), i64, st, vp]
            L.forge_wgrad_opt.restype = st
            L.forge_wgrad_adamw_sr.argtypes = [vp, vp, vp, ForgeMoment, ForgeMoment, i64, i64,
                                               i64, f32, f32, f32, f32, f32, i64, st,
                                               ctypes.c_uint64, vp]
            L.forge_wgrad_adamw_sr.restype = st
            L.forge_wgrad_accumulate.argtypes = [vp, vp, vp, f32, i64, i64, i64, vp]
            L.forge_wgrad_accumulate.restype = st
            L.forge_wgrad_adamw_grouped.argtypes = [ctypes.POINTER(ForgeLinear), st, i64,
                                                    f32, f32, f32, f32, f32, i64, st, vp]
            L.forge_wgrad_adamw_grouped.restype = st
            L.forge_wgrad.argtypes = [vp, vp, vp, st, i64, i64, i64, vp]
            L.forge_wgrad.restype = st
            L.forge_adamw.argtypes = [vp, st, vp, ForgeMoment, ForgeMoment, i64, i64,
                                      f32, f32, f32, f32, f32, i64, st, vp]
            L.forge_adamw.restype = st
            L.forge_dgrad.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            L.forge_dgrad.restype = st
            L.forge_dgrad_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            L.forge_dgrad_noalloc.restype = st
            L.forge_linear_backward.argtypes = [vp, vp, vp, vp, ForgeMoment, ForgeMoment, i64,
                                                i64, i64, f32, f32, f32, f32, f32, i64, st, vp]
            L.forge_linear_backward.restype = st
            L.forge_device_error.argtypes = [vp]
            L.forge_device_error.restype = st
            L.forge_status_string.argtypes = [st]
            L.forge_status_string.restype = ctypes.c_char_p
            L.forge_describe_config.argtypes = [i64, i64, i64, st, ctypes.c_char_p, st]
            L.forge_describe_config.restype = st
            L.forge_describe_dgrad_config.argtypes = [i64, i64, i64, ctypes.c_char_p, st]
            L.forge_describe_dgrad_config.restype = st
            L.forge_debug_timeout_site.argtypes = []
            L.forge_debug_timeout_site.restype = st
            L.forge_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.forge_set_wait_limit_ns.restype = None
            L.forge_debug_drop_first_arrival.argtypes = [st]
            L.forge_debug_drop_first_arrival.restype = None
            _lib = L
        return _lib


def header_functions() -> list[str]:
    """Names of the functions include/forge.h declares."""
    src = open(HEADER_PATH).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(forge_[a-z0-9_]+)\s*\(", src)))


def status_string(status: int) -> str:
    try:
        return lib().forge_status_string(int(status)).decode()
    except Exception:
        return STATUS_NAMES.get(int(status), f"status {status}")


def _check(status: int, what: str) -> None:
    if status != FORGE_OK:
        raise ForgeError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dense(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def moment_format(m: torch.Tensor) -> int:
    if m.dtype == torch.float32:
        return MOM_FP32
    if m.dtype == torch.bfloat16:
        return MOM_BF16
    if m.dtype == torch.int8:
        return MOM_INT8_B128
    raise ValueError(f"unsupported moment dtype {m.dtype}")


def _moment(data: torch.Tensor, scale: Optional[torch.Tensor]) -> ForgeMoment:
    return ForgeMoment(_ptr(data), _ptr(scale))


def wgrad_adamw(X: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, m: torch.Tensor,
                v: torch.Tensor, *, lr: float, beta1: float, beta2: float, eps: float,
                weight_decay: float, step: int, m_scale: Optional[torch.Tensor] = None,
                v_scale: Optional[torch.Tensor] = None, stream=None) -> None:
    """One fused step: G = dY^T X, AdamW on G, W/m/v (and int8 scales) updated
    in place.  X [bt, d_in] and dY [bt, d_out] bf16; W [d_out, d_in] bf16;
    m, v fp32, bf16 or int8 (with fp32 scales [d_out, d_in/128])."""
    for t, n in ((X, "X"), (dY, "dY"), (W, "W"), (m, "m"), (v, "v")):
        _dense(t, n)
    bt, d_in = X.shape
    d_out = dY.shape[1]
    fmt = moment_format(m)
    st = lib().forge_wgrad_adamw(
        _ptr(X), _ptr(dY), _ptr(W), _moment(m, m_scale), _moment(v, v_scale), bt, d_in, d_out,
        lr, beta1, beta2, eps, weight_decay, step, fmt, _stream(stream))
    _check(st, "forge_wgrad_adamw")


def wgrad_opt(X: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, opt: int,
              s1: Optional[torch.Tensor] = None, s2: Optional[torch.Tensor] = None, *,
              lr: float, weight_decay: float, step: int, beta1: float = 0.9,
              beta2: float = 0.999, eps: float = 1e-8, momentum: float = 0.9,
              alpha: float = 0.99, momentum_decay: float = 4e-3, stream=None) -> None:
    """One fused step with optimizer `opt` (OPT_*) in place of AdamW: W and the
    optimizer's states s1, s2 (fp32 or bf16, as many as OPT_STATES says)
    updated in place."""
    for t, n in ((X, "X"), (dY, "dY"), (W, "W")):
        _dense(t, n)
    states = [s for s in (s1, s2) if s is not None]
    for s in states:
        _dense(s, "state")
    fmt = moment_format(states[0]) if states else MOM_FP32
    bt, d_in = X.shape
    d_out = dY.shape[1]
    h = ForgeOptHyper(lr, weight_decay, beta1, beta2, eps, momentum, alpha, momentum_decay)
    st = lib().forge_wgrad_opt(_ptr(X), _ptr(dY), _ptr(W), _moment(s1, None), _moment(s2, None),
                               bt, d_in, d_out, opt, ctypes.byref(h), step, fmt,
                               _stream(stream))
    _check(st, "forge_wgrad_opt")


def wgrad_accumulate(X: torch.Tensor, dY: torch.Tensor, B: torch.Tensor, beta: float,
                     stream=None) -> None:
    """B = beta * B + dY^T X (B fp32 [d_out, d_in], updated in place; not
    read when beta is 0)."""
    for t, n in ((X, "X"), (dY, "dY"), (B, "B")):
        _dense(t, n)
    if B.dtype != torch.float32:
        raise TypeError("B must be fp32")
    bt, d_in = X.shape
    d_out = dY.shape[1]
    _check(lib().forge_wgrad_accumulate(_ptr(X), _ptr(dY), _ptr(B), beta, bt, d_in, d_out,
                                        _stream(stream)), "forge_wgrad_accumulate")


def alloc_states(opt: int, d_out: int, d_in: int, fmt: int = MOM_FP32, device="cuda"):
    """Zero-initialised states (s1, s2; None where the optimizer has fewer)."""
    dt = {MOM_FP32: torch.float32, MOM_BF16: torch.bfloat16}[fmt]
    n = OPT_STATES[opt]
    return tuple(torch.zeros((d_out, d_in), dtype=dt, device=device) if i < n else None
                 for i in range(2))


def wgrad_adamw_sr(X: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, m: torch.Tensor,
                   v: torch.Tensor, *, lr: float, beta1: float, beta2: float, eps: float,
                   weight_decay: float, step: int, seed: int, stream=None) -> None:
    """wgrad_adamw with W committed by stochastic rounding (Philox4x64-10
    random bits from `seed`, the weight index and the step); fp32 or bf16 moments."""
    for t, n in ((X, "X"), (dY, "dY"), (W, "W"), (m, "m"), (v, "v")):
        _dense(t, n)
    bt, d_in = X.shape
    d_out = dY.shape[1]
    st = lib().forge_wgrad_adamw_sr(
        _ptr(X), _ptr(dY), _ptr(W), _moment(m, None), _moment(v, None), bt, d_in, d_out,
        lr, beta1, beta2, eps, weight_decay, step, moment_format(m), seed, _stream(stream))
    _check(st, "forge_wgrad_adamw_sr")


def wgrad_adamw_grouped(layers, *, lr: float, beta1: float, beta2: float, eps: float,
                        weight_decay: float, step: int, stream=None) -> None:
    """The fused step on several linear layers (same token count, moment
    format and hyperparameters) in one launch.  `layers` is a sequence of
    dicts with keys X, dY, W, m, v and, for int8 moments, m_scale, v_scale."""
    n = len(layers)
    arr = (ForgeLinear * max(n, 1))()
    fmt = None
    bt = None
    for i, ly in enumerate(layers):
        for k in ("X", "dY", "W", "m", "v"):
            _dense(ly[k], k)
        f = moment_format(ly["m"])
        if fmt is not None and f != fmt:
            raise ValueError("all layers of a group need the same moment format")
        fmt = f
        b = ly["X"].shape[0]
        if bt is not None and b != bt:
            raise ValueError("all layers of a group need the same token count")
        bt = b
        arr[i] = ForgeLinear(_ptr(ly["X"]), _ptr(ly["dY"]), _ptr(ly["W"]),
                             _moment(ly["m"], ly.get("m_scale")),
                             _moment(ly["v"], ly.get("v_scale")),
                             ly["X"].shape[1], ly["dY"].shape[1])
    st = lib().forge_wgrad_adamw_grouped(arr, n, bt or 0, lr, beta1, beta2, eps, weight_decay,
                                         step, fmt if fmt is not None else 0, _stream(stream))
    _check(st, "forge_wgrad_adamw_grouped")


def wgrad(X: torch.Tensor, dY: torch.Tensor, dW: torch.Tensor, stream=None) -> None:
    """dW = dY^T X stored (fp32 or bf16 by dW's dtype)."""
    for t, n in ((X, "X"), (dY, "dY"), (dW, "dW")):
        _dense(t, n)
    bt, d_in = X.shape
    d_out = dY.shape[1]
    dt = {torch.float32: DT_FP32, torch.bfloat16: DT_BF16}[dW.dtype]
    _check(lib().forge_wgrad(_ptr(X), _ptr(dY), _ptr(dW), dt, bt, d_in, d_out, _stream(stream)),
           "forge_wgrad")


def dgrad(dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor, stream=None) -> None:
    """dX = dY W (bf16): the layer's input gradient.  dY [bt, d_out],
    W [d_out, d_in], dX [bt, d_in], all bf16."""
    for t, n in ((dY, "dY"), (W, "W"), (dX, "dX")):
        _dense(t, n)
    if dX.dtype != torch.bfloat16:
        raise TypeError("dX must be bf16")
    bt, d_out = dY.shape
    d_in = W.shape[1]
    _check(lib().forge_dgrad(_ptr(dY), _ptr(W), _ptr(dX), bt, d_in, d_out, _stream(stream)),
           "forge_dgrad")


def dgrad_noalloc(dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor, stream=None) -> None:
    """dgrad with its split partials in the library's static scratch (no
    allocation); calls of it on one device must not overlap in time."""
    for t, n in ((dY, "dY"), (W, "W"), (dX, "dX")):
        _dense(t, n)
    if dX.dtype != torch.bfloat16:
        raise TypeError("dX must be bf16")
    bt, d_out = dY.shape
    d_in = W.shape[1]
    _check(lib().forge_dgrad_noalloc(_ptr(dY), _ptr(W), _ptr(dX), bt, d_in, d_out,
                                     _stream(stream)), "forge_dgrad_noalloc")


def linear_backward(X: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor,
                    m: torch.Tensor, v: torch.Tensor, *, lr: float, beta1: float, beta2: float,
                    eps: float, weight_decay: float, step: int,
                    m_scale: Optional[torch.Tensor] = None,
                    v_scale: Optional[torch.Tensor] = None, stream=None) -> None:
    """The layer's backward step: dX = dY W from the weight before the update,
    then the fused weight-gradient + AdamW step (W, m, v updated in place)."""
    for t, n in ((X, "X"), (dY, "dY"), (W, "W"), (dX, "dX"), (m, "m"), (v, "v")):
        _dense(t, n)
    if dX.dtype != torch.bfloat16:
        raise TypeError("dX must be bf16")
    bt, d_in = X.shape
    d_out = dY.shape[1]
    fmt = moment_format(m)
    st = lib().forge_linear_backward(
        _ptr(X), _ptr(dY), _ptr(W), _ptr(dX), _moment(m, m_scale), _moment(v, v_scale), bt,
        d_in, d_out, lr, beta1, beta2, eps, weight_decay, step, fmt, _stream(stream))
    _check(st, "forge_linear_backward")


def adamw(dW: Optional[torch.Tensor], W: torch.Tensor, m: torch.Tensor, v: torch.Tensor, *,
          lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, step: int,
          m_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
          stream=None) -> None:
    """The unfused optimizer step on a stored gradient (None = zero gradient)."""
    for t, n in ((W, "W"), (m, "m"), (v, "v")):
        _dense(t, n)
    dt = DT_FP32
    if dW is not None:
        _dense(dW, "dW")
        dt = {torch.float32: DT_FP32, torch.bfloat16: DT_BF16}[dW.dtype]
    d_out, d_in = W.shape
    st = lib().forge_adamw(_ptr(dW), dt, _ptr(W), _moment(m, m_scale), _moment(v, v_scale),
                           d_in, d_out, lr, beta1, beta2, eps, weight_decay, step,
                           moment_format(m), _stream(stream))
    _check(st, "forge_adamw")


def device_error(stream=None) -> int:
    """Synchronise and return (and clear) the device error status."""
    return lib().forge_device_error(_stream(stream))


def describe_config(bt: int, d_in: int, d_out: int, fmt: int = MOM_FP32) -> str:
    n = lib().forge_describe_config(bt, d_in, d_out, fmt, None, 0)
    if n < 0:
        raise ValueError("invalid shape or format")
    buf = ctypes.create_string_buffer(n)
    lib().forge_describe_config(bt, d_in, d_out, fmt, buf, n)
    return buf.value.decode()


def describe_dgrad_config(bt: int, d_in: int, d_out: int) -> str:
    """The configuration forge_dgrad would use for dY [bt, d_out], W [d_out, d_in]."""
    n = lib().forge_describe_dgrad_config(bt, d_in, d_out, None, 0)
    if n < 0:
        raise ValueError("invalid shape")
    buf = ctypes.create_string_buffer(n)
    lib().forge_describe_dgrad_config(bt, d_in, d_out, buf, n)
    return buf.value.decode()


def timeout_site() -> int:
    """Where the first timed-out wait happened (see forge.h), 0 if none."""
    return lib().forge_debug_timeout_site()


def set_wait_limit_ns(ns: int) -> None:
    lib().forge_set_wait_limit_ns(int(ns))


def debug_drop_first_arrival(enable: bool = True) -> None:
    lib().forge_debug_drop_first_arrival(1 if enable else 0)


def alloc_moments(d_out: int, d_in: int, fmt: int, device="cuda"):
    """Zero-initialised (m, v, m_scale, v_scale) for a [d_out, d_in] weight."""
    if fmt == MOM_FP32:
        z = lambda: torch.zeros((d_out, d_in), dtype=torch.float32, device=device)  # noqa: E731
        return z(), z(), None, None
    if fmt == MOM_BF16:
        z = lambda: torch.zeros((d_out, d_in), dtype=torch.bfloat16, device=device)  # noqa: E731
        return z(), z(), None, None
    if fmt == MOM_INT8_B128:
        if d_in % 128:
            raise ValueError("int8 moments need d_in % 128 == 0")
        q = lambda: torch.zeros((d_out, d_in), dtype=torch.int8, device=device)  # noqa: E731
        s = lambda: torch.zeros((d_out, d_in // 128), dtype=torch.float32, device=device)  # noqa: E731
        return q(), q(), s(), s()
    raise ValueError(f"unknown moment format {fmt}")
