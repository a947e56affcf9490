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
MOM_FP32, MOM_BF16, MOM_INT8_B128, MOM_FP8_E4M3 = 0, 1, 2, 3
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


class ForgeAccumItem(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("dY", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("d_in", ctypes.c_int64), ("d_out", ctypes.c_int64)]


class ForgeDgradItem(ctypes.Structure):
    _fields_ = [("dY", ctypes.c_void_p), ("W", ctypes.c_void_p), ("dX", ctypes.c_void_p),
                ("d_in", ctypes.c_int64), ("d_out", ctypes.c_int64)]

# forge_profile values
PROFILES = {"auto": -1, "stream": 0, "mma": 1, "balanced": 2, "deep": 3}


class ForgeTuning(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int) for k in ("profile", "cta_group", "bn", "group_m",
                                            "poll_store", "splits", "l2_hints",
                                            "state_prefetch")]


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
            sz = ctypes.c_size_t
            L.forge_wgrad_opt_grouped.argtypes = [ctypes.POINTER(ForgeLinear), st, i64, st,
                                                  ctypes.POINTER(ForgeOptHyper), i64, st, vp]
            L.forge_wgrad_opt_grouped.restype = st
            L.forge_wgrad_adamw_sr_grouped.argtypes = [ctypes.POINTER(ForgeLinear),
                                                       ctypes.POINTER(ctypes.c_uint64), st, i64,
                                                       f32, f32, f32, f32, f32, i64, st, vp]
            L.forge_wgrad_adamw_sr_grouped.restype = st
            L.forge_wgrad_accumulate_grouped.argtypes = [ctypes.POINTER(ForgeAccumItem), st, i64,
                                                         f32, vp]
            L.forge_wgrad_accumulate_grouped.restype = st
            L.forge_dgrad_grouped.argtypes = [ctypes.POINTER(ForgeDgradItem), st, i64, vp, sz, vp]
            L.forge_dgrad_grouped.restype = st
            L.forge_dgrad_workspace_bytes.argtypes = [ctypes.POINTER(ForgeDgradItem), st, i64]
            L.forge_dgrad_workspace_bytes.restype = sz
            L.forge_linear_backward_grouped.argtypes = [ctypes.POINTER(ForgeLinear),
                                                        ctypes.POINTER(vp), st, i64, f32, f32,
                                                        f32, f32, f32, i64, st, vp, sz, vp]
            L.forge_linear_backward_grouped.restype = st
            L.forge_wgrad_adamw_acc.argtypes = [vp, vp, vp, ForgeMoment, ForgeMoment, vp, i64,
                                                i64, i64, f32, f32, f32, f32, f32, i64, st, vp]
            L.forge_wgrad_adamw_acc.restype = st
            L.forge_wgrad_adamw_acc_grouped.argtypes = [ctypes.POINTER(ForgeLinear),
                                                        ctypes.POINTER(vp), st, i64, f32, f32,
                                                        f32, f32, f32, i64, st, vp]
            L.forge_wgrad_adamw_acc_grouped.restype = st
            L.forge_fp8_roll_scales.argtypes = [vp, st, f32, vp]
            L.forge_fp8_roll_scales.restype = st
            L.forge_set_tuning.argtypes = [ctypes.POINTER(ForgeTuning)]
            L.forge_set_tuning.restype = None
            L.forge_get_tuning.argtypes = [ctypes.POINTER(ForgeTuning)]
            L.forge_get_tuning.restype = None
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
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur} "
                         f"(the library runs on the current device)")


def _want(t: Optional[torch.Tensor], name: str, shape, dtypes) -> None:
    """Shape and dtype of one argument, checked before anything reaches the
    library: the kernels size their tensor maps from the shapes they are
    given, so a short buffer would be read or written past its end."""
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {list(dtypes)}")


_BF16 = (torch.bfloat16,)
_F32 = (torch.float32,)
_MOM = (torch.float32, torch.bfloat16, torch.int8, torch.float8_e4m3fn)


def _operands(X: torch.Tensor, dY: torch.Tensor):
    """bt, d_in, d_out of X [bt, d_in] and dY [bt, d_out] (both bf16)."""
    if X.dim() != 2 or dY.dim() != 2:
        raise ValueError("X and dY must be 2-D")
    bt, d_in = X.shape
    d_out = dY.shape[1]
    _want(X, "X", (bt, d_in), _BF16)
    _want(dY, "dY", (bt, d_out), _BF16)
    return bt, d_in, d_out


def _moments(m, v, m_scale, v_scale, d_out: int, d_in: int, dtypes=_MOM) -> int:
    """Checks AdamW moments (and int8 scales) of a [d_out, d_in] weight;
    returns the moment format."""
    _want(m, "m", (d_out, d_in), dtypes)
    _want(v, "v", (d_out, d_in), (m.dtype,))
    fmt = moment_format(m)
    if fmt == MOM_INT8_B128:
        if d_in % 128:
            raise ValueError("int8 moments need d_in % 128 == 0")
        _want(m_scale, "m_scale", (d_out, d_in // 128), _F32)
        _want(v_scale, "v_scale", (d_out, d_in // 128), _F32)
    elif fmt == MOM_FP8_E4M3:
        if d_in % 16:
            raise ValueError("fp8 moments need d_in % 16 == 0")
        _want(m_scale, "m_scale", (4,), _F32)     # forge_fp8_scales
        _want(v_scale, "v_scale", (4,), _F32)
    return fmt


def _on_device(**tensors) -> None:
    for n, t in tensors.items():
        if t is not None:
            _dense(t, n)


def moment_format(m: torch.Tensor) -> int:
    if m.dtype == torch.float32:
        return MOM_FP32
    if m.dtype == torch.bfloat16:
        return MOM_BF16
    if m.dtype == torch.int8:
        return MOM_INT8_B128
    if m.dtype == torch.float8_e4m3fn:
        return MOM_FP8_E4M3
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
    bt, d_in, d_out = _operands(X, dY)
    _want(W, "W", (d_out, d_in), _BF16)
    fmt = _moments(m, v, m_scale, v_scale, d_out, d_in)
    _on_device(X=X, dY=dY, W=W, m=m, v=v, m_scale=m_scale, v_scale=v_scale)
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
    bt, d_in, d_out = _operands(X, dY)
    _want(W, "W", (d_out, d_in), _BF16)
    n_st = OPT_STATES.get(opt)
    if n_st is None:
        raise ValueError(f"unknown optimizer {opt}")
    states = [s1, s2][:n_st]
    for i, st_t in enumerate(states):
        _want(st_t, f"s{i + 1}", (d_out, d_in),
              (states[0].dtype,) if i else (torch.float32, torch.bfloat16))
    _on_device(X=X, dY=dY, W=W, **{f"s{i + 1}": t for i, t in enumerate(states)})
    fmt = moment_format(states[0]) if states else MOM_FP32
    h = ForgeOptHyper(lr, weight_decay, beta1, beta2, eps, momentum, alpha, momentum_decay)
    st = lib().forge_wgrad_opt(_ptr(X), _ptr(dY), _ptr(W), _moment(s1, None), _moment(s2, None),
                               bt, d_in, d_out, opt, ctypes.byref(h), step, fmt,
                               _stream(stream))
    _check(st, "forge_wgrad_opt")


def wgrad_accumulate(X: torch.Tensor, dY: torch.Tensor, B: torch.Tensor, beta: float,
                     stream=None) -> None:
    """B = beta * B + dY^T X (B fp32 [d_out, d_in], updated in place; not
    read when beta is 0)."""
    bt, d_in, d_out = _operands(X, dY)
    _want(B, "B", (d_out, d_in), _F32)
    _on_device(X=X, dY=dY, B=B)
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
    bt, d_in, d_out = _operands(X, dY)
    _want(W, "W", (d_out, d_in), _BF16)
    _moments(m, v, None, None, d_out, d_in, (torch.float32, torch.bfloat16))
    _on_device(X=X, dY=dY, W=W, m=m, v=v)
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
    if n > MAX_GROUP:
        raise ValueError(f"at most {MAX_GROUP} layers per grouped call")
    for i, ly in enumerate(layers):
        b, d_in, d_out = _operands(ly["X"], ly["dY"])
        _want(ly["W"], "W", (d_out, d_in), _BF16)
        f = _moments(ly["m"], ly["v"], ly.get("m_scale"), ly.get("v_scale"), d_out, d_in)
        _on_device(X=ly["X"], dY=ly["dY"], W=ly["W"], m=ly["m"], v=ly["v"],
                   m_scale=ly.get("m_scale"), v_scale=ly.get("v_scale"))
        if fmt is not None and f != fmt:
            raise ValueError("all layers of a group need the same moment format")
        fmt = f
        if bt is not None and b != bt:
            raise ValueError("all layers of a group need the same token count")
        bt = b
        arr[i] = ForgeLinear(_ptr(ly["X"]), _ptr(ly["dY"]), _ptr(ly["W"]),
                             _moment(ly["m"], ly.get("m_scale")),
                             _moment(ly["v"], ly.get("v_scale")), d_in, d_out)
    st = lib().forge_wgrad_adamw_grouped(arr, n, bt or 0, lr, beta1, beta2, eps, weight_decay,
                                         step, fmt if fmt is not None else 0, _stream(stream))
    _check(st, "forge_wgrad_adamw_grouped")


def wgrad(X: torch.Tensor, dY: torch.Tensor, dW: torch.Tensor, stream=None) -> None:
    """dW = dY^T X stored (fp32 or bf16 by dW's dtype)."""
    bt, d_in, d_out = _operands(X, dY)
    _want(dW, "dW", (d_out, d_in), (torch.float32, torch.bfloat16))
    _on_device(X=X, dY=dY, dW=dW)
    dt = {torch.float32: DT_FP32, torch.bfloat16: DT_BF16}[dW.dtype]
    _check(lib().forge_wgrad(_ptr(X), _ptr(dY), _ptr(dW), dt, bt, d_in, d_out, _stream(stream)),
           "forge_wgrad")


def _dgrad_shapes(dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor):
    """bt, d_out, d_in of dY [bt, d_out], W [d_out, d_in], dX [bt, d_in] (bf16)."""
    if dY.dim() != 2 or W.dim() != 2:
        raise ValueError("dY and W must be 2-D")
    bt, d_out = dY.shape
    d_in = W.shape[1]
    _want(dY, "dY", (bt, d_out), _BF16)
    _want(W, "W", (d_out, d_in), _BF16)
    _want(dX, "dX", (bt, d_in), _BF16)
    _on_device(dY=dY, W=W, dX=dX)
    return bt, d_out, d_in


def dgrad(dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor, stream=None) -> None:
    """dX = dY W (bf16): the layer's input gradient.  dY [bt, d_out],
    W [d_out, d_in], dX [bt, d_in], all bf16."""
    bt, d_out, d_in = _dgrad_shapes(dY, W, dX)
    _check(lib().forge_dgrad(_ptr(dY), _ptr(W), _ptr(dX), bt, d_in, d_out, _stream(stream)),
           "forge_dgrad")


def dgrad_noalloc(dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor, stream=None) -> None:
    """dgrad with its split partials in the library's static scratch (no
    allocation); calls of it on one device must not overlap in time."""
    bt, d_out, d_in = _dgrad_shapes(dY, W, dX)
    _check(lib().forge_dgrad_noalloc(_ptr(dY), _ptr(W), _ptr(dX), bt, d_in, d_out,
                                     _stream(stream)), "forge_dgrad_noalloc")


def linear_backward(X: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, dX: torch.Tensor,
                    m: torch.Tensor, v: torch.Tensor, *, lr: float, beta1: float, beta2: float,
                    eps: float, weight_decay: float, step: int,
                    m_scale: Optional[torch.Tensor] = None,
                    v_scale: Optional[torch.Tensor] = None, stream=None) -> None:
    """The layer's backward step: dX = dY W from the weight before the update,
    then the fused weight-gradient + AdamW step (W, m, v updated in place)."""
    bt, d_in, d_out = _operands(X, dY)
    _want(W, "W", (d_out, d_in), _BF16)
    _want(dX, "dX", (bt, d_in), _BF16)
    fmt = _moments(m, v, m_scale, v_scale, d_out, d_in)
    _on_device(X=X, dY=dY, W=W, dX=dX, m=m, v=v, m_scale=m_scale, v_scale=v_scale)
    st = lib().forge_linear_backward(
        _ptr(X), _ptr(dY), _ptr(W), _ptr(dX), _moment(m, m_scale), _moment(v, v_scale), bt,
        d_in, d_out, lr, beta1, beta2, eps, weight_decay, step, fmt, _stream(stream))
    _check(st, "forge_linear_backward")


def adamw(dW: Optional[torch.Tensor], W: torch.Tensor, m: torch.Tensor, v: torch.Tensor, *,
          lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, step: int,
          m_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
          stream=None) -> None:
    """The unfused optimizer step on a stored gradient (None = zero gradient)."""
    if W.dim() != 2:
        raise ValueError("W must be 2-D")
    d_out, d_in = W.shape
    _want(W, "W", (d_out, d_in), _BF16)
    fmt = _moments(m, v, m_scale, v_scale, d_out, d_in)
    dt = DT_FP32
    if dW is not None:
        _want(dW, "dW", (d_out, d_in), (torch.float32, torch.bfloat16))
        dt = {torch.float32: DT_FP32, torch.bfloat16: DT_BF16}[dW.dtype]
    _on_device(W=W, m=m, v=v, dW=dW, m_scale=m_scale, v_scale=v_scale)
    st = lib().forge_adamw(_ptr(dW), dt, _ptr(W), _moment(m, m_scale), _moment(v, v_scale),
                           d_in, d_out, lr, beta1, beta2, eps, weight_decay, step, fmt,
                           _stream(stream))
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


def get_tuning() -> dict:
    """The tuning overrides in force (see forge_set_tuning in forge.h)."""
    t = ForgeTuning()
    lib().forge_get_tuning(ctypes.byref(t))
    names = {v: k for k, v in PROFILES.items()}
    return dict(profile=names.get(t.profile, "auto"), cg=t.cta_group, bn=t.bn,
                group_m=t.group_m, poll_store=t.poll_store, splits=t.splits,
                l2_hints=t.l2_hints, state_prefetch=t.state_prefetch)


def set_tuning(profile: str = "auto", cg: int = 0, bn: int = 0, group_m: int = 0,
               poll_store: int = -1, splits: int = 0, l2_hints: int = -1,
               state_prefetch: int = -1) -> None:
    """Replace the tuning overrides (the defaults leave every choice to the
    library).  profile: auto|stream|balanced|mma|deep; cg: 1 or 2 CTAs per
    tile; bn: 128 or 256; group_m: 1..64; poll_store: 0 or 1; splits: 1..8;
    l2_hints: 0..3; state_prefetch: 0..32 slices."""
    if profile not in PROFILES:
        raise ValueError(f"unknown profile {profile}")
    t = ForgeTuning(PROFILES[profile], int(cg), int(bn), int(group_m), int(poll_store),
                    int(splits), int(l2_hints), int(state_prefetch))
    lib().forge_set_tuning(ctypes.byref(t))


class tuning:
    """Context manager: tuning overrides for the calls inside the block,
    the previous ones restored afterwards.  Fields not given keep their
    current value."""

    def __init__(self, **kw):
        self.kw = kw

    def __enter__(self):
        self.saved = get_tuning()
        set_tuning(**{**self.saved, **self.kw})
        return self

    def __exit__(self, *exc):
        set_tuning(**self.saved)
        return False


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
    if fmt == MOM_FP8_E4M3:
        if d_in % 16:
            raise ValueError("fp8 moments need d_in % 16 == 0")
        q = lambda: torch.zeros((d_out, d_in), dtype=torch.float8_e4m3fn, device=device)  # noqa: E731
        sc = alloc_fp8_scales(2, device=device)
        return q(), q(), sc[0], sc[1]
    raise ValueError(f"unknown moment format {fmt}")


def alloc_fp8_scales(n: int, read_scale: float = 1.0, write_scale: float = 1.0,
                     device="cuda") -> torch.Tensor:
    """n forge_fp8_scales records as one fp32 [n, 4] tensor (read scale,
    write scale, amax, unused); row i is the `m_scale`/`v_scale` of one fp8
    moment."""
    t = torch.zeros((n, 4), dtype=torch.float32, device=device)
    t[:, 0] = read_scale
    t[:, 1] = write_scale
    return t


def fp8_roll_scales(scales: torch.Tensor, headroom: float = 1.0, stream=None) -> None:
    """The scale roll between two steps of fp8 moments, on the device:
    read <- write, write <- amax * headroom / 448 (kept when amax is 0),
    amax <- 0, for every record of `scales` ([n, 4] or [4] fp32)."""
    if scales.dtype != torch.float32 or scales.shape[-1] != 4 or scales.dim() > 2:
        raise ValueError("scales must be fp32 [n, 4] or [4]")
    _dense(scales, "scales")
    n = 1 if scales.dim() == 1 else scales.shape[0]
    _check(lib().forge_fp8_roll_scales(_ptr(scales), n, headroom, _stream(stream)),
           "forge_fp8_roll_scales")


# ---------------------------------------------------------------------------
# grouped calls: several linear layers with one token count in one launch
# ---------------------------------------------------------------------------

def _group_arr(layers, m_key="m", v_key="v", scales=True):
    """ForgeLinear array, token count and the layers' (d_in, d_out)."""
    n = len(layers)
    if not 1 <= n <= MAX_GROUP:
        raise ValueError(f"1 to {MAX_GROUP} layers per grouped call")
    arr = (ForgeLinear * n)()
    bt = None
    for i, ly in enumerate(layers):
        b, d_in, d_out = _operands(ly["X"], ly["dY"])
        if bt is not None and b != bt:
            raise ValueError("all layers of a group need the same token count")
        bt = b
        _want(ly["W"], "W", (d_out, d_in), _BF16)
        m, v = ly.get(m_key), ly.get(v_key)
        _on_device(X=ly["X"], dY=ly["dY"], W=ly["W"], m=m, v=v,
                   m_scale=ly.get("m_scale") if scales else None,
                   v_scale=ly.get("v_scale") if scales else None)
        arr[i] = ForgeLinear(_ptr(ly["X"]), _ptr(ly["dY"]), _ptr(ly["W"]),
                             _moment(m, ly.get("m_scale") if scales else None) if m is not None
                             else ForgeMoment(None, None),
                             _moment(v, ly.get("v_scale") if scales else None) if v is not None
                             else ForgeMoment(None, None), d_in, d_out)
    return arr, n, bt


def wgrad_adamw_acc(X: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, m: torch.Tensor,
                    v: torch.Tensor, B: torch.Tensor, *, lr: float, beta1: float, beta2: float,
                    eps: float, weight_decay: float, step: int, stream=None) -> None:
    """The step at the final micro-batch of the exact-accumulation mode: AdamW
    on fp32(B + dY^T X), B being the fp32 accumulator of the earlier
    micro-batches (read, not written); W, m, v updated in place; fp32 or bf16
    moments."""
    wgrad_adamw_acc_grouped([dict(X=X, dY=dY, W=W, m=m, v=v, B=B)], lr=lr, beta1=beta1,
                            beta2=beta2, eps=eps, weight_decay=weight_decay, step=step,
                            stream=stream)


def wgrad_adamw_acc_grouped(layers, *, lr: float, beta1: float, beta2: float, eps: float,
                            weight_decay: float, step: int, stream=None) -> None:
    """wgrad_adamw_acc on several layers in one launch; each layer is a dict
    with X, dY, W, m, v and its accumulator B (fp32 [d_out, d_in])."""
    arr, n, bt = _group_arr(layers, scales=False)
    fmt = None
    bs = (ctypes.c_void_p * n)()
    for i, ly in enumerate(layers):
        d_out, d_in = ly["W"].shape
        f = _moments(ly["m"], ly["v"], None, None, d_out, d_in)
        if f not in (MOM_FP32, MOM_BF16):
            raise ValueError("the final micro-batch's step takes fp32 or bf16 moments")
        if fmt is not None and f != fmt:
            raise ValueError("all layers of a group need the same moment format")
        fmt = f
        _want(ly["B"], "B", (d_out, d_in), (torch.float32,))
        _on_device(B=ly["B"])
        bs[i] = _ptr(ly["B"])
    st = lib().forge_wgrad_adamw_acc_grouped(arr, bs, n, bt or 0, lr, beta1, beta2, eps,
                                             weight_decay, step, fmt, _stream(stream))
    _check(st, "forge_wgrad_adamw_acc_grouped")


def wgrad_opt_grouped(layers, opt: int, *, lr: float, weight_decay: float, step: int,
                      beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                      momentum: float = 0.9, alpha: float = 0.99, momentum_decay: float = 4e-3,
                      stream=None) -> None:
    """wgrad_opt on several layers in one launch; each layer is a dict with X,
    dY, W and the optimizer's states s1, s2 (as many as OPT_STATES says)."""
    n_st = OPT_STATES.get(opt)
    if n_st is None:
        raise ValueError(f"unknown optimizer {opt}")
    fmt = MOM_FP32
    for ly in layers:
        d_out, d_in = ly["W"].shape
        sts = [ly.get("s1"), ly.get("s2")][:n_st]
        for i, t in enumerate(sts):
            _want(t, f"s{i + 1}", (d_out, d_in),
                  (sts[0].dtype,) if i else (torch.float32, torch.bfloat16))
        if sts:
            fmt = moment_format(sts[0])
    arr, n, bt = _group_arr([dict(ly, s1=ly.get("s1") if n_st >= 1 else None,
                                  s2=ly.get("s2") if n_st >= 2 else None) for ly in layers],
                            "s1", "s2", scales=False)
    h = ForgeOptHyper(lr, weight_decay, beta1, beta2, eps, momentum, alpha, momentum_decay)
    _check(lib().forge_wgrad_opt_grouped(arr, n, bt, opt, ctypes.byref(h), step, fmt,
                                         _stream(stream)), "forge_wgrad_opt_grouped")


def wgrad_adamw_sr_grouped(layers, seeds, *, lr: float, beta1: float, beta2: float, eps: float,
                           weight_decay: float, step: int, stream=None) -> None:
    """wgrad_adamw_sr on several layers in one launch; layer i uses seeds[i]."""
    fmt = None
    for ly in layers:
        d_out, d_in = ly["W"].shape
        f = _moments(ly["m"], ly["v"], None, None, d_out, d_in, (torch.float32, torch.bfloat16))
        if fmt is not None and f != fmt:
            raise ValueError("all layers of a group need the same moment format")
        fmt = f
    arr, n, bt = _group_arr(layers, scales=False)
    if len(seeds) != n:
        raise ValueError("one seed per layer")
    sd = (ctypes.c_uint64 * n)(*[int(x) for x in seeds])
    _check(lib().forge_wgrad_adamw_sr_grouped(arr, sd, n, bt, lr, beta1, beta2, eps,
                                              weight_decay, step, fmt, _stream(stream)),
           "forge_wgrad_adamw_sr_grouped")


def wgrad_accumulate_grouped(items, beta: float, stream=None) -> None:
    """wgrad_accumulate on several layers (dicts with X, dY, B) in one launch."""
    n = len(items)
    if not 1 <= n <= MAX_GROUP:
        raise ValueError(f"1 to {MAX_GROUP} layers per grouped call")
    arr = (ForgeAccumItem * n)()
    bt = None
    for i, it in enumerate(items):
        b, d_in, d_out = _operands(it["X"], it["dY"])
        if bt is not None and b != bt:
            raise ValueError("all layers of a group need the same token count")
        bt = b
        _want(it["B"], "B", (d_out, d_in), _F32)
        _on_device(X=it["X"], dY=it["dY"], B=it["B"])
        arr[i] = ForgeAccumItem(_ptr(it["X"]), _ptr(it["dY"]), _ptr(it["B"]), d_in, d_out)
    _check(lib().forge_wgrad_accumulate_grouped(arr, n, bt, beta, _stream(stream)),
           "forge_wgrad_accumulate_grouped")


def _dgrad_arr(items):
    n = len(items)
    if not 1 <= n <= MAX_GROUP:
        raise ValueError(f"1 to {MAX_GROUP} projections per grouped call")
    arr = (ForgeDgradItem * n)()
    bt = None
    for i, it in enumerate(items):
        b, d_out, d_in = _dgrad_shapes(it["dY"], it["W"], it["dX"])
        if bt is not None and b != bt:
            raise ValueError("all projections of a group need the same token count")
        bt = b
        arr[i] = ForgeDgradItem(_ptr(it["dY"]), _ptr(it["W"]), _ptr(it["dX"]), d_in, d_out)
    return arr, n, bt


def dgrad_workspace_bytes(items) -> int:
    """Workspace bytes dgrad_grouped wants for these projections (dicts with
    dY, W, dX), 0 if it would not split."""
    arr, n, bt = _dgrad_arr(items)
    return int(lib().forge_dgrad_workspace_bytes(arr, n, bt))


def dgrad_grouped(items, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """dX = dY W for several projections (dicts with dY, W, dX) in one launch;
    split partials go to `workspace` (a device tensor; none: unsplit)."""
    arr, n, bt = _dgrad_arr(items)
    if workspace is not None:
        _dense(workspace, "workspace")
    _check(lib().forge_dgrad_grouped(arr, n, bt, _ptr(workspace),
                                     0 if workspace is None else workspace.numel() *
                                     workspace.element_size(), _stream(stream)),
           "forge_dgrad_grouped")


def linear_backward_grouped(layers, *, lr: float, beta1: float, beta2: float, eps: float,
                            weight_decay: float, step: int,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """linear_backward on several layers in one grouped dX launch and one
    grouped fused launch.  Each layer is a dict with X, dY, W, dX, m, v (and
    m_scale, v_scale for int8 or fp8 moments)."""
    fmt = None
    for ly in layers:
        d_out, d_in = ly["W"].shape
        f = _moments(ly["m"], ly["v"], ly.get("m_scale"), ly.get("v_scale"), d_out, d_in)
        if fmt is not None and f != fmt:
            raise ValueError("all layers of a group need the same moment format")
        fmt = f
        _want(ly["dX"], "dX", (ly["X"].shape[0], d_in), _BF16)
        _on_device(dX=ly["dX"])
    arr, n, bt = _group_arr(layers)
    dx = (ctypes.c_void_p * n)(*[_ptr(ly["dX"]) for ly in layers])
    if workspace is not None:
        _dense(workspace, "workspace")
    _check(lib().forge_linear_backward_grouped(
        arr, dx, n, bt, lr, beta1, beta2, eps, weight_decay, step, fmt, _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)), "forge_linear_backward_grouped")
