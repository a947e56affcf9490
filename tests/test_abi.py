"""The C-ABI library builds, loads without a GPU and exports every function
include/forge.h declares; host-side argument checks answer before any device
call.  No compute runs here."""
import ctypes
import subprocess

import pytest
import torch

from weight_gradient_gemm_gb300 import _build
from weight_gradient_gemm_gb300 import forge as F


@pytest.fixture(scope="module")
def L():
    _build.build()
    return F.lib()


def test_header_declares_the_boundary():
    names = F.header_functions()
    for n in ("forge_wgrad_adamw", "forge_wgrad", "forge_adamw", "forge_device_error",
              "forge_status_string", "forge_wgrad_adamw_grouped", "forge_dgrad",
              "forge_linear_backward", "forge_describe_dgrad_config", "forge_dgrad_noalloc",
              "forge_wgrad_opt", "forge_wgrad_accumulate", "forge_wgrad_adamw_sr",
              "forge_fp8_roll_scales", "forge_set_tuning", "forge_get_tuning",
              "forge_wgrad_adamw_acc", "forge_wgrad_adamw_acc_grouped"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", F.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in F.header_functions():
        assert name in exported, name
        assert hasattr(L, name)


def test_status_strings(L):
    for code, name in F.STATUS_NAMES.items():
        assert F.status_string(code).startswith(name)
    assert "unknown" in F.status_string(99)


def test_describe_config_without_gpu(L):
    s = F.describe_config(512, 4096, 4096, F.MOM_FP32)
    assert "tile=128x128" in s and "bk=64" in s
    assert "slice=128" in F.describe_config(4096, 4096, 1024, F.MOM_INT8_B128)
    with pytest.raises(ValueError):
        F.describe_config(512, 4097, 4096)


def test_dgrad_split_choice_without_gpu(L, tune):
    # host logic only (152 SMs assumed without a device).  dX of the
    # Llama-3.1-8B gate/up projections (d_out = 14336, d_in = 4096): at 512
    # tokens 32 pair tiles for 76 SM pairs, so the reduction over d_out is
    # split; from 1024 tokens on the cost estimate keeps it whole
    tune(splits=0)
    s = F.describe_dgrad_config(512, 4096, 14336)
    assert "tile=256x256" in s and "ctas=2" in s and "splits=2" in s, s
    assert "grid=128" in s, s                       # 64 units -> 64 pairs
    for bt in (1024, 2048, 4096, 8192):
        assert "splits=1" in F.describe_dgrad_config(bt, 4096, 14336)
    # the k projection (d_out = 1024: 16 k-steps) is too short to split
    assert "splits=1" in F.describe_dgrad_config(512, 4096, 1024)
    # the override is clamped to splits of at least 8 k-steps
    tune(splits=8)
    assert "splits=8" in F.describe_dgrad_config(512, 4096, 14336)
    assert "splits=2" in F.describe_dgrad_config(512, 4096, 1024)
    assert "splits=1" in F.describe_dgrad_config(512, 4096, 512)
    with pytest.raises(ValueError):
        F.describe_dgrad_config(512, 4097, 4096)


A = 1 << 20      # fake, 16-byte aligned addresses: never dereferenced
B = 1 << 30
C = 1 << 34
D = 1 << 38


def fused(L, X=A, dY=B, W=C, m=(D, None), v=(D + (1 << 36), None), bt=64, d_in=256, d_out=128,
          lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.01, step=1, fmt=0):
    return L.forge_wgrad_adamw(X, dY, W, F.ForgeMoment(*m), F.ForgeMoment(*v), bt, d_in, d_out,
                               lr, b1, b2, eps, wd, step, fmt, None)


def test_fused_argument_errors(L):
    assert fused(L, X=None) == 1                     # FORGE_ERR_NULL
    assert fused(L, W=None) == 1
    assert fused(L, m=(None, None)) == 1
    assert fused(L, fmt=2) == 1                      # int8 without scales
    assert fused(L, X=A + 8) == 2                    # FORGE_ERR_ALIGN
    assert fused(L, d_in=260) == 3                   # FORGE_ERR_SHAPE
    assert fused(L, d_out=0) == 3
    assert fused(L, bt=-1) == 3
    assert fused(L, d_in=264, fmt=2, m=(D, A), v=(D + (1 << 36), B)) == 3   # int8 needs 128 | d_in
    assert fused(L, fmt=7) == 4                      # FORGE_ERR_FORMAT
    assert fused(L, step=0) == 5                     # FORGE_ERR_HYPER
    assert fused(L, b1=1.0) == 5
    assert fused(L, b2=-0.1) == 5
    assert fused(L, lr=float("nan")) == 5
    assert fused(L, eps=-1.0) == 5
    assert fused(L, eps=1e-40) == 5          # eps: 0 or a normal number ...
    assert fused(L, eps=2.0 ** 65) == 5      # ... at most 2^64
    assert fused(L, X=C) == 6                        # FORGE_ERR_ALIAS: X is W
    assert fused(L, dY=D + 64) == 6                  # dY inside m
    assert fused(L, v=(D, None)) == 6                # m and v the same buffer


def test_fp8_argument_errors(L):
    # fp8 moments: the scale records are required and 16-byte aligned, rows
    # of codes must be 16-byte aligned (d_in % 16), and the record of one
    # moment must not overlap the other's
    E = (1 << 40)
    fp8 = dict(fmt=3, m=(D, E), v=(D + (1 << 36), E + 16))
    assert fused(L, **fp8) in (0, 7, 10)             # valid: stops at the device check
    assert fused(L, fmt=3) == 1                      # no scale records
    assert fused(L, **dict(fp8, m=(D, E + 4))) == 2  # record not 16-byte aligned
    assert fused(L, **dict(fp8, d_in=264)) == 3      # 264 % 16 != 0
    assert fused(L, **dict(fp8, v=(D + (1 << 36), E))) == 6   # both moments share one record
    assert fused(L, **dict(fp8, X=E)) == 6           # X over a record
    assert L.forge_wgrad_adamw_sr(A, B, C, F.ForgeMoment(D, E), F.ForgeMoment(D + (1 << 36), E + 16),
                                  64, 256, 128, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 3, 1, None) == 4
    assert L.forge_fp8_roll_scales(None, 2, 1.0, None) == 1
    assert L.forge_fp8_roll_scales(E + 4, 2, 1.0, None) == 2
    assert L.forge_fp8_roll_scales(E, -1, 1.0, None) == 3
    assert L.forge_fp8_roll_scales(E, 2, 0.5, None) == 5
    assert L.forge_fp8_roll_scales(E, 2, float("inf"), None) == 5
    assert L.forge_fp8_roll_scales(None, 0, 1.0, None) == 0   # nothing to roll


def test_fused_valid_arguments_reach_the_device_check(L):
    # valid arguments get past validation and stop at the device query, which
    # fails on a machine without a GPU (FORGE_ERR_CUDA) or with another GPU
    st = fused(L)
    assert st in (7, 10) or st == 0


def test_wgrad_and_adamw_argument_errors(L):
    assert L.forge_wgrad(A, B, None, 0, 64, 256, 128, None) == 1
    assert L.forge_wgrad(A, B, C, 5, 64, 256, 128, None) == 4
    assert L.forge_wgrad(A, B, A, 0, 64, 256, 128, None) == 6
    assert L.forge_wgrad(A, B, C + 4, 0, 64, 256, 128, None) == 2
    m, v = F.ForgeMoment(D, None), F.ForgeMoment(D + (1 << 36), None)
    assert L.forge_adamw(C, 0, C, m, v, 256, 128, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 0, None) == 6
    assert L.forge_adamw(A, 3, C, m, v, 256, 128, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 0, None) == 4
    assert L.forge_adamw(A, 0, C, m, v, 256, 128, 1e-3, 0.9, 0.999, 1e-8, 0.01, 0, 0, None) == 5


def test_dgrad_and_linear_backward_argument_errors(L):
    # codes: 1 NULL, 2 ALIGN, 3 SHAPE, 5 HYPER, 6 ALIAS
    assert L.forge_dgrad(B, C, None, 64, 256, 128, None) == 1
    assert L.forge_dgrad(B, C + 4, A, 64, 256, 128, None) == 2
    assert L.forge_dgrad(B, C, A, 64, 250, 128, None) == 3
    assert L.forge_dgrad(B, C, C, 64, 256, 128, None) == 6          # dX over W
    assert L.forge_dgrad(None, None, None, 0, 256, 128, None) == 0  # no tokens: nothing to do
    # the variant without allocation checks its arguments the same way
    assert L.forge_dgrad_noalloc(B, C, None, 64, 256, 128, None) == 1
    assert L.forge_dgrad_noalloc(B, C + 4, A, 64, 256, 128, None) == 2
    assert L.forge_dgrad_noalloc(B, C, A, 64, 250, 128, None) == 3
    assert L.forge_dgrad_noalloc(B, C, C, 64, 256, 128, None) == 6
    assert L.forge_dgrad_noalloc(None, None, None, 0, 256, 128, None) == 0
    m, v = F.ForgeMoment(D, None), F.ForgeMoment(D + (1 << 36), None)
    args = (256, 128, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert L.forge_linear_backward(A, B, C, None, m, v, 64, *args, 1, 0, None) == 1
    assert L.forge_linear_backward(A, B, C, A, m, v, 64, *args, 1, 0, None) == 6   # dX over X
    assert L.forge_linear_backward(A, B, C, C, m, v, 64, *args, 1, 0, None) == 6   # dX over W
    assert L.forge_linear_backward(A, B, C, G + 4, m, v, 64, *args, 1, 0, None) == 2
    # a bad step is caught before the input gradient is enqueued
    assert L.forge_linear_backward(A, B, C, G, m, v, 64, *args, 0, 0, None) == 5


def opt_call(L, opt=1, s1=D, s2=None, X=A, dY=B, W=C, bt=64, d_in=256, d_out=128, step=1,
             fmt=0, **hk):
    h = dict(lr=1e-3, weight_decay=0.01, beta1=0.9, beta2=0.999, eps=1e-8, momentum=0.9,
             alpha=0.99, momentum_decay=4e-3)
    h.update(hk)
    hp = F.ForgeOptHyper(*[h[k] for k in ("lr", "weight_decay", "beta1", "beta2", "eps",
                                          "momentum", "alpha", "momentum_decay")])
    return L.forge_wgrad_opt(X, dY, W, F.ForgeMoment(s1, None), F.ForgeMoment(s2, None), bt,
                             d_in, d_out, opt, ctypes.byref(hp), step, fmt, None)


def test_wgrad_opt_argument_errors(L):
    # codes: 1 NULL, 2 ALIGN, 3 SHAPE, 4 FORMAT, 5 HYPER, 6 ALIAS; 10 = valid
    # arguments that reached the device query (no GPU here)
    assert opt_call(L) == 10
    assert opt_call(L, opt=0, s1=None) == 10                 # SGD keeps no state
    assert opt_call(L, opt=5, s2=D + (1 << 36)) == 10        # NAdam: two states
    assert opt_call(L, s1=None) == 1                         # momentum buffer missing
    assert opt_call(L, opt=6) == 1                           # RAdam needs s2 too
    assert opt_call(L, W=None) == 1
    assert opt_call(L, s1=D + 4) == 2
    assert opt_call(L, d_in=250) == 3
    assert opt_call(L, fmt=2) == 4                           # no int8 state here
    assert opt_call(L, opt=7) == 5
    assert opt_call(L, step=0) == 5
    assert opt_call(L, opt=4, beta1=1.0) == 5                # Lion betas in [0, 1)
    assert opt_call(L, opt=2, eps=-1.0) == 5                 # Adagrad eps >= 0
    assert opt_call(L, opt=3, eps=1e-40) == 5                # RMSprop eps subnormal
    assert opt_call(L, opt=3, alpha=1.0) == 5                # RMSprop alpha < 1
    assert opt_call(L, momentum=float("nan")) == 5
    assert opt_call(L, lr=float("inf")) == 5
    assert opt_call(L, s1=C) == 6                            # state over W
    assert opt_call(L, X=C) == 6                             # input over W
    assert opt_call(L, opt=5, s1=D, s2=D) == 6               # the two states overlap
    assert L.forge_wgrad_opt(A, B, C, F.ForgeMoment(D, None), F.ForgeMoment(None, None), 64,
                             256, 128, 1, None, 1, 0, None) == 5    # no hyperparameters


def test_wgrad_adamw_sr_argument_errors(L):
    m, v = F.ForgeMoment(D, None), F.ForgeMoment(D + (1 << 36), None)
    args = (64, 256, 128, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    sr = L.forge_wgrad_adamw_sr
    assert sr(A, B, C, m, v, *args, 1, 0, 7, None) == 10          # valid: reached the device
    assert sr(A, B, C, m, v, *args, 1, 2, 7, None) in (1, 4)      # int8: no scales / format
    ms, vs = F.ForgeMoment(D, G), F.ForgeMoment(D + (1 << 36), G + (1 << 20))
    assert sr(A, B, C, ms, vs, *args, 1, 2, 7, None) == 4         # int8 moments: not here
    assert sr(A, B, C, m, v, *args, 0, 0, 7, None) == 5           # step 0
    assert sr(A, B, C, m, v, *args, 1 << 31, 0, 7, None) == 5     # step beyond 32 bits
    assert sr(A, B, None, m, v, *args, 1, 0, 7, None) == 1
    assert sr(A, B, A, m, v, *args, 1, 0, 7, None) == 6           # W over X


def test_wgrad_accumulate_argument_errors(L):
    # codes: 1 NULL, 2 ALIGN, 3 SHAPE, 5 HYPER, 6 ALIAS; 10 = reached the device query
    acc = L.forge_wgrad_accumulate
    assert acc(A, B, C, 1.0, 64, 256, 128, None) == 10
    assert acc(A, B, None, 1.0, 64, 256, 128, None) == 1
    assert acc(None, B, C, 1.0, 64, 256, 128, None) == 1
    assert acc(None, None, C, 0.9, 0, 256, 128, None) == 10    # no tokens: X, dY unused
    assert acc(A, B, C + 8, 1.0, 64, 256, 128, None) == 2
    assert acc(A, B, C, 1.0, 64, 256, 124, None) == 3
    assert acc(A, B, C, float("nan"), 64, 256, 128, None) == 5
    assert acc(A, B, C, float("inf"), 64, 256, 128, None) == 5
    assert acc(A, B, A, 1.0, 64, 256, 128, None) == 6          # B over X


def grouped(L, layers, bt=64, step=1, fmt=0):
    arr = (F.ForgeLinear * max(1, len(layers)))(*layers)
    return L.forge_wgrad_adamw_grouped(arr, len(layers), bt, 1e-3, 0.9, 0.999, 1e-8, 0.01, step,
                                       fmt, None)


def lin(X, dY, W, m, v, d_in=256, d_out=128, ms=None, vs=None):
    return F.ForgeLinear(X, dY, W, F.ForgeMoment(m, ms), F.ForgeMoment(v, vs), d_in, d_out)


G = 1 << 40


def test_grouped_argument_errors(L):
    assert L.forge_wgrad_adamw_grouped(None, 1, 64, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 0, None) == 1
    a = lin(A, B, C, D, D + G)
    b = lin(A, B, C + 2 * G, D + 3 * G, D + 4 * G)     # shares X and dY with a: allowed
    assert grouped(L, []) == 3                          # n = 0
    assert grouped(L, [a] * 9) == 3                     # n > FORGE_MAX_GROUP
    assert grouped(L, [a, lin(A, B, C, D + 5 * G, D + 6 * G)]) == 6   # two layers share W
    assert grouped(L, [a, lin(C, B, C + 2 * G, D + 3 * G, D + 4 * G)]) == 6  # X of one is W of other
    assert grouped(L, [a, lin(A, B, C + 2 * G, D + 3 * G, D + 4 * G, d_in=260)]) == 3
    assert grouped(L, [a, b], step=0) == 5
    assert grouped(L, [a, b]) in (0, 7, 10)            # valid: stops at the device query here


# ---------------------------------------------------------------------------
# The Python binding checks every tensor's shape, dtype and device before it
# calls into the library (the kernels size their tensor maps from the shapes
# they are given, so a short buffer would be read or written past its end).
# The checks run on the host: CPU tensors reach the shape and dtype checks,
# and a tensor of the right shape on the CPU is then refused as not a CUDA
# tensor.
# ---------------------------------------------------------------------------

def _t(shape, dt=torch.bfloat16):
    return torch.zeros(shape, dtype=dt)


HY = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)


def test_binding_rejects_mismatched_shapes_and_dtypes():
    bt, d_in, d_out = 64, 256, 128
    X, dY = _t((bt, d_in)), _t((bt, d_out))
    W = _t((d_out, d_in))
    m, v = _t((d_out, d_in), torch.float32), _t((d_out, d_in), torch.float32)
    with pytest.raises(ValueError, match="W has shape"):
        F.wgrad_adamw(X, dY, _t((d_out, d_in - 8)), m, v, **HY)
    with pytest.raises(ValueError, match="dY has shape"):
        F.wgrad_adamw(X, _t((bt - 1, d_out)), W, m, v, **HY)
    with pytest.raises(ValueError, match="m has shape"):
        F.wgrad_adamw(X, dY, W, _t((d_out, 8), torch.float32), v, **HY)
    with pytest.raises(TypeError, match="v has dtype"):
        F.wgrad_adamw(X, dY, W, m, _t((d_out, d_in)), **HY)
    with pytest.raises(TypeError, match="X has dtype"):
        F.wgrad_adamw(_t((bt, d_in), torch.float32), dY, W, m, v, **HY)
    with pytest.raises(ValueError, match="m_scale is required"):
        F.wgrad_adamw(X, dY, W, _t((d_out, d_in), torch.int8), _t((d_out, d_in), torch.int8),
                      **HY)
    with pytest.raises(ValueError, match="v_scale has shape"):
        F.wgrad_adamw(X, dY, W, _t((d_out, d_in), torch.int8), _t((d_out, d_in), torch.int8),
                      m_scale=_t((d_out, 2), torch.float32), v_scale=_t((d_out, 1), torch.float32),
                      **HY)
    with pytest.raises(ValueError, match="dX has shape"):
        F.dgrad(dY, W, _t((bt, d_in + 8)))
    with pytest.raises(ValueError, match="W has shape"):
        F.dgrad(dY, _t((d_out + 8, d_in)), _t((bt, d_in)))
    with pytest.raises(ValueError, match="dX has shape"):
        F.dgrad_noalloc(dY, W, _t((bt - 1, d_in)))
    with pytest.raises(ValueError, match="dX has shape"):
        F.linear_backward(X, dY, W, _t((bt, d_out)), m, v, **HY)
    with pytest.raises(ValueError, match="dW has shape"):
        F.wgrad(X, dY, _t((d_in, d_out), torch.float32))
    with pytest.raises(TypeError, match="B has dtype"):
        F.wgrad_accumulate(X, dY, _t((d_out, d_in)), 1.0)
    with pytest.raises(ValueError, match="s2 is required"):
        F.wgrad_opt(X, dY, W, F.OPT_NADAM, m, None, lr=1e-3, weight_decay=0.0, step=1)
    with pytest.raises(ValueError, match="s1 has shape"):
        F.wgrad_opt(X, dY, W, F.OPT_LION, _t((d_out, 8), torch.float32), lr=1e-3,
                    weight_decay=0.0, step=1)
    with pytest.raises(ValueError, match="dW has shape"):
        F.adamw(_t((d_out, 8), torch.float32), W, m, v, **HY)
    with pytest.raises(TypeError, match="m has dtype"):
        F.wgrad_adamw_sr(X, dY, W, _t((d_out, d_in), torch.int8), _t((d_out, d_in), torch.int8),
                         seed=1, **HY)
    with pytest.raises(ValueError, match="W has shape"):
        F.wgrad_adamw_grouped([dict(X=X, dY=dY, W=_t((d_in, d_out)), m=m, v=v)], **HY)


def test_binding_refuses_host_tensors():
    bt, d_in, d_out = 64, 256, 128
    X, dY, W = _t((bt, d_in)), _t((bt, d_out)), _t((d_out, d_in))
    m, v = _t((d_out, d_in), torch.float32), _t((d_out, d_in), torch.float32)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        F.wgrad_adamw(X, dY, W, m, v, **HY)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        F.dgrad(dY, W, _t((bt, d_in)))


def test_tuning_round_trip_without_gpu(L, tune):
    tune(profile="deep", cg=2, bn=256, group_m=8, poll_store=0, splits=3, l2_hints=1,
         state_prefetch=4)
    t = F.get_tuning()
    assert t == dict(profile="deep", cg=2, bn=256, group_m=8, poll_store=0, splits=3,
                     l2_hints=1, state_prefetch=4)
    # the override reaches the host's configuration choice
    assert "profile=deep" in F.describe_config(512, 4096, 4096, F.MOM_FP32)
    assert "group_m=8" in F.describe_config(512, 4096, 4096, F.MOM_FP32)
    with F.tuning(profile="stream"):
        assert "profile=stream" in F.describe_config(4096, 4096, 4096, F.MOM_FP32)
    assert F.get_tuning()["profile"] == "deep"
    F.set_tuning()
    assert F.get_tuning() == dict(profile="auto", cg=0, bn=0, group_m=0, poll_store=-1,
                                  splits=0, l2_hints=-1, state_prefetch=-1)
    with pytest.raises(ValueError):
        F.set_tuning(profile="fast")


def test_grouped_calls_argument_errors(L):
    # codes: 1 NULL, 2 ALIGN, 3 SHAPE, 4 FORMAT, 5 HYPER, 6 ALIAS
    lin = F.ForgeLinear(A, B, C, F.ForgeMoment(D, None), F.ForgeMoment(D + (1 << 36), None),
                        256, 128)
    arr = (F.ForgeLinear * 2)(lin, lin)
    h = F.ForgeOptHyper(1e-3, 0.0, 0.9, 0.999, 1e-8, 0.9, 0.99, 4e-3)
    assert L.forge_wgrad_opt_grouped(None, 1, 64, 1, ctypes.byref(h), 1, 0, None) == 1
    assert L.forge_wgrad_opt_grouped(arr, 0, 64, 1, ctypes.byref(h), 1, 0, None) == 3
    assert L.forge_wgrad_opt_grouped(arr, 1, 64, 1, ctypes.byref(h), 0, 0, None) == 5
    assert L.forge_wgrad_opt_grouped(arr, 1, 64, 1, ctypes.byref(h), 1, 2, None) == 4
    assert L.forge_wgrad_opt_grouped(arr, 2, 64, 1, ctypes.byref(h), 1, 0, None) == 6  # same W twice
    seeds = (ctypes.c_uint64 * 2)(1, 2)
    assert L.forge_wgrad_adamw_sr_grouped(arr, None, 1, 64, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 0,
                                          None) == 1
    assert L.forge_wgrad_adamw_sr_grouped(arr, seeds, 2, 64, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 0,
                                          None) == 6
    acc = (F.ForgeAccumItem * 2)(F.ForgeAccumItem(A, B, C, 256, 128),
                                 F.ForgeAccumItem(A, B, C + 64, 256, 128))
    assert L.forge_wgrad_accumulate_grouped(acc, 2, 64, 1.0, None) == 6    # B's overlap
    assert L.forge_wgrad_accumulate_grouped(acc, 1, 64, float("inf"), None) == 5
    dg = (F.ForgeDgradItem * 2)(F.ForgeDgradItem(B, C, A, 256, 128),
                                F.ForgeDgradItem(B, C, A, 256, 128))
    assert L.forge_dgrad_grouped(dg, 2, 64, None, 0, None) == 6             # same dX twice
    assert L.forge_dgrad_grouped(dg, 9, 64, None, 0, None) == 3
    assert L.forge_dgrad_grouped(dg, 1, 64, A + 4, 1024, None) == 2        # workspace alignment
    assert L.forge_dgrad_workspace_bytes(dg, 1, 0) == 0
    dx = (ctypes.c_void_p * 2)(A, A)
    assert L.forge_linear_backward_grouped(arr, None, 1, 64, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 0,
                                           None, 0, None) == 1
    assert L.forge_linear_backward_grouped(arr, dx, 1, 64, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 0,
                                           None, 0, None) == 6             # dX over X


def final_step(L, X=A, dY=B, W=C, m=(D, None), v=(D + (1 << 36), None), Bacc=(1 << 40),
               bt=64, d_in=256, d_out=128, eps=1e-8, fmt=0):
    return L.forge_wgrad_adamw_acc(X, dY, W, F.ForgeMoment(*m), F.ForgeMoment(*v), Bacc, bt,
                                   d_in, d_out, 1e-3, 0.9, 0.999, eps, 0.01, 1, fmt, None)


def test_final_micro_batch_step_argument_errors(L):
    # codes: 1 NULL, 2 ALIGN, 3 SHAPE, 4 FORMAT, 5 HYPER, 6 ALIAS; 10 = valid
    # arguments that reached the device query (no GPU here)
    assert final_step(L) == 10
    assert final_step(L, fmt=1) == 10                     # bf16 moments
    assert final_step(L, Bacc=None) == 1
    assert final_step(L, Bacc=(1 << 40) + 4) == 2
    assert final_step(L, d_in=260) == 3
    assert final_step(L, fmt=2, m=(D, A), v=(D + (1 << 36), B)) == 4   # int8: not this step
    assert final_step(L, fmt=3) == 4
    assert final_step(L, eps=1e-40) == 5
    assert final_step(L, Bacc=C + 64) == 6                # the accumulator inside W
    assert final_step(L, Bacc=D + 64) == 6                # ... inside m
    assert final_step(L, Bacc=B) == 10                    # over dY: both are read only
