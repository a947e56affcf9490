"""GPU parity of forge_wgrad_opt (SGD, SGD with momentum, Adagrad, RMSprop,
Lion, NAdam, RAdam fused into the weight-gradient epilogue) against the
regime-1 oracle, under the bars of ``tests/parity.py`` (``check_opt_step``).
Every compared step starts from the oracle's own rounded state."""
import numpy as np
import pytest
import torch

import oracle as O
from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import bf16_bits, bits_to_bf16, make_step_inputs

from .gpu_util import DEV, mom_from_dev, mom_to_dev, require_gpu
from .parity import check_opt_step

pytestmark = pytest.mark.gpu

# the appendix table's settings where it gives them (betas, eps), with a
# larger learning rate so that the weight visibly moves in one step
H = O.OptHyper(lr=1e-3, weight_decay=0.01, beta1=0.9, beta2=0.999, eps=1e-8, momentum=0.9,
               alpha=0.99, momentum_decay=4e-3)
LION = O.OptHyper(lr=1e-4, weight_decay=1.0, beta1=0.9, beta2=0.99)


def hyper_for(opt):
    return LION if opt == O.OPT_LION else H


def kwargs(h: O.OptHyper):
    return dict(lr=h.lr, weight_decay=h.weight_decay, beta1=h.beta1, beta2=h.beta2, eps=h.eps,
                momentum=h.momentum, alpha=h.alpha, momentum_decay=h.momentum_decay)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def initial_states(opt, fmt, d_out, d_in, seed):
    """Warm, plausible states: signed momenta, positive second-moment sums."""
    rng = np.random.default_rng(seed)
    n = O.OPT_STATES[opt]
    out = []
    for i in range(n):
        if opt == O.OPT_ADAGRAD:
            x = rng.uniform(1e-8, 1e-6, (d_out, d_in))
        elif opt == O.OPT_RMSPROP or i == 1:
            x = rng.uniform(1e-10, 1e-8, (d_out, d_in))
        else:
            x = rng.normal(0, 1e-4, (d_out, d_in))
        out.append(O.encode_moment(fmt, x, False))
    return out + [None] * (2 - n)


def run_gpu(opt, fmt, x, dy, w_bits, states, h, t):
    W = bits_to_bf16(w_bits).to(DEV)
    dev = [mom_to_dev(s)[0] if s is not None else None for s in states]
    F.wgrad_opt(x.to(DEV), dy.to(DEV), W, opt, dev[0], dev[1], step=t, **kwargs(h))
    assert F.device_error() == 0
    return bf16_bits(W.cpu()), [mom_from_dev(fmt, s, None) if s is not None else None
                                for s in dev]


def compare(opt, fmt, bt, d_in, d_out, t, seed, label=""):
    s = make_step_inputs(200 + seed, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True,
                         spike_frac=0.01)
    w_bits = bf16_bits(s.w)
    states = initial_states(opt, fmt, d_out, d_in, seed)
    h = hyper_for(opt)
    gw, gs = run_gpu(opt, fmt, s.x, s.dy, w_bits, states, h, t)
    xb, db = bf16_bits(s.x), bf16_bits(s.dy)
    ref = dict(G=O.wgrad(xb, db), S=O.wgrad_abs(xb, db), W_bits=w_bits, states=states)
    rep = check_opt_step(gw, gs, ref, opt, h, t, fmt, bt, label=label)
    print(label, {k: str(v) for k, v in rep.items()})


OPTS = list(range(7))
IDS = [O.OPT_NAMES[o] for o in OPTS]


@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("opt", OPTS, ids=IDS)
@pytest.mark.parametrize("bt,d_in,d_out,t", [(200, 264, 136, 3), (1000, 384, 264, 7)],
                         ids=["cta", "pair"])
def test_opt_against_oracle(opt, fmt, bt, d_in, d_out, t):
    # t = 3 and t = 7 put RAdam on both sides of its rectification threshold
    compare(opt, fmt, bt, d_in, d_out, t, seed=opt + 10 * fmt, label=f"{O.OPT_NAMES[opt]}")


@pytest.fixture(params=[("stream", "128", "1"), ("stream", "256", "1"), ("balanced", "256", "1"),
                        ("deep", "256", "2"), ("mma", "256", "2")],
                ids=lambda p: f"{p[0]}-bn{p[1]}-cta{p[2]}")
def forced(request, tune):
    tune(profile=request.param[0], bn=int(request.param[1]), cg=int(request.param[2]))
    return request.param


@pytest.mark.parametrize("opt", [O.OPT_SGD, O.OPT_LION, O.OPT_NADAM], ids=["sgd", "lion", "nadam"])
def test_opt_under_every_slot_layout(opt, forced):
    # none, one and two states in full and half-tile state slots
    compare(opt, O.FMT_FP32, 130, 264, 392, 5, seed=50 + opt, label=str(forced))


@pytest.mark.parametrize("opt", [O.OPT_ADAGRAD, O.OPT_LION, O.OPT_RADAM],
                         ids=["adagrad", "lion", "radam"])
def test_opt_without_tokens(opt):
    # G = 0: decay and the state-driven part of the update only
    compare(opt, O.FMT_FP32, 0, 256, 128, 4, seed=70 + opt, label="bt=0")


@pytest.mark.parametrize("opt", [O.OPT_LION, O.OPT_RADAM], ids=["lion", "radam"])
def test_opt_gate_projection_sampled_rows(opt):
    # Llama-3.1-8B gate projection (14336 x 4096) at 512 tokens; the oracle
    # computes sampled weight rows
    bt, d_out, d_in, t = 512, 14336, 4096, 12
    s = make_step_inputs(300 + opt, 4, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True)
    w_bits = bf16_bits(s.w)
    states = initial_states(opt, O.FMT_FP32, d_out, d_in, 300 + opt)
    h = hyper_for(opt)
    gw, gs = run_gpu(opt, O.FMT_FP32, s.x, s.dy, w_bits, states, h, t)
    rows = np.array(sorted({0, 127, 128, 255, 256, 7000, 8191, 14335}))
    xb, db = bf16_bits(s.x), bf16_bits(s.dy)
    ref = dict(G=O.wgrad(xb, db, rows), S=O.wgrad_abs(xb, db, rows), W_bits=w_bits[rows],
               states=[st.rows(rows) if st is not None else None for st in states])
    check_opt_step(gw[rows], [g.rows(rows) if g is not None else None for g in gs], ref, opt, h,
                   t, O.FMT_FP32, bt, label="gate")


def test_opt_is_deterministic_and_leaves_unused_states_alone():
    # SGD keeps no state: buffers passed for s1, s2 are neither read nor written
    s = make_step_inputs(400, 0, 1, 256, 512, 256, dy_std=1e-3, with_w=True)
    X, dY = s.x.to(DEV), s.dy.to(DEV)
    outs = []
    for _ in range(2):
        W = s.w.to(DEV)
        guard = torch.full((256, 512), 7.0, device=DEV)
        F.wgrad_opt(X, dY, W, O.OPT_SGD, guard, guard.clone(), step=1, **kwargs(H))
        assert F.device_error() == 0
        assert torch.all(guard == 7.0)
        outs.append(W.view(torch.int16).clone())
    assert torch.equal(outs[0], outs[1])
