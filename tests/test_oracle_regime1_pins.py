"""Pins of the regime-1 optimizer oracle (``oracle/regime1.py``) to things
other than itself:

* SGD, SGD with momentum, Adagrad, RMSprop, NAdam and RAdam: PyTorch's own
  ``torch.optim`` implementations in float64 (independent code), over twelve
  steps so that RAdam passes its rectification threshold (step 6 at
  beta2 = 0.999) and NAdam's momentum schedule moves;
* Lion (not in torch.optim): closed forms of the sign update;
* special cases: zero gradient and state, the first momentum step, row subsets
  and the one rounding per stored value.
"""
import numpy as np
import pytest
import torch

import oracle as O

H = O.OptHyper(lr=1e-3, weight_decay=0.01, beta1=0.9, beta2=0.999, eps=1e-8, momentum=0.9,
               alpha=0.99, momentum_decay=4e-3)
SHAPE = (6, 10)


def _torch_opt(opt, p, h):
    if opt == O.OPT_SGD:
        return torch.optim.SGD([p], lr=h["lr"], weight_decay=h["weight_decay"]), []
    if opt == O.OPT_SGD_MOMENTUM:
        return (torch.optim.SGD([p], lr=h["lr"], momentum=h["momentum"],
                                weight_decay=h["weight_decay"]), ["momentum_buffer"])
    if opt == O.OPT_ADAGRAD:
        return (torch.optim.Adagrad([p], lr=h["lr"], eps=h["eps"],
                                    weight_decay=h["weight_decay"]), ["sum"])
    if opt == O.OPT_RMSPROP:
        return (torch.optim.RMSprop([p], lr=h["lr"], alpha=h["alpha"], eps=h["eps"],
                                    weight_decay=h["weight_decay"]), ["square_avg"])
    if opt == O.OPT_NADAM:
        return (torch.optim.NAdam([p], lr=h["lr"], betas=(h["beta1"], h["beta2"]), eps=h["eps"],
                                  weight_decay=h["weight_decay"],
                                  momentum_decay=h["momentum_decay"]), ["exp_avg", "exp_avg_sq"])
    if opt == O.OPT_RADAM:
        return (torch.optim.RAdam([p], lr=h["lr"], betas=(h["beta1"], h["beta2"]), eps=h["eps"],
                                  weight_decay=h["weight_decay"]), ["exp_avg", "exp_avg_sq"])
    raise ValueError(opt)


TORCH_OPTS = [O.OPT_SGD, O.OPT_SGD_MOMENTUM, O.OPT_ADAGRAD, O.OPT_RMSPROP, O.OPT_NADAM,
              O.OPT_RADAM]


@pytest.fixture
def f64_default():
    # torch.optim keeps per-step scalars (NAdam's running mu product, the step
    # count) in the default dtype; float64 makes the reference fp64 throughout
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


@pytest.mark.parametrize("opt", TORCH_OPTS, ids=[O.OPT_NAMES[o] for o in TORCH_OPTS])
def test_matches_torch_optim_f64(opt, f64_default):
    rng = np.random.default_rng(100 + opt)
    h = H.as_f64()
    W = rng.normal(0, 0.02, SHAPE)
    p = torch.tensor(W.copy(), dtype=torch.float64, requires_grad=True)
    topt, names = _torch_opt(opt, p, h)
    n = O.OPT_STATES[opt]
    assert n == len(names)
    s1 = np.zeros(SHAPE) if n >= 1 else None
    s2 = np.zeros(SHAPE) if n >= 2 else None
    for t in range(1, 13):
        G = rng.normal(0, 1e-3, SHAPE)
        p.grad = torch.tensor(G, dtype=torch.float64)
        topt.step()
        W, s1, s2 = O.opt_f64(opt, G, W, s1, s2, H, t)
        np.testing.assert_allclose(W, p.detach().numpy(), rtol=1e-12, atol=1e-18,
                                   err_msg=f"W at t={t}")
        st = topt.state[p]
        for name, mine in zip(names, (s1, s2)):
            np.testing.assert_allclose(mine, st[name].numpy(), rtol=1e-12, atol=1e-24,
                                       err_msg=f"{name} at t={t}")


def test_radam_rectification_starts_at_step_six():
    h = H.as_f64()
    assert [O.radam_scalars(h, t)[0] for t in range(1, 8)] == [False] * 5 + [True] * 2


def test_lion_closed_forms():
    h = H.as_f64()
    lr, wd, b1, b2 = h["lr"], h["weight_decay"], h["beta1"], h["beta2"]
    rng = np.random.default_rng(7)
    W = rng.normal(0, 0.02, SHAPE)
    G = rng.normal(0, 1e-3, SHAPE)
    G[0, :3] = 0.0
    # step 1 from m = 0: the direction is sign(G); sign(0) = 0 leaves pure decay
    W1, m1, s2 = O.opt_f64(O.OPT_LION, G, W, np.zeros(SHAPE), None, H, 1)
    assert s2 is None
    np.testing.assert_array_equal(W1, (1 - lr * wd) * W - lr * np.sign(G))
    np.testing.assert_array_equal(m1, (1 - b2) * G)
    assert np.all(W1[0, :3] == (1 - lr * wd) * W[0, :3])
    # the direction mixes the old state with beta1, the new state with beta2:
    # a large positive m against a small negative G still moves W down
    m = np.full(SHAPE, 1e-2)
    G2 = np.full(SHAPE, -1e-3)
    W2, m2, _ = O.opt_f64(O.OPT_LION, G2, W, m, None, H, 5)
    np.testing.assert_array_equal(W2, (1 - lr * wd) * W - lr)
    np.testing.assert_array_equal(m2, b2 * m + (1 - b2) * G2)
    # and a G that outweighs beta1 m turns it around: c = 0.9e-2 - 0.1 * 0.2 < 0
    G3 = np.full(SHAPE, -0.2)
    W3, _, _ = O.opt_f64(O.OPT_LION, G3, W, m, None, H, 5)
    np.testing.assert_array_equal(W3, (1 - lr * wd) * W + lr)


def test_first_momentum_step_is_sgd_and_zero_gradient_cases():
    rng = np.random.default_rng(3)
    W = rng.normal(0, 0.02, SHAPE)
    G = rng.normal(0, 1e-3, SHAPE)
    a, _, _ = O.opt_f64(O.OPT_SGD, G, W, None, None, H, 1)
    b, buf, _ = O.opt_f64(O.OPT_SGD_MOMENTUM, G, W, np.zeros(SHAPE), None, H, 1)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(buf, G + H.as_f64()["weight_decay"] * W)
    # without decay and gradient nothing moves, whatever the optimizer
    h0 = O.OptHyper(weight_decay=0.0)
    Z = np.zeros(SHAPE)
    for opt in TORCH_OPTS:
        n = O.OPT_STATES[opt]
        W1, s1, s2 = O.opt_f64(opt, Z, W, Z if n >= 1 else None, Z if n >= 2 else None, h0, 3)
        np.testing.assert_array_equal(W1, W)


@pytest.mark.parametrize("opt", range(7), ids=[O.OPT_NAMES[o] for o in range(7)])
@pytest.mark.parametrize("fmt", [O.FMT_FP32, O.FMT_BF16])
def test_opt_step_rounds_once_and_rows_are_exact_subsets(opt, fmt):
    from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs
    s = make_step_inputs(40 + opt, 0, 1, 32, 128, 24, dy_std=1e-3, with_w=True)
    xb, dyb, wb = bf16_bits(s.x), bf16_bits(s.dy), bf16_bits(s.w)
    rng = np.random.default_rng(opt)
    n = O.OPT_STATES[opt]
    st = [O.encode_moment(fmt, np.abs(rng.normal(0, 1e-4, (24, 128))), False) for _ in range(n)]
    st += [None] * (2 - n)
    W1, a1, a2, (G, Wf, f1, f2) = O.opt_step(opt, xb, dyb, wb, st[0], st[1], H, 4,
                                             return_f64=True)
    np.testing.assert_array_equal(W1, O.f64_to_bf16(Wf))
    for got, f in ((a1, f1), (a2, f2)):
        if f is not None:
            np.testing.assert_array_equal(got.data, O.encode_moment(fmt, f, False).data)
    rows = np.array([0, 5, 23])
    Wr, r1, r2 = O.opt_step(opt, xb, dyb, wb[rows], st[0].rows(rows) if n >= 1 else None,
                            st[1].rows(rows) if n >= 2 else None, H, 4, rows=rows)
    np.testing.assert_array_equal(Wr, W1[rows])
    if n >= 1:
        np.testing.assert_array_equal(r1.data, a1.data[rows])
    if n >= 2:
        np.testing.assert_array_equal(r2.data, a2.data[rows])
