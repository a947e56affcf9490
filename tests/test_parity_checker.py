"""The bf16 weight bar of the GPU parity tests (tests/parity.py, check_w),
checked on the CPU: it accepts the oracle's own rounded result, rejects a
well-conditioned entry 3 ulp away, and holds an entry whose update cancels
most of W to the fp32 bound of the arithmetic."""
import numpy as np
import pytest

import oracle as O

from .parity import check_w


def _case():
    rng = np.random.default_rng(0)
    W0 = O.bf16_to_f64(O.f64_to_bf16(rng.normal(0, 0.02, 20000)))
    Wn = W0 * (1 - 1e-5) - 1e-3 * np.sign(rng.normal(size=W0.size))
    # entry 0: the update cancels W almost exactly (W' ~ 1e-9)
    W0[0] = O.bf16_to_f64(O.f64_to_bf16(np.array([1e-3])))[0]
    Wn[0] = W0[0] * (1 - 1e-5) - (W0[0] * (1 - 1e-5) - 1.3e-9)
    return W0, [Wn - 1e-12, Wn, Wn + 1e-12]


def test_accepts_the_oracles_rounding():
    W0, outs = _case()
    rep = check_w(O.f64_to_bf16(outs[1]), outs, W0)
    assert rep.cancelling >= 1 and rep.violations == 0


def test_rejects_three_ulp_on_a_well_conditioned_entry():
    W0, outs = _case()
    g = O.f64_to_bf16(outs[1]).astype(np.int64)
    g[5] += 3 if g[5] < 0x8000 else -3        # three steps away from the value
    with pytest.raises(AssertionError):
        check_w(g.astype(np.uint16), outs, W0)


def test_cancelling_entry_held_to_the_fp32_bound():
    W0, outs = _case()
    delta = 2.0 ** -21 * (abs(W0[0]) + abs(W0[0] - outs[1][0]))
    ok = O.f64_to_bf16(outs[1])
    ok[0] = O.f64_to_bf16(np.array([outs[1][0] + 0.5 * delta]))[0]
    check_w(ok, outs, W0)                      # within delta: accepted
    bad = O.f64_to_bf16(outs[1])
    bad[0] = O.f64_to_bf16(np.array([outs[1][0] + 4 * delta]))[0]
    with pytest.raises(AssertionError):
        check_w(bad, outs, W0)
