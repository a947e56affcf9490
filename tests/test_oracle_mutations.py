"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, through monkeypatch)
and checks that at least one pin in ``test_oracle_pins`` then fails.
"""
import numpy as np
import pytest

import oracle as O
import oracle.forge_oracle as F
from tests import test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(F, name, fn)
    monkeypatch.setattr(O, name, fn)


def _adamw_variant(kind):
    def f(G, W, m, v, hyper, t):
        lr, b1, b2, eps, wd = hyper.as_f64()
        m1 = b1 * m + (1 - b1) * G
        v1 = b2 * v + (1 - b2) * G * G
        bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
        if kind == "no_bias_correction":
            bc1 = bc2 = 1.0
        if kind == "eps_inside_sqrt":
            W1 = (1 - lr * wd) * W - lr * (m1 / bc1) / np.sqrt(v1 / bc2 + eps)
        elif kind == "coupled_decay":
            m1 = b1 * m + (1 - b1) * (G + wd * W)
            v1 = b2 * v + (1 - b2) * (G + wd * W) ** 2
            W1 = W - lr * (m1 / bc1) / (np.sqrt(v1 / bc2) + eps)
        elif kind == "decay_after_update":
            W1 = (1 - lr * wd) * (W - lr * (m1 / bc1) / (np.sqrt(v1 / bc2) + eps))
        elif kind == "wrong_sign":
            W1 = (1 - lr * wd) * W + lr * (m1 / bc1) / (np.sqrt(v1 / bc2) + eps)
        elif kind == "swapped_betas":
            m1 = b2 * m + (1 - b2) * G
            v1 = b1 * v + (1 - b1) * G * G
            W1 = (1 - lr * wd) * W - lr * (m1 / bc1) / (np.sqrt(v1 / bc2) + eps)
        else:
            W1 = (1 - lr * wd) * W - lr * (m1 / bc1) / (np.sqrt(v1 / bc2) + eps)
        return W1, m1, v1
    return f


ADAMW_PINS = [
    lambda: P.test_adamw_matches_torch_optim_adamw_f64(10),
    P.test_step1_moves_each_weight_by_lr_times_sign,
    P.test_step1_with_eps_is_close_to_sign_step,
    P.test_no_tokens_decays_moments,
]


def _fails_one(pins):
    for pin in pins:
        try:
            pin()
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("kind", ["no_bias_correction", "eps_inside_sqrt",
                                  "coupled_decay", "decay_after_update",
                                  "wrong_sign", "swapped_betas"])
def test_adamw_mistakes_are_caught(monkeypatch, kind):
    _patch(monkeypatch, "adamw_f64", _adamw_variant(kind))
    assert _fails_one(ADAMW_PINS)


def test_unmutated_adamw_variant_passes(monkeypatch):
    _patch(monkeypatch, "adamw_f64", _adamw_variant("none"))
    assert not _fails_one(ADAMW_PINS)


@pytest.mark.parametrize("kind", ["transposed", "x_first", "dropped_token"])
def test_wgrad_mistakes_are_caught(monkeypatch, kind):
    def wg(x_bits, dy_bits, rows=None):
        X, dY = F.bf16_to_f64(x_bits), F.bf16_to_f64(dy_bits)
        if rows is not None:
            dY = dY[:, rows]
        if kind == "transposed":
            return (dY.T @ X).T.copy() if X.shape[1] != dY.shape[1] else (dY.T @ X).T
        if kind == "x_first":
            return X.T @ dY
        return dY[1:].T @ X[1:]
    _patch(monkeypatch, "wgrad", wg)
    pins = [lambda: P.test_wgrad_exact_rational_bruteforce(7, 3, 5),
            P.test_wgrad_one_hot_closed_form]
    assert _fails_one(pins)


@pytest.mark.parametrize("kind", ["truncate", "half_away", "via_float32"])
def test_bf16_rounding_mistakes_are_caught(monkeypatch, kind):
    good = F.f64_to_bf16

    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        if kind == "via_float32":     # double rounding
            f = x.astype(np.float32)
            return good(f.astype(np.float64))
        a = np.abs(x)
        _, e = np.frexp(a)
        q = np.where(e - 1 >= -126, e - 8, -133).astype(np.int32)
        s = np.ldexp(a, -q)
        r = np.floor(s) if kind == "truncate" else np.floor(s + 0.5)
        return good(np.copysign(np.ldexp(r, q), x))
    _patch(monkeypatch, "f64_to_bf16", bad)
    pins = [P.test_bf16_midpoints_round_to_even, P.test_bf16_overflow_and_subnormals]
    assert _fails_one(pins)


@pytest.mark.parametrize("kind", ["columns", "qmax_128", "no_floor", "block_64"])
def test_int8_mistakes_are_caught(monkeypatch, kind):
    def quant(x, floor_one):
        x = np.asarray(x, dtype=np.float64)
        rows, cols = x.shape
        blk = 64 if kind == "block_64" else 128
        if kind == "columns":
            a = np.repeat(np.max(np.abs(x), axis=0, keepdims=True), rows, axis=0)
            a = a.reshape(rows, cols // 128, 128).max(axis=2)
        else:
            a = np.max(np.abs(x.reshape(rows, cols // blk, blk)), axis=2)
            if blk == 64:
                a = a.reshape(rows, cols // 128, 2).max(axis=2) * 0 + a[:, ::2]
        qmax = 128.0 if kind == "qmax_128" else 127.0
        s = a / qmax
        sb = np.repeat(s, 128, axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.where(sb > 0, np.rint(x / np.where(sb > 0, sb, 1)), 0)
        q = np.clip(q, -127, 127)
        if floor_one and kind != "no_floor":
            q = np.where(sb > 0, np.maximum(q, 1), q)
        return q.astype(np.int8), s.astype(np.float32)
    _patch(monkeypatch, "quantize_int8_blocks", quant)
    pins = [P.test_int8_exactly_representable_block_round_trips,
            P.test_int8_error_within_half_a_step,
            P.test_int8_blocks_are_128_wide_along_rows,
            P.test_int8_second_moment_floor]
    assert _fails_one(pins)


@pytest.mark.parametrize("kind", ["w_transposed", "flipped_rows", "dropped_output"])
def test_dgrad_mistakes_are_caught(monkeypatch, kind):
    def dg(dy_bits, w_bits, rows=None):
        dY, W = F.bf16_to_f64(dy_bits), F.bf16_to_f64(w_bits)
        if rows is not None:
            dY = dY[rows]
        if kind == "w_transposed":
            return dY @ (W.T if W.shape[0] == W.shape[1] else W[::-1])
        if kind == "flipped_rows":
            return dY @ W[::-1]
        return dY[:, 1:] @ W[1:]
    _patch(monkeypatch, "dgrad", dg)
    pins = [lambda: P.test_dgrad_exact_rational_bruteforce(5, 3, 4),
            lambda: P.test_dgrad_one_hot_closed_form(7, 7),
            P.test_dgrad_and_wgrad_are_adjoint_to_the_forward_pass]
    assert _fails_one(pins)


# ---------------------------------------------------------------------------
# regime-1 optimizers (oracle/regime1.py)
# ---------------------------------------------------------------------------

import oracle.regime1 as R  # noqa: E402
from tests import test_oracle_regime1_pins as PR  # noqa: E402

_ORIG_OPT = R.opt_f64


def _opt_variant(kind):
    def f(opt, G, W, s1, s2, hyper, t):
        h = hyper.as_f64()
        lr, wd, eps, b1, b2 = h["lr"], h["weight_decay"], h["eps"], h["beta1"], h["beta2"]
        g = G + wd * W
        if kind == "momentum_dampened" and opt == R.OPT_SGD_MOMENTUM:
            b = h["momentum"] * s1 + (1 - h["momentum"]) * g
            return W - lr * b, b, None
        if kind == "adagrad_no_accumulation" and opt == R.OPT_ADAGRAD:
            s = g * g
            return W - lr * g / (np.sqrt(s) + eps), s1 + g * g, None
        if kind == "rmsprop_alpha_swapped" and opt == R.OPT_RMSPROP:
            s = (1 - h["alpha"]) * s1 + h["alpha"] * g * g
            return W - lr * g / (np.sqrt(s) + eps), s, None
        if kind == "rmsprop_decoupled_decay" and opt == R.OPT_RMSPROP:
            s = h["alpha"] * s1 + (1 - h["alpha"]) * G * G
            return (1 - lr * wd) * W - lr * G / (np.sqrt(s) + eps), s, None
        if kind == "lion_sign_of_new_state" and opt == R.OPT_LION:
            m = b2 * s1 + (1 - b2) * G
            return (1 - lr * wd) * W - lr * np.sign(m), m, None
        if kind == "lion_coupled_decay" and opt == R.OPT_LION:
            c = b1 * s1 + (1 - b1) * g
            return W - lr * np.sign(c), b2 * s1 + (1 - b2) * g, None
        if kind.startswith("nadam") and opt == R.OPT_NADAM:
            m = b1 * s1 + (1 - b1) * g
            v = b2 * s2 + (1 - b2) * g * g
            mu_t, mu_next, prod = R.nadam_scalars(h, t)
            if kind == "nadam_mu_next_is_mu_t":
                mu_next = mu_t
            bc2 = 1.0 if kind == "nadam_no_bias_correction" else 1 - b2 ** t
            d = np.sqrt(v / bc2) + eps
            return (W - lr * (1 - mu_t) / (1 - prod) * g / d
                    - lr * mu_next / (1 - prod * mu_next) * m / d), m, v
        if kind.startswith("radam") and opt == R.OPT_RADAM:
            m = b1 * s1 + (1 - b1) * g
            v = b2 * s2 + (1 - b2) * g * g
            mhat = m if kind == "radam_no_bias_correction" else m / (1 - b1 ** t)
            rect, r = R.radam_scalars(h, t)
            if kind == "radam_never_rectified":
                rect = False
            if rect:
                return W - lr * mhat * r * np.sqrt(1 - b2 ** t) / (np.sqrt(v) + eps), m, v
            return W - lr * mhat, m, v
        return _ORIG_OPT(opt, G, W, s1, s2, hyper, t)
    return f


@pytest.mark.parametrize("kind", [
    "momentum_dampened", "adagrad_no_accumulation", "rmsprop_alpha_swapped",
    "rmsprop_decoupled_decay", "lion_sign_of_new_state", "lion_coupled_decay",
    "nadam_mu_next_is_mu_t", "nadam_no_bias_correction", "radam_no_bias_correction",
    "radam_never_rectified"])
def test_regime1_mistakes_are_caught(monkeypatch, kind):
    f = _opt_variant(kind)
    monkeypatch.setattr(R, "opt_f64", f)
    monkeypatch.setattr(O, "opt_f64", f)
    torch_pins = [(lambda o=o: _with_f64_default(lambda: PR.test_matches_torch_optim_f64(o, None)))
                  for o in PR.TORCH_OPTS]
    pins = torch_pins + [PR.test_lion_closed_forms,
                         PR.test_first_momentum_step_is_sgd_and_zero_gradient_cases]
    assert _fails_one(pins)


def _with_f64_default(fn):
    import torch
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    try:
        fn()
    finally:
        torch.set_default_dtype(old)


def test_regime1_pins_pass_on_the_unmodified_oracle():
    # the control for the cases above: with nothing planted no pin fails
    pins = [(lambda o=o: _with_f64_default(lambda: PR.test_matches_torch_optim_f64(o, None)))
            for o in PR.TORCH_OPTS]
    pins += [PR.test_lion_closed_forms, PR.test_first_momentum_step_is_sgd_and_zero_gradient_cases]
    assert not _fails_one(pins)


# ---------------------------------------------------------------------------
# accumulate mode (oracle/accum.py)
# ---------------------------------------------------------------------------

import oracle.accum as A  # noqa: E402
from tests import test_oracle_accumulate_pins as PA  # noqa: E402


def _acc_variant(kind):
    def f(x_bits, dy_bits, B, beta, rows=None, return_f64=False):
        G = F.wgrad(x_bits, dy_bits, rows)
        b = float(np.float32(beta))
        Bf = np.asarray(B, dtype=np.float64)
        if kind == "beta_on_gradient":
            exact = G if b == 0.0 else Bf + b * G
        elif kind == "buffer_ignored":
            exact = G
        elif kind == "transposed":
            exact = G if b == 0.0 else b * Bf + (G.T if G.shape[0] == G.shape[1] else G[::-1])
        else:   # rounded twice
            exact = G if b == 0.0 else b * Bf + G
            out = F.f64_to_f32(F.f64_to_f32(b * Bf).astype(np.float64) + G) if b != 0.0 \
                else F.f64_to_f32(G)
            return (out, exact) if return_f64 else out
        out = F.f64_to_f32(exact)
        return (out, exact) if return_f64 else out
    return f


ACC_PINS = [PA.test_beta_zero_is_the_gradient_and_ignores_the_buffer,
            PA.test_integer_micro_batches_sum_to_the_whole_batch_exactly,
            lambda: PA.test_muon_momentum_closed_form_on_one_hot_inputs(3, 7),
            PA.test_no_tokens_scales_the_buffer_and_rounds_once]


@pytest.mark.parametrize("kind", ["beta_on_gradient", "buffer_ignored", "transposed",
                                  "rounded_twice"])
def test_accumulate_mistakes_are_caught(monkeypatch, kind):
    f = _acc_variant(kind)
    monkeypatch.setattr(A, "accumulate", f)
    monkeypatch.setattr(O, "accumulate", f)
    assert _fails_one(ACC_PINS)


def test_accumulate_pins_pass_on_the_unmodified_oracle():
    assert not _fails_one(ACC_PINS)


FINAL_PINS = [PA.test_final_step_moves_each_weight_against_the_sign_of_the_whole_sum,
              PA.test_final_step_with_a_zero_accumulator_is_the_plain_step,
              PA.test_final_step_reads_the_gradient_rounded_to_fp32]


def _final_variant(kind):
    def f(x_bits, dy_bits, w_bits, m, v, B, hyper, t, rows=None, return_f64=False):
        if kind == "accumulator_ignored":
            return F.step(x_bits, dy_bits, w_bits, m, v, hyper, t, rows, return_f64=return_f64)
        G = F.wgrad(x_bits, dy_bits, rows)
        Bf = np.asarray(B, dtype=np.float64)
        g = Bf - G if kind == "accumulator_subtracted" else Bf + G
        if kind != "not_rounded_to_fp32":
            g = F.f64_to_f32(g).astype(np.float64)
        W = F.bf16_to_f64(w_bits)
        W1, m1, v1 = F.adamw_f64(g, W, F.decode_moment(m, False), F.decode_moment(v, True),
                                 hyper, t)
        out = (F.f64_to_bf16(W1), F.encode_moment(m.fmt, m1, False),
               F.encode_moment(v.fmt, v1, True))
        return out + ((g, W1, m1, v1),) if return_f64 else out
    return f


@pytest.mark.parametrize("kind", ["accumulator_ignored", "accumulator_subtracted",
                                  "not_rounded_to_fp32"])
def test_final_step_mistakes_are_caught(monkeypatch, kind):
    f = _final_variant(kind)
    monkeypatch.setattr(A, "step_accumulated", f)
    monkeypatch.setattr(O, "step_accumulated", f)
    assert _fails_one(FINAL_PINS)


def test_final_step_pins_pass_on_the_unmodified_oracle():
    assert not _fails_one(FINAL_PINS)


# ---------------------------------------------------------------------------
# stochastic-rounding store (oracle/sr.py)
# ---------------------------------------------------------------------------

import oracle.sr as SRM  # noqa: E402
from tests import test_oracle_sr_pins as PS  # noqa: E402

_ORIG_PHILOX = SRM.philox4x64_10
_ORIG_SR = SRM.sr_to_bf16


def _philox_variant(kind):
    M = (1 << 64) - 1

    def f(counter, key):
        c0, c1, c2, c3 = (int(x) & M for x in counter)
        k0, k1 = (int(x) & M for x in key)
        m0 = 0xD2E7470EE14C6C93 if kind != "wrong_multiplier" else 0xD2E7470EE14C6C95
        for r in range(10):
            if r and kind != "no_key_bump":
                k0 = (k0 + 0x9E3779B97F4A7C15) & M
                k1 = (k1 + 0xBB67AE8584CAA73B) & M
            p0, p1 = m0 * c0, 0xCA5A826395121157 * c2
            if kind == "no_permutation":
                c0, c1, c2, c3 = p0 >> 64 ^ c1 ^ k0, p0 & M, p1 >> 64 ^ c3 ^ k1, p1 & M
            else:
                c0, c1, c2, c3 = (p1 >> 64) ^ c1 ^ k0, p1 & M, (p0 >> 64) ^ c3 ^ k1, p0 & M
        return c0, c1, c2, c3
    return f


def _sr_variant(kind):
    def f(x32, r16):
        r = np.asarray(r16, dtype=np.uint64)
        if kind == "nearest":
            r = np.full(r.shape, 0x8000, np.uint64)
        elif kind == "fifteen_bits":
            r = r >> np.uint64(1)
        return _ORIG_SR(x32, r)
    return f


SR_PINS = [lambda: PS.test_philox_matches_numpy((0, 0), (0, 0, 0, 0)),
           lambda: PS.test_philox_matches_numpy((42, 0), ((1 << 64) - 1, (1 << 64) - 1, 0, 9)),
           PS.test_sr_specials_and_extreme_draws, PS.test_sr_is_unbiased_exactly]


@pytest.mark.parametrize("kind", ["wrong_multiplier", "no_key_bump", "no_permutation"])
def test_philox_mistakes_are_caught(monkeypatch, kind):
    f = _philox_variant(kind)
    monkeypatch.setattr(SRM, "philox4x64_10", f)
    monkeypatch.setattr(O, "philox4x64_10", f)
    assert _fails_one(SR_PINS)


@pytest.mark.parametrize("kind", ["nearest", "fifteen_bits"])
def test_stochastic_rounding_mistakes_are_caught(monkeypatch, kind):
    f = _sr_variant(kind)
    monkeypatch.setattr(SRM, "sr_to_bf16", f)
    monkeypatch.setattr(O, "sr_to_bf16", f)
    assert _fails_one(SR_PINS)


def test_sr_pins_pass_on_the_unmodified_oracle():
    assert not _fails_one(SR_PINS)


# ---------------------------------------------------------------------------
# fp8 moments (oracle/fp8.py)
# ---------------------------------------------------------------------------

import oracle.fp8 as F8  # noqa: E402
from tests import test_oracle_fp8_pins as P8  # noqa: E402

_ORIG_TO_E4M3 = F8.f64_to_e4m3
_ORIG_FROM_E4M3 = F8.e4m3_to_f64


def _fp8_variant(kind):
    if kind == "bias_eight":
        def dec(codes):
            return _ORIG_FROM_E4M3(codes) / 2.0
        return "e4m3_to_f64", dec

    def enc(x):
        x = np.asarray(x, dtype=np.float64)
        if kind == "truncating":
            a = np.abs(x)
            _, e = np.frexp(a)
            q = np.where(e - 1 >= -6, e - 1 - 3, -9)
            t = np.ldexp(np.floor(np.ldexp(a, -q)), q)
            return _ORIG_TO_E4M3(np.copysign(t, x))
        with np.errstate(over="ignore", invalid="ignore"):   # no saturation: wraps past 448
            c = _ORIG_TO_E4M3(x).astype(np.int64)
            big = np.abs(x) > 448
            return np.where(big, (c & 0x80) | 0x7F, c).astype(np.uint8)
    return "f64_to_e4m3", enc


@pytest.mark.parametrize("kind", ["bias_eight", "truncating", "no_saturation"])
def test_fp8_mistakes_are_caught(monkeypatch, kind):
    name, f = _fp8_variant(kind)
    monkeypatch.setattr(F8, name, f)
    monkeypatch.setattr(O, name, f)
    pins = [P8.test_encoding_matches_torch_float8_e4m3fn,
            P8.test_decoding_all_codes_matches_torch_and_round_trips,
            P8.test_saturation_and_power_of_two_scales]
    assert _fails_one(pins)


def test_fp8_pins_pass_on_the_unmodified_oracle():
    assert not _fails_one([P8.test_encoding_matches_torch_float8_e4m3fn,
                           P8.test_decoding_all_codes_matches_torch_and_round_trips,
                           P8.test_saturation_and_power_of_two_scales])


_ORIG_ROLL = F8.roll_fp8_scales


def _roll_variant(kind):
    def roll(read_scale, write_scale, amax, headroom):
        if kind == "read_not_rolled":
            return np.float32(read_scale), _ORIG_ROLL(read_scale, write_scale, amax, headroom)[1]
        if kind == "int8_range":
            return np.float32(write_scale), np.float32(np.float32(amax) * headroom / 127.0)
        # headroom ignored
        return _ORIG_ROLL(read_scale, write_scale, amax, 1.0)
    return roll


@pytest.mark.parametrize("kind", ["read_not_rolled", "int8_range", "no_headroom"])
def test_fp8_scale_roll_mistakes_are_caught(monkeypatch, kind):
    f = _roll_variant(kind)
    monkeypatch.setattr(F8, "roll_fp8_scales", f)
    monkeypatch.setattr(O, "roll_fp8_scales", f)
    assert _fails_one([P8.test_scale_roll_closed_forms])
    monkeypatch.setattr(O, "roll_fp8_scales", _ORIG_ROLL)
    assert not _fails_one([P8.test_scale_roll_closed_forms])
