"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (stated bar, with the GEMM's own rounding accounted for):

* tau: the GPU forms each G_pq in fp32 as ceil(BT/16) tensor-core
  accumulations of 16 exact bf16 products; the oracle forms it in fp64.  Their
  difference is bounded by ``tau = (ceil(BT/16) + 8) * 2**-23 * S_pq`` with
  ``S_pq = sum_t |dY_tp X_tq|``: at most one fp32 unit of roundoff (2^-23
  relative, truncation included) per accumulation, plus margin for the
  summation inside one MMA.
* W (bf16): the GPU result must lie within 1 ulp of the range of oracle
  results over G in [G - tau, G + tau]; among entries whose oracle result does
  not move within that range, at least 99.99% must be within 1 ulp of the
  oracle and none more than 2 ulp.
  Entries where the update cancels most of W are held to the fp32 bound of
  the arithmetic instead (see check_w).
* fp32 moments: ``|d| <= 1e-5 |ref| + (propagated tau)``.
* bf16 moments: within 1 ulp of the oracle range over G +- tau.
* int8 moments: codes within 1 level of the oracle range over G +- tau,
  scales within 1e-5 relative plus the propagated tau.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

import oracle as O


def bf16_ordered(bits) -> np.ndarray:
    """Monotone integer image of bf16 bit patterns (+0 and -0 both map to 0)."""
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_diff(a_bits, b_bits) -> np.ndarray:
    return np.abs(bf16_ordered(a_bits) - bf16_ordered(b_bits))


def tau_bound(S: np.ndarray, bt: int) -> np.ndarray:
    return (math.ceil(bt / 16) + 8) * 2.0 ** -23 * S


@dataclass
class Report:
    n: int
    frac_within_1: float
    max_ulp: int
    sensitive: int
    violations: int
    cancelling: int = 0

    def __str__(self):
        return (f"n={self.n} within1={100 * self.frac_within_1:.4f}% max={self.max_ulp} "
                f"sensitive={self.sensitive} cancelling={self.cancelling} "
                f"violations={self.violations}")


def check_w(gpu_w_bits, w_outs, W0, label=""):
    """The bf16 weight bar.  w_outs: the oracle's fp64 W' at the points of
    g_points (at G first); W0: the weight before the step (fp64).

    The GPU forms W' = (1 - lr wd) W - lr u in fp32: its error is at most a few
    units of 2^-24 of the terms, bounded here by delta = 2^-21 (|W| + |W - W'|)
    (2^-24 for the decay product and the final rounding, 2^-22 for the update
    u, whose reciprocal and square root run on the special-function unit,
    2^-23 for moments the GPU decodes in fp32).  Where that bound is below
    half a bf16 ulp of the result, the stated bar holds: within 1 ulp of the
    oracle's range on at least 99.99 % of entries and never beyond 2 ulp
    (entries whose result moves over the range, "sensitive", count as within
    when inside it).  Where the update cancels most of W, so that delta is
    larger than that ("cancelling": W' << W), no fp32 evaluation can promise
    a bf16 ulp of the small result; those entries are counted and must lie
    within delta + 1 ulp of the range."""
    wb = [bf16_ordered(O.f64_to_bf16(x)) for x in w_outs]
    wlo, whi = np.minimum.reduce(wb), np.maximum.reduce(wb)
    g = bf16_ordered(gpu_w_bits)
    dist = np.maximum(np.maximum(wlo - g, g - whi), 0)
    mid = w_outs[0]
    delta = 2.0 ** -21 * (np.abs(W0) + np.abs(W0 - mid))
    ulp_mid = np.exp2(np.floor(np.log2(np.maximum(np.abs(mid), 2.0 ** -126))) - 7)
    cancel = delta > 0.5 * ulp_mid
    well = ~cancel
    # the cancelling entries, in value space
    gv = O.bf16_to_f64(np.asarray(gpu_w_bits, dtype=np.uint16))
    vlo = np.minimum.reduce([O.bf16_to_f64(O.f64_to_bf16(x)) for x in w_outs])
    vhi = np.maximum.reduce([O.bf16_to_f64(O.f64_to_bf16(x)) for x in w_outs])
    excess = np.maximum(np.maximum(vlo - gv, gv - vhi), 0.0)
    ulp_g = np.exp2(np.floor(np.log2(np.maximum(np.abs(gv), 2.0 ** -126))) - 7)
    bad_cancel = cancel & (excess > delta + ulp_g)
    sensitive = (whi > wlo) & well
    frac1 = float(np.mean(dist[well] <= 1)) if well.any() else 1.0
    mx = int(dist[well].max()) if well.any() else 0
    rep = Report(int(g.size), frac1, mx, int(sensitive.sum()),
                 int(np.sum(well & (dist > 2)) + bad_cancel.sum()), int(cancel.sum()))
    assert rep.violations == 0, f"{label} W: {rep}"
    assert rep.frac_within_1 >= 0.9999 and rep.max_ulp <= 2, f"{label} W: {rep}"
    return rep


def g_points(G, tau, extra=()):
    """Gradients at which the oracle is evaluated to span its results over
    [G - tau, G + tau]: G first, then eight more points across the interval,
    g = 0 where the interval holds it (the second moment is smallest there),
    and each array in `extra` clipped into the interval (an interior
    extremum of the update).  The update is not monotonic in g, so the end
    points alone do not bound it."""
    pts = [G] + [G + f * tau for f in (-1.0, -0.75, -0.5, -0.25, 0.25, 0.5, 0.75, 1.0)]
    pts.append(np.where(np.abs(G) <= tau, 0.0, G))
    for e in extra:
        pts.append(np.clip(e, G - tau, G + tau))
    return pts


def adamw_extremum(m, v, hyper):
    """The gradient at which u(g) = (b1 m + (1 - b1) g) / sqrt(b2 v + (1 - b2) g^2)
    is extremal (without eps): g* = (1 - b1) b2 v / (b1 m (1 - b2)); NaN where
    m = 0."""
    b1, b2 = hyper.beta1, hyper.beta2
    den = b1 * m * (1.0 - b2)
    safe = np.where(den != 0.0, den, 1.0)
    return np.where(den != 0.0, (1.0 - b1) * b2 * v / safe, np.nan)


def oracle_outs(G, tau, W, m, v, hyper, t):
    """The oracle's fp64 (W', m', v') at the points of g_points (G first),
    the update's interior extremum among them."""
    gs = adamw_extremum(m, v, hyper)
    pts = g_points(G, tau, extra=(np.where(np.isnan(gs), G, gs),))
    return [O.adamw_f64(g, W, m, v, hyper, t) for g in pts]


def check_step(gpu_w_bits, gpu_m, gpu_v, ref_inputs, hyper, t, fmt, bt, label=""):
    """Compare one GPU step with the oracle.

    ref_inputs: dict with G, S (fp64 [R, Din]), W_bits, m (Moment), v (Moment):
    the state and gradient the step started from, for the compared rows.
    gpu_m / gpu_v: Moment objects holding the GPU's stored moments (same rows).
    Raises AssertionError with a report when a bound is broken."""
    G, S = ref_inputs["G"], ref_inputs["S"]
    # a caller whose gradient is not the plain dY^T X (the final micro-batch's
    # fp32(B + G), R28) passes the bound of that gradient instead
    tau = ref_inputs["tau"] if "tau" in ref_inputs else tau_bound(S, bt)
    W = O.bf16_to_f64(ref_inputs["W_bits"])
    m0 = O.decode_moment(ref_inputs["m"], False)
    v0 = O.decode_moment(ref_inputs["v"], True)
    outs = oracle_outs(G, tau, W, m0, v0, hyper, t)
    reports = {}

    # ---- W (bf16)
    reports["W"] = check_w(gpu_w_bits, [x[0] for x in outs], W, label)

    # ---- moments
    if fmt == O.FMT_FP32:
        for which, idx, beta_term in (("m", 1, None), ("v", 2, None)):
            ref = outs[0][idx]
            got = (gpu_m if which == "m" else gpu_v).data.astype(np.float64)
            spread = np.max(np.stack([np.abs(x[idx] - ref) for x in outs]), axis=0)
            allow = 1e-5 * np.abs(ref) + spread + 1e-38
            err = np.abs(got - ref)
            nv = int(np.sum(err > allow))
            reports[which] = f"max rel {float(np.max(err / np.maximum(np.abs(ref), 1e-30))):.2e} violations={nv}"
            assert nv == 0, f"{label} {which}: {reports[which]}"
    elif fmt == O.FMT_BF16:
        for which, idx in (("m", 1), ("v", 2)):
            rb = [bf16_ordered(O.f64_to_bf16(x[idx])) for x in outs]
            rlo, rhi = np.minimum.reduce(rb), np.maximum.reduce(rb)
            got = bf16_ordered((gpu_m if which == "m" else gpu_v).data)
            nv = int(np.sum((got < rlo - 1) | (got > rhi + 1)))
            reports[which] = f"max ulp {int(np.max(np.abs(got - rb[0])))} violations={nv}"
            assert nv == 0, f"{label} {which}: {reports[which]}"
    else:
        for which, idx in (("m", 1), ("v", 2)):
            second = which == "v"
            encs = [O.encode_moment(O.FMT_INT8, x[idx], second) for x in outs]
            mom = gpu_m if which == "m" else gpu_v
            # scales: within 1e-5 relative of the oracle's range
            sc = np.stack([e.scale.astype(np.float64) for e in encs])
            slo, shi = sc.min(axis=0), sc.max(axis=0)
            gs = mom.scale.astype(np.float64)
            s_bad = (gs < slo * (1 - 1e-5)) | (gs > shi * (1 + 1e-5))
            # codes: within one level of the codes the oracle range gives
            cs = np.stack([e.data.astype(np.int64) for e in encs])
            clo, chi = cs.min(axis=0), cs.max(axis=0)
            gc = mom.data.astype(np.int64)
            c_bad = (gc < clo - 1) | (gc > chi + 1)
            if second:
                blk_nz = np.repeat(gs > 0, O.INT8_BLOCK, axis=1)
                c_bad |= blk_nz & (gc < 1)
            reports[which] = (f"scale violations={int(s_bad.sum())} code violations={int(c_bad.sum())}"
                              f" max code diff={int(np.max(np.abs(gc - cs[0])))}")
            assert not s_bad.any() and not c_bad.any(), f"{label} {which}: {reports[which]}"
    return reports


def check_opt_step(gpu_w_bits, gpu_states, ref_inputs, opt, hyper, t, fmt, bt, label=""):
    """check_step for the other optimizers (oracle/regime1.py): W within 1 ulp
    of the oracle range over G +- tau (and the same share within 1 ulp as for
    AdamW), fp32 states within 1e-5 relative plus the propagated tau, bf16
    states within 1 ulp of the range.

    "Relative" for an fp32 state is taken against the larger of the result
    and the magnitude of the terms it is formed from (the same update on
    |G| + tau, |W| and |state|): a state such as m' = beta1 m + (1 - beta1) g
    can cancel, and fp32 arithmetic errs by a unit of its terms, not of the
    result.  With tokens the tau spread already covers this; without tokens
    (G = 0) it is the only allowance.

    ref_inputs: G, S, W_bits and states [Moment or None, Moment or None] the
    step started from; gpu_states the GPU's states (Moment or None)."""
    G, S = ref_inputs["G"], ref_inputs["S"]
    tau = tau_bound(S, bt)
    W = O.bf16_to_f64(ref_inputs["W_bits"])
    n = O.OPT_STATES[opt]
    st0 = [O.decode_moment(s, False) if i < n else None
           for i, s in enumerate(ref_inputs["states"])]
    outs = [O.opt_f64(opt, g, W, st0[0], st0[1], hyper, t) for g in g_points(G, tau)]
    mag = O.opt_f64(opt, np.abs(G) + tau, np.abs(W),
                    None if st0[0] is None else np.abs(st0[0]),
                    None if st0[1] is None else np.abs(st0[1]), hyper, t)
    rep = check_w(gpu_w_bits, [x[0] for x in outs], W, label)
    reports = {"W": rep}
    for i in range(n):
        idx = i + 1
        name = f"s{idx}"
        if fmt == O.FMT_FP32:
            ref = outs[0][idx]
            got = gpu_states[i].data.astype(np.float64)
            spread = np.max(np.stack([np.abs(x[idx] - ref) for x in outs]), axis=0)
            err = np.abs(got - ref)
            scale = np.maximum(np.abs(ref), np.abs(mag[idx]))
            nv = int(np.sum(err > 1e-5 * scale + spread + 1e-38))
            reports[name] = f"max rel {float(np.max(err / np.maximum(np.abs(ref), 1e-30))):.2e} violations={nv}"
        else:
            rb = [bf16_ordered(O.f64_to_bf16(x[idx])) for x in outs]
            rlo, rhi = np.minimum.reduce(rb), np.maximum.reduce(rb)
            got = bf16_ordered(gpu_states[i].data)
            nv = int(np.sum((got < rlo - 1) | (got > rhi + 1)))
            reports[name] = f"max ulp {int(np.max(np.abs(got - rb[0])))} violations={nv}"
        assert nv == 0, f"{label} {name}: {reports[name]}"
    return reports
