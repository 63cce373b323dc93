"""ORACLE — test infrastructure, not product code.

Comparison of one layer computed on the device with the oracle: the rule
every parity test and the bench's parity spot check apply.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs use it.

What is compared, for sampled tokens of a layer (device arrays in, numpy):

  exact      q8_K codes and scales of x; expert ids (a token whose oracle gap
             l_(k) - l_(k+1), or a gap between two of its selected logits,
             is below NEAR_TIE, or below twice the device's own logit error
             of that token (checked against the bound below), may differ:
             counted as a near-tie, not failed); the bucket order (perm) of
             the device's own ids.
  logits     (when the device's logits are given) against the oracle's fp64
             logits: |dl| <= (H + 8) * u * sum_h |w_eh x_h| + u * |bias_e|,
             the forward error bound of an fp32 dot product of length H in
             any summation order.
  gates      the device's fp32 gates against the oracle's fp64 gates of the
             same ids: |dg| <= g * (2 * max_s |dl_s| + 16 u) + GATE_ATOL, the
             first-order change of a renormalised softmax or sigmoid gate
             under the device's own logit errors dl plus the rounding of its
             exp and division (without the device's logits: GATE_RTOL * g +
             GATE_ATOL).
  h codes    the q8_K codes and block scales of the device's h against the
             oracle's q8_K of its own h (fp64 rounded to fp32).  A code whose
             h sits within rounding of a .5 boundary may flip: flips are
             counted and reported (Pulsar README, "Fidelity notes": results of
             two dot orders agree to a tolerance, not bit for bit).
  y, out     against the oracle evaluated on the DEVICE's h codes and gates,
             so both sides sum the same exact integer sub-block sums:
               |y_dev - y_ref|     <= (nb_I + 8) * u * C
               |out_dev - out_ref| <= (nb_I + 8 + k + S + 1) * u * A
             u = 2^-24 (fp32 unit roundoff); C = the sum of the magnitudes of
             the super-block terms of that down row (oracle.qmatvec_absterms);
             A = |residual| + sum_s |g_s| C_s + sum_shared C_sh.  The factor is
             the number of fp32 roundings on the device's longest path to one
             output (per super-block term: the int->fp32 conversion of the
             scaled sum, the min-term product, the fused multiply-add and the
             block scale, then one addition per term and up to 8 more for a
             cross-warp reduction; then one rounding per slot, shared expert
             and residual in the combine): a first-order forward error bound.
  relative   out against the oracle's own fp64 layer (its h codes, its
             gates): max_i |d_i| <= REL_TOL * ||ref_row||_2 on every row.

The stated float tolerance is 1e-3 of the output row's L2 norm and 1e-4
absolute per element.  The fp32 output itself cannot hold 1e-4 above 2048
(its spacing there is 2.4e-4; the decode workload's outputs reach ~2100 and
the wide workload's ~16000), so the absolute check is the fp32 bound above,
which is below 1e-4 wherever A < 1e-4 / (m u) (about 80 for m = 20), and the
count of elements within 1e-4 of the oracle is reported beside it.
"""
from __future__ import annotations

import numpy as np

from . import bucket, expert_ffn, layer_forward, q8k_quantize, qmatvec, qmatvec_absterms, route

NEAR_TIE = 1e-5
REL_TOL = 1e-3
ABS_TOL = 1e-4
GATE_RTOL = 1e-5
GATE_ATOL = 1e-6
U32 = 2.0 ** -24
MAX_FLIP_FRAC = 1e-2


def _routing(gpu_ids, oracle_ids, gap, logits, tie):
    """(near-tie tokens whose ids differ, hard mismatches [token indices]).
    tie [T]: per token, the logit gap below which an order may differ."""
    mism = (gpu_ids != oracle_ids).any(axis=1)
    allowed = gap < tie
    sel = np.take_along_axis(logits, oracle_ids, axis=1)
    same_set = (np.sort(gpu_ids, axis=1) == np.sort(oracle_ids, axis=1)).all(axis=1)
    if sel.shape[1] > 1:
        inner = np.abs(np.diff(sel, axis=1)).min(axis=1) < tie
    else:
        inner = np.zeros(len(sel), bool)
    allowed = allowed | (same_set & inner)
    return int((mism & allowed).sum()), np.nonzero(mism & ~allowed)[0]


def check_layer(fmt, H, I, E, k, S, route_kind, experts, wr, bias, x, residual, dev, tokens, nthreads=None):
    """Compare one device layer with the oracle on rows `tokens` of a T-token call.

    experts: host list of E + S (gate, up, down) byte arrays (None where not
    present); every expert the device selected for a sampled token must be
    given.  x, residual: the layer's fp32 inputs [T, H] (residual may be None).
    dev: device results as numpy arrays over all T tokens:
      ids [T, k], gates [T, k], perm [P] (bucket position -> slot index),
      h [P, I] (bucket order), y [P, H] (by slot index), out [T, H];
      optional xq [T, H], logits [T, E].
    Returns (metrics dict, list of failure strings)."""
    tokens = np.asarray(tokens, np.int64)
    T = x.shape[0]
    P = T * (k + S)
    nbI = I // 256
    m_y = nbI + 8
    m_out = m_y + k + S + 1
    fails = []
    xs = np.ascontiguousarray(x[tokens])
    res = None if residual is None else np.ascontiguousarray(residual[tokens])
    xq, xd, _ = q8k_quantize(xs)
    if "xq" in dev and not np.array_equal(dev["xq"][tokens], xq):
        fails.append(f"q8_K codes of x differ at {int((dev['xq'][tokens] != xq).sum())} positions")
    logits, rids, _, gap = route(xs, wr, bias, k, route_kind)
    # fp32 error bound of each logit: (H + 8) u sum_h |w x| + u |bias|
    lbound = (H + 8) * U32 * (np.abs(xs.astype(np.float64)) @ np.abs(wr.astype(np.float64)).T)
    if bias is not None:
        lbound += U32 * np.abs(np.asarray(bias, np.float64))[None, :]
    gids = np.ascontiguousarray(dev["ids"][tokens]).astype(np.int32)
    lerr = None
    if "logits" in dev:
        l_dev = np.asarray(dev["logits"][tokens], np.float64)
        lerr = np.abs(l_dev - logits)
        if (lerr > lbound).any():
            t, e = np.unravel_index(np.argmax(lerr - lbound), lerr.shape)
            fails.append(f"logit of token {int(tokens[t])} expert {e}: |dl| {lerr[t, e]:.3e} > bound {lbound[t, e]:.3e}")
    # a selection may differ only where the oracle's gap is below NEAR_TIE or
    # below twice the device's own (bounded) logit error of that token
    tie = NEAR_TIE if lerr is None else np.maximum(NEAR_TIE, 2 * lerr.max(axis=1))
    near, hard = _routing(gids, rids, gap, logits, tie)
    if len(hard):
        t = int(hard[0])
        fails.append(f"routing differs at token {int(tokens[t])} (gap {gap[t]:.3e}): gpu {gids[t]} oracle {rids[t]}")
    _, _, g_or, _ = route(xs, wr, bias, k, route_kind, forced_ids=gids)
    g_dev = np.asarray(dev["gates"][tokens], np.float64)
    if lerr is not None:
        dl = np.take_along_axis(lerr, gids, axis=1).max(axis=1, keepdims=True)
        gtol = np.abs(g_or) * (2 * dl + 16 * U32) + GATE_ATOL
    else:
        gtol = GATE_RTOL * np.abs(g_or) + GATE_ATOL
    if (np.abs(g_dev - g_or) > gtol).any():
        t, s_ = np.unravel_index(np.argmax(np.abs(g_dev - g_or) - gtol), g_dev.shape)
        fails.append(f"gate of token {int(tokens[t])} slot {s_}: |dg| {abs(g_dev[t, s_] - g_or[t, s_]):.3e} > "
                     f"{gtol[t, s_]:.3e}")
    # bucketing of every token of the call, from the device's own ids
    _, _, rperm = bucket(np.ascontiguousarray(dev["ids"]).astype(np.int32), E, S)
    perm = np.asarray(dev["perm"], np.int64)[:P]
    bucket_exact = bool(np.array_equal(perm, rperm))
    if not bucket_exact:
        fails.append(f"bucket order differs at {int((perm != rperm).sum())} positions")
    inv = np.empty(P, np.int64)
    inv[rperm] = np.arange(P)
    # oracle evaluated on the device's h codes and gates, per sampled token
    n_codes = flips = scale_flips = 0
    y_ratio = 0.0
    out_ref = np.zeros((len(tokens), H))
    A = np.zeros((len(tokens), H))
    if res is not None:
        out_ref += res.astype(np.float64)
        A += np.abs(res.astype(np.float64))
    for ti, t in enumerate(tokens):
        pairs = [(int(t) * k + s, int(gids[ti, s]), float(g_dev[ti, s])) for s in range(k)]
        pairs += [(T * k + sh * T + int(t), E + sh, 1.0) for sh in range(S)]
        for p, e, g in pairs:
            if experts[e] is None:
                continue
            gate_w, up_w, down_w = experts[e]
            _, _, hq_or, hd_or = expert_ffn(gate_w, up_w, down_w, fmt, H, I, xq[ti:ti + 1], xd[ti:ti + 1],
                                            nthreads, return_h=True)
            hq_d, hd_d, _ = q8k_quantize(np.asarray(dev["h"][inv[p]], np.float32)[None, :])
            n_codes += hq_d.size
            flips += int((hq_d != hq_or).sum())
            scale_flips += int((hd_d != hd_or).sum())
            y_ref = qmatvec(down_w, fmt, H, I, hq_d, hd_d, nthreads)[0]
            C = qmatvec_absterms(down_w, fmt, H, I, hq_d, hd_d, nthreads)[0]
            y_dev = np.asarray(dev["y"][p], np.float64)
            err = np.abs(y_dev - y_ref)
            y_ratio = max(y_ratio, float((err / np.maximum(U32 * C, 1e-300)).max()))
            if (err > m_y * U32 * C).any():
                i = int(np.argmax(err - m_y * U32 * C))
                fails.append(f"y of token {int(t)} slot {p} (expert {e}) elt {i}: |d| {err[i]:.3e} > "
                             f"{m_y} u C = {m_y * U32 * C[i]:.3e}")
            out_ref[ti] += g * y_ref
            A[ti] += abs(g) * C
    out_dev = np.asarray(dev["out"][tokens], np.float64)
    err_c = np.abs(out_dev - out_ref)
    out_ratio = float((err_c / np.maximum(U32 * A, 1e-300)).max())
    if (err_c > m_out * U32 * A).any():
        i = np.unravel_index(np.argmax(err_c - m_out * U32 * A), err_c.shape)
        fails.append(f"out of token {int(tokens[i[0]])} elt {i[1]}: |d| {err_c[i]:.3e} > {m_out} u A = "
                     f"{m_out * U32 * A[i]:.3e}")
    if n_codes and flips > MAX_FLIP_FRAC * n_codes:
        fails.append(f"{flips} of {n_codes} h codes differ from the oracle's")
    # the oracle's own layer (its gates, its h codes), the device's ids forced
    ref, _, _, _ = layer_forward(fmt, H, I, E, k, S, route_kind, experts, wr, bias, xs, residual=res,
                                 forced_ids=gids, nthreads=nthreads)
    err = np.abs(out_dev - ref)
    norm = np.maximum(np.linalg.norm(ref, axis=1), 1e-300)
    rel = err.max(axis=1) / norm
    if (rel > REL_TOL).any():
        t = int(np.argmax(rel))
        fails.append(f"token {int(tokens[t])}: max |d| / ||ref|| = {rel[t]:.3e} > {REL_TOL:g}")
    metrics = {
        "tokens": int(len(tokens)),
        "max_logit_err": None if lerr is None else float(lerr.max()),
        "max_abs_err": float(err.max()),
        "max_rel_l2_err": float(rel.max()),
        "frac_within_1e-4": float((err <= ABS_TOL).mean()),
        "max_abs_ref": float(np.abs(ref).max()),
        "near_ties": near,
        "h_codes": int(n_codes),
        "h_code_flips": int(flips),
        "h_scale_flips": int(scale_flips),
        "bucket_exact": bucket_exact,
        "y_err_over_u_C": y_ratio,
        "out_err_over_u_A": out_ratio,
        "bound_factors": {"y": m_y, "out": m_out},
    }
    return metrics, fails


def merge(metrics):
    """Totals / maxima of several check_layer metrics dicts."""
    if not metrics:
        return {}
    out = {"layers_checked": len(metrics)}
    for key in ("tokens", "near_ties", "h_codes", "h_code_flips", "h_scale_flips"):
        out[key] = int(sum(m[key] for m in metrics))
    for key in ("max_abs_err", "max_rel_l2_err", "max_abs_ref", "y_err_over_u_C", "out_err_over_u_A"):
        out[key] = float(max(m[key] for m in metrics))
    out["frac_within_1e-4"] = float(min(m["frac_within_1e-4"] for m in metrics))
    le = [m["max_logit_err"] for m in metrics if m.get("max_logit_err") is not None]
    out["max_logit_err"] = float(max(le)) if le else None
    out["bucket_exact"] = all(m["bucket_exact"] for m in metrics)
    return out
