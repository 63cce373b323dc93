"""Helpers of the GPU parity tests: device copies of synthetic inputs and the
relative tolerance rule.

Relative bound (floating-point outputs): per token row t and element i,
|gpu - oracle| <= 1e-3 * ||oracle_row_t||_2, the row's L2 norm being the
"output's L2 norm" of the stated bound.  The absolute side of the rule (the
fp32 forward-error bound, and the count of elements within 1e-4) needs the
oracle's per-slot terms and is applied by oracle.parity.check_layer.
Integer results (q8_K codes, expert ids, bucket order, sub-block sums) are
compared bit for bit."""
from __future__ import annotations

import numpy as np

from oracle.parity import NEAR_TIE, REL_TOL  # noqa: F401  (one definition of the rule)


def tol_rows(ref: np.ndarray) -> np.ndarray:
    return REL_TOL * np.linalg.norm(ref, axis=-1, keepdims=True)


def assert_close_rows(got, ref, what="output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > tol_rows(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol_rows(ref)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements beyond tolerance; worst at {i}: gpu {got[i]} "
                             f"oracle {ref[i]} |d|={err[i]:.3e} tol={tol_rows(ref)[i[:-1]][0]:.3e}")
    return float(err.max()), float((err / np.maximum(np.linalg.norm(ref, axis=-1, keepdims=True), 1e-30)).max())


def to_dev(a, torch, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def routing_ok(gpu_ids, oracle_ids, gap, logits=None, tie=None):
    """ids must match the oracle's except at near-ties: tokens whose oracle
    gap l_(k) - l_(k+1) is below the tie threshold may select a different
    set, and tokens whose selected logits hold two within it of each other
    may order them differently.  The threshold is NEAR_TIE, or per token
    `tie` (the parity rule's max(NEAR_TIE, twice the device's logit error)).
    Returns the number of such near-tie tokens whose ids differ (reported,
    not failed)."""
    gpu_ids = np.asarray(gpu_ids)
    oracle_ids = np.asarray(oracle_ids)
    tie = np.full(len(gpu_ids), NEAR_TIE) if tie is None else np.asarray(tie)
    mism = (gpu_ids != oracle_ids).any(axis=1)
    allowed = np.asarray(gap) < tie
    if logits is not None:
        sel = np.take_along_axis(np.asarray(logits), oracle_ids, axis=1)
        same_set = (np.sort(gpu_ids, axis=1) == np.sort(oracle_ids, axis=1)).all(axis=1)
        inner = np.abs(np.diff(sel, axis=1)).min(axis=1) < tie if sel.shape[1] > 1 else np.zeros(len(sel), bool)
        allowed |= same_set & inner
    hard = mism & ~allowed
    if hard.any():
        t = int(np.nonzero(hard)[0][0])
        raise AssertionError(f"routing differs at token {t} (gap {gap[t]:.3e}): gpu {gpu_ids[t]} oracle {oracle_ids[t]}")
    return int((mism & allowed).sum())
