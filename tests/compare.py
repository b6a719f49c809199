"""Comparator used by every parity test (CUDA path vs oracle).

Tolerances:
* expert ids: exact, as ordered lists (descending logit, ties to the lower
  index).  A swap between two experts is accepted only where their oracle F32
  logits differ by no more than ``tie_bound`` = 1e-5 * max|logit| of the token,
  about ten times the real error of an F32 router sum at these sizes (~1e-6);
  there both choices are correct results of an F32 router, and the caller
  re-evaluates the oracle on the kernel's selection before comparing values and
  reports the tokens it did that for.  At the fixed seeds of the five workloads
  every 8th/9th gap is far above the bound, so the tests there require that no
  token needed it.
* routing weights: max |w - w_ref| <= 1e-5.
* outputs: max |out - ref| / max |ref| over the whole tensor
  (2e-3 for the fp32-accumulating decode path, 5e-3 for the half-precision
  tensor-core prefill path).
"""
from __future__ import annotations

import numpy as np

TOL_FP32 = 2e-3
TOL_BF16 = 5e-3
TOL_W = 1e-5


def rel_err(out, ref) -> float:
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(out - ref).max() / den) if den > 0 else float(np.abs(out - ref).max())


TIE_REL = 1e-5


def tie_bound(logits_ref) -> np.ndarray:
    """Per-token near-tie allowance: 1e-5 * max|logit| of the token."""
    lg = np.atleast_2d(np.asarray(logits_ref, dtype=np.float64))
    return TIE_REL * np.abs(lg).max(axis=1)


def ids_match(ids, ids_ref, logits_ref, bound) -> tuple[bool, list]:
    """Exact match of ordered id lists, or swaps confined to near-ties.

    Returns (ok, near_tie_tokens).  A token whose selected *set* differs from the
    reference is accepted only if every expert that entered or left the set has
    an oracle logit within ``bound`` of the k-th largest logit; an order
    difference inside the set is accepted only between logits within ``bound``.
    """
    ids = np.asarray(ids)
    ids_ref = np.asarray(ids_ref)
    logits_ref = np.asarray(logits_ref, dtype=np.float64)
    bound = np.broadcast_to(np.asarray(bound, dtype=np.float64), (ids.shape[0],))
    ties = []
    for t in range(ids.shape[0]):
        if np.array_equal(ids[t], ids_ref[t]):
            continue
        lg = logits_ref[t]
        if len(set(ids[t].tolist())) != ids.shape[1]:
            return False, ties
        kth = lg[ids_ref[t]].min()
        changed = set(ids[t].tolist()) ^ set(ids_ref[t].tolist())
        if any(abs(lg[e] - kth) > bound[t] for e in changed):
            return False, ties
        # order inside the set must be non-increasing up to the bound
        vals = lg[ids[t]]
        if np.any(np.diff(vals) > bound[t]):
            return False, ties
        ties.append(t)
    return True, ties


def min_gap(logits_ref, K) -> float:
    """Smallest gap between the K-th and (K+1)-th largest logit over tokens."""
    lg = np.sort(np.asarray(logits_ref, dtype=np.float64), axis=1)[:, ::-1]
    if lg.shape[1] <= K:
        return float("inf")
    return float((lg[:, K - 1] - lg[:, K]).min())
