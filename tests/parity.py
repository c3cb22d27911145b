"""Parity rules between the GPU path and the oracle (test helper, no method arithmetic).

Top-k rule (per query row, on the oracle's float64 scores s):
  * the row holds exactly min(k, L) distinct offsets in [0, L), then only -1;
  * with s sorted descending, if s_(k) - s_(k+1) > 1e-3 * max(|s_(k)|, |s_(k+1)|) the GPU set
    equals the oracle set exactly;
  * otherwise every selected offset has s >= s_(k) - margin, and every offset with
    s > s_(k) + margin is selected.
Attention rule: max-abs difference against the float64 oracle fed the GPU's own indices.
"""
from __future__ import annotations

import numpy as np

REL_TIE = 1e-3


def check_topk_row(gpu_row: np.ndarray, scores: np.ndarray, k: int, oracle_row: np.ndarray | None = None) -> str | None:
    """Return None when the row satisfies the rule, else a description of the violation."""
    gpu_row = np.asarray(gpu_row).astype(np.int64)
    L = scores.shape[0]
    kt = min(k, L)
    valid = gpu_row[gpu_row >= 0]
    if valid.size != kt:
        return f"count {valid.size} != min(k, L) = {kt}"
    if np.any(gpu_row[:kt] < 0) or np.any(gpu_row[kt:] != -1):
        return "-1 padding not confined to the tail"
    if np.unique(valid).size != valid.size:
        return "duplicate offsets"
    if np.any(np.diff(valid) <= 0):
        return "offsets not in ascending order"
    if valid.size and (valid.min() < 0 or valid.max() >= L):
        return f"offset outside [0, {L})"
    if kt == L:
        return None
    order = np.lexsort((np.arange(L), -scores))
    sk, sk1 = scores[order[kt - 1]], scores[order[kt]]
    margin = REL_TIE * max(abs(sk), abs(sk1))
    if sk - sk1 > margin:
        want = set(order[:kt].tolist()) if oracle_row is None else set(oracle_row[oracle_row >= 0].tolist())
        if set(valid.tolist()) != want:
            return f"set differs from the oracle's (gap {sk - sk1:.3e} > margin {margin:.3e})"
        return None
    if np.any(scores[valid] < sk - margin):
        return f"selected score below threshold {sk:.6e} - {margin:.3e}"
    must = np.nonzero(scores > sk + margin)[0]
    if not set(must.tolist()) <= set(valid.tolist()):
        return "a score clearly above the threshold was not selected"
    return None


def check_topk(gpu_idx: np.ndarray, score_rows, k: int, rows) -> list:
    bad = []
    for n, t in enumerate(rows):
        err = check_topk_row(gpu_idx[t], score_rows[n], k)
        if err:
            bad.append((int(t), err))
    return bad
