"""Brute-force formulation used to check the oracle on tiny inputs (T <= 64).

TEST INFRASTRUCTURE ONLY (see ``oracle/dsa_oracle.py``).  It deliberately computes the
same quantities a different way:

* scores: a dense [T, T] matrix by explicit einsum over (head, dim), then a causal mask;
* top-k: a full argsort of every row, turned into a boolean selection mask, exactly the
  ``indexer_mask`` the MaxText page feeds to dense attention ("add glm5.2 indexshare",
  Code Review, the ``jax.lax.cond`` over ``_run_full`` / ``_run_shared``);
* attention: dense masked softmax over all T keys for every head at once.

It shares no code with ``dsa_oracle`` except the bf16/RoPE helpers, which are pinned
separately.
"""
from __future__ import annotations

import numpy as np


def dense_scores(q_rot: np.ndarray, k_rot: np.ndarray, w: np.ndarray,
                 ks: np.ndarray, ke: np.ndarray) -> np.ndarray:
    """S[t, j] for every query t and key j; -inf outside [ks_t, ke_t)."""
    dots = np.einsum("thd,jd->thj", q_rot, k_rot)
    s = np.einsum("th,thj->tj", w, np.where(dots > 0.0, dots, 0.0))
    j = np.arange(k_rot.shape[0])[None, :]
    inside = (j >= ks[:, None]) & (j < ke[:, None])
    return np.where(inside, s, -np.inf)


def topk_mask(scores: np.ndarray, ks: np.ndarray, ke: np.ndarray, topk: int) -> np.ndarray:
    """Boolean mask [T, n_kv]: True for the min(topk, L_t) best keys of each row.

    Full argsort per row, stable, on (-score) so equal scores keep ascending key order.
    """
    T, n = scores.shape
    mask = np.zeros((T, n), dtype=bool)
    for t in range(T):
        L = int(ke[t] - ks[t])
        order = np.argsort(-scores[t], kind="stable")
        mask[t, order[:min(topk, L)]] = True
    return mask


def dense_masked_attn(q: np.ndarray, kv: np.ndarray, mask: np.ndarray, scale: float,
                      d_v: int = 512):
    """o[t, h] = softmax over masked keys of scale * q[t, h] . kv[j], times kv[j, :d_v]."""
    logits = scale * np.einsum("thd,jd->thj", q, kv)
    logits = np.where(mask[:, None, :], logits, -np.inf)
    m = logits.max(axis=2, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(logits - m)
    l = p.sum(axis=2, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.einsum("thj,jd->thd", p, kv[:, :d_v]) / l
        lse = (m + np.log(l))[..., 0]
    o = np.where(l > 0, o, 0.0)
    return o, lse
