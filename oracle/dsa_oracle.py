"""CPU oracle for the DSA indexer -> causal top-k -> IndexShare -> sparse MLA attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module: only the
tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` use it.  It shares no code with the CUDA library and imports nothing from it.

Everything here is plain NumPy in float64, written from the problem statement on three
public pages:

* "add glm5.2 indexshare" (MaxText pull request; sections Description, Key Changes,
  Code Review),
* "GLM-5/5.1/5.2 DSA + LoRA enablement" (Megatron-Bridge pull request; the commit
  messages on the indexer RoPE half swap, on capping top-k for short sequences and on
  cross-layer top-k sharing),
* "GLM-5.2 IndexShare" (explainer; sections 1 "What DSA does before sharing",
  2 "What IndexShare changes", "Layer execution pattern", "Public config evidence",
  "What is actually shared?", "Implementation checklist").

Readings taken where the pages are silent:

* index RoPE rotates the LAST ``r`` dims of each index head (Megatron convention), with
  rotate-half pairing (i, i + r/2) inside those dims, inv_freq_i = theta^(-2i/r) and
  angle = position * inv_freq_i evaluated in float64;  the rotated value is rounded to
  bf16 (round-to-nearest-even) because that is the precision the contraction consumes;
* the causal prefix of query t is the key range [ks_t, ke_t) and includes the query
  token itself, so it is never empty for a prefill row;
* ties in the top-k are broken towards the lower key index;
* returned indices are offsets relative to ks_t, sorted ascending, padded with -1;
* V is the first ``d_v`` (= 512) dims of the same 576-dim latent row;  the softmax scale
  is a parameter (default 1/sqrt(576));  the log-sum-exp uses the natural log.

Function status: every public function below is pinned by ``tests/test_oracle_pins.py``
against closed forms, library routines, brute force or the pages' printed values; no
function is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np

FULL = "full"
SHARED = "shared"


class NoDonorError(ValueError):
    """A shared layer has no full layer before it, so there is no index set to reuse.

    The Megatron-Bridge page ("assert a pipeline stage starts on a computing layer")
    makes this a hard error at build time rather than a silent fallback.
    """


# --------------------------------------------------------------------------------------
# bf16 helpers (exact in float64)
# --------------------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw bf16 bit patterns (uint16) into float64, exactly."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64.

    bf16 keeps 8 significant bits.  With x = m * 2**e (0.5 <= |m| < 1) the rounded value
    is rint(m * 2**8) * 2**(e - 8);  ``np.rint`` rounds halfway cases to even.  Subnormal
    and overflow ranges are not reached by this path's values.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


# --------------------------------------------------------------------------------------
# a1: RoPE on the last r dims of each index head
# --------------------------------------------------------------------------------------

def rope_inv_freq(rope_dim: int, theta: float) -> np.ndarray:
    """inv_freq_i = theta ** (-2 i / r) for i in [0, r/2)."""
    if rope_dim % 2:
        raise ValueError("rope_dim must be even")
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / rope_dim)


def rope_rotate_f64(x: np.ndarray, pos: np.ndarray, rope_dim: int, theta: float) -> np.ndarray:
    """Rotate the last ``rope_dim`` dims of ``x`` (float64, no rounding).

    x: [..., n, d] or [n, ..., d] with the token axis given by ``pos`` broadcasting
    against ``x[..., 0]``.  The first d - r dims pass through unchanged (the
    Megatron-Bridge page, indexer RoPE half-swap commit: RoPE sits in the last
    ``qk_pos_emb_head_dim`` dims of each index head).  Inside the last r dims, element i
    pairs with element i + r/2.
    """
    x = np.asarray(x, dtype=np.float64)
    if rope_dim == 0:
        return x.copy()
    d = x.shape[-1]
    if not (0 < rope_dim <= d):
        raise ValueError("rope_dim out of range")
    half = rope_dim // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(rope_dim, theta)
    c, s = np.cos(ang), np.sin(ang)
    y = x.copy()
    x1 = x[..., d - rope_dim: d - half]
    x2 = x[..., d - half:]
    y[..., d - rope_dim: d - half] = x1 * c - x2 * s
    y[..., d - half:] = x2 * c + x1 * s
    return y


def apply_index_rope(x: np.ndarray, pos: np.ndarray, rope_dim: int, theta: float) -> np.ndarray:
    """Index-head RoPE followed by the bf16 rounding the contraction consumes.

    ``pos`` must broadcast against ``x[..., 0]``: for q [n, H, d] pass pos[:, None];
    for k [n, d] pass pos.
    """
    return round_to_bf16(rope_rotate_f64(x, pos, rope_dim, theta))


# --------------------------------------------------------------------------------------
# a2: indexer scores
# --------------------------------------------------------------------------------------

def indexer_scores_row(q_rot: np.ndarray, k_rot: np.ndarray, w: np.ndarray) -> np.ndarray:
    """s[j] = sum_h w[h] * max(0, q_rot[h] . k_rot[j]) for one query row.

    q_rot: [H_I, d]   k_rot: [L, d]   w: [H_I]   ->   s: [L]
    The weighted ReLU sum over index heads with one key head shared by all index heads
    (Megatron-Bridge page: one ``wk``/``k_norm`` per index head dim;  ``weights_proj``
    is a per-head scalar).
    """
    dots = q_rot @ k_rot.T                      # [H_I, L]
    return w @ np.maximum(dots, 0.0)            # [L]


# --------------------------------------------------------------------------------------
# a3: causal top-k
# --------------------------------------------------------------------------------------

def topk_row(scores: np.ndarray, topk: int) -> np.ndarray:
    """Offsets of the min(topk, L) largest scores, ties to the lower offset.

    Returned sorted ascending and padded with -1 to width ``topk`` (Megatron-Bridge page,
    commit capping ``torch.topk`` at the sequence length and padding back with -1).
    """
    L = scores.shape[0]
    kt = min(topk, L)
    order = np.lexsort((np.arange(L), -scores))   # primary: score desc, secondary: index asc
    sel = np.sort(order[:kt])
    out = np.full(topk, -1, dtype=np.int64)
    out[:kt] = sel
    return out


def indexer_topk(q_idx: np.ndarray, k_idx: np.ndarray, w: np.ndarray,
                 q_pos: np.ndarray, k_pos: np.ndarray, ks: np.ndarray, ke: np.ndarray,
                 rope_dim: int, theta: float, topk: int,
                 rope_q: bool = True, rope_k: bool = True,
                 rows: Sequence[int] | None = None, return_scores: bool = False):
    """Lightning-indexer scores + causal top-k for the query rows ``rows`` (default all).

    q_idx: [n_q, H_I, d] float64 holding bf16 values;  k_idx: [n_kv, d];  w: [n_q, H_I];
    ks/ke: [n_q] key row range of each query.  Returns idx [len(rows), topk] (offsets
    relative to ks, -1 padded) and, if asked, the list of score rows.
    """
    if rows is None:
        rows = range(q_idx.shape[0])
    rows = list(rows)
    k_rot = apply_index_rope(k_idx, k_pos, rope_dim, theta) if rope_k else np.asarray(k_idx, np.float64)
    out = np.full((len(rows), topk), -1, dtype=np.int64)
    score_rows = []
    for n, t in enumerate(rows):
        q_t = np.asarray(q_idx[t], np.float64)
        q_rot = apply_index_rope(q_t, np.full(q_t.shape[0], q_pos[t]), rope_dim, theta) if rope_q else q_t
        s = indexer_scores_row(q_rot, k_rot[ks[t]:ke[t]], np.asarray(w[t], np.float64))
        out[n] = topk_row(s, topk)
        if return_scores:
            score_rows.append(s)
    return (out, score_rows) if return_scores else out


# --------------------------------------------------------------------------------------
# a5: MLA-absorbed sparse attention
# --------------------------------------------------------------------------------------

def sparse_attn_row(q_t: np.ndarray, kv: np.ndarray, idx_t: np.ndarray, ks_t: int,
                    scale: float, d_v: int = 512):
    """Attention of all heads of one query over its selected latent rows.

    q_t: [H, D_qk]   kv: [n_kv, D_qk]   idx_t: [topk] offsets (relative to ks_t, -1 = none)
    o[h] = sum_j softmax_j(scale * q[h] . kv[j]) * kv[j, :d_v];  lse[h] = log sum_j exp(.)
    Every head of the token reads the same rows; V is the first d_v dims of each row.
    A row with no valid index yields o = 0 and lse = -inf.
    """
    sel = idx_t[idx_t >= 0].astype(np.int64) + ks_t
    H = q_t.shape[0]
    if sel.size == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    rows = np.asarray(kv[sel], np.float64)                 # [n, D_qk]
    logits = scale * (np.asarray(q_t, np.float64) @ rows.T)  # [H, n]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ rows[:, :d_v]) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def sparse_attn(q: np.ndarray, kv: np.ndarray, idx: np.ndarray, ks: np.ndarray,
                scale: float, d_v: int = 512, rows: Sequence[int] | None = None):
    """Sparse attention for query rows ``rows`` (default all).  Returns (o, lse).

    ``idx`` holds one index row per entry of ``rows``, in the same order.
    """
    if rows is None:
        rows = range(q.shape[0])
    rows = list(rows)
    if idx.shape[0] != len(rows):
        raise ValueError("idx must hold one row per requested query row")
    H = q.shape[1]
    o = np.zeros((len(rows), H, d_v))
    lse = np.zeros((len(rows), H))
    for n, t in enumerate(rows):
        o[n], lse[n] = sparse_attn_row(q[t], kv, idx[n], int(ks[t]), scale, d_v)
    return o, lse


# --------------------------------------------------------------------------------------
# a4: IndexShare schedule and index cache
# --------------------------------------------------------------------------------------

def donor_table(indexer_types: Sequence[str]) -> list[int]:
    """donor[l] = l for a full layer, else the nearest preceding full layer.

    "GLM-5.2 IndexShare" explainer, "Layer execution pattern": shared layers reuse the
    nearest preceding full layer's top-k;  "Public config evidence": follow
    ``indexer_types`` instead of hard-coding a pattern.  Raises NoDonorError when a shared
    layer has no full layer before it.
    """
    donors, last_full = [], None
    for l, t in enumerate(indexer_types):
        if t == FULL:
            last_full = l
            donors.append(l)
        elif t == SHARED:
            if last_full is None:
                raise NoDonorError(f"layer {l} is shared but no full layer precedes it")
            donors.append(last_full)
        else:
            raise ValueError(f"layer {l}: unknown indexer type {t!r}")
    return donors


def layers_forward(indexer_types: Sequence[str], layers: Sequence[dict],
                   q_pos, k_pos, ks, ke, rope_dim: int, theta: float, topk: int,
                   scale: float, d_v: int = 512, rope_q: bool = True, rope_k: bool = True,
                   rows: Sequence[int] | None = None):
    """Run the IndexShare layer loop.

    layers[l] holds 'q', 'kv' (every layer) and, on full layers, 'q_idx', 'k_idx', 'w'.
    Full layers compute and cache their index set; shared layers take the donor's set
    unchanged ("What is actually shared?": top-k indices yes, attention no).  Returns
    (idx per layer, o per layer, lse per layer).
    """
    donors = donor_table(indexer_types)
    cache: dict[int, np.ndarray] = {}
    idx_l, o_l, lse_l = [], [], []
    for l, t in enumerate(indexer_types):
        if t == FULL:
            L = layers[l]
            cache[l] = indexer_topk(L["q_idx"], L["k_idx"], L["w"], q_pos, k_pos, ks, ke,
                                    rope_dim, theta, topk, rope_q, rope_k, rows=rows)
        idx = cache[donors[l]]
        o, lse = sparse_attn(layers[l]["q"], layers[l]["kv"], idx, ks, scale, d_v, rows=rows)
        idx_l.append(idx)
        o_l.append(o)
        lse_l.append(lse)
    return idx_l, o_l, lse_l


def mtp_indexshare_steps(steps: Sequence[dict], q_pos_steps: Sequence, k_pos, ks, ke_steps: Sequence,
                         rope_dim: int, theta: float, topk: int, scale: float, d_v: int = 512,
                         rope_q: bool = True, rope_k: bool = True, rows: Sequence[int] | None = None):
    """Multi-step MTP drafting with IndexShare.

    "GLM-5.2 IndexShare" (explainer), section "MTP path: IndexShare + KVShare": for multi-step
    MTP the indexer is placed at the first step and the following steps reuse its top-k
    indices.  steps[s] holds 'q' and 'kv' (every step) and, at step 0, 'q_idx', 'k_idx', 'w';
    q_pos_steps[s] / ke_steps[s] are the query positions and key-range ends of step s (the
    range start ks is common, the indices being offsets from it).  Returns (idx of step 0,
    o per step, lse per step).
    """
    s0 = steps[0]
    idx = indexer_topk(s0["q_idx"], s0["k_idx"], s0["w"], q_pos_steps[0], k_pos, ks, ke_steps[0],
                       rope_dim, theta, topk, rope_q, rope_k, rows=rows)
    o_l, lse_l = [], []
    for st in steps:
        o, lse = sparse_attn(st["q"], st["kv"], idx, ks, scale, d_v, rows=rows)
        o_l.append(o)
        lse_l.append(lse)
    return idx, o_l, lse_l


def unpage_rows(cache: np.ndarray, block_table: np.ndarray, seq_len: np.ndarray, page_rows: int):
    """Gather each row's logical keys out of a paged cache into one packed array.

    Layout of the paged decode caches: query row t's logical key j (j < seq_len[t]) is cache
    row block_table[t, j // page_rows] * page_rows + j % page_rows.  Returns (packed, ks, ke)
    with row t's keys at packed[ks[t]:ke[t]] in logical order, so the contiguous-cache
    functions above apply unchanged and their offsets are logical positions.
    """
    parts, ks, ke, off = [], [], [], 0
    for t in range(len(seq_len)):
        L = int(seq_len[t])
        j = np.arange(L)
        rows = block_table[t, j // page_rows].astype(np.int64) * page_rows + j % page_rows
        parts.append(cache[rows])
        ks.append(off)
        ke.append(off + L)
        off += L
    packed = np.concatenate(parts, axis=0) if parts else cache[:0]
    return packed, np.asarray(ks, np.int64), np.asarray(ke, np.int64)


def indexer_projections(x: np.ndarray, q_latent: np.ndarray, wq_b: np.ndarray, wk: np.ndarray,
                        k_norm_w: np.ndarray, k_norm_b: np.ndarray, w_proj: np.ndarray,
                        n_heads: int, head_dim: int, eps: float):
    """The indexer's input projections of one full layer.

    "GLM-5/5.1/5.2 DSA + LoRA enablement" (Megatron-Bridge pull request), indexer RoPE
    half-swap commit: wq_b gives the index queries, wk the shared index key, k_norm (a
    LayerNorm with weight and bias) is applied to the key before RoPE, weights_proj gives one
    scalar per index head.  Read here as q_idx = q_latent wq_b^T, k_idx = LayerNorm(x wk^T)
    (biased variance, epsilon inside the square root) * k_norm_w + k_norm_b, w = x
    weights_proj^T, with q_idx and k_idx rounded to bf16 once (what the indexer consumes).
    Returns (q_idx [T, H, d], k_idx [T, d], w [T, H]) as float64.
    """
    T = x.shape[0]
    q = round_to_bf16(np.asarray(q_latent, np.float64) @ np.asarray(wq_b, np.float64).T).reshape(T, n_heads, head_dim)
    y = np.asarray(x, np.float64) @ np.asarray(wk, np.float64).T
    mu = y.mean(axis=1, keepdims=True)
    var = ((y - mu) ** 2).mean(axis=1, keepdims=True)
    k = round_to_bf16((y - mu) / np.sqrt(var + eps) * np.asarray(k_norm_w, np.float64) + np.asarray(k_norm_b, np.float64))
    w = np.asarray(x, np.float64) @ np.asarray(w_proj, np.float64).T
    return q, k, w


def sparse_attn_backward(q: np.ndarray, kv: np.ndarray, idx: np.ndarray, ks: np.ndarray, scale: float,
                         d_o: np.ndarray, d_lse: np.ndarray | None = None, d_v: int = 512):
    """Gradients of the sparse attention above with respect to q and the latent rows.

    Differentiates exactly what sparse_attn computes.  No page defines a backward: "GLM-5/5.1/5.2
    DSA + LoRA enablement" (Megatron-Bridge pull request #15), in the commit that vendors the
    fused training kernels, only names one.  For token t, head h and selected rows j,
        s_j = scale q . kv_j,  p_j = exp(s_j - lse),  o = sum_j p_j kv_j[:d_v],
    given the upstream d_o (and d_lse, optional):
        dp_j = d_o . kv_j[:d_v],  D = sum_j p_j dp_j,  ds_j = p_j (dp_j - D + d_lse),
        dq += scale sum_j ds_j kv_j,
        dkv_j += scale ds_j q  (+ p_j d_o on the first d_v dims),
    summed over every (token, head) that selects row j.  Returns (dq [T, H, D], dkv [n_kv, D]).
    """
    q = np.asarray(q, np.float64)
    kv = np.asarray(kv, np.float64)
    T, H, Dq = q.shape
    dq = np.zeros_like(q)
    dkv = np.zeros_like(kv)
    for t in range(T):
        sel = idx[t][idx[t] >= 0]
        if sel.size == 0:
            continue
        rows = int(ks[t]) + sel
        K = kv[rows]                                    # [n, D]
        s = scale * (q[t] @ K.T)                        # [H, n]
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        p /= p.sum(axis=1, keepdims=True)               # = exp(s - lse)
        dp = np.asarray(d_o[t], np.float64) @ K[:, :d_v].T   # [H, n]
        D = (p * dp).sum(axis=1, keepdims=True)
        g = 0.0 if d_lse is None else np.asarray(d_lse[t], np.float64)[:, None]
        ds = p * (dp - D + g)
        dq[t] = scale * ds @ K
        contrib = scale * ds.T @ q[t]                   # [n, D]
        contrib[:, :d_v] += p.T @ np.asarray(d_o[t], np.float64)
        np.add.at(dkv, rows, contrib)
    return dq, dkv


# --------------------------------------------------------------------------------------
# lightning-indexer backward (a2 differentiated)
# --------------------------------------------------------------------------------------

def indexer_backward(q_idx: np.ndarray, k_idx: np.ndarray, w: np.ndarray,
                     q_pos: np.ndarray, k_pos: np.ndarray, ks: np.ndarray,
                     idx: np.ndarray, d_score: np.ndarray, rope_dim: int, theta: float,
                     rope_q: bool = True, rope_k: bool = True, round_rotated: bool = True,
                     rows: Sequence[int] | None = None, key_rows: Sequence[int] | None = None):
    """Gradients of the selected indexer scores with respect to q_idx, k_idx and w.

    "GLM-5/5.1/5.2 DSA + LoRA enablement" (Megatron-Bridge pull request), in the commit that
    vendors the fused lighting_indexer "with fwd/bwd", names this backward without defining
    it; it is the derivative of indexer_scores_row.  For query t, selected offset j
    (idx[t, n] = j >= 0, key row ks_t + j) and upstream gradient g = d_score[t, n]:
        x_h = q~[t, h] . k~[ks_t + j],    s = sum_h w[t, h] max(0, x_h)
        dw[t, h]        += g max(0, x_h)
        dq~[t, h]       += g w[t, h] [x_h > 0] k~[ks_t + j]
        dk~[ks_t + j]   += g sum_h w[t, h] [x_h > 0] q~[t, h]
    (ReLU'(0) = 0), then back through the rotation: dq = R(q_pos)^T dq~ when rope_q,
    dk = R(k_pos)^T dk~ when rope_k, R^T being the rotation by the negated angle.  The bf16
    rounding of the rotated values is taken as the identity in the derivative; with
    round_rotated=False the forward it differentiates has no rounding at all (the form the
    finite-difference pin uses).

    rows: the query rows whose dq / dw to return (default all); key_rows: the key rows whose
    dk to return (default all).  dk sums over EVERY query of idx whatever ``rows`` is.
    Returns (dq [len(rows), H_I, d], dk [len(key_rows), d], dw [len(rows), H_I]).
    """
    rot = (lambda x, p: apply_index_rope(x, p, rope_dim, theta)) if round_rotated else \
          (lambda x, p: rope_rotate_f64(x, p, rope_dim, theta))
    q_idx = np.asarray(q_idx, np.float64)
    k_idx = np.asarray(k_idx, np.float64)
    w = np.asarray(w, np.float64)
    n_q, H, d = q_idx.shape
    rows = list(range(n_q)) if rows is None else list(rows)
    key_rows = list(range(k_idx.shape[0])) if key_rows is None else list(key_rows)
    k_rot = rot(k_idx, k_pos) if rope_k else k_idx
    want_key = {int(j): n for n, j in enumerate(key_rows)}
    want_row = {int(t): n for n, t in enumerate(rows)}
    dq_rot = np.zeros((len(rows), H, d))
    dk_rot = np.zeros((len(key_rows), d))
    dw = np.zeros((len(rows), H))
    for t in range(n_q):
        sel_n = np.nonzero(idx[t] >= 0)[0]
        if sel_n.size == 0:
            continue
        keys = int(ks[t]) + idx[t][sel_n]
        hit = [m for m, j in enumerate(keys) if int(j) in want_key]
        if t not in want_row and not hit:
            continue
        q_rot = rot(q_idx[t], np.full(H, q_pos[t])) if rope_q else q_idx[t]
        cols = np.arange(keys.size) if t in want_row else np.asarray(hit, dtype=np.int64)
        K = k_rot[keys[cols]]                            # [n, d]
        g = np.asarray(d_score[t], np.float64)[sel_n[cols]]
        x = q_rot @ K.T                                  # [H, n]
        G = (x > 0) * w[t][:, None] * g[None, :]         # [H, n]
        if t in want_row:
            r = want_row[t]
            dw[r] = np.maximum(x, 0.0) @ g
            dq_rot[r] = G @ K
        for c, m in enumerate(cols):
            if int(keys[m]) in want_key:
                dk_rot[want_key[int(keys[m])]] += G[:, c] @ q_rot
    if rope_q:
        dq = rope_rotate_f64(dq_rot, -np.asarray(q_pos, np.float64)[rows][:, None], rope_dim, theta)
    else:
        dq = dq_rot
    if rope_k:
        dk = rope_rotate_f64(dk_rot, -np.asarray(k_pos, np.float64)[key_rows], rope_dim, theta)
    else:
        dk = dk_rot
    return dq, dk, dw
