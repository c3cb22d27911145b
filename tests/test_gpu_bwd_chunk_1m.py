"""Both backward kernels at chunk_1m's full size (4096 queries over a 1,048,576-key prefix, 64
heads, k = 2048), checked on sampled rows against the oracle.

Selections are drawn here (2048 distinct offsets of each query's prefix, uniform), so every key
row is selected by a handful of queries and the backward walks take their long-cache forms: the
attention backward's gather walk and the indexer backward's transposed dK.  The oracle sees
only the rows it needs: for a sampled query, its own selected rows; for a sampled key row, every
query that selects it (found from idx), so those gradients are exact sums.  Tolerances as in
the small-case tests of each kernel.
"""
import math

import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV
from oracle import dsa_oracle as O

pytestmark = pytest.mark.gpu

T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.fixture(scope="module")
def case():
    w = synth.WORKLOADS["chunk_1m"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device=DEV)
    rng = np.random.default_rng(41)
    n_q, k = w.n_q, w.topk
    idx = np.empty((n_q, k), dtype=np.int32)
    for t in range(n_q):
        Lt = int(geo.ke[t] - geo.ks[t])
        cand = np.unique(rng.integers(0, Lt, size=k + 256))
        idx[t] = np.sort(rng.permutation(cand)[:k])
    return w, geo, L, idx


def _selecting(idx, ks, rows):
    """Queries whose selection contains latent row r, for each r in rows."""
    absrow = idx.astype(np.int64) + ks.astype(np.int64)[:, None]
    return {int(r): np.nonzero((absrow == r).any(axis=1))[0] for r in rows}


def _rel_rows(got, ref):
    got = got.reshape(got.shape[0], -1)
    ref = ref.reshape(ref.shape[0], -1)
    den = np.linalg.norm(ref, axis=1)
    floor = 0.25 * float(np.median(den[den > 0])) if (den > 0).any() else 1.0
    return float((np.linalg.norm(got - ref, axis=1) / np.maximum(den, floor)).max())


def _subset(idx, ks, tokens, kv_rows):
    """Selections of `tokens` remapped into the union of their latent rows (ks = 0)."""
    absrow = idx[tokens].astype(np.int64) + ks[tokens].astype(np.int64)[:, None]
    uniq, inv = np.unique(absrow, return_inverse=True)
    return uniq, inv.reshape(absrow.shape).astype(np.int32), np.zeros(len(tokens), np.int32)


def test_attention_backward_chunk_1m_sampled(case):
    w, geo, L, idx = case
    n_q, H = w.n_q, w.n_heads
    desc = D.attn_desc(n_q, geo.n_kv, H, w.topk, w.softmax_scale)
    idx_d, ks_d = T(idx), T(geo.ks)
    out = torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((n_q, H), dtype=torch.float32, device=DEV)
    assert D.dsa_workspace_status(D.dsa_sparse_attn(desc, L["q"], L["kv"], idx_d, ks_d, out, lse)) == 0
    g = torch.Generator(device=DEV)
    g.manual_seed(43)
    d_out = torch.randn((n_q, H, 512), generator=g, device=DEV).to(torch.bfloat16)
    dq = torch.empty((n_q, H, 576), dtype=torch.float32, device=DEV)
    dkv = torch.empty((geo.n_kv, 576), dtype=torch.float32, device=DEV)
    ws = D.dsa_sparse_attn_backward(desc, L["q"], L["kv"], idx_d, ks_d, out, lse, d_out, dq, dkv)
    assert D.dsa_workspace_status(ws) == 0
    f = synth.to_f64
    # dq of sampled tokens
    toks = np.array([0, 1, 2047, 4095])
    uniq, sub, ks0 = _subset(idx, geo.ks, toks, None)
    kv_sub = f(L["kv"][torch.as_tensor(uniq, device=DEV)])
    q_s, do_s = f(L["q"][torch.as_tensor(toks, device=DEV)]), f(d_out[torch.as_tensor(toks, device=DEV)])
    dq_ref, _ = O.sparse_attn_backward(q_s, kv_sub, sub, ks0, w.softmax_scale, do_s)
    assert _rel_rows(dq[torch.as_tensor(toks, device=DEV)].double().cpu().numpy(), dq_ref) <= 5e-2
    # dkv of sampled latent rows: every query selecting them
    rows = [int(geo.ks[100]) + int(idx[100, 5]), int(geo.ks[3000]) + int(idx[3000, 1000])]
    sel = _selecting(idx, geo.ks, rows)
    toks2 = np.unique(np.concatenate([sel[r] for r in rows]))
    uniq2, sub2, ks02 = _subset(idx, geo.ks, toks2, None)
    kv_sub2 = f(L["kv"][torch.as_tensor(uniq2, device=DEV)])
    q2, do2 = f(L["q"][torch.as_tensor(toks2, device=DEV)]), f(d_out[torch.as_tensor(toks2, device=DEV)])
    _, dkv_ref = O.sparse_attn_backward(q2, kv_sub2, sub2, ks02, w.softmax_scale, do2)
    pos = [int(np.searchsorted(uniq2, r)) for r in rows]
    assert _rel_rows(dkv[torch.as_tensor(rows, device=DEV)].double().cpu().numpy(), dkv_ref[pos]) <= 5e-2


def test_indexer_backward_chunk_1m_sampled(case):
    w, geo, L, idx = case
    n_q = w.n_q
    flags = D.DSA_IDX_ROPE_Q | (D.DSA_IDX_ROPE_K if w.rope_k else 0)
    desc = D.indexer_desc(n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len, flags)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(47)
    d_score = torch.randn((n_q, w.topk), generator=g, device=DEV)
    dq = torch.empty((n_q, w.n_heads_idx, w.head_dim_idx), dtype=torch.float32, device=DEV)
    dk = torch.empty((geo.n_kv, w.head_dim_idx), dtype=torch.float32, device=DEV)
    dw = torch.empty((n_q, w.n_heads_idx), dtype=torch.float32, device=DEV)
    ws = D.dsa_indexer_backward(desc, L["q_idx"], L["k_idx"], L["w"], T(geo.q_pos), T(geo.k_pos), T(geo.ks),
                                T(geo.ke), rope, T(idx), d_score, dq, dk, dw)
    assert D.dsa_workspace_status(ws) == 0
    f = synth.to_f64
    ds = d_score.double().cpu().numpy()
    rows_k = [int(geo.ks[7]) + int(idx[7, 0]), int(geo.ks[2222]) + int(idx[2222, 2047])]
    sel = _selecting(idx, geo.ks, rows_k)
    toks = np.unique(np.concatenate([np.array([0, 2048, 4095])] + [sel[r] for r in rows_k]))
    uniq, sub, ks0 = _subset(idx, geo.ks, toks, None)
    tsel = torch.as_tensor(toks, device=DEV)
    dq_ref, dk_ref, dw_ref = O.indexer_backward(
        f(L["q_idx"][tsel]), f(L["k_idx"][torch.as_tensor(uniq, device=DEV)]), f(L["w"][tsel]), geo.q_pos[toks],
        geo.k_pos[uniq], ks0, sub, ds[toks], w.rope_dim, w.theta, rope_q=True, rope_k=bool(w.rope_k),
        key_rows=[int(np.searchsorted(uniq, r)) for r in rows_k])
    assert _rel_rows(dq[tsel].double().cpu().numpy(), dq_ref) <= 1e-2
    assert _rel_rows(dw[tsel].double().cpu().numpy(), dw_ref) <= 2e-3
    assert _rel_rows(dk[torch.as_tensor(rows_k, device=DEV)].double().cpu().numpy(), dk_ref) <= 1e-2
