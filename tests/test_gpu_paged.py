"""GPU parity of the paged decode caches (dsa_indexer_topk_paged, dsa_sparse_attn_paged).

The same decode-shaped data is laid out twice: packed (contiguous ranges) and in shuffled
128-row pages behind a block table.  The paged calls must give bit-identical indices, scores
and attention outputs to the contiguous calls (the same keys meet the same arithmetic), agree
with the oracle on an un-paged copy, and report (not fault on) a block-table entry outside the
cache.
"""
import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV
from oracle import dsa_oracle as O
from parity import check_topk

pytestmark = pytest.mark.gpu
P = D.DSA_PAGE_ROWS


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()
    assert torch.cuda.is_available()


def _paged_layout(geo, seed=3, spare=5):
    """Physical page of every (row, logical page), shuffled; returns block table, seq_len,
    n_pages and the physical cache row of every packed row."""
    lens = (geo.ke - geo.ks).astype(np.int64)
    n_pp = (lens + P - 1) // P
    n_pages = int(n_pp.sum()) + spare
    perm = np.random.default_rng(seed).permutation(n_pages)
    bt = np.full((lens.size, int(n_pp.max())), -1, dtype=np.int32)
    phys = np.zeros(int(lens.sum()), dtype=np.int64)
    k = 0
    for t, L in enumerate(lens):
        for p in range(n_pp[t]):
            bt[t, p] = perm[k]
            k += 1
        j = np.arange(L)
        phys[geo.ks[t] + j] = bt[t, j // P].astype(np.int64) * P + j % P
    return bt, lens.astype(np.int32), n_pages, phys


@pytest.mark.parametrize("n_seqs,len_lo,len_hi,topk,H", [(12, 900, 9000, 2048, 128), (8, 1, 700, 256, 64)])
def test_paged_equals_contiguous_and_oracle(n_seqs, len_lo, len_hi, topk, H):
    w = synth.Workload("paged", "decode", n_seqs, ("full",), 64, 128, 64, 8e6, topk, H, n_seqs=n_seqs,
                       len_lo=len_lo, len_hi=len_hi, rope_k=False)
    geo = synth.geometry(w, seed=11)
    L = synth.layer_inputs(w, geo, 0, device=DEV, attn_scale="unit")
    bt, seq_len, n_pages, phys = _paged_layout(geo)
    phys_t = torch.from_numpy(phys).to(DEV)
    k_cache = torch.zeros((n_pages * P, 128), dtype=torch.bfloat16, device=DEV)
    kv_cache = torch.zeros((n_pages * P, 576), dtype=torch.bfloat16, device=DEV)
    k_cache[phys_t] = L["k_idx"]
    kv_cache[phys_t] = L["kv"]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    bt_d, sl_d = t(bt), t(seq_len)
    pages = D.paged_cache(bt_d, sl_d, n_pages)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)
    flags = D.DSA_IDX_ROPE_Q | D.DSA_IDX_INDEPENDENT_ROWS
    n_q = w.n_q
    # contiguous reference run
    idesc_c = D.indexer_desc(n_q, geo.n_kv, 64, 128, 64, topk, geo.max_len, flags)
    idx_c = torch.empty((n_q, topk), dtype=torch.int32, device=DEV)
    sc_c = torch.empty((n_q, topk), dtype=torch.float32, device=DEV)
    ws = D.dsa_indexer_topk(idesc_c, L["q_idx"], L["k_idx"], L["w"], t(geo.q_pos), t(geo.k_pos), t(geo.ks),
                            t(geo.ke), rope, idx_c, sc_c)
    assert D.dsa_workspace_status(ws) == 0
    # paged run
    idesc_p = D.indexer_desc(n_q, n_pages * P, 64, 128, 64, topk, geo.max_len, flags)
    idx_p = torch.full((n_q, topk), -9, dtype=torch.int32, device=DEV)
    sc_p = torch.empty((n_q, topk), dtype=torch.float32, device=DEV)
    ws = D.dsa_indexer_topk_paged(idesc_p, L["q_idx"], k_cache, L["w"], t(geo.q_pos), pages, rope, idx_p, sc_p)
    assert D.dsa_workspace_status(ws) == 0
    assert torch.equal(idx_p, idx_c)
    assert torch.equal(sc_p, sc_c)
    # oracle on an un-paged copy of the paged cache
    packed, ks, ke = O.unpage_rows(synth.to_f64(k_cache), bt, seq_len, P)
    rows = list(range(n_q))
    _, score_rows = O.indexer_topk(synth.to_f64(L["q_idx"]), packed, synth.to_f64(L["w"]), geo.q_pos, None, ks, ke,
                                   64, w.theta, topk, rope_q=True, rope_k=False, rows=rows, return_scores=True)
    bad = check_topk(idx_p.cpu().numpy(), score_rows, topk, rows)
    assert not bad, f"{len(bad)} rows violate the top-k rule, first: {bad[:3]}"
    # attention: paged == contiguous, bit for bit
    adesc_c = D.attn_desc(n_q, geo.n_kv, H, topk, w.softmax_scale)
    out_c = torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=DEV)
    lse_c = torch.empty((n_q, H), dtype=torch.float32, device=DEV)
    ws = D.dsa_sparse_attn(adesc_c, L["q"], L["kv"], idx_c, t(geo.ks), out_c, lse_c)
    assert D.dsa_workspace_status(ws) == 0
    adesc_p = D.attn_desc(n_q, n_pages * P, H, topk, w.softmax_scale)
    out_p = torch.empty_like(out_c)
    lse_p = torch.empty_like(lse_c)
    ws = D.dsa_sparse_attn_paged(adesc_p, L["q"], kv_cache, idx_p, pages, out_p, lse_p)
    assert D.dsa_workspace_status(ws) == 0
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    # a block-table entry outside the cache is counted, not dereferenced (scores requested, so
    # every row is scored, including a row short enough to keep all its keys)
    bt_bad = bt.copy()
    bt_bad[0, 0] = n_pages + 3
    bad_pages = D.paged_cache(t(bt_bad), sl_d, n_pages)
    ws = D.dsa_indexer_topk_paged(idesc_p, L["q_idx"], k_cache, L["w"], t(geo.q_pos), bad_pages, rope, idx_p, sc_p)
    assert D.dsa_workspace_status(ws, raise_on_fault=False) != 0
    ws = D.dsa_sparse_attn_paged(adesc_p, L["q"], kv_cache, idx_c, bad_pages, out_p, lse_p)
    assert D.dsa_workspace_status(ws, raise_on_fault=False) != 0
