"""GPU parity of the sparse-attention backward (dsa_sparse_attn_backward) against the oracle.

The kernel takes D = d_out . out from the forward's bf16 output (the oracle uses the exact
product), so gradients agree to bf16-level relative error: max-abs within 2e-2 of the largest
reference gradient.  Covers rows shorter than k (-1 padding), rows shared by many tokens (the
dkv scatter), a head count that is not a multiple of the 16-head block, and an index outside
the cache (counted, skipped).
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()
    assert torch.cuda.is_available()


# the kernel walks each token's k slots in chunks of 64 rows, double-buffered: k > 64 covers the
# buffer alternation and dQ accumulated across chunks, k = 136 a ragged last chunk, and the gap
# rows an all-empty chunk between two selected ones
@pytest.mark.parametrize("n_q,n_kv,H,topk", [(48, 200, 16, 64), (30, 120, 40, 48), (17, 90, 4, 40),
                                             (20, 700, 16, 200), (12, 500, 40, 136),
                                             (8, 300, 64, 128), (6, 300, 128, 128),   # decode / chunk head counts
                                             (3, 100, 16, 40)])   # fewer than 64 (token, head) rows: per-token kernel
def test_backward_matches_oracle(n_q, n_kv, H, topk):
    rng = np.random.default_rng(n_q + H)
    ks = rng.integers(0, n_kv // 3, size=n_q).astype(np.int32)
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        L = int(rng.integers(1, min(topk, n_kv - ks[t]) + 1))
        idx[t, :L] = np.sort(rng.choice(n_kv - ks[t], size=L, replace=False))
    if topk > 128:
        tail = min(20, topk - 128)
        for t in (1, 4):   # slots 64..127 empty, selections before and after them
            idx[t] = -1
            sel = np.sort(rng.choice(n_kv - ks[t], size=20 + tail, replace=False))
            idx[t, :20], idx[t, 128:128 + tail] = sel[:20], sel[20:]
    g = torch.Generator(device=DEV)
    g.manual_seed(n_q * 3 + H)
    q = torch.randn((n_q, H, 576), generator=g, device=DEV).to(torch.bfloat16)
    kv = torch.randn((n_kv, 576), generator=g, device=DEV).to(torch.bfloat16)
    d_out = torch.randn((n_q, H, 512), generator=g, device=DEV).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(576)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    desc = D.attn_desc(n_q, n_kv, H, topk, scale)
    out = torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((n_q, H), dtype=torch.float32, device=DEV)
    ws = D.dsa_sparse_attn(desc, q, kv, t(idx), t(ks), out, lse)
    assert D.dsa_workspace_status(ws) == 0
    dq = torch.empty((n_q, H, 576), dtype=torch.float32, device=DEV)
    dkv = torch.full((n_kv, 576), 7.0, dtype=torch.float32, device=DEV)   # the call zeroes it
    ws = D.dsa_sparse_attn_backward(desc, q, kv, t(idx), t(ks), out, lse, d_out, dq, dkv)
    assert D.dsa_workspace_status(ws) == 0
    f = synth.to_f64
    dq_ref, dkv_ref = O.sparse_attn_backward(f(q), f(kv), idx, ks, scale, f(d_out))
    assert np.abs(dq.double().cpu().numpy() - dq_ref).max() <= 2e-2 * np.abs(dq_ref).max()
    assert np.abs(dkv.double().cpu().numpy() - dkv_ref).max() <= 2e-2 * np.abs(dkv_ref).max()
    # per (token, head) row of dq: relative L2 error (the bound above is relative to the largest
    # gradient and would hide errors confined to small rows).  A row's error comes from D taken
    # as dO . O from the bf16 output: an error dD moves every ds_j = p_j (dp_j - D) by -p_j dD,
    # so dq moves by -tau dD sum_j p_j kv_j, whatever the size of the row's own (possibly
    # cancelling) sum.  Rows whose norm falls below a quarter of the median row norm compare
    # against that floor; measured worst rows reach ~3.5e-2, typical ones ~2e-3.
    got = dq.double().cpu().numpy().reshape(n_q * H, -1)
    ref = dq_ref.reshape(n_q * H, -1)
    den = np.linalg.norm(ref, axis=1)
    floor = 0.25 * float(np.median(den[den > 0])) if (den > 0).any() else 1.0
    rel = np.linalg.norm(got - ref, axis=1) / np.maximum(den, floor)
    assert rel.max() <= 5e-2, (float(rel.max()), int(rel.argmax()), float(den[rel.argmax()]), floor)
    # an index past the cache is counted and skipped
    bad = idx.copy()
    bad[0, 0] = n_kv + 5
    ws = D.dsa_sparse_attn_backward(desc, q, kv, t(bad), t(ks), out, lse, d_out, dq, dkv)
    assert D.dsa_workspace_status(ws, raise_on_fault=False) != 0


def _fwd_bwd(q, kv, idx, ks, scale, d_out):
    """Forward (for out / lse) then backward through the library; returns dq, dkv, status bits."""
    n_q, H = q.shape[0], q.shape[1]
    n_kv, topk = kv.shape[0], idx.shape[1]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    desc = D.attn_desc(n_q, n_kv, H, topk, scale)
    out = torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((n_q, H), dtype=torch.float32, device=DEV)
    ws = D.dsa_sparse_attn(desc, q, kv, t(idx), t(ks), out, lse)
    assert D.dsa_workspace_status(ws) == 0
    dq = torch.full((n_q, H, 576), 5.0, dtype=torch.float32, device=DEV)   # every row is written
    dkv = torch.full((n_kv, 576), 7.0, dtype=torch.float32, device=DEV)    # the call zeroes it
    ws = D.dsa_sparse_attn_backward(desc, q, kv, t(idx), t(ks), out, lse, d_out, dq, dkv)
    return dq, dkv, D.dsa_workspace_status(ws, raise_on_fault=False)


def _rel_rows(got, ref):
    """Largest relative L2 error over rows, rows below a quarter of the median norm against that floor."""
    got = got.reshape(got.shape[0], -1)
    ref = ref.reshape(ref.shape[0], -1)
    den = np.linalg.norm(ref, axis=1)
    floor = 0.25 * float(np.median(den[den > 0])) if (den > 0).any() else 1.0
    return float((np.linalg.norm(got - ref, axis=1) / np.maximum(den, floor)).max())


def _causal_idx(n_q, topk, rng, offset=0):
    """Row t selects a random min(k, t + offset + 1) of its causal prefix (ks = 0), -1 padded."""
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        L = t + offset + 1
        kt = min(topk, L)
        idx[t, :kt] = np.sort(rng.permutation(L)[:kt])
    return idx


# the tensor-core (block-dense) walk for every head count it takes: 1, 2 and 8 heads (64, 32
# and 8 tokens an item), including a last item with fewer tokens than the others
@pytest.mark.parametrize("n_q,n_kv,H,topk", [(70, 300, 1, 64), (40, 1000, 2, 300), (33, 400, 8, 100)])
def test_backward_block_dense_head_counts(n_q, n_kv, H, topk):
    assert D.lib() is not None
    rng = np.random.default_rng(n_q * 11 + H)
    ks = rng.integers(0, n_kv // 4, size=n_q).astype(np.int32)
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        L = int(rng.integers(1, min(topk, n_kv - ks[t]) + 1))
        idx[t, :L] = np.sort(rng.choice(n_kv - ks[t], size=L, replace=False))
    idx[5] = -1   # a token that selects nothing: zero dq rows
    g = torch.Generator(device=DEV)
    g.manual_seed(n_q + 7 * H)
    q = torch.randn((n_q, H, 576), generator=g, device=DEV).to(torch.bfloat16)
    kv = torch.randn((n_kv, 576), generator=g, device=DEV).to(torch.bfloat16)
    d_out = torch.randn((n_q, H, 512), generator=g, device=DEV).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(576)
    dq, dkv, bits = _fwd_bwd(q, kv, idx, ks, scale, d_out)
    assert bits == 0
    f = synth.to_f64
    dq_ref, dkv_ref = O.sparse_attn_backward(f(q), f(kv), idx, ks, scale, f(d_out))
    dq_g, dkv_g = dq.double().cpu().numpy(), dkv.double().cpu().numpy()
    assert np.abs(dq_g - dq_ref).max() <= 2e-2 * np.abs(dq_ref).max()
    assert np.abs(dkv_g - dkv_ref).max() <= 2e-2 * np.abs(dkv_ref).max()
    assert _rel_rows(dq_g, dq_ref) <= 5e-2
    assert not dq_g[5].any()
    used = {int(ks[t]) + int(j) for t in range(n_q) for j in idx[t] if j >= 0}
    unused = sorted(set(range(n_kv)) - used)
    assert unused and not dkv_g[unused].any()


def test_backward_block_dense_causal_many_tiles():
    # 512 causal tokens over a 512-row cache, 16 heads, k = 256: items of 4 tokens walk up to
    # eight 64-row tiles (ragged last tiles), rows shared by hundreds of tokens
    n_q = n_kv = 512
    H, topk = 16, 256
    rng = np.random.default_rng(3)
    idx = _causal_idx(n_q, topk, rng)
    ks = np.zeros(n_q, dtype=np.int32)
    g = torch.Generator(device=DEV)
    g.manual_seed(21)
    q = (torch.randn((n_q, H, 576), generator=g, device=DEV) / 24.0).to(torch.bfloat16)
    kv = (torch.randn((n_kv, 576), generator=g, device=DEV) / 24.0).to(torch.bfloat16)
    d_out = torch.randn((n_q, H, 512), generator=g, device=DEV).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(576)
    dq, dkv, bits = _fwd_bwd(q, kv, idx, ks, scale, d_out)
    assert bits == 0
    f = synth.to_f64
    dq_ref, dkv_ref = O.sparse_attn_backward(f(q), f(kv), idx, ks, scale, f(d_out))
    assert _rel_rows(dq.double().cpu().numpy(), dq_ref) <= 5e-2
    assert _rel_rows(dkv.double().cpu().numpy(), dkv_ref) <= 5e-2


def test_backward_prefill_4k_sampled():
    # prefill_4k's first attention layer: 4096 causal tokens, 16 heads of 576 / 512, k = 2048,
    # each token selecting a random min(k, t + 1) of its prefix.  dq is checked on sampled tokens;
    # dkv on the last 96 rows, which only the last 96 tokens can select, so the oracle over those
    # tokens gives their exact gradient.
    w = synth.WORKLOADS["prefill_4k"]
    geo = synth.geometry(w)
    assert (geo.ks == 0).all()
    L = synth.layer_inputs(w, geo, 0, device=DEV)
    n_q, topk, H = w.n_q, w.topk, w.n_heads
    rng = np.random.default_rng(17)
    idx = _causal_idx(n_q, topk, rng)
    g = torch.Generator(device=DEV)
    g.manual_seed(23)
    d_out = torch.randn((n_q, H, 512), generator=g, device=DEV).to(torch.bfloat16)
    scale = w.softmax_scale
    dq, dkv, bits = _fwd_bwd(L["q"], L["kv"], idx, geo.ks, scale, d_out)
    assert bits == 0
    f = synth.to_f64
    q64, kv64, do64 = f(L["q"]), f(L["kv"]), f(d_out)
    rows = [0, 1, 63, 64, 2047, 2048, 3001, 4095]
    dq_ref, _ = O.sparse_attn_backward(q64[rows], kv64, idx[rows], geo.ks[rows], scale, do64[rows])
    assert _rel_rows(dq[torch.as_tensor(rows, device=DEV)].double().cpu().numpy(), dq_ref) <= 5e-2
    tail = list(range(n_q - 96, n_q))
    _, dkv_ref = O.sparse_attn_backward(q64[tail], kv64, idx[tail], geo.ks[tail], scale, do64[tail])
    assert _rel_rows(dkv[n_q - 96:].double().cpu().numpy(), dkv_ref[n_q - 96:]) <= 5e-2


def test_backward_gather_walk_long_rows():
    # the tcgen05 gather walk: 64 tokens x 64 heads, each selecting up to k = 2048 random rows of
    # a 20000-row cache (32 tiles of 64 slots, rows shared by a few tokens), some rows shorter
    # than k, one token selecting nothing
    n_q, n_kv, H, topk = 64, 20000, 64, 2048
    rng = np.random.default_rng(29)
    ks = np.zeros(n_q, dtype=np.int32)
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        L = topk if t % 5 else int(rng.integers(1, topk))
        idx[t, :L] = np.sort(rng.choice(n_kv, size=L, replace=False))
    idx[9] = -1
    g = torch.Generator(device=DEV)
    g.manual_seed(31)
    q = (torch.randn((n_q, H, 576), generator=g, device=DEV) / 24.0).to(torch.bfloat16)
    kv = (torch.randn((n_kv, 576), generator=g, device=DEV) / 24.0).to(torch.bfloat16)
    d_out = torch.randn((n_q, H, 512), generator=g, device=DEV).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(576)
    dq, dkv, bits = _fwd_bwd(q, kv, idx, ks, scale, d_out)
    assert bits == 0
    f = synth.to_f64
    dq_ref, dkv_ref = O.sparse_attn_backward(f(q), f(kv), idx, ks, scale, f(d_out))
    dq_g, dkv_g = dq.double().cpu().numpy(), dkv.double().cpu().numpy()
    assert _rel_rows(dq_g, dq_ref) <= 5e-2
    used = np.unique(idx[idx >= 0])
    assert _rel_rows(dkv_g[used], dkv_ref[used]) <= 5e-2
    assert not dq_g[9].any()
    unused = np.setdiff1d(np.arange(n_kv), used)
    assert not dkv_g[unused].any()
