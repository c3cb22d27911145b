"""Failure detection on the GPU without a fault: the bounded pipeline waits.

The test hook (dsa_debug_pipeline) makes the TMA producers of the indexer and attention
kernels stop after a few tiles and bounds every pipeline wait at 1 ms.  The waits behind the
stopped producer run out, the kernel records a timeout in the workspace status word and
returns (copies already in flight land first), so the context stays usable: the status maps
to DSA_ERR_TIMEOUT, and the next normal call on the same workspace is clean and gives the
same results as a call made before the hook was set, which in turn match the oracle.
"""
import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth

from gpu_cases import device_geometry, oracle_attn, oracle_scores, rope_table_dev
from parity import check_topk

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 1


@pytest.fixture
def hook():
    yield
    D.dsa_debug_pipeline(-1, 0)


def _indexer_call(w, geo, L, ws, idx):
    q_pos, k_pos, ks, ke = device_geometry(geo)
    desc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len,
                          D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    if ws is None:
        ws = torch.empty(D.dsa_indexer_workspace_size(desc), dtype=torch.uint8, device="cuda")
    D.dsa_indexer_topk(desc, L["q_idx"], L["k_idx"], L["w"], q_pos, k_pos, ks, ke, rope_table_dev(w, geo), idx,
                       ws=ws)
    return ws


def test_indexer_wait_runs_out_then_the_workspace_is_clean(hook):
    # rows of up to 1024 keys: eight 128-key tiles per unit, so producers stopped after two
    # leave their consumers waiting
    w = synth.WORKLOADS["tiny"].replace(n_q=1024, topk=48)
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device="cuda", with_attn=False)
    ref = torch.empty((w.n_q, w.topk), dtype=torch.int32, device="cuda")
    ws_ref = _indexer_call(w, geo, L, None, ref)
    assert D.dsa_workspace_status(ws_ref) == 0

    D.dsa_debug_pipeline(stop_after_tiles=2, wait_ns=1_000_000)
    idx = torch.full((w.n_q, w.topk), -7, dtype=torch.int32, device="cuda")
    ws = _indexer_call(w, geo, L, None, idx)
    bits = D.dsa_workspace_status(ws, raise_on_fault=False)
    assert bits & TIMEOUT_BIT, f"status bits 0x{bits:x}: no wait ran out"
    with pytest.raises(D.DsaError) as e:
        D.dsa_workspace_status(ws)
    assert e.value.name == "DSA_ERR_TIMEOUT"

    D.dsa_debug_pipeline(-1, 0)
    idx2 = torch.full((w.n_q, w.topk), -7, dtype=torch.int32, device="cuda")
    _indexer_call(w, geo, L, ws, idx2)          # the same workspace, now a normal call
    assert D.dsa_workspace_status(ws) == 0
    assert torch.equal(idx2, ref)
    rows = [0, 47, 48, 500, 1023]
    sr = oracle_scores(w, geo, L, rows)
    bad = check_topk(idx2.cpu().numpy(), sr, w.topk, rows)
    assert not bad, bad


@pytest.mark.parametrize("heads", [4, 64])   # block-dense walk (4 heads) and per-token gathers (64)
def test_attention_wait_runs_out_then_the_workspace_is_clean(hook, heads):
    w = synth.WORKLOADS["tiny"].replace(n_q=512, topk=128, n_heads=heads)
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device="cuda", attn_scale="unit")
    rng = np.random.default_rng(3)
    idx_np = np.full((w.n_q, w.topk), -1, dtype=np.int32)
    for t in range(w.n_q):
        k = min(w.topk, t + 1)
        idx_np[t, :k] = np.sort(rng.choice(t + 1, size=k, replace=False))
    idx = torch.from_numpy(idx_np).cuda()
    ks = torch.from_numpy(geo.ks).cuda()
    desc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    out_ref = torch.empty((w.n_q, w.n_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty((w.n_q, w.n_heads), dtype=torch.float32, device="cuda")
    ws_ref = D.dsa_sparse_attn(desc, L["q"], L["kv"], idx, ks, out_ref, lse_ref)
    assert D.dsa_workspace_status(ws_ref) == 0

    D.dsa_debug_pipeline(stop_after_tiles=2, wait_ns=1_000_000)
    out = torch.zeros_like(out_ref)
    lse = torch.zeros_like(lse_ref)
    ws = D.dsa_sparse_attn(desc, L["q"], L["kv"], idx, ks, out, lse)
    bits = D.dsa_workspace_status(ws, raise_on_fault=False)
    assert bits & TIMEOUT_BIT, f"status bits 0x{bits:x}: no wait ran out"

    D.dsa_debug_pipeline(-1, 0)
    D.dsa_sparse_attn(desc, L["q"], L["kv"], idx, ks, out, lse, ws=ws)
    assert D.dsa_workspace_status(ws) == 0
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    rows = [0, 1, 127, 128, 511]
    o_ref, l_ref = oracle_attn(w, geo, L, idx_np, rows)
    got = synth.to_f64(out[torch.as_tensor(rows, device="cuda")])
    assert float(np.abs(got - o_ref).max()) <= 1e-2


@pytest.mark.parametrize("heads", [16, 64])   # the backward's block-dense walk (16 heads) and gather walk (64)
def test_attention_backward_wait_runs_out_then_the_workspace_is_clean(hook, heads):
    import math
    n_q, n_kv, topk = 512, 512, 256
    rng = np.random.default_rng(heads)
    idx_np = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        k = min(topk, t + 1)
        idx_np[t, :k] = np.sort(rng.permutation(t + 1)[:k])
    idx = torch.from_numpy(idx_np).cuda()
    ks = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(heads)
    q = (torch.randn((n_q, heads, 576), generator=g, device="cuda") / 24.0).to(torch.bfloat16)
    kv = (torch.randn((n_kv, 576), generator=g, device="cuda") / 24.0).to(torch.bfloat16)
    d_out = torch.randn((n_q, heads, 512), generator=g, device="cuda").to(torch.bfloat16)
    desc = D.attn_desc(n_q, n_kv, heads, topk, 1.0 / math.sqrt(576))
    out = torch.empty((n_q, heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n_q, heads), dtype=torch.float32, device="cuda")
    assert D.dsa_workspace_status(D.dsa_sparse_attn(desc, q, kv, idx, ks, out, lse)) == 0

    def bwd(ws=None):
        dq = torch.full((n_q, heads, 576), 5.0, dtype=torch.float32, device="cuda")
        dkv = torch.full((n_kv, 576), 7.0, dtype=torch.float32, device="cuda")
        ws = D.dsa_sparse_attn_backward(desc, q, kv, idx, ks, out, lse, d_out, dq, dkv, ws=ws)
        return dq, dkv, ws

    dq_ref, dkv_ref, ws_ref = bwd()
    assert D.dsa_workspace_status(ws_ref) == 0
    D.dsa_debug_pipeline(stop_after_tiles=2, wait_ns=1_000_000)
    _, _, ws = bwd()
    bits = D.dsa_workspace_status(ws, raise_on_fault=False)
    assert bits & TIMEOUT_BIT, f"status bits 0x{bits:x}: no wait ran out"
    with pytest.raises(D.DsaError) as e:
        D.dsa_workspace_status(ws)
    assert e.value.name == "DSA_ERR_TIMEOUT"

    D.dsa_debug_pipeline(-1, 0)
    dq2, dkv2, _ = bwd(ws)                       # the same workspace, now a normal call
    assert D.dsa_workspace_status(ws) == 0
    assert torch.equal(dq2, dq_ref)              # written once per (token, head) row
    # fp32 reductions in a different order: last bits of each sum, cancellation included
    torch.testing.assert_close(dkv2, dkv_ref, rtol=1e-4, atol=1e-5 * float(dkv_ref.abs().max()))
