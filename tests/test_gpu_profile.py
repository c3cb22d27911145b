"""Per-phase profiling of the indexer call (GPU): same results with and without it."""
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth

from gpu_cases import run_indexer

pytestmark = pytest.mark.gpu


def test_profiled_indexer_call_reports_phases_and_keeps_results():
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device="cuda")
    idx_plain, _, bits = run_indexer(w, geo, L)
    assert bits == 0
    D.dsa_profile_enable(True)
    try:
        idx_prof, _, bits = run_indexer(w, geo, L)
        ms = D.dsa_profile_indexer_last()
    finally:
        D.dsa_profile_enable(False)
    assert bits == 0
    assert torch.equal(idx_plain, idx_prof)
    assert len(ms) == 4 and all(m >= 0.0 for m in ms)
    assert ms[2] > 0.0                    # the score kernel ran
    assert sum(ms) < 1000.0


def test_launch_log_lists_every_kernel_of_a_layer_loop_in_order():
    """With profiling on, the launch log holds one record per kernel launch of the library, in
    launch order: per full layer RoPE (q, k), ranges, scores, select; per layer the attention
    pre-pass and kernel."""
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    from gpu_cases import device_geometry, rope_table_dev
    q_pos, k_pos, ks, ke = device_geometry(geo)
    layers = []
    for l in range(len(w.layers)):
        L = synth.layer_inputs(w, geo, l, device="cuda")
        L["out"] = torch.empty((w.n_q, w.n_heads, 512), dtype=torch.bfloat16, device="cuda")
        layers.append(L)
    cache = D.IndexCache(w.layers, w.n_q, w.topk, device="cuda")
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len,
                           D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = rope_table_dev(w, geo)
    D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache)
    D.dsa_profile_enable(True)
    try:
        ws = D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache)
        log = D.dsa_profile_read()
    finally:
        D.dsa_profile_enable(False)
    assert D.dsa_workspace_status(ws) == 0
    kinds = [k for k, _ in log]
    n_full = sum(t == "full" for t in w.layers)
    assert kinds.count("attn") == len(w.layers)
    assert kinds.count("indexer") <= n_full
    assert kinds[0] == "rope" and "attn" in kinds
    assert all(ms >= 0.0 for _, ms in log)
    # switching profiling on again empties the log
    D.dsa_profile_enable(True)
    D.dsa_profile_enable(False)
    assert D.dsa_profile_read() == []
    cache.close()
