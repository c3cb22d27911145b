"""GPU parity of multi-step MTP drafting with IndexShare (dsa_mtp_indexshare_step).

"GLM-5.2 IndexShare" (explainer), "MTP path: IndexShare + KVShare": the indexer runs at the
first MTP step and the following steps reuse its top-k.  Checked here: step 0's indices
against the oracle's scores (tie rule of tests/parity.py); the index buffer is left
bit-identical by the later steps; every step's attention (its own q, the growing key range)
matches the oracle fed step 0's GPU indices within 1e-2 on unit-scale inputs.
"""
import math

import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV, attn_errors
from oracle import dsa_oracle as O
from parity import check_topk

pytestmark = pytest.mark.gpu

ATOL_OUT = 1e-2
ATOL_LSE = 4e-3   # bf16 softmax weights in the denominator (as in test_gpu_parity)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("n_seqs,len_lo,len_hi,H_I,d,r,theta,topk,H,steps", [
    (8, 40, 300, 4, 64, 16, 1e4, 32, 4, 3),            # small: rows shorter and longer than k
    (16, 2500, 9000, 64, 128, 64, 8e6, 2048, 128, 3),  # decode shape: 64 x 128 index heads, 128 heads
])
def test_mtp_steps_reuse_the_first_step_indices(n_seqs, len_lo, len_hi, H_I, d, r, theta, topk, H, steps):
    w = synth.Workload("mtp", "decode", n_seqs, ("full",), H_I, d, r, theta, topk, H, n_seqs=n_seqs,
                       len_lo=len_lo, len_hi=len_hi, rope_k=False)
    geos = synth.mtp_geometry(w, steps, seed=7)
    g0 = geos[0]
    n_q, n_kv = w.n_q, g0.n_kv
    L0 = synth.layer_inputs(w, g0, 0, device=DEV, attn_scale="unit")
    gen = torch.Generator(device=DEV)
    gen.manual_seed(4242)
    q_steps = [L0["q"]] + [torch.randn((n_q, H, 576), generator=gen, device=DEV).to(torch.bfloat16)
                           for _ in range(steps - 1)]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    ks, k_pos = t(g0.ks), t(g0.k_pos)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, max(gg.max_pos for gg in geos)).to(DEV)
    idesc = D.indexer_desc(n_q, n_kv, H_I, d, r, topk, g0.max_len, D.DSA_IDX_ROPE_Q | D.DSA_IDX_INDEPENDENT_ROWS)
    mtp_idx = torch.full((n_q, topk), -7, dtype=torch.int32, device=DEV)
    outs, idx0 = [], None
    for s, gs in enumerate(geos):
        adesc = D.attn_desc(n_q, n_kv, H, topk, w.softmax_scale)
        layer = {"q": q_steps[s], "kv": L0["kv"],
                 "out": torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=DEV),
                 "lse": torch.empty((n_q, H), dtype=torch.float32, device=DEV)}
        if s == 0:
            layer.update(q_idx=L0["q_idx"], k_idx=L0["k_idx"], w=L0["w"])
        ws = D.dsa_mtp_indexshare_step(idesc, adesc, s, layer, ks, t(gs.ke), t(gs.q_pos), k_pos, rope, mtp_idx)
        assert D.dsa_workspace_status(ws) == 0
        if s == 0:
            idx0 = mtp_idx.clone()
        outs.append(layer)
    assert torch.equal(mtp_idx, idx0), "a later MTP step changed the step-0 indices"
    # step 0's selection against the oracle's scores
    rows = list(range(n_q))
    _, score_rows = O.indexer_topk(synth.to_f64(L0["q_idx"]), synth.to_f64(L0["k_idx"]), synth.to_f64(L0["w"]),
                                   g0.q_pos, g0.k_pos, g0.ks, g0.ke, r, theta, topk, rope_q=True, rope_k=False,
                                   rows=rows, return_scores=True)
    idx_np = idx0.cpu().numpy()
    bad = check_topk(idx_np, score_rows, topk, rows)
    assert not bad, f"{len(bad)} rows violate the top-k rule, first: {bad[:3]}"
    # every step attends over step 0's rows with its own q
    kv64 = synth.to_f64(L0["kv"])
    for s in range(steps):
        q64 = synth.to_f64(q_steps[s])
        o_ref = np.zeros((n_q, H, 512))
        lse_ref = np.zeros((n_q, H))
        for b in rows:
            o_ref[b], lse_ref[b] = O.sparse_attn_row(q64[b], kv64, idx_np[b], int(g0.ks[b]), w.softmax_scale)
        e_o, e_l = attn_errors(outs[s]["out"], outs[s]["lse"], o_ref, lse_ref, rows)
        assert e_o <= ATOL_OUT and e_l <= ATOL_LSE, (s, e_o, e_l)
    assert not torch.equal(outs[0]["out"], outs[1]["out"])
