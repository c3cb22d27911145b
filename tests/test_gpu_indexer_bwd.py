"""GPU parity of the lightning-indexer backward (dsa_indexer_backward) against the oracle.

The tensor-core products take G = g w [x > 0] in bf16 (relative rounding 2^-9 per term) with
fp32 accumulation, so dq and dk agree with the float64 oracle to a relative row error well
under 1e-2.  dw is summed in fp32 from the fp32 scores; its bound, 2e-3, covers the rotated
inputs, which the library rotates in fp32 and the oracle in float64 before both round to
bf16, so an element can differ by one bf16 ulp (2^-8 relative).  Index sets are
drawn here with numpy (any set is a valid input to the backward), so nothing the oracle reads
comes from the CUDA path.  Covers ragged tiles (slots not a multiple of 128), -1 padding, rows
with nothing selected, keys no row selects, 32 and 64 heads, RoPE on and off, an offset past
the row's range (flagged and skipped), and a prefill_4k-sized case checked on sampled rows.
"""
import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV
from oracle import dsa_oracle as O

pytestmark = pytest.mark.gpu

T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _rel_rows(got, ref):
    """Largest relative L2 error over rows (rows of zero reference compare absolutely)."""
    got = got.reshape(got.shape[0], -1)
    ref = ref.reshape(ref.shape[0], -1)
    num = np.linalg.norm(got - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    scale = max(float(den.max()), 1e-30)
    return float(np.max(num / np.maximum(den, 1e-3 * scale)))


def _case(n_q, n_kv, H, topk, r, seed, flags=D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K):
    rng = np.random.default_rng(seed)
    d = 128
    ks = rng.integers(0, n_kv // 4, size=n_q).astype(np.int32)
    ke = np.minimum(ks + rng.integers(1, n_kv, size=n_q), n_kv).astype(np.int32)
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        kt = min(topk, int(ke[t] - ks[t]))
        n = int(rng.integers(0, kt + 1)) if t % 7 else kt
        if t == 3:
            n = 0   # nothing selected
        idx[t, :n] = np.sort(rng.choice(int(ke[t] - ks[t]), size=n, replace=False))
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    q = (torch.randn((n_q, H, d), generator=g, device=DEV) / d ** 0.5).to(torch.bfloat16)
    k = (torch.randn((n_kv, d), generator=g, device=DEV) / d ** 0.5).to(torch.bfloat16)
    w = torch.randn((n_q, H), generator=g, device=DEV)
    d_score = torch.randn((n_q, topk), generator=g, device=DEV)
    q_pos = rng.integers(0, 5000, size=n_q).astype(np.int32)
    k_pos = rng.integers(0, 5000, size=n_kv).astype(np.int32)
    theta = 8e6
    desc = D.indexer_desc(n_q, n_kv, H, d, r, topk, int(max(1, (ke - ks).max())), flags)
    rope = D.dsa_rope_table(theta, r, 5000).to(DEV) if r else None
    return dict(desc=desc, q=q, k=k, w=w, d_score=d_score, idx=idx, ks=ks, ke=ke, q_pos=q_pos, k_pos=k_pos,
                rope=rope, theta=theta, r=r, n_q=n_q, n_kv=n_kv, H=H, d=d, topk=topk,
                rope_q=bool(flags & D.DSA_IDX_ROPE_Q), rope_k=bool(flags & D.DSA_IDX_ROPE_K))


def _run(c, idx=None):
    dq = torch.full((c["n_q"], c["H"], c["d"]), 5.0, dtype=torch.float32, device=DEV)   # written
    dk = torch.full((c["n_kv"], c["d"]), 7.0, dtype=torch.float32, device=DEV)          # zeroed by the call
    dw = torch.full((c["n_q"], c["H"]), 3.0, dtype=torch.float32, device=DEV)
    ws = D.dsa_indexer_backward(c["desc"], c["q"], c["k"], c["w"], T(c["q_pos"]), T(c["k_pos"]), T(c["ks"]),
                                T(c["ke"]), c["rope"], T(c["idx"] if idx is None else idx), c["d_score"], dq, dk, dw)
    return dq, dk, dw, D.dsa_workspace_status(ws, raise_on_fault=False)


def _oracle(c, rows=None, key_rows=None):
    f = synth.to_f64
    return O.indexer_backward(f(c["q"]), f(c["k"]), f(c["w"]), c["q_pos"], c["k_pos"], c["ks"], c["idx"],
                              f(c["d_score"]), c["r"], c["theta"], rope_q=c["rope_q"], rope_k=c["rope_k"],
                              rows=rows, key_rows=key_rows)


@pytest.mark.parametrize("n_q,n_kv,H,topk,r,flags", [
    (40, 600, 64, 256, 64, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K),
    (33, 900, 32, 300, 64, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K),   # ragged last tile, 32 heads
    (25, 400, 64, 130, 0, 0),                                       # no RoPE
    (20, 500, 16, 200, 64, D.DSA_IDX_ROPE_Q),                      # q rotated, k given rotated
])
def test_indexer_backward_matches_oracle(n_q, n_kv, H, topk, r, flags):
    c = _case(n_q, n_kv, H, topk, r, seed=n_q * 7 + H, flags=flags)
    dq, dk, dw, bits = _run(c)
    assert bits == 0, f"device status 0x{bits:x}"
    dq_ref, dk_ref, dw_ref = _oracle(c)
    dq_g, dk_g, dw_g = (x.double().cpu().numpy() for x in (dq, dk, dw))
    assert _rel_rows(dq_g, dq_ref) <= 1e-2
    assert _rel_rows(dk_g, dk_ref) <= 1e-2
    assert _rel_rows(dw_g, dw_ref) <= 2e-3
    # nothing selected: zero gradients; keys nobody selects: zero rows
    assert not dq_g[3].any() and not dw_g[3].any()
    used = {int(c["ks"][t]) + int(j) for t in range(n_q) for j in c["idx"][t] if j >= 0}
    unused = sorted(set(range(n_kv)) - used)
    assert unused and not dk_g[unused].any()


def test_indexer_backward_offset_past_the_row_is_flagged_and_skipped():
    c = _case(12, 300, 64, 128, 64, seed=5)
    bad = c["idx"].copy()
    t = 1
    n = int((bad[t] >= 0).sum())
    assert n > 0
    bad[t, 0] = int(c["ke"][t] - c["ks"][t]) + 3   # outside the row's key range
    dq, dk, dw, bits = _run(c, bad)
    assert bits != 0
    # the other slots of the row still count: compare with the oracle without the bad slot
    ref_idx = bad.copy()
    ref_idx[t, 0] = -1
    c2 = dict(c, idx=ref_idx)
    dq_ref, dk_ref, dw_ref = _oracle(c2)
    assert _rel_rows(dq.double().cpu().numpy(), dq_ref) <= 1e-2
    assert _rel_rows(dw.double().cpu().numpy(), dw_ref) <= 2e-3


def test_indexer_backward_prefill_4k_sampled_rows():
    # prefill_4k's first layer shapes: 4096 causal rows, 32 x 128 index heads, r = 64, k = 2048,
    # each row selecting a random min(k, t + 1) of its prefix
    w = synth.WORKLOADS["prefill_4k"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device=DEV, with_attn=False)
    rng = np.random.default_rng(11)
    n_q, topk = w.n_q, w.topk
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    for t in range(n_q):
        Lt = int(geo.ke[t] - geo.ks[t])
        kt = min(topk, Lt)
        idx[t, :kt] = np.sort(rng.permutation(Lt)[:kt])
    g = torch.Generator(device=DEV)
    g.manual_seed(17)
    d_score = torch.randn((n_q, topk), generator=g, device=DEV)
    flags = D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K
    desc = D.indexer_desc(n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, topk, geo.max_len, flags)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)
    dq = torch.empty((n_q, w.n_heads_idx, w.head_dim_idx), dtype=torch.float32, device=DEV)
    dk = torch.empty((geo.n_kv, w.head_dim_idx), dtype=torch.float32, device=DEV)
    dw = torch.empty((n_q, w.n_heads_idx), dtype=torch.float32, device=DEV)
    ws = D.dsa_indexer_backward(desc, L["q_idx"], L["k_idx"], L["w"], T(geo.q_pos), T(geo.k_pos), T(geo.ks),
                                T(geo.ke), rope, T(idx), d_score, dq, dk, dw)
    assert D.dsa_workspace_status(ws) == 0
    rows = [0, 1, 2046, 2047, 2048, 3000, 4095]
    keys = [0, 1, 2047, 4000, 4095]
    f = synth.to_f64
    dq_ref, dk_ref, dw_ref = O.indexer_backward(f(L["q_idx"]), f(L["k_idx"]), f(L["w"]), geo.q_pos, geo.k_pos,
                                                geo.ks, idx, f(d_score), w.rope_dim, w.theta, rows=rows,
                                                key_rows=keys)
    sel_r = torch.as_tensor(rows, device=DEV)
    assert _rel_rows(dq[sel_r].double().cpu().numpy(), dq_ref) <= 1e-2
    assert _rel_rows(dw[sel_r].double().cpu().numpy(), dw_ref) <= 2e-3
    assert _rel_rows(dk[torch.as_tensor(keys, device=DEV)].double().cpu().numpy(), dk_ref) <= 1e-2
