"""Pins for the CPU oracle: each test checks it against something other than itself.

Sources of truth used here: closed forms of the rotation and of the softmax, library
routines (torch rounding, torch.topk, torch matmul, torch scaled-dot-product attention),
a brute-force dense formulation on tiny inputs, and the values the pages print about the
IndexShare schedule (``tests/golden/indexshare_facts.json``).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import brute
from oracle import dsa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "indexshare_facts.json")


def facts():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------------------- bf16 rounding

def test_round_to_bf16_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, -1.0]]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), ref)


def test_round_to_bf16_halfway_goes_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even mantissa (1.0)
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6)
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)])
    np.testing.assert_array_equal(O.round_to_bf16(x), [1.0, 1 + 2.0 ** -6, -1.0])
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), ref)


def test_bf16_bits_decode():
    bits = np.array([0x3F80, 0xBF80, 0x4000, 0x0000, 0x3E80], dtype=np.uint16)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), [1.0, -1.0, 2.0, 0.0, 0.25])


# ---------------------------------------------------------------------------- RoPE

def test_rope_zero_dims_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 3, 64))
    np.testing.assert_array_equal(O.rope_rotate_f64(x, np.arange(5)[:, None], 0, 1e4), x)


def test_rope_leaves_the_first_d_minus_r_dims_alone():
    # RoPE sits in the LAST r dims of each index head (Megatron convention).
    x = np.random.default_rng(2).standard_normal((7, 128))
    y = O.rope_rotate_f64(x, np.arange(7) * 1000 + 3, 64, 8e6)
    np.testing.assert_array_equal(y[:, :64], x[:, :64])
    assert not np.allclose(y[:, 64:], x[:, 64:])


def test_rope_closed_form_on_unit_vectors():
    # e at rotary slot i of the first half -> (cos(p f_i), sin(p f_i)) at slots (i, i + r/2).
    d, r, theta, p = 64, 16, 1e4, 37
    f = {0: 1.0, 1: 1.0 / math.sqrt(10.0), 4: 0.01}     # 1e4^(-2i/16): i=1 -> 10^-0.5, i=4 -> 10^-2
    for i, fi in f.items():
        e = np.zeros(d)
        e[d - r + i] = 1.0
        y = O.rope_rotate_f64(e, np.array(p), r, theta)
        expect = np.zeros(d)
        expect[d - r + i] = math.cos(p * fi)
        expect[d - r // 2 + i] = math.sin(p * fi)
        np.testing.assert_allclose(y, expect, atol=1e-15)
    # a unit vector in the second half rotates the other way: (-sin, cos)
    e = np.zeros(d)
    e[d - r // 2 + 1] = 1.0
    y = O.rope_rotate_f64(e, np.array(p), r, theta)
    assert y[d - r + 1] == pytest.approx(-math.sin(p * f[1]), abs=1e-15)
    assert y[d - r // 2 + 1] == pytest.approx(math.cos(p * f[1]), abs=1e-15)


def test_rope_preserves_norm_and_depends_on_relative_position_only():
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal(128), rng.standard_normal(128)
    r, th = 64, 8e6
    ra = lambda v, p: O.rope_rotate_f64(v, np.array(p), r, th)
    assert np.linalg.norm(ra(a, 123456)) == pytest.approx(np.linalg.norm(a), rel=1e-13)
    d0 = ra(a, 1000) @ ra(b, 990)
    for shift in (1, 77, 500000, 1048575 - 1000):
        assert ra(a, 1000 + shift) @ ra(b, 990 + shift) == pytest.approx(d0, rel=1e-9, abs=1e-9)


def test_apply_index_rope_rounds_to_bf16():
    rng = np.random.default_rng(4)
    x = O.round_to_bf16(rng.standard_normal((3, 4, 64)) / 8)
    y = O.apply_index_rope(x, np.array([5, 6, 7])[:, None], 16, 1e4)
    np.testing.assert_array_equal(y, O.round_to_bf16(y))
    np.testing.assert_array_equal(y[..., :48], x[..., :48])


# ---------------------------------------------------------------------------- indexer scores

def test_scores_single_head_unit_weight_is_relu_matmul():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 32))
    k = rng.standard_normal((50, 32))
    s = O.indexer_scores_row(q, k, np.array([1.0]))
    ref = torch.relu(torch.from_numpy(k) @ torch.from_numpy(q[0])).numpy()
    np.testing.assert_allclose(s, ref, rtol=1e-14, atol=1e-14)


def test_scores_weighted_head_sum_and_sign():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, 16))
    k = rng.standard_normal((20, 16))
    s = O.indexer_scores_row(q, k, np.array([2.0, 0.0, -1.0]))
    tq, tk = torch.from_numpy(q), torch.from_numpy(k)
    ref = 2.0 * torch.relu(tk @ tq[0]) - torch.relu(tk @ tq[2])
    np.testing.assert_allclose(s, ref.numpy(), rtol=1e-13, atol=1e-13)
    # negative weights make negative scores possible
    assert (s < 0).any()


# ---------------------------------------------------------------------------- top-k

def test_topk_distinct_scores_matches_torch_topk_set():
    rng = np.random.default_rng(7)
    for L, k in ((100, 10), (4096, 2048), (50, 49)):
        s = rng.standard_normal(L)
        got = O.topk_row(s, k)
        ref = torch.topk(torch.from_numpy(s), k).indices.numpy()
        assert set(got.tolist()) == set(ref.tolist())
        assert np.all(np.diff(got) > 0)


def test_topk_ties_go_to_lower_index():
    s = np.array([1.0, 5.0, 3.0, 5.0, 3.0, 3.0, 0.0])
    np.testing.assert_array_equal(O.topk_row(s, 3), [1, 2, 3])
    np.testing.assert_array_equal(O.topk_row(s, 4), [1, 2, 3, 4])
    np.testing.assert_array_equal(O.topk_row(np.zeros(6), 2), [0, 1])


def test_topk_short_row_pads_with_minus_one():
    pad = facts()["short_sequence_topk"]["pad_value"]
    s = np.array([0.3, -2.0, 7.0])
    np.testing.assert_array_equal(O.topk_row(s, 5), [0, 1, 2, pad, pad])
    np.testing.assert_array_equal(O.topk_row(np.zeros(0), 3), [pad, pad, pad])


def test_indexer_topk_causal_first_row_sees_only_itself():
    rng = np.random.default_rng(8)
    T, H, d = 6, 2, 16
    q = O.round_to_bf16(rng.standard_normal((T, H, d)))
    k = O.round_to_bf16(rng.standard_normal((T, d)))
    w = rng.standard_normal((T, H))
    pos = np.arange(T)
    idx = O.indexer_topk(q, k, w, pos, pos, np.zeros(T, int), pos + 1, 4, 1e4, 3)
    np.testing.assert_array_equal(idx[0], [0, -1, -1])
    np.testing.assert_array_equal(idx[1], [0, 1, -1])
    assert (idx[5] >= 0).sum() == 3 and idx[5].max() <= 5


# ---------------------------------------------------------------------------- attention

def test_attn_equal_logits_give_the_mean_of_v():
    rng = np.random.default_rng(9)
    kv = rng.standard_normal((30, 576))
    q = np.zeros((2, 576))
    idx = np.array([3, 7, 11, 29, -1, -1])
    o, lse = O.sparse_attn_row(q, kv, idx, 0, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(kv[[3, 7, 11, 29], :512].mean(0), (2, 512)), rtol=1e-13)
    np.testing.assert_allclose(lse, [math.log(4)] * 2, rtol=1e-14)


def test_attn_single_row_and_empty_row():
    rng = np.random.default_rng(10)
    kv = rng.standard_normal((10, 576))
    q = rng.standard_normal((3, 576))
    o, lse = O.sparse_attn_row(q, kv, np.array([-1, -1]), 4, 0.1)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    o, lse = O.sparse_attn_row(q, kv, np.array([2, -1]), 4, 0.1)      # row 4 + 2 = 6
    np.testing.assert_allclose(o, np.broadcast_to(kv[6, :512], (3, 512)), rtol=1e-14)
    np.testing.assert_allclose(lse, 0.1 * q @ kv[6], rtol=1e-13)


def test_sparse_equals_dense_causal_when_k_covers_the_prefix():
    # Short rows "degenerate to dense": with k >= L_t the selection is the whole prefix.
    rng = np.random.default_rng(11)
    T, H, scale = 40, 4, 1.0 / math.sqrt(576)
    q = rng.standard_normal((T, H, 576))
    kv = rng.standard_normal((T, 576))
    idx = np.stack([O.topk_row(rng.standard_normal(t + 1), 64) for t in range(T)])
    o, lse = O.sparse_attn(q, kv, idx, np.zeros(T, int), scale)
    tq = torch.from_numpy(q).permute(1, 0, 2)                           # [H, T, 576]
    tk = torch.from_numpy(kv)[None].expand(H, T, 576)
    tv = torch.from_numpy(kv[:, :512])[None].expand(H, T, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
    # lse of the first row is its single logit
    np.testing.assert_allclose(lse[0], scale * q[0] @ kv[0], rtol=1e-12)


# ---------------------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed,T,H_I,d,r,k,H", [(0, 48, 4, 64, 16, 8, 4), (1, 64, 8, 32, 8, 16, 2),
                                                  (2, 33, 1, 16, 0, 40, 3), (3, 64, 4, 64, 16, 32, 4)])
def test_oracle_matches_brute_force(seed, T, H_I, d, r, k, H):
    rng = np.random.default_rng(seed)
    q_idx = O.round_to_bf16(rng.standard_normal((T, H_I, d)) / math.sqrt(d))
    k_idx = O.round_to_bf16(rng.standard_normal((T, d)) / math.sqrt(d))
    w = rng.standard_normal((T, H_I))
    pos = np.arange(T)
    ks, ke = np.zeros(T, int), pos + 1
    idx, rows = O.indexer_topk(q_idx, k_idx, w, pos, pos, ks, ke, r, 1e4, k, return_scores=True)
    # brute force: dense scores from the same rotated inputs, full argsort, mask
    q_rot = O.apply_index_rope(q_idx, pos[:, None], r, 1e4)
    k_rot = O.apply_index_rope(k_idx, pos, r, 1e4)
    S = brute.dense_scores(q_rot, k_rot, w, ks, ke)
    for t in range(T):
        np.testing.assert_allclose(rows[t], S[t, :t + 1], rtol=1e-12, atol=1e-12)
    mask = brute.topk_mask(S, ks, ke, k)
    for t in range(T):
        assert set(idx[t][idx[t] >= 0].tolist()) == set(np.nonzero(mask[t])[0].tolist())
    q = rng.standard_normal((T, H, 576))
    kv = rng.standard_normal((T, 576))
    o, lse = O.sparse_attn(q, kv, idx, ks, 1 / math.sqrt(576))
    ob, lseb = brute.dense_masked_attn(q, kv, mask, 1 / math.sqrt(576))
    np.testing.assert_allclose(o, ob, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=1e-12)


# ---------------------------------------------------------------------------- IndexShare

def test_donor_table_on_the_78_layer_fsss_schedule():
    f = facts()["glm52_schedule"]
    types = [O.FULL if l % 4 == 0 else O.SHARED for l in range(f["n_layers"])]
    donors = O.donor_table(types)
    full = [l for l in range(len(types)) if donors[l] == l]
    assert len(full) == f["n_full"] and len(types) - len(full) == f["n_shared"]
    assert full[:3] == f["full_layers_prefix"]
    assert [l for l in range(8) if donors[l] != l] == f["shared_layers_prefix"]
    assert round(100.0 * f["n_shared"] / f["n_layers"], 1) == f["pruned_percent_1dp"]
    ex = facts()["donor_example"]
    for l in ex["layers"]:
        assert donors[l] == ex["donor"] != ex["wrong_donor"]


def test_donor_table_follows_the_released_indexer_types():
    types = facts()["released_config"]["indexer_types_prefix"]
    assert O.donor_table(types) == [0, 1, 2, 2, 2, 2, 6, 6, 6, 6]


def test_shared_layer_without_donor_is_an_error():
    with pytest.raises(O.NoDonorError):
        O.donor_table([O.SHARED, O.FULL])
    with pytest.raises(ValueError):
        O.donor_table([O.FULL, "sometimes"])


def test_layers_forward_reuses_donor_indices_and_runs_own_attention():
    rng = np.random.default_rng(12)
    T, H_I, d, H = 24, 2, 32, 2
    types = [O.FULL, O.SHARED, O.FULL, O.SHARED]
    layers = []
    for t in types:
        L = {"q": rng.standard_normal((T, H, 576)), "kv": rng.standard_normal((T, 576))}
        if t == O.FULL:
            L.update(q_idx=O.round_to_bf16(rng.standard_normal((T, H_I, d))),
                     k_idx=O.round_to_bf16(rng.standard_normal((T, d))),
                     w=rng.standard_normal((T, H_I)))
        layers.append(L)
    pos = np.arange(T)
    idx, o, lse = O.layers_forward(types, layers, pos, pos, np.zeros(T, int), pos + 1, 8, 1e4, 6,
                                   1 / 24.0)
    assert idx[1] is idx[0] and idx[3] is idx[2]
    assert not np.array_equal(idx[0], idx[2])
    assert not np.allclose(o[0], o[1])
    # each layer's output is its own attention over the shared index set
    o1, _ = O.sparse_attn(layers[1]["q"], layers[1]["kv"], idx[0], np.zeros(T, int), 1 / 24.0)
    np.testing.assert_array_equal(o[1], o1)


# ---------------------------------------------------------------------------- MTP IndexShare

def test_mtp_steps_attend_with_the_first_step_selection_brute_force():
    # "MTP path: IndexShare + KVShare": the indexer runs at the first MTP step and the later
    # steps reuse its top-k.  Brute force: dense step-0 scores, full argsort mask, and dense
    # masked attention of every step's q over that same mask (the later steps' longer ranges
    # must not enter).
    rng = np.random.default_rng(21)
    lens, steps, H_I, d, r, k, H = np.array([6, 11, 17, 23]), 3, 2, 16, 8, 5, 2
    span = lens + steps - 1
    off = np.concatenate([[0], np.cumsum(span)[:-1]])
    n_kv = int(span.sum())
    k_pos = np.arange(n_kv) - np.repeat(off, span)
    ks = off
    ke_steps = [off + lens + s for s in range(steps)]
    q_pos_steps = [lens - 1 + s for s in range(steps)]
    B = lens.size
    kv = rng.standard_normal((n_kv, 24))
    st = [{"q": rng.standard_normal((B, H, 24)), "kv": kv} for _ in range(steps)]
    st[0].update(q_idx=O.round_to_bf16(rng.standard_normal((B, H_I, d)) / 4),
                 k_idx=O.round_to_bf16(rng.standard_normal((n_kv, d)) / 4), w=rng.standard_normal((B, H_I)))
    idx, o, lse = O.mtp_indexshare_steps(st, q_pos_steps, k_pos, ks, ke_steps, r, 1e4, k, 0.3, d_v=16)
    q_rot = O.apply_index_rope(st[0]["q_idx"], q_pos_steps[0][:, None], r, 1e4)
    k_rot = O.apply_index_rope(st[0]["k_idx"], k_pos, r, 1e4)
    S = brute.dense_scores(q_rot, k_rot, st[0]["w"], ks, ke_steps[0])
    mask = brute.topk_mask(S, ks, ke_steps[0], k)
    for b in range(B):
        assert set((idx[b][idx[b] >= 0] + ks[b]).tolist()) == set(np.nonzero(mask[b])[0].tolist())
        assert idx[b].max() < lens[b]                      # inside step 0's causal range
    for s in range(steps):
        ob, lseb = brute.dense_masked_attn(st[s]["q"], kv, mask, 0.3, d_v=16)
        np.testing.assert_allclose(o[s], ob, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[s], lseb, rtol=1e-12)
    assert not np.allclose(o[1], o[0])                     # each step runs its own attention


# ---------------------------------------------------------------------------- paged caches

def test_unpage_rows_hand_example_and_round_trip():
    # 2 rows, pages of 2 rows; row 0 = keys 0..2 on pages (3, 1), row 1 = keys 0..3 on (0, 2)
    cache = np.arange(8 * 3, dtype=np.float64).reshape(8, 3)      # cache row r = [3r, 3r+1, 3r+2]
    bt = np.array([[3, 1], [0, 2]])
    packed, ks, ke = O.unpage_rows(cache, bt, np.array([3, 4]), 2)
    assert ks.tolist() == [0, 3] and ke.tolist() == [3, 7]
    np.testing.assert_array_equal(packed[:, 0] / 3, [6, 7, 2, 0, 1, 4, 5])
    # scattering a packed cache into shuffled pages and gathering it back is the identity
    rng = np.random.default_rng(5)
    lens = np.array([5, 1, 9, 4])
    P = 4
    n_pages_row = (lens + P - 1) // P
    perm = rng.permutation(int(n_pages_row.sum()) + 3)
    bt = np.full((lens.size, int(n_pages_row.max())), -1)
    src = rng.standard_normal((int(lens.sum()), 5))
    paged = np.zeros((perm.size * P, 5))
    k, off = 0, 0
    for t, L in enumerate(lens):
        for p in range(n_pages_row[t]):
            bt[t, p] = perm[k]
            n = min(P, L - p * P)
            paged[perm[k] * P: perm[k] * P + n] = src[off + p * P: off + p * P + n]
            k += 1
        off += L
    back, ks, ke = O.unpage_rows(paged, bt, lens, P)
    np.testing.assert_array_equal(back, src)


# ---------------------------------------------------------------------------- projections

def test_projections_layer_norm_matches_torch_and_closed_forms():
    rng = np.random.default_rng(31)
    T, D, Dq, H, d, eps = 5, 64, 64, 2, 8, 1e-6
    x = rng.standard_normal((T, D))
    ql = rng.standard_normal((T, Dq))
    wk = rng.standard_normal((d, D))
    g, b = rng.standard_normal(d), rng.standard_normal(d)
    # one-hot weights select input columns: q_idx[t, h, i] = q_latent[t, sel[h * d + i]]
    sel = rng.integers(0, Dq, size=H * d)
    wq = np.zeros((H * d, Dq))
    wq[np.arange(H * d), sel] = 1.0
    wp = np.zeros((H, D))
    wp[0, 3], wp[1, 7] = 1.0, -2.0
    q, k, w = O.indexer_projections(x, ql, wq, wk, g, b, wp, H, d, eps)
    np.testing.assert_array_equal(q.reshape(T, H * d), O.round_to_bf16(ql[:, sel]))
    np.testing.assert_array_equal(w, np.stack([x[:, 3], -2.0 * x[:, 7]], axis=1))
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x @ wk.T), (d,), torch.from_numpy(g), torch.from_numpy(b),
                                         eps=eps).numpy()
    np.testing.assert_array_equal(k, O.round_to_bf16(ref))
    # a row whose projected key is constant normalises to the bias
    x2 = np.zeros((1, D))
    wk2 = np.ones((d, D))
    _, k2, _ = O.indexer_projections(x2 + 1.0, ql[:1], wq, wk2, g, b, wp, H, d, eps)
    np.testing.assert_allclose(k2[0], O.round_to_bf16(b), rtol=0, atol=0)


# ---------------------------------------------------------------------------- attention backward

def test_sparse_attn_backward_matches_finite_differences():
    # central differences of L = sum d_o . o + sum d_lse . lse through the forward oracle; rows
    # shared by several tokens (the scatter of dkv) and -1 padding included
    rng = np.random.default_rng(41)
    T, H, D, dv, n_kv, k = 4, 2, 12, 8, 9, 5
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((n_kv, D))
    ks = np.array([0, 1, 2, 0])
    idx = np.full((T, k), -1)
    for t in range(T):
        L = int(rng.integers(2, k + 1))
        idx[t, :L] = np.sort(rng.choice(n_kv - ks[t], size=L, replace=False))
    d_o = rng.standard_normal((T, H, dv))
    d_lse = rng.standard_normal((T, H))
    scale = 0.4

    def loss(q_, kv_):
        o, lse = O.sparse_attn(q_, kv_, idx, ks, scale, d_v=dv)
        return float((d_o * o).sum() + (d_lse * lse).sum())

    dq, dkv = O.sparse_attn_backward(q, kv, idx, ks, scale, d_o, d_lse, d_v=dv)
    h = 1e-6
    fq = np.zeros_like(q)
    for i in np.ndindex(q.shape):
        qp, qm = q.copy(), q.copy()
        qp[i] += h
        qm[i] -= h
        fq[i] = (loss(qp, kv) - loss(qm, kv)) / (2 * h)
    fk = np.zeros_like(kv)
    for i in np.ndindex(kv.shape):
        kp, km = kv.copy(), kv.copy()
        kp[i] += h
        km[i] -= h
        fk[i] = (loss(q, kp) - loss(q, km)) / (2 * h)
    np.testing.assert_allclose(dq, fq, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dkv, fk, rtol=1e-6, atol=1e-7)
    # a row no token selects gets no gradient
    unused = sorted(set(range(n_kv)) - {int(ks[t]) + int(j) for t in range(T) for j in idx[t] if j >= 0})
    for r in unused:
        assert not dkv[r].any()


def test_sparse_attn_backward_single_row_closed_form():
    # one selected row: p = 1 and D = dp, so ds = d_lse exactly; with no d_lse dq vanishes and
    # the row's value dims receive d_o summed over heads
    rng = np.random.default_rng(43)
    T, H, D, dv, n_kv = 3, 4, 10, 6, 7
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((n_kv, D))
    ks = np.array([0, 2, 1])
    idx = np.array([[3, -1, -1], [0, -1, -1], [5, -1, -1]])
    d_o = rng.standard_normal((T, H, dv))
    d_lse = rng.standard_normal((T, H))
    scale = 0.7
    dq, dkv = O.sparse_attn_backward(q, kv, idx, ks, scale, d_o, d_v=dv)
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)
    want = np.zeros_like(kv)
    for t in range(T):
        want[ks[t] + idx[t, 0], :dv] += d_o[t].sum(axis=0)
    np.testing.assert_allclose(dkv, want, atol=1e-12)
    dq, dkv = O.sparse_attn_backward(q, kv, idx, ks, scale, d_o, d_lse, d_v=dv)
    for t in range(T):
        r = ks[t] + idx[t, 0]
        np.testing.assert_allclose(dq[t], scale * d_lse[t][:, None] * kv[r][None, :], atol=1e-12)
        want[r] += scale * d_lse[t] @ q[t]
    np.testing.assert_allclose(dkv, want, atol=1e-12)


def test_sparse_attn_backward_identical_rows_closed_form():
    # n selected rows with equal contents: p = 1/n and dp_j = D for every j, so ds = 0: dq
    # vanishes and each row receives d_o / n (summed over heads) on its value dims only
    rng = np.random.default_rng(44)
    H, D, dv, n = 3, 10, 6, 4
    q = rng.standard_normal((1, H, D))
    row = rng.standard_normal(D)
    kv = np.tile(row, (n + 2, 1))
    idx = np.array([[0, 2, 3, 5]])
    d_o = rng.standard_normal((1, H, dv))
    dq, dkv = O.sparse_attn_backward(q, kv, idx, np.array([0]), 0.5, d_o, d_v=dv)
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)
    for r in range(n + 2):
        want = np.zeros(D)
        if r in (0, 2, 3, 5):
            want[:dv] = d_o[0].sum(axis=0) / n
        np.testing.assert_allclose(dkv[r], want, atol=1e-12)


def test_rope_inverse_frequencies_closed_form():
    # theta^(-2i/r): pair 0 turns once per position, consecutive pairs differ by theta^(-2/r),
    # and the last pair sits at theta^(-(r-2)/r); a rotary width must be even
    for r, theta in ((64, 8e6), (32, 1e4), (2, 5.0)):
        f = O.rope_inv_freq(r, theta)
        assert f.shape == (r // 2,) and f[0] == 1.0
        np.testing.assert_allclose(f[1:] / f[:-1], theta ** (-2.0 / r), rtol=1e-14)
        np.testing.assert_allclose(f[-1], theta ** (-(r - 2) / r), rtol=1e-14)
    with pytest.raises(ValueError):
        O.rope_inv_freq(63, 1e4)


# ---------------------------------------------------------------------------- indexer backward

def _indexer_bwd_case(seed, n_q=5, n_kv=14, H=3, d=8, r=4, k=6):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n_q, H, d))
    kk = rng.standard_normal((n_kv, d))
    w = rng.standard_normal((n_q, H))
    q_pos = rng.integers(0, 50, n_q)
    k_pos = rng.integers(0, 50, n_kv)
    ks = rng.integers(0, 3, n_q)
    idx = np.full((n_q, k), -1)
    for t in range(n_q):
        n = int(rng.integers(1, k + 1))
        idx[t, :n] = np.sort(rng.choice(n_kv - ks[t], size=n, replace=False))
    g = rng.standard_normal((n_q, k))
    return q, kk, w, q_pos, k_pos, ks, idx, g


def _indexer_loss(q, kk, w, q_pos, k_pos, ks, idx, g, r, theta):
    # L = sum over selected entries of g * s, through the oracle's own forward (no rounding)
    k_rot = O.rope_rotate_f64(kk, k_pos, r, theta)
    total = 0.0
    for t in range(q.shape[0]):
        q_rot = O.rope_rotate_f64(q[t], np.full(q.shape[1], q_pos[t]), r, theta)
        s = O.indexer_scores_row(q_rot, k_rot[ks[t]:], w[t])
        for n, j in enumerate(idx[t]):
            if j >= 0:
                total += g[t, n] * s[j]
    return total


def test_indexer_backward_matches_finite_differences():
    # central differences of sum g * s through indexer_scores_row and the rotation, keys shared
    # by several queries (the scatter of dk) and -1 padding included
    r, theta = 4, 1e4
    q, kk, w, q_pos, k_pos, ks, idx, g = _indexer_bwd_case(7)
    args = (q_pos, k_pos, ks, idx, g, r, theta)
    dq, dk, dw = O.indexer_backward(q, kk, w, q_pos, k_pos, ks, idx, g, r, theta, round_rotated=False)
    h = 1e-6
    num = []
    for arr, pos in ((q, 0), (kk, 1), (w, 2)):
        f = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[i] += h
            am[i] -= h
            vp = [q, kk, w]
            vm = [q, kk, w]
            vp[pos], vm[pos] = ap, am
            f[i] = (_indexer_loss(*vp, *args) - _indexer_loss(*vm, *args)) / (2 * h)
        num.append(f)
    np.testing.assert_allclose(dq, num[0], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dk, num[1], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, num[2], rtol=1e-6, atol=1e-7)
    used = {int(ks[t]) + int(j) for t in range(q.shape[0]) for j in idx[t] if j >= 0}
    for row in set(range(kk.shape[0])) - used:
        assert not dk[row].any()


def test_indexer_backward_single_head_is_relu_matmul_autograd():
    # H_I = 1, w = 1, no RoPE: s = relu(q . k_j), differentiated by torch autograd
    rng = np.random.default_rng(3)
    n_q, n_kv, d, k = 4, 9, 6, 5
    q = rng.standard_normal((n_q, 1, d))
    kk = rng.standard_normal((n_kv, d))
    w = np.ones((n_q, 1))
    ks = np.zeros(n_q, dtype=np.int64)
    idx = np.stack([np.sort(rng.choice(n_kv, size=k, replace=False)) for _ in range(n_q)])
    g = rng.standard_normal((n_q, k))
    dq, dk, dw = O.indexer_backward(q, kk, w, np.zeros(n_q), np.zeros(n_kv), ks, idx, g, 0, 1e4,
                                    rope_q=False, rope_k=False)
    tq = torch.tensor(q[:, 0], dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(kk, dtype=torch.float64, requires_grad=True)
    s = torch.relu(tq @ tk.T)                                # [n_q, n_kv]
    sel = torch.gather(s, 1, torch.tensor(idx))
    (sel * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(dq[:, 0], tq.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw[:, 0], (torch.gather(s, 1, torch.tensor(idx)).detach().numpy() * g).sum(1),
                               rtol=1e-12)


def test_indexer_backward_euler_identity_and_row_subsets():
    # s is positively homogeneous of degree 1 in each of q~, k~ and w, so
    # sum q~.dq~ = sum k~.dk~ = sum w.dw = sum g s; the rotation is orthogonal, so the same
    # holds for the unrotated q, k and their gradients (no rounding).  Row and key subsets
    # return the matching slices of the full result.
    r, theta = 4, 1e4
    q, kk, w, q_pos, k_pos, ks, idx, g = _indexer_bwd_case(11, n_q=6, n_kv=16, H=4, d=8, k=7)
    L = _indexer_loss(q, kk, w, q_pos, k_pos, ks, idx, g, r, theta)
    dq, dk, dw = O.indexer_backward(q, kk, w, q_pos, k_pos, ks, idx, g, r, theta, round_rotated=False)
    assert abs(float((q * dq).sum()) - L) <= 1e-10 * max(1.0, abs(L))
    assert abs(float((kk * dk).sum()) - L) <= 1e-10 * max(1.0, abs(L))
    assert abs(float((w * dw).sum()) - L) <= 1e-10 * max(1.0, abs(L))
    rows, keys = [4, 1], [3, 0, 15]
    dq2, dk2, dw2 = O.indexer_backward(q, kk, w, q_pos, k_pos, ks, idx, g, r, theta, round_rotated=False,
                                       rows=rows, key_rows=keys)
    np.testing.assert_allclose(dq2, dq[rows], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dw2, dw[rows], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk2, dk[keys], rtol=1e-13, atol=1e-15)
