"""GPU parity: the C-ABI path (libdsa.so) against the float64 oracle on the same bytes.

Top-k: the tie rule of tests/parity.py.  Attention: max-abs <= 1e-2 against the oracle fed
the GPU's own indices, on unit-scale inputs (N(0,1) q / kv) and on the workloads'
N(0,1)/sqrt(576) inputs (relative to the output's scale there).
"""
import math

import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV, attn_errors, oracle_attn, oracle_scores, run_attn, run_indexer
from parity import check_topk

pytestmark = pytest.mark.gpu

ATOL_OUT = 1e-2
# The softmax weights enter the second product as bf16 (relative rounding <= 2^-9) and the
# denominator sums those same rounded weights, so the log-sum-exp the kernel reports is
# log(sum of rounded weights): within log(1 + 2^-9) ~ 2e-3 of the exact value, plus fp32
# accumulation error.  4e-3 leaves a factor 2.
ATOL_LSE = 4e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()
    assert torch.cuda.is_available()


def _check_indexer(w, geo, L, rows):
    idx, sc, bits = run_indexer(w, geo, L, want_scores=True)
    assert bits == 0, f"device status bits {bits:#x}"
    score_rows = oracle_scores(w, geo, L, rows)
    idx_np = idx.cpu().numpy()
    bad = check_topk(idx_np, score_rows, w.topk, rows)
    assert not bad, f"{len(bad)} rows violate the top-k rule, first: {bad[:3]}"
    # reported scores of the selected keys agree with the oracle's
    sc_np = sc.cpu().numpy()
    for n, t in enumerate(rows):
        sel = idx_np[t][idx_np[t] >= 0]
        ref = score_rows[n][sel]
        got = sc_np[t][: sel.size]
        if sel.size:
            np.testing.assert_allclose(got, ref, rtol=2e-3, atol=2e-3 * (np.abs(ref).max() + 1e-30))
        assert np.all(np.isneginf(sc_np[t][sel.size:]))
    return idx


def test_indexer_tiny_every_row():
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device=DEV)
    _check_indexer(w, geo, L, list(range(w.n_q)))


def test_indexer_prefill_4k_sampled_rows():
    w = synth.WORKLOADS["prefill_4k"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device=DEV, with_attn=False)
    _check_indexer(w, geo, L, synth.sample_rows(w.n_q, 192, w.topk))


@pytest.mark.parametrize("H_I,d,r,topk", [(16, 128, 64, 100), (64, 128, 64, 300), (8, 64, 16, 1), (32, 64, 0, 2048)])
def test_indexer_ragged_ranges(H_I, d, r, topk):
    # rows not a multiple of the group, empty rows, rows shorter than k, ragged key tail
    rng = np.random.default_rng(H_I + topk)
    n_q, n_kv = 77, 2600
    ks = rng.integers(0, 600, n_q).astype(np.int32)
    ln = rng.integers(0, 2000, n_q)
    ln[[0, 5, 40]] = 0
    ln[7] = 2000
    ke = np.minimum(ks + ln, n_kv).astype(np.int32)
    geo = synth.Geometry(n_kv, rng.integers(0, 5000, n_q).astype(np.int32), rng.integers(0, 5000, n_kv).astype(np.int32),
                         ks, ke)
    w = synth.Workload("ragged", "prefill", n_q, ("full",), H_I, d, r, 1e4, topk, 4)
    L = synth.layer_inputs(w, geo, 0, device=DEV, with_attn=False)
    _check_indexer(w, geo, L, list(range(n_q)))


@pytest.mark.parametrize("topk", [512, 2048])
def test_indexer_filtered_rows_in_the_dense_select(topk):
    """Rows of 4100-8192 keys in one chunk (608 groups of 4 rows: the chunk is the whole row):
    the indexer filters them (more than 4096 keys in the chunk), so the final select sees only
    the keys at or above each row's threshold, and since no row is longer than 8192 keys it
    takes the dense path (one score key per offset of the row), where many offsets hold no
    entry.  With and without scores requested, the same keys are selected."""
    rng = np.random.default_rng(31 + topk)
    n_q, n_kv = 2432, 8192
    ks = np.zeros(n_q, np.int32)
    ke = rng.integers(4100, n_kv + 1, n_q).astype(np.int32)
    ke[3] = n_kv
    geo = synth.Geometry(n_kv, rng.integers(0, 9000, n_q).astype(np.int32),
                         rng.integers(0, 9000, n_kv).astype(np.int32), ks, ke)
    w = synth.Workload("filtered", "prefill", n_q, ("full",), 64, 128, 64, 1e4, topk, 4)
    L = synth.layer_inputs(w, geo, 0, device=DEV, with_attn=False)
    idx = _check_indexer(w, geo, L, [0, 3, 100, 777, 1500, n_q - 1] + list(range(5, n_q, 97)))
    idx2, _, bits = run_indexer(w, geo, L, want_scores=False)
    assert bits == 0 and torch.equal(idx, idx2)


def test_indexer_independent_rows_decode_shape():
    # batched decode: each row is its own sequence in a packed, already-rotated key cache
    w = synth.Workload("decode_small", "decode", 6, ("full",), 64, 128, 64, 8e6, 256, 8, n_seqs=6, len_lo=1,
                       len_hi=3000, rope_k=False)
    geo = synth.geometry(w, seed=5)
    L = synth.layer_inputs(w, geo, 0, device=DEV, with_attn=False)
    _check_indexer(w, geo, L, list(range(w.n_q)))


def _attn_case(w, geo, idx, rows, attn_scale, layer=1):
    L = synth.layer_inputs(w, geo, layer, device=DEV, attn_scale=attn_scale)
    out, lse, bits = run_attn(w, geo, L, idx)
    assert bits == 0, f"device status bits {bits:#x}"
    o_ref, lse_ref = oracle_attn(w, geo, L, idx.cpu().numpy(), rows)
    e_o, e_l = attn_errors(out, lse, o_ref, lse_ref, rows)
    return e_o, e_l, float(np.abs(o_ref).max())


@pytest.mark.parametrize("name", ["tiny", "prefill_4k"])
def test_attention_unit_scale_and_config_scale(name):
    w = synth.WORKLOADS[name]
    geo = synth.geometry(w)
    Li = synth.layer_inputs(w, geo, 0, device=DEV, with_attn=False)
    idx, _, bits = run_indexer(w, geo, Li)
    assert bits == 0
    rows = list(range(w.n_q)) if w.n_q <= 256 else synth.sample_rows(w.n_q, 96, w.topk)
    e_o, e_l, _ = _attn_case(w, geo, idx, rows, "unit")
    assert e_o <= ATOL_OUT and e_l <= ATOL_LSE, (e_o, e_l)
    e_o, e_l, scale = _attn_case(w, geo, idx, rows, "config")
    assert e_o <= ATOL_OUT * scale and e_l <= ATOL_LSE, (e_o, e_l, scale)


@pytest.mark.parametrize("H", [1, 4, 16, 40, 64, 128])
def test_attention_head_blocks_and_bad_indices(H):
    rng = np.random.default_rng(H)
    n_q, n_kv, topk = 9, 700, 200
    ks = rng.integers(0, 100, n_q).astype(np.int32)
    idx = np.stack([rng.permutation(600)[:topk] for _ in range(n_q)]).astype(np.int32)   # distinct offsets
    idx[rng.random((n_q, topk)) < 0.2] = -1          # scattered unused slots
    idx[2, :] = -1                                   # a row with nothing selected
    idx[3, 150:] = -1                                # a ragged row
    idx[4, 7] = 650                                  # ks + 650 >= n_kv for ks >= 50 -> skipped, counted
    geo = synth.Geometry(n_kv, np.zeros(n_q, np.int32), np.zeros(n_kv, np.int32), ks, ks)
    w = synth.Workload("heads", "prefill", n_q, ("full", "shared"), 4, 64, 0, 1e4, topk, H)
    L = synth.layer_inputs(w, geo, 1, device=DEV, attn_scale="unit")
    out, lse, bits = run_attn(w, geo, L, torch.from_numpy(idx).to(DEV))
    bad_expected = int(ks[4]) + 650 >= n_kv
    assert (bits != 0) == bad_expected
    idx_ref = idx.copy()
    if bad_expected:
        idx_ref[4, 7] = -1
    o_ref, lse_ref = oracle_attn(w, geo, L, idx_ref, range(n_q))
    e_o, e_l = attn_errors(out, lse, o_ref, lse_ref, range(n_q))
    assert e_o <= ATOL_OUT and e_l <= ATOL_LSE, (e_o, e_l)
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))


@pytest.mark.parametrize("name", ["tiny", "prefill_4k"])
def test_layers_forward_against_oracle(name):
    w = synth.WORKLOADS[name]
    geo = synth.geometry(w)
    q_pos, k_pos, ks, ke = (torch.from_numpy(a).to(DEV) for a in (geo.q_pos, geo.k_pos, geo.ks, geo.ke))
    layers = []
    for l in range(len(w.layers)):
        L = synth.layer_inputs(w, geo, l, device=DEV, attn_scale="unit")
        L["out"] = torch.empty((w.n_q, w.n_heads, 512), dtype=torch.bfloat16, device=DEV)
        L["lse"] = torch.empty((w.n_q, w.n_heads), dtype=torch.float32, device=DEV)
        layers.append(L)
    cache = D.IndexCache(w.layers, w.n_q, w.topk)
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len,
                           D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)
    ws = D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache)
    assert D.dsa_workspace_status(ws) == 0
    donors = D.dsa_donor_table(w.layers)
    rows = list(range(w.n_q)) if w.n_q <= 256 else synth.sample_rows(w.n_q, 48, w.topk)
    for l, t in enumerate(w.layers):
        assert cache.donor(l) == donors[l]
        assert cache.indices_ptr(l) == cache.buffers[donors[l]].data_ptr()
        if t == "full":
            score_rows = oracle_scores(w, geo, layers[l], rows)
            bad = check_topk(cache.buffers[l].cpu().numpy(), score_rows, w.topk, rows)
            assert not bad, (l, bad[:3])
        idx_np = cache.buffers[donors[l]].cpu().numpy()
        o_ref, lse_ref = oracle_attn(w, geo, layers[l], idx_np, rows)
        e_o, e_l = attn_errors(layers[l]["out"], layers[l]["lse"], o_ref, lse_ref, rows)
        assert e_o <= ATOL_OUT and e_l <= ATOL_LSE, (l, e_o, e_l)
    cache.close()


@pytest.mark.parametrize("H", [4, 16])
def test_attention_gather_walk_for_small_heads(H):
    # a long key range with a short index row takes the per-token gather walk
    rng = np.random.default_rng(100 + H)
    n_q, n_kv, topk = 37, 5000, 128
    ks = rng.integers(0, 1000, n_q).astype(np.int32)
    idx = np.stack([rng.permutation(3900)[:topk] for _ in range(n_q)]).astype(np.int32)
    idx[rng.random((n_q, topk)) < 0.1] = -1
    idx[5, :] = -1
    geo = synth.Geometry(n_kv, np.zeros(n_q, np.int32), np.zeros(n_kv, np.int32), ks, ks)
    w = synth.Workload("gather", "prefill", n_q, ("full", "shared"), 4, 64, 0, 1e4, topk, H)
    L = synth.layer_inputs(w, geo, 1, device=DEV, attn_scale="unit")
    out, lse, bits = run_attn(w, geo, L, torch.from_numpy(idx).to(DEV))
    assert bits == 0
    o_ref, lse_ref = oracle_attn(w, geo, L, idx, range(n_q))
    e_o, e_l = attn_errors(out, lse, o_ref, lse_ref, range(n_q))
    assert e_o <= ATOL_OUT and e_l <= ATOL_LSE, (e_o, e_l)
    assert torch.all(out[5] == 0) and torch.all(torch.isneginf(lse[5]))


@pytest.mark.parametrize("H", [64, 128])
def test_attention_gather_walk_split_over_ctas(H):
    # few tokens with long index rows: each (token, head block) is split over several CTAs whose
    # partial outputs a combine pass merges; rows of 1 to 32 tiles give splits with no tile at
    # all, one token selects nothing
    rng = np.random.default_rng(200 + H)
    n_q, n_kv, topk = 5, 9000, 2048
    ks = rng.integers(0, 500, n_q).astype(np.int32)
    idx = np.full((n_q, topk), -1, dtype=np.int32)
    lengths = [2048, 1, 300, 0, 1111]
    for t, L in enumerate(lengths):
        idx[t, :L] = rng.permutation(8000)[:L]
    idx[0, rng.random(topk) < 0.05] = -1     # scattered unused slots
    geo = synth.Geometry(n_kv, np.zeros(n_q, np.int32), np.zeros(n_kv, np.int32), ks, ks)
    w = synth.Workload("split", "decode", n_q, ("full", "shared"), 4, 64, 0, 1e4, topk, H)
    L = synth.layer_inputs(w, geo, 1, device=DEV, attn_scale="unit")
    out, lse, bits = run_attn(w, geo, L, torch.from_numpy(idx).to(DEV))
    assert bits == 0
    o_ref, lse_ref = oracle_attn(w, geo, L, idx, range(n_q))
    e_o, e_l = attn_errors(out, lse, o_ref, lse_ref, range(n_q))
    assert e_o <= ATOL_OUT and e_l <= ATOL_LSE, (e_o, e_l)
    assert torch.all(out[3] == 0) and torch.all(torch.isneginf(lse[3]))
    # the same call without lse writes the same output
    out2, _, bits2 = run_attn(w, geo, L, torch.from_numpy(idx).to(DEV), lse=False)
    assert bits2 == 0 and torch.equal(out, out2)


def test_indexer_rising_scores_cut_back_the_buffer():
    """Scores that rise along the keys beat every streaming threshold, so a long row's
    candidate buffer fills up and has to be cut back to its exact top-k (ties to the lower
    key index) again and again; the result is still exactly the oracle's set.  Here every
    head sees s_j = k_j[0], which rises with j in steps of bf16 rounding, so long runs of
    equal scores exercise the tie rule as well.  The buffers have room for every key of a
    chunk up to 64K keys, so the rows here span one chunk of up to 100K keys: a lane quarter
    of it (25K keys) overflows its 16K entries."""
    from oracle import dsa_oracle as O
    n_q, n_kv, H, d, topk = 2432, 100000, 64, 128, 2048   # 608 groups of 4 rows: one chunk per row
    q = torch.zeros((n_q, H, d), dtype=torch.float32)
    q[:, :, 0] = 1.0
    k = torch.zeros((n_kv, d), dtype=torch.float32)
    k[:, 0] = (torch.arange(n_kv, dtype=torch.float32) + 1.0) / n_kv
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    w = torch.full((n_q, H), 1.0 / 64.0, dtype=torch.float32)
    ks = np.zeros(n_q, np.int32)
    ke = (n_kv - (np.arange(n_q) % 7) * 1000).astype(np.int32)
    pos = np.arange(n_kv, dtype=np.int32)
    q_pos = (ke - 1).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    desc = D.indexer_desc(n_q, n_kv, H, d, 0, topk, n_kv, 0)
    idx = torch.empty((n_q, topk), dtype=torch.int32, device=DEV)
    ws = D.dsa_indexer_topk(desc, q.to(DEV), k.to(DEV), w.to(DEV), dev(q_pos), dev(pos), dev(ks), dev(ke), None, idx)
    assert D.dsa_workspace_status(ws) == 0
    rows = [0, 1, 6, 1000, n_q - 1]
    ref = O.indexer_topk(synth.to_f64(q), synth.to_f64(k), synth.to_f64(w), q_pos, pos, ks, ke, 0, 1e4, topk,
                         rope_q=False, rope_k=False, rows=rows)
    got = idx.cpu().numpy()
    for n, t in enumerate(rows):
        assert np.array_equal(got[t], ref[n]), f"row {t}"


def test_indexer_negative_scores_use_the_signed_histogram():
    """Head weights all negative make every score <= 0, so each row's k-th largest score is
    negative: the streaming threshold must rise through the negative half of the histogram
    (a positive-only map would keep every key and cut its buffers back again and again).  Long
    filtered rows (over 4096 keys in their chunk), checked against the oracle on sampled rows
    with the near-tie rule."""
    from oracle import dsa_oracle as O
    n_q, n_kv, H, d, topk = 256, 30000, 64, 128, 512
    g = torch.Generator()
    g.manual_seed(21)
    q = (torch.randn((n_q, H, d), generator=g) / d ** 0.5).to(torch.bfloat16)
    k = (torch.randn((n_kv, d), generator=g) / d ** 0.5).to(torch.bfloat16)
    w = -torch.rand((n_q, H), generator=g) - 0.05
    ks = np.zeros(n_q, np.int32)
    ke = (n_kv - (np.arange(n_q) * 97) % 9000).astype(np.int32)
    pos = np.arange(n_kv, dtype=np.int32)
    q_pos = (ke - 1).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    desc = D.indexer_desc(n_q, n_kv, H, d, 0, topk, n_kv, 0)
    idx = torch.empty((n_q, topk), dtype=torch.int32, device=DEV)
    ws = D.dsa_indexer_topk(desc, q.to(DEV), k.to(DEV), w.to(DEV), dev(q_pos), dev(pos), dev(ks), dev(ke), None, idx)
    assert D.dsa_workspace_status(ws) == 0
    rows = [0, 1, 77, 128, n_q - 1]
    _, sr = O.indexer_topk(synth.to_f64(q), synth.to_f64(k), synth.to_f64(w), q_pos, pos, ks, ke, 0, 1e4, topk,
                           rope_q=False, rope_k=False, rows=rows, return_scores=True)
    assert all(float(np.sort(s)[-topk]) < 0.0 for s in sr), "the k-th largest score should be negative"
    bad = check_topk(idx.cpu().numpy(), sr, topk, rows)
    assert not bad, bad
