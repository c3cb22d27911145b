"""GPU parity on the large workloads at full size, on sampled query rows.

long_32k (T=32768, biased keys), decode_64 (64 independent sequences up to 131072 keys,
rotated key cache, 128 heads) and chunk_1m (4096 queries over a 1,048,576-key prefix).
The oracle computes the sampled rows one by one; attention is checked with the oracle fed
the GPU's own indices, gathering only the selected latent rows to the host.
"""
import numpy as np
import pytest
import torch

from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV, oracle_scores, run_attn, run_indexer
from oracle import dsa_oracle as O
from parity import check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()


def attn_check_rows(w, geo, L, idx, out, lse, rows):
    """Oracle attention for `rows`, moving only each row's selected latent rows to the host."""
    err_o = err_l = 0.0
    idx_np = idx.cpu().numpy()
    for t in rows:
        sel = idx_np[t][idx_np[t] >= 0].astype(np.int64) + int(geo.ks[t])
        kv_rows = synth.to_f64(L["kv"][torch.from_numpy(sel).to(DEV)]) if sel.size else np.zeros((0, 576))
        q_t = synth.to_f64(L["q"][t])
        o, l = O.sparse_attn_row(q_t, kv_rows, np.arange(sel.size), 0, w.softmax_scale)
        got = synth.to_f64(out[t])
        err_o = max(err_o, float(np.abs(got - o).max()))
        gl = lse[t].double().cpu().numpy()
        fin = np.isfinite(l)
        assert np.array_equal(np.isfinite(gl), fin)
        if fin.any():
            err_l = max(err_l, float(np.abs(gl[fin] - l[fin]).max()))
    return err_o, err_l


@pytest.mark.parametrize("name,n_rows", [("long_32k", 24), ("decode_64", 64), ("chunk_1m", 12)])
def test_full_size_workload(name, n_rows):
    w = synth.WORKLOADS[name]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device=DEV, attn_scale="unit")
    idx, _, bits = run_indexer(w, geo, L)
    assert bits == 0, f"device status {bits:#x}"
    rows = synth.sample_rows(w.n_q, n_rows, w.topk)
    score_rows = oracle_scores(w, geo, L, rows)
    bad = check_topk(idx.cpu().numpy(), score_rows, w.topk, rows)
    assert not bad, bad[:3]
    # every row selects exactly min(k, L_t) keys (all rows, not only the sampled ones)
    cnt = (idx >= 0).sum(dim=1).cpu().numpy()
    np.testing.assert_array_equal(cnt, np.minimum(w.topk, geo.ke - geo.ks))
    out, lse, bits = run_attn(w, geo, L, idx)
    assert bits == 0
    e_o, e_l = attn_check_rows(w, geo, L, idx, out, lse, rows[: max(4, n_rows // 2)])
    assert e_o <= 1e-2 and e_l <= 4e-3, (e_o, e_l)
