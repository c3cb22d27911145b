"""Shared helpers of the GPU parity tests: run the C-ABI path and the oracle on the same bytes."""
from __future__ import annotations

import math

import numpy as np
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from oracle import dsa_oracle as O

DEV = "cuda"


def device_geometry(geo: synth.Geometry):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke)


def rope_table_dev(w: synth.Workload, geo: synth.Geometry):
    if w.rope_dim == 0:
        return None
    return D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)


def run_indexer(w: synth.Workload, geo: synth.Geometry, L: dict, want_scores: bool = False):
    q_pos, k_pos, ks, ke = device_geometry(geo)
    flags = D.DSA_IDX_ROPE_Q | (D.DSA_IDX_ROPE_K if w.rope_k else 0)
    if w.kind == "decode":
        flags |= D.DSA_IDX_INDEPENDENT_ROWS
    desc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, max(1, geo.max_len), flags)
    idx = torch.empty((w.n_q, w.topk), dtype=torch.int32, device=DEV)
    sc = torch.empty((w.n_q, w.topk), dtype=torch.float32, device=DEV) if want_scores else None
    ws = D.dsa_indexer_topk(desc, L["q_idx"], L["k_idx"], L["w"], q_pos, k_pos, ks, ke, rope_table_dev(w, geo), idx, sc)
    bits = D.dsa_workspace_status(ws, raise_on_fault=False)
    return idx, sc, bits


def oracle_scores(w: synth.Workload, geo: synth.Geometry, L: dict, rows):
    """Oracle score rows for `rows`, one row at a time on that row's own key slice.

    Only the row's query heads and its key range [ks_t, ke_t) are moved to the host, so the
    largest workloads (a million keys, or a 4.5 M-row decode cache) stay within host memory.
    """
    out = []
    for t in rows:
        a, b = int(geo.ks[t]), int(geo.ke[t])
        q_t = synth.to_f64(L["q_idx"][t:t + 1])
        w_t = synth.to_f64(L["w"][t:t + 1])
        k_sub = synth.to_f64(L["k_idx"][a:b]) if b > a else np.zeros((0, w.head_dim_idx))
        _, sr = O.indexer_topk(q_t, k_sub, w_t, geo.q_pos[t:t + 1], geo.k_pos[a:b], np.zeros(1, np.int64),
                               np.array([b - a]), w.rope_dim, w.theta, w.topk, rope_q=True, rope_k=w.rope_k,
                               return_scores=True)
        out.append(sr[0])
    return out


def run_attn(w: synth.Workload, geo: synth.Geometry, L: dict, idx: torch.Tensor, lse: bool = True):
    ks = torch.from_numpy(geo.ks).to(DEV)
    desc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    out = torch.empty((w.n_q, w.n_heads, 512), dtype=torch.bfloat16, device=DEV)
    lse_t = torch.empty((w.n_q, w.n_heads), dtype=torch.float32, device=DEV) if lse else None
    ws = D.dsa_sparse_attn(desc, L["q"], L["kv"], idx, ks, out, lse_t)
    bits = D.dsa_workspace_status(ws, raise_on_fault=False)
    return out, lse_t, bits


def oracle_attn(w: synth.Workload, geo: synth.Geometry, L: dict, idx_np: np.ndarray, rows):
    rows = list(rows)
    q = L["q"][torch.as_tensor(rows, device=L["q"].device)]
    q64 = synth.to_f64(q)
    kv64 = synth.to_f64(L["kv"])
    o = np.zeros((len(rows), w.n_heads, 512))
    lse = np.zeros((len(rows), w.n_heads))
    for n, t in enumerate(rows):
        o[n], lse[n] = O.sparse_attn_row(q64[n], kv64, idx_np[t], int(geo.ks[t]), w.softmax_scale)
    return o, lse


def attn_errors(out: torch.Tensor, lse_t, o_ref: np.ndarray, lse_ref: np.ndarray, rows):
    rows = list(rows)
    got = synth.to_f64(out[torch.as_tensor(rows, device=out.device)])
    err_o = float(np.max(np.abs(got - o_ref))) if got.size else 0.0
    err_l = 0.0
    if lse_t is not None:
        gl = lse_t[torch.as_tensor(rows, device=out.device)].double().cpu().numpy()
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(gl), fin), "lse finiteness differs"
        err_l = float(np.max(np.abs(gl[fin] - lse_ref[fin]))) if fin.any() else 0.0
    return err_o, err_l
