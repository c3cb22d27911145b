"""GPU test of dsa_indexer_topk_static, the entry point for callers that cannot allocate.

Some callers cannot give the library a workspace (a plugin handed only its input and
output buffers by a host framework that owns the allocator, or a loop that cannot afford
cudaMalloc's implicit synchronisation).  dsa_indexer_topk_static runs the same kernels on
a static device array instead.  This test calls it through the C ABI twice in a row and
checks both results against the workspace entry point.  The file is named so that pytest
collects it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()


def _inputs(w, geo):
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    L = synth.layer_inputs(w, geo, 0, device=dev, with_attn=False)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(dev)
    desc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len,
                          D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    return desc, L, t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke), rope


@pytest.mark.parametrize("n_q", [256, 1024])
def test_static_scratch_matches_workspace_entry_point_twice(n_q):
    w = synth.WORKLOADS["tiny"].replace(n_q=n_q, topk=48)
    geo = synth.geometry(w)
    desc, L, q_pos, k_pos, ks, ke, rope = _inputs(w, geo)
    ref_idx = torch.empty((w.n_q, w.topk), dtype=torch.int32, device="cuda")
    ref_sc = torch.empty((w.n_q, w.topk), dtype=torch.float32, device="cuda")
    ws = D.dsa_indexer_topk(desc, L["q_idx"], L["k_idx"], L["w"], q_pos, k_pos, ks, ke, rope, ref_idx, ref_sc)
    assert D.dsa_workspace_status(ws) == 0
    lib = D.lib()
    for call in range(2):
        idx = torch.full((w.n_q, w.topk), -7, dtype=torch.int32, device="cuda")
        sc = torch.zeros((w.n_q, w.topk), dtype=torch.float32, device="cuda")
        st = lib.dsa_indexer_topk_static(C.byref(desc), L["q_idx"].data_ptr(), L["k_idx"].data_ptr(),
                                         L["w"].data_ptr(), q_pos.data_ptr(), k_pos.data_ptr(), ks.data_ptr(),
                                         ke.data_ptr(), rope.data_ptr(), rope.shape[0], idx.data_ptr(),
                                         sc.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, lib.dsa_last_error().decode()
        torch.cuda.synchronize()
        # the same kernels on the same inputs: indices identical, scores within the tests' tolerance
        assert torch.equal(idx, ref_idx), f"call {call}: indices differ"
        fin = torch.isfinite(ref_sc)
        assert torch.equal(torch.isfinite(sc), fin)
        np.testing.assert_allclose(sc[fin].cpu().numpy(), ref_sc[fin].cpu().numpy(), rtol=2e-3, atol=1e-6)


def test_static_scratch_rejects_problems_beyond_its_size():
    w = synth.WORKLOADS["prefill_4k"]
    desc = D.indexer_desc(w.n_q, w.n_q, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, w.n_q,
                          D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    assert D.dsa_indexer_workspace_size(desc) > (32 << 20)
    z = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = z.data_ptr()
    lib = D.lib()
    st = lib.dsa_indexer_topk_static(C.byref(desc), p, p, p, p, p, p, p, p, 1, p, None,
                                     torch.cuda.current_stream().cuda_stream)
    assert _lib.STATUS_NAMES[st] == "DSA_ERR_WORKSPACE"


def test_static_scratch_reports_device_faults_through_its_status_query():
    """A key range outside [0, n_kv) is flagged on the device; the static variant's status
    query reports it, and the next clean call clears it."""
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    desc, L, q_pos, k_pos, ks, ke, rope = _inputs(w, geo)
    idx = torch.empty((w.n_q, w.topk), dtype=torch.int32, device="cuda")
    bad_ke = ke.clone()
    bad_ke[5] = geo.n_kv + 10
    D.dsa_indexer_topk_static(desc, L["q_idx"], L["k_idx"], L["w"], q_pos, k_pos, ks, bad_ke, rope, idx)
    bits = D.dsa_indexer_static_status(raise_on_fault=False)
    assert bits != 0
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_static_status()
    assert e.value.name == "DSA_ERR_DEVICE"
    D.dsa_indexer_topk_static(desc, L["q_idx"], L["k_idx"], L["w"], q_pos, k_pos, ks, ke, rope, idx)
    assert D.dsa_indexer_static_status() == 0
