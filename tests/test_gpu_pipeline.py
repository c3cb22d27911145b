"""The host pipeline (dsa_indexer_cross_gb300.pipeline) against the device-resident layer loop.

Same kernels, same order on the compute stream, only the transfers move to other streams: the
outputs that reach host memory must equal indexshare_layers_forward's bit for bit, over two
consecutive passes (the second uses the other device set), and over three passes enqueued back
to back (each uploads while the one before computes; the third reuses the first one's set).
"""
import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from dsa_indexer_cross_gb300.pipeline import HostLayerPipeline
from gpu_cases import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", ["tiny", "prefill_4k"])
def test_host_pipeline_equals_device_layer_loop(name):
    w = synth.WORKLOADS[name]
    geo = synth.geometry(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    q_pos, k_pos, ks, ke = t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke)
    layers = []
    for l in range(len(w.layers)):
        L = synth.layer_inputs(w, geo, l, device=DEV, attn_scale="unit")
        L["out"] = torch.empty((w.n_q, w.n_heads, 512), dtype=torch.bfloat16, device=DEV)
        layers.append(L)
    cache = D.IndexCache(w.layers, w.n_q, w.topk, device=DEV)
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len,
                           D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)
    ws = D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache)
    assert D.dsa_workspace_status(ws) == 0
    host_in = [{k: v.cpu().pin_memory() for k, v in L.items() if k in ("q_idx", "k_idx", "w", "q", "kv")}
               for L in layers]
    host_out = [torch.zeros(L["out"].shape, dtype=torch.bfloat16).pin_memory() for L in layers]
    pipe = HostLayerPipeline(idesc, adesc, w.layers, host_in, DEV)
    for _ in range(2):
        for h in host_out:
            h.zero_()
        pipe.forward(host_in, host_out, ks, ke, q_pos, k_pos, rope).synchronize()
        assert D.dsa_workspace_status(pipe.iws) == 0 and D.dsa_workspace_status(pipe.aws) == 0
        for l, L in enumerate(layers):
            assert torch.equal(host_out[l], L["out"].cpu()), f"layer {l}"
    cache.close()


def test_back_to_back_passes_overlap_without_hazards():
    """Three passes enqueued without a host sync between them, each with its own inputs (another
    seed per pass) and its own host outputs: every pass must produce exactly what the
    device-resident loop gives on its inputs."""
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    q_pos, k_pos, ks, ke = t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke)
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len,
                           D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(DEV)
    passes, expected = [], []
    for p in range(3):
        layers = []
        for l in range(len(w.layers)):
            L = synth.layer_inputs(w, geo, l, seed=1234 + 17 * p, device=DEV, attn_scale="unit")
            L["out"] = torch.empty((w.n_q, w.n_heads, 512), dtype=torch.bfloat16, device=DEV)
            layers.append(L)
        cache = D.IndexCache(w.layers, w.n_q, w.topk, device=DEV)
        ws = D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache)
        assert D.dsa_workspace_status(ws) == 0
        expected.append([L["out"].cpu() for L in layers])
        cache.close()
        passes.append([{k: v.cpu().pin_memory() for k, v in L.items() if k in ("q_idx", "k_idx", "w", "q", "kv")}
                       for L in layers])
    host_out = [[torch.zeros((w.n_q, w.n_heads, 512), dtype=torch.bfloat16).pin_memory() for _ in w.layers]
                for _ in range(3)]
    pipe = HostLayerPipeline(idesc, adesc, w.layers, passes[0], DEV)
    ends = [pipe.forward(passes[p], host_out[p], ks, ke, q_pos, k_pos, rope) for p in range(3)]
    ends[-1].synchronize()
    torch.cuda.synchronize()
    assert D.dsa_workspace_status(pipe.iws) == 0 and D.dsa_workspace_status(pipe.aws) == 0
    for p in range(3):
        for l in range(len(w.layers)):
            assert torch.equal(host_out[p][l], expected[p][l]), f"pass {p} layer {l}"
