"""The IndexShare layer loop on inputs held in pinned host memory, with transfers overlapped.

Every step still runs in libdsa's kernels through the C ABI (dsa_indexer_topk on full layers,
dsa_sparse_attn on every layer, each layer attending with its donor's indices, as
indexshare_layers_forward does).  What this adds is the schedule of the transfers around
them: layer l's inputs are uploaded on an upload stream while earlier layers compute, and
layer l's output is downloaded on a download stream as soon as its attention is done, so the
two copy directions and the kernels overlap instead of running one after the other.
"""
from __future__ import annotations

from typing import Sequence

import torch

from . import _lib as L

_IN_KEYS = ("q_idx", "k_idx", "w", "q", "kv")


class HostLayerPipeline:
    """Device buffers and streams for repeated host-to-host layer-loop calls of one shape.

    host_layers[l]: pinned CPU tensors 'q', 'kv' (every layer) and 'q_idx', 'k_idx', 'w' (full
    layers); host_out[l]: pinned CPU tensor [n_q, n_heads, 512] bf16 that receives layer l's
    attention output.
    """

    def __init__(self, idesc: L.IndexerDesc, adesc: L.AttnDesc, indexer_types: Sequence, host_layers: Sequence[dict],
                 device):
        self.idesc, self.adesc = idesc, adesc
        self.types = L.types_to_u8(indexer_types)
        self.donors = L.dsa_donor_table(indexer_types)
        self.device = torch.device(device)
        self.dev = [{k: torch.empty_like(v, device=self.device) for k, v in H.items() if k in _IN_KEYS}
                    for H in host_layers]
        n_q, topk = idesc.n_q, idesc.topk
        self.idx = {l: torch.empty((n_q, topk), dtype=torch.int32, device=self.device)
                    for l, t in enumerate(self.types) if t == L.DSA_LAYER_FULL}
        self.out = [torch.empty((adesc.n_q, adesc.n_heads, adesc.d_v), dtype=torch.bfloat16, device=self.device)
                    for _ in host_layers]
        self.iws = torch.empty(L.dsa_indexer_workspace_size(idesc), dtype=torch.uint8, device=self.device)
        self.aws = torch.empty(L.dsa_sparse_attn_workspace_size(adesc), dtype=torch.uint8, device=self.device)
        self.up = torch.cuda.Stream(device=self.device)
        self.down = torch.cuda.Stream(device=self.device)

    def forward(self, host_layers: Sequence[dict], host_out: Sequence[torch.Tensor], ks, ke, q_pos, k_pos, rope_cs,
                stream=None) -> torch.cuda.Event:
        """Enqueue one pass; returns an event on `stream` (default: the current stream) that
        completes once every output has reached host memory.  Work starts after everything
        already enqueued on `stream`."""
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        start = torch.cuda.Event()
        start.record(st)
        self.up.wait_event(start)
        self.down.wait_event(start)
        uploaded = []
        with torch.cuda.stream(self.up):
            for H, Dv in zip(host_layers, self.dev):
                for k, v in Dv.items():
                    v.copy_(H[k], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(self.up)
                uploaded.append(ev)
        for l, t in enumerate(self.types):
            st.wait_event(uploaded[l])
            Dv = self.dev[l]
            if t == L.DSA_LAYER_FULL:
                L.dsa_indexer_topk(self.idesc, Dv["q_idx"], Dv["k_idx"], Dv["w"], q_pos, k_pos, ks, ke, rope_cs,
                                   self.idx[l], None, ws=self.iws, stream=st)
            L.dsa_sparse_attn(self.adesc, Dv["q"], Dv["kv"], self.idx[self.donors[l]], ks, self.out[l], None,
                              ws=self.aws, stream=st)
            done = torch.cuda.Event()
            done.record(st)
            self.down.wait_event(done)
            with torch.cuda.stream(self.down):
                host_out[l].copy_(self.out[l], non_blocking=True)
        finished = torch.cuda.Event()
        finished.record(self.down)
        st.wait_event(finished)
        end = torch.cuda.Event()
        end.record(st)
        return end
