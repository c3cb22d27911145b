"""The IndexShare layer loop on inputs held in pinned host memory, with transfers overlapped.

Every step still runs in libdsa's kernels through the C ABI (dsa_indexer_topk on full layers,
dsa_sparse_attn on every layer, each layer attending with its donor's indices, as
indexshare_layers_forward does).  What this adds is the schedule of the transfers around
them:
- layer l's inputs are uploaded on an upload stream while earlier layers compute; a full
  layer's indexer inputs (q_idx, k_idx, w) go first and its indexer starts as soon as they
  have landed, while the attention inputs (q, kv) are still on their way;
- layer l's output is downloaded on a download stream as soon as its attention is done;
- the device copies of the inputs and outputs come in two sets used by alternate passes, so
  the next pass's uploads run while this pass's kernels still read the other set.
The two copy directions and the kernels of consecutive passes thus overlap instead of running
one after the other.
"""
from __future__ import annotations

from typing import Sequence

import torch

from . import _lib as L

_IDX_KEYS = ("q_idx", "k_idx", "w")
_ATTN_KEYS = ("q", "kv")


class HostLayerPipeline:
    """Device buffers and streams for repeated host-to-host layer-loop calls of one shape.

    host_layers[l]: pinned CPU tensors 'q', 'kv' (every layer) and 'q_idx', 'k_idx', 'w' (full
    layers); host_out[l]: pinned CPU tensor [n_q, n_heads, 512] bf16 that receives layer l's
    attention output.  n_sets device copies of the inputs and outputs (two by default: a pass
    uploads into one while the previous pass computes from the other).
    """

    def __init__(self, idesc: L.IndexerDesc, adesc: L.AttnDesc, indexer_types: Sequence, host_layers: Sequence[dict],
                 device, n_sets: int = 2):
        if n_sets < 1:
            raise ValueError("n_sets must be at least 1")
        self.idesc, self.adesc = idesc, adesc
        self.types = L.types_to_u8(indexer_types)
        self.donors = L.dsa_donor_table(indexer_types)
        self.device = torch.device(device)
        keys = _IDX_KEYS + _ATTN_KEYS
        self.dev = [[{k: torch.empty_like(v, device=self.device) for k, v in H.items() if k in keys}
                     for H in host_layers] for _ in range(n_sets)]
        n_q, topk = idesc.n_q, idesc.topk
        self.idx = {l: torch.empty((n_q, topk), dtype=torch.int32, device=self.device)
                    for l, t in enumerate(self.types) if t == L.DSA_LAYER_FULL}
        self.out = [[torch.empty((adesc.n_q, adesc.n_heads, adesc.d_v), dtype=torch.bfloat16, device=self.device)
                     for _ in host_layers] for _ in range(n_sets)]
        self.iws = torch.empty(L.dsa_indexer_workspace_size(idesc), dtype=torch.uint8, device=self.device)
        self.aws = torch.empty(L.dsa_sparse_attn_workspace_size(adesc), dtype=torch.uint8, device=self.device)
        self.up = torch.cuda.Stream(device=self.device)
        self.down = torch.cuda.Stream(device=self.device)
        self.calls = 0
        self.inputs_free = [None] * n_sets   # compute stream: the last kernel reading set s
        self.outs_free = [None] * n_sets     # download stream: the last copy out of set s

    def forward(self, host_layers: Sequence[dict], host_out: Sequence[torch.Tensor], ks, ke, q_pos, k_pos, rope_cs,
                stream=None) -> torch.cuda.Event:
        """Enqueue one pass; returns an event (on the download stream, with timing enabled) that
        completes once every output of the pass has reached host memory.  The kernels run on
        `stream` (default: the current stream) after everything already enqueued there; the
        uploads start as soon as the pass's device set is no longer read by the pass before
        the previous one.  host_layers must not change until the pass has completed, nor may
        host_out be read before then."""
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        s = self.calls % len(self.dev)
        self.calls += 1
        dev, out = self.dev[s], self.out[s]
        if self.inputs_free[s] is not None:
            self.up.wait_event(self.inputs_free[s])
        ready = []
        with torch.cuda.stream(self.up):
            for H, Dv in zip(host_layers, dev):
                evs = []
                for keys in (_IDX_KEYS, _ATTN_KEYS):
                    for k in keys:
                        if k in Dv:
                            Dv[k].copy_(H[k], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(self.up)
                    evs.append(ev)
                ready.append(evs)
        if self.outs_free[s] is not None:
            st.wait_event(self.outs_free[s])
        for l, t in enumerate(self.types):
            Dv = dev[l]
            if t == L.DSA_LAYER_FULL:
                st.wait_event(ready[l][0])
                L.dsa_indexer_topk(self.idesc, Dv["q_idx"], Dv["k_idx"], Dv["w"], q_pos, k_pos, ks, ke, rope_cs,
                                   self.idx[l], None, ws=self.iws, stream=st)
            st.wait_event(ready[l][1])
            L.dsa_sparse_attn(self.adesc, Dv["q"], Dv["kv"], self.idx[self.donors[l]], ks, out[l], None,
                              ws=self.aws, stream=st)
            done = torch.cuda.Event()
            done.record(st)
            self.down.wait_event(done)
            with torch.cuda.stream(self.down):
                host_out[l].copy_(out[l], non_blocking=True)
        free = torch.cuda.Event()
        free.record(st)
        self.inputs_free[s] = free
        finished = torch.cuda.Event(enable_timing=True)
        finished.record(self.down)
        self.outs_free[s] = finished
        return finished
