"""ctypes binding of libdsa.so (include/dsa.h).  Argument marshalling only.

Every function keeps the C name.  Tensors are torch tensors on the GPU (their data pointers
are passed through); the stream defaults to torch's current stream.  A non-OK status raises
DsaError carrying the library's message.  There is no fallback: if the shared library is
missing the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_LAYER_SHARED = 0
DSA_LAYER_FULL = 1
DSA_IDX_ROPE_Q = 1 << 0
DSA_IDX_ROPE_K = 1 << 1
DSA_IDX_INDEPENDENT_ROWS = 1 << 2

STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_ARG", 2: "DSA_ERR_SHAPE", 3: "DSA_ERR_NO_DONOR", 4: "DSA_ERR_UNSUPPORTED",
                5: "DSA_ERR_CUDA", 6: "DSA_ERR_WORKSPACE", 7: "DSA_ERR_TIMEOUT", 8: "DSA_ERR_DEVICE"}
EXPORTED = ("dsa_status_string", "dsa_last_error", "dsa_donor_table", "dsa_rope_table", "dsa_indexer_workspace_size",
            "dsa_indexer_topk", "dsa_sparse_attn_workspace_size", "dsa_sparse_attn", "dsa_index_cache_create",
            "dsa_index_cache_donor", "dsa_index_cache_indices", "dsa_index_cache_destroy",
            "dsa_layers_workspace_size", "indexshare_layers_forward", "dsa_workspace_status",
            "dsa_indexer_topk_static", "dsa_profile_enable", "dsa_profile_indexer_last", "dsa_mtp_indexshare_step",
            "dsa_indexer_topk_paged", "dsa_sparse_attn_paged", "dsa_indexer_projections", "dsa_sparse_attn_backward",
            "dsa_indexer_static_status", "dsa_profile_read", "dsa_debug_pipeline",
            "dsa_indexer_backward_workspace_size", "dsa_indexer_backward",
            "dsa_sparse_attn_backward_workspace_size")

PROFILE_KINDS = {0: "rope", 1: "ranges", 2: "indexer", 3: "select", 4: "attn_prep", 5: "attn", 6: "attn_bwd",
                 7: "proj", 8: "indexer_bwd"}


class DsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.name}: {message}")


class IndexerDesc(C.Structure):
    _fields_ = [("n_q", C.c_int32), ("n_kv", C.c_int32), ("n_heads", C.c_int32), ("head_dim", C.c_int32),
                ("rope_dim", C.c_int32), ("topk", C.c_int32), ("max_len", C.c_int32), ("flags", C.c_uint32)]


class AttnDesc(C.Structure):
    _fields_ = [("n_q", C.c_int32), ("n_kv", C.c_int32), ("n_heads", C.c_int32), ("d_qk", C.c_int32),
                ("d_v", C.c_int32), ("topk", C.c_int32), ("softmax_scale", C.c_float), ("flags", C.c_uint32)]


class ProfileRecord(C.Structure):
    _fields_ = [("kind", C.c_int32), ("ms", C.c_float)]


class LayerIO(C.Structure):
    _fields_ = [("q_idx", C.c_void_p), ("k_idx", C.c_void_p), ("w", C.c_void_p), ("q", C.c_void_p),
                ("kv", C.c_void_p), ("out", C.c_void_p), ("lse", C.c_void_p)]


_lib: Optional[C.CDLL] = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run dsa_indexer_cross_gb300.build.build() first")
        L = C.CDLL(LIB_PATH)
        st, vp, i32, u32, sz = C.c_int, C.c_void_p, C.c_int32, C.c_uint32, C.c_size_t
        P = C.POINTER
        L.dsa_status_string.restype = C.c_char_p
        L.dsa_status_string.argtypes = [st]
        L.dsa_last_error.restype = C.c_char_p
        L.dsa_last_error.argtypes = []
        L.dsa_donor_table.restype = st
        L.dsa_donor_table.argtypes = [i32, P(C.c_uint8), P(i32)]
        L.dsa_rope_table.restype = st
        L.dsa_rope_table.argtypes = [C.c_double, i32, i32, P(C.c_float)]
        L.dsa_indexer_workspace_size.restype = st
        L.dsa_indexer_workspace_size.argtypes = [P(IndexerDesc), P(sz)]
        L.dsa_indexer_topk.restype = st
        L.dsa_indexer_topk.argtypes = [P(IndexerDesc), vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        L.dsa_sparse_attn_workspace_size.restype = st
        L.dsa_sparse_attn_workspace_size.argtypes = [P(AttnDesc), P(sz)]
        L.dsa_sparse_attn.restype = st
        L.dsa_sparse_attn.argtypes = [P(AttnDesc), vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dsa_index_cache_create.restype = st
        L.dsa_index_cache_create.argtypes = [i32, P(C.c_uint8), i32, i32, P(vp), P(vp)]
        L.dsa_index_cache_donor.restype = st
        L.dsa_index_cache_donor.argtypes = [vp, i32, P(i32)]
        L.dsa_index_cache_indices.restype = vp
        L.dsa_index_cache_indices.argtypes = [vp, i32]
        L.dsa_index_cache_destroy.restype = None
        L.dsa_index_cache_destroy.argtypes = [vp]
        L.dsa_layers_workspace_size.restype = st
        L.dsa_layers_workspace_size.argtypes = [P(IndexerDesc), P(AttnDesc), P(sz)]
        L.indexshare_layers_forward.restype = st
        L.indexshare_layers_forward.argtypes = [P(IndexerDesc), P(AttnDesc), i32, P(C.c_uint8), P(LayerIO), vp, vp,
                                                vp, vp, vp, i32, vp, vp, sz, vp]
        L.dsa_workspace_status.restype = st
        L.dsa_workspace_status.argtypes = [vp, vp, P(u32)]
        L.dsa_profile_enable.restype = st
        L.dsa_profile_enable.argtypes = [i32]
        L.dsa_profile_indexer_last.restype = st
        L.dsa_profile_indexer_last.argtypes = [P(C.c_float), i32]
        L.dsa_indexer_topk_static.restype = st
        L.dsa_indexer_topk_static.argtypes = [P(IndexerDesc), vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp]
        L.dsa_indexer_static_status.restype = st
        L.dsa_indexer_static_status.argtypes = [vp, P(u32)]
        L.dsa_debug_pipeline.restype = st
        L.dsa_debug_pipeline.argtypes = [i32, C.c_uint64]
        L.dsa_profile_read.restype = st
        L.dsa_profile_read.argtypes = [P(ProfileRecord), i32, P(i32)]
        L.dsa_sparse_attn_backward.restype = st
        L.dsa_sparse_attn_backward_workspace_size.restype = st
        L.dsa_sparse_attn_backward_workspace_size.argtypes = [P(AttnDesc), P(sz)]
        L.dsa_sparse_attn_backward.argtypes = [P(AttnDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dsa_indexer_backward_workspace_size.restype = st
        L.dsa_indexer_backward_workspace_size.argtypes = [P(IndexerDesc), P(sz)]
        L.dsa_indexer_backward.restype = st
        L.dsa_indexer_backward.argtypes = [P(IndexerDesc), vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                           sz, vp]
        L.dsa_indexer_projections.restype = st
        L.dsa_indexer_projections.argtypes = [P(ProjDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dsa_indexer_topk_paged.restype = st
        L.dsa_indexer_topk_paged.argtypes = [P(IndexerDesc), vp, vp, vp, vp, P(PagedCache), vp, i32, vp, vp, vp, sz, vp]
        L.dsa_sparse_attn_paged.restype = st
        L.dsa_sparse_attn_paged.argtypes = [P(AttnDesc), vp, vp, vp, P(PagedCache), vp, vp, vp, sz, vp]
        L.dsa_mtp_indexshare_step.restype = st
        L.dsa_mtp_indexshare_step.argtypes = [P(IndexerDesc), P(AttnDesc), i32, P(LayerIO), vp, vp, vp, vp, vp, i32,
                                              vp, vp, sz, vp]
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise DsaError(status, lib().dsa_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    """Device address of a contiguous CUDA tensor (every tensor argument of libdsa's GPU calls is
    device memory; a host tensor is refused here rather than handed to a kernel)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libdsa must be CUDA tensors (device memory)")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdsa must be contiguous")
    return t.data_ptr()


def _want(t: torch.Tensor, dtype, numel: int, name: str) -> None:
    """Refuse a tensor of the wrong type or too few elements before its address reaches a kernel
    (the C ABI takes bare pointers and cannot check either)."""
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, has {t.numel()}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _u8(types: Sequence[int]):
    return (C.c_uint8 * len(types))(*[int(x) for x in types])


def types_to_u8(indexer_types: Sequence) -> list:
    """'full'/'shared' strings (as in a released config) or 0/1 ints -> 0/1 ints."""
    out = []
    for t in indexer_types:
        if isinstance(t, str):
            out.append(DSA_LAYER_FULL if t == "full" else DSA_LAYER_SHARED if t == "shared" else 255)
        else:
            out.append(int(t))
    return out


# ------------------------------------------------------------------------------ schedule

def dsa_donor_table(indexer_types: Sequence) -> list:
    types = types_to_u8(indexer_types)
    donors = (C.c_int32 * max(1, len(types)))()
    _check(lib().dsa_donor_table(len(types), _u8(types), donors))
    return list(donors)[:len(types)]


def dsa_rope_table(theta: float, rope_dim: int, n_pos: int) -> torch.Tensor:
    """Host float32 tensor [n_pos, rope_dim/2, 2] of (cos, sin)."""
    out = torch.empty((n_pos, max(rope_dim // 2, 1), 2), dtype=torch.float32)
    _check(lib().dsa_rope_table(float(theta), int(rope_dim), int(n_pos),
                                C.cast(out.data_ptr(), C.POINTER(C.c_float))))
    return out


# ------------------------------------------------------------------------------ indexer

def indexer_desc(n_q, n_kv, n_heads, head_dim, rope_dim, topk, max_len, flags) -> IndexerDesc:
    return IndexerDesc(n_q, n_kv, n_heads, head_dim, rope_dim, topk, max_len, flags)


def dsa_indexer_workspace_size(desc: IndexerDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dsa_indexer_workspace_size(C.byref(desc), C.byref(n)))
    return n.value


def _indexer_args(desc: IndexerDesc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx_out, score_out) -> None:
    n_q, n_kv, H, d, k = desc.n_q, desc.n_kv, desc.n_heads, desc.head_dim, desc.topk
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for t, dt, n, name in ((q_idx, bf, n_q * H * d, "q_idx"), (k_idx, bf, n_kv * d, "k_idx"), (w, f32, n_q * H, "w"),
                           (q_pos, i32, n_q, "q_pos"), (k_pos, i32, n_kv, "k_pos"), (ks, i32, n_q, "ks"),
                           (ke, i32, n_q, "ke"), (rope_cs, f32, 0, "rope_cs"), (idx_out, i32, n_q * k, "idx_out"),
                           (score_out, f32, n_q * k, "score_out")):
        if t is not None:
            _want(t, dt, n, name)


def dsa_indexer_topk(desc: IndexerDesc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx_out, score_out=None,
                     ws=None, stream=None) -> torch.Tensor:
    _indexer_args(desc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx_out, score_out)
    if ws is None:
        ws = torch.empty(dsa_indexer_workspace_size(desc), dtype=torch.uint8, device=idx_out.device)
    n_pos = rope_cs.shape[0] if rope_cs is not None else 0
    _check(lib().dsa_indexer_topk(C.byref(desc), _ptr(q_idx), _ptr(k_idx), _ptr(w), _ptr(q_pos), _ptr(k_pos),
                                  _ptr(ks), _ptr(ke), _ptr(rope_cs), n_pos, _ptr(idx_out), _ptr(score_out),
                                  _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def dsa_indexer_topk_static(desc: IndexerDesc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx_out,
                            score_out=None, stream=None) -> None:
    """dsa_indexer_topk with the library's static device scratch instead of a workspace."""
    _indexer_args(desc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx_out, score_out)
    n_pos = rope_cs.shape[0] if rope_cs is not None else 0
    _check(lib().dsa_indexer_topk_static(C.byref(desc), _ptr(q_idx), _ptr(k_idx), _ptr(w), _ptr(q_pos), _ptr(k_pos),
                                         _ptr(ks), _ptr(ke), _ptr(rope_cs), n_pos, _ptr(idx_out), _ptr(score_out),
                                         _stream(stream)))


def dsa_indexer_backward_workspace_size(desc: IndexerDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dsa_indexer_backward_workspace_size(C.byref(desc), C.byref(n)))
    return n.value


def dsa_indexer_backward(desc: IndexerDesc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx, d_score, dq_idx,
                         dk_idx, dw, ws=None, stream=None) -> torch.Tensor:
    """Gradients of the selected scores: dq_idx (written), dk_idx and dw (zeroed, then
    accumulated), fp32, for the upstream d_score aligned with the forward's idx."""
    _indexer_args(desc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, idx, None)
    n_q, n_kv, H, d, k = desc.n_q, desc.n_kv, desc.n_heads, desc.head_dim, desc.topk
    f32 = torch.float32
    for t, n, name in ((d_score, n_q * k, "d_score"), (dq_idx, n_q * H * d, "dq_idx"), (dk_idx, n_kv * d, "dk_idx"),
                       (dw, n_q * H, "dw")):
        _want(t, f32, n, name)
    if ws is None:
        ws = torch.empty(dsa_indexer_backward_workspace_size(desc), dtype=torch.uint8, device=dq_idx.device)
    n_pos = rope_cs.shape[0] if rope_cs is not None else 0
    _check(lib().dsa_indexer_backward(C.byref(desc), _ptr(q_idx), _ptr(k_idx), _ptr(w), _ptr(q_pos), _ptr(k_pos),
                                      _ptr(ks), _ptr(ke), _ptr(rope_cs), n_pos, _ptr(idx), _ptr(d_score),
                                      _ptr(dq_idx), _ptr(dk_idx), _ptr(dw), _ptr(ws), ws.numel(), _stream(stream)))
    return ws


# ------------------------------------------------------------------------------ attention

def attn_desc(n_q, n_kv, n_heads, topk, softmax_scale, d_qk=576, d_v=512) -> AttnDesc:
    return AttnDesc(n_q, n_kv, n_heads, d_qk, d_v, topk, softmax_scale, 0)


def dsa_sparse_attn_workspace_size(desc: AttnDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dsa_sparse_attn_workspace_size(C.byref(desc), C.byref(n)))
    return n.value


def dsa_sparse_attn(desc: AttnDesc, q, kv, idx, ks, out, lse=None, ws=None, stream=None) -> torch.Tensor:
    n_q, n_kv, H, k = desc.n_q, desc.n_kv, desc.n_heads, desc.topk
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for t, dt, n, name in ((q, bf, n_q * H * desc.d_qk, "q"), (kv, bf, n_kv * desc.d_qk, "kv"), (idx, i32, n_q * k, "idx"),
                           (ks, i32, n_q, "ks"), (out, bf, n_q * H * desc.d_v, "out"), (lse, f32, n_q * H, "lse")):
        if t is not None:
            _want(t, dt, n, name)
    if ws is None:
        ws = torch.empty(dsa_sparse_attn_workspace_size(desc), dtype=torch.uint8, device=out.device)
    _check(lib().dsa_sparse_attn(C.byref(desc), _ptr(q), _ptr(kv), _ptr(idx), _ptr(ks), _ptr(out), _ptr(lse),
                                 _ptr(ws), ws.numel(), _stream(stream)))
    return ws


# ------------------------------------------------------------------------------ index cache

class IndexCache:
    """Owns a dsa_index_cache handle and the per-full-layer device index buffers."""

    def __init__(self, indexer_types: Sequence, n_q: int, topk: int, device="cuda"):
        self.types = types_to_u8(indexer_types)
        self.n_q, self.topk = n_q, topk
        self.buffers = [torch.full((n_q, topk), -1, dtype=torch.int32, device=device)
                        if t == DSA_LAYER_FULL else None for t in self.types]
        ptrs = (C.c_void_p * len(self.types))(*[b.data_ptr() if b is not None else None for b in self.buffers])
        h = C.c_void_p()
        _check(lib().dsa_index_cache_create(len(self.types), _u8(self.types), n_q, topk, ptrs, C.byref(h)))
        self.handle = h

    def donor(self, layer: int) -> int:
        d = C.c_int32(0)
        _check(lib().dsa_index_cache_donor(self.handle, layer, C.byref(d)))
        return d.value

    def indices_ptr(self, layer: int) -> int:
        p = lib().dsa_index_cache_indices(self.handle, layer)
        if not p:
            raise DsaError(1, lib().dsa_last_error().decode())
        return p

    def indices(self, layer: int) -> torch.Tensor:
        return self.buffers[self.donor(layer)]

    def close(self):
        if getattr(self, "handle", None):
            lib().dsa_index_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------------------ layer loop

def dsa_layers_workspace_size(idesc: IndexerDesc, adesc: AttnDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dsa_layers_workspace_size(C.byref(idesc), C.byref(adesc), C.byref(n)))
    return n.value


def indexshare_layers_forward(idesc: IndexerDesc, adesc: AttnDesc, indexer_types: Sequence, layers: Sequence[dict],
                              ks, ke, q_pos, k_pos, rope_cs, cache: IndexCache, ws=None, stream=None):
    """layers[l]: dict with 'q', 'kv', 'out' (+ 'lse') and, on full layers, 'q_idx', 'k_idx', 'w'."""
    types = types_to_u8(indexer_types)
    io = (LayerIO * len(layers))()
    for l, L in enumerate(layers):
        io[l] = LayerIO(_ptr(L.get("q_idx")), _ptr(L.get("k_idx")), _ptr(L.get("w")), _ptr(L["q"]), _ptr(L["kv"]),
                        _ptr(L["out"]), _ptr(L.get("lse")))
    if ws is None:
        ws = torch.empty(dsa_layers_workspace_size(idesc, adesc), dtype=torch.uint8, device=layers[0]["q"].device)
    n_pos = rope_cs.shape[0] if rope_cs is not None else 0
    _check(lib().indexshare_layers_forward(C.byref(idesc), C.byref(adesc), len(types), _u8(types), io, _ptr(ks),
                                           _ptr(ke), _ptr(q_pos), _ptr(k_pos), _ptr(rope_cs), n_pos, cache.handle,
                                           _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def dsa_sparse_attn_backward_workspace_size(desc: AttnDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dsa_sparse_attn_backward_workspace_size(C.byref(desc), C.byref(n)))
    return n.value


def dsa_sparse_attn_backward(desc: AttnDesc, q, kv, idx, ks, out, lse, d_out, dq, dkv, ws=None, stream=None):
    """dq (written) and dkv (zeroed, then accumulated), fp32, for the upstream gradient d_out."""
    n_q, n_kv, H, k = desc.n_q, desc.n_kv, desc.n_heads, desc.topk
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for t, dt, n, name in ((q, bf, n_q * H * desc.d_qk, "q"), (kv, bf, n_kv * desc.d_qk, "kv"), (idx, i32, n_q * k, "idx"),
                           (ks, i32, n_q, "ks"), (out, bf, n_q * H * desc.d_v, "out"), (lse, f32, n_q * H, "lse"),
                           (d_out, bf, n_q * H * desc.d_v, "d_out"), (dq, f32, n_q * H * desc.d_qk, "dq"),
                           (dkv, f32, n_kv * desc.d_qk, "dkv")):
        _want(t, dt, n, name)
    if ws is None:
        ws = torch.empty(dsa_sparse_attn_backward_workspace_size(desc), dtype=torch.uint8, device=q.device)
    _check(lib().dsa_sparse_attn_backward(C.byref(desc), _ptr(q), _ptr(kv), _ptr(idx), _ptr(ks), _ptr(out), _ptr(lse),
                                          _ptr(d_out), _ptr(dq), _ptr(dkv), _ptr(ws), ws.numel(), _stream(stream)))
    return ws


class ProjDesc(C.Structure):
    _fields_ = [("n_tokens", C.c_int32), ("d_hidden", C.c_int32), ("d_q", C.c_int32), ("n_heads", C.c_int32),
                ("head_dim", C.c_int32), ("ln_eps", C.c_float)]


def dsa_indexer_projections(desc: "ProjDesc", x, q_latent, wq_b, wk, k_norm_w, k_norm_b, weights_proj, q_idx, k_idx,
                            w, ws=None, stream=None):
    """q_idx = q_latent wq_b^T, k_idx = LayerNorm(x wk^T) (k_norm weight / bias), w = x weights_proj^T."""
    T, dh, dq, H, d = desc.n_tokens, desc.d_hidden, desc.d_q, desc.n_heads, desc.head_dim
    bf, f32 = torch.bfloat16, torch.float32
    for t, dt, n, name in ((x, bf, T * dh, "x"), (q_latent, bf, T * dq, "q_latent"), (wq_b, bf, H * d * dq, "wq_b"),
                           (wk, bf, d * dh, "wk"), (k_norm_w, f32, d, "k_norm_w"), (k_norm_b, f32, d, "k_norm_b"),
                           (weights_proj, bf, H * dh, "weights_proj"), (q_idx, bf, T * H * d, "q_idx"),
                           (k_idx, bf, T * d, "k_idx"), (w, f32, T * H, "w")):
        _want(t, dt, n, name)
    if ws is None:
        ws = torch.zeros(256, dtype=torch.uint8, device=x.device)
    _check(lib().dsa_indexer_projections(C.byref(desc), _ptr(x), _ptr(q_latent), _ptr(wq_b), _ptr(wk), _ptr(k_norm_w),
                                         _ptr(k_norm_b), _ptr(weights_proj), _ptr(q_idx), _ptr(k_idx), _ptr(w),
                                         _ptr(ws), ws.numel(), _stream(stream)))
    return ws


DSA_PAGE_ROWS = 128


class PagedCache(C.Structure):
    """dsa_paged_cache: row t's logical key j sits at cache row
    block_table[t, j // page_rows] * page_rows + j % page_rows, valid for j < seq_len[t]."""
    _fields_ = [("block_table", C.c_void_p), ("seq_len", C.c_void_p), ("max_pages", C.c_int32),
                ("n_pages", C.c_int32), ("page_rows", C.c_int32)]


def paged_cache(block_table: torch.Tensor, seq_len: torch.Tensor, n_pages: int) -> PagedCache:
    """block_table: int32 [n_q, max_pages] device tensor; seq_len: int32 [n_q] (kept alive by the caller)."""
    return PagedCache(_ptr(block_table), _ptr(seq_len), block_table.shape[1], n_pages, DSA_PAGE_ROWS)


def _paged_args(pages: PagedCache) -> None:
    if not pages.block_table or not pages.seq_len:
        raise ValueError("paged cache: block_table and seq_len must be set")


def dsa_indexer_topk_paged(desc: IndexerDesc, q_idx, k_cache, w, q_pos, pages: PagedCache, rope_cs, idx_out,
                           score_out=None, ws=None, stream=None):
    n_q, H, d, k = desc.n_q, desc.n_heads, desc.head_dim, desc.topk
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for t, dt, n, name in ((q_idx, bf, n_q * H * d, "q_idx"), (k_cache, bf, desc.n_kv * d, "k_cache"),
                           (w, f32, n_q * H, "w"), (q_pos, i32, n_q, "q_pos"), (rope_cs, f32, 0, "rope_cs"),
                           (idx_out, i32, n_q * k, "idx_out"), (score_out, f32, n_q * k, "score_out")):
        if t is not None:
            _want(t, dt, n, name)
    _paged_args(pages)
    if ws is None:
        ws = torch.empty(dsa_indexer_workspace_size(desc), dtype=torch.uint8, device=q_idx.device)
    n_pos = rope_cs.shape[0] if rope_cs is not None else 0
    _check(lib().dsa_indexer_topk_paged(C.byref(desc), _ptr(q_idx), _ptr(k_cache), _ptr(w), _ptr(q_pos),
                                        C.byref(pages), _ptr(rope_cs), n_pos, _ptr(idx_out), _ptr(score_out),
                                        _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def dsa_sparse_attn_paged(desc: AttnDesc, q, kv_cache, idx, pages: PagedCache, out, lse=None, ws=None, stream=None):
    n_q, H, k = desc.n_q, desc.n_heads, desc.topk
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for t, dt, n, name in ((q, bf, n_q * H * desc.d_qk, "q"), (kv_cache, bf, desc.n_kv * desc.d_qk, "kv_cache"),
                           (idx, i32, n_q * k, "idx"), (out, bf, n_q * H * desc.d_v, "out"), (lse, f32, n_q * H, "lse")):
        if t is not None:
            _want(t, dt, n, name)
    _paged_args(pages)
    if ws is None:
        ws = torch.empty(dsa_sparse_attn_workspace_size(desc), dtype=torch.uint8, device=q.device)
    _check(lib().dsa_sparse_attn_paged(C.byref(desc), _ptr(q), _ptr(kv_cache), _ptr(idx), C.byref(pages), _ptr(out),
                                       _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def dsa_mtp_indexshare_step(idesc: IndexerDesc, adesc: AttnDesc, step: int, layer: dict, ks, ke, q_pos, k_pos,
                            rope_cs, mtp_idx, ws=None, stream=None):
    """One MTP draft step: step 0 runs the indexer into mtp_idx and attends with it; later
    steps attend with mtp_idx unchanged.  layer: 'q', 'kv', 'out' (+ 'lse') and, at step 0,
    'q_idx', 'k_idx', 'w'."""
    L = layer
    n_q, H, k = adesc.n_q, adesc.n_heads, adesc.topk
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for key, dt, n in (("q", bf, n_q * H * adesc.d_qk), ("kv", bf, adesc.n_kv * adesc.d_qk),
                       ("out", bf, n_q * H * adesc.d_v), ("lse", f32, n_q * H)):
        if L.get(key) is not None:
            _want(L[key], dt, n, key)
    _want(mtp_idx, i32, n_q * k, "mtp_idx")
    for t, dt, n, name in ((ks, i32, n_q, "ks"), (ke, i32, n_q, "ke"), (q_pos, i32, n_q, "q_pos")):
        _want(t, dt, n, name)
    if step == 0:
        _indexer_args(idesc, L.get("q_idx"), L.get("k_idx"), L.get("w"), None, k_pos, None, None, rope_cs, None, None)
    io = LayerIO(_ptr(L.get("q_idx")), _ptr(L.get("k_idx")), _ptr(L.get("w")), _ptr(L["q"]), _ptr(L["kv"]),
                 _ptr(L["out"]), _ptr(L.get("lse")))
    if ws is None:
        ws = torch.empty(dsa_layers_workspace_size(idesc, adesc), dtype=torch.uint8, device=L["q"].device)
    n_pos = rope_cs.shape[0] if rope_cs is not None else 0
    _check(lib().dsa_mtp_indexshare_step(C.byref(idesc), C.byref(adesc), int(step), C.byref(io), _ptr(ks), _ptr(ke),
                                         _ptr(q_pos), _ptr(k_pos), _ptr(rope_cs), n_pos, _ptr(mtp_idx), _ptr(ws),
                                         ws.numel(), _stream(stream)))
    return ws


def dsa_workspace_status(ws: torch.Tensor, stream=None, raise_on_fault: bool = True) -> int:
    """Synchronise and read the device status bits of a workspace.

    Raises DsaError on a device fault unless raise_on_fault is False, in which case the raw
    bits are returned (0 = clean).  A CUDA error always raises.
    """
    bits = C.c_uint32(0)
    st = lib().dsa_workspace_status(_ptr(ws), _stream(stream), C.byref(bits))
    if st not in (0, 7, 8) or (st != 0 and raise_on_fault):
        _check(st)
    return bits.value


def dsa_profile_enable(on: bool) -> None:
    """Turn per-phase event recording of indexer calls on or off (process-wide)."""
    _check(lib().dsa_profile_enable(1 if on else 0))


def dsa_profile_indexer_last() -> list:
    """Device milliseconds of the last profiled indexer call on the current device:
    [RoPE, key-range plan, scores + streaming top-k, final select]."""
    ms = (C.c_float * 4)()
    _check(lib().dsa_profile_indexer_last(ms, 4))
    return [float(x) for x in ms]


def dsa_indexer_static_status(stream=None, raise_on_fault: bool = True) -> int:
    """Status bits of the last dsa_indexer_topk_static call on the current device (synchronises
    the stream).  Raises DsaError on a device fault unless raise_on_fault is False."""
    bits = C.c_uint32(0)
    st = lib().dsa_indexer_static_status(_stream(stream), C.byref(bits))
    if st not in (0, 7, 8) or (st != 0 and raise_on_fault):
        _check(st)
    return bits.value


def dsa_profile_read(cap: int = 8192) -> list:
    """[(kind name, device ms)] of every launch logged on the current device since profiling was
    switched on, in launch order (waits for them to finish)."""
    buf = (ProfileRecord * cap)()
    n = C.c_int32(0)
    _check(lib().dsa_profile_read(buf, cap, C.byref(n)))
    return [(PROFILE_KINDS.get(buf[i].kind, str(buf[i].kind)), float(buf[i].ms)) for i in range(min(n.value, cap))]


def dsa_debug_pipeline(stop_after_tiles: int = -1, wait_ns: int = 0) -> None:
    """Test hook: bound every pipeline wait at wait_ns (0: the default 2 s) and make the TMA
    producers stop after stop_after_tiles tiles (-1: never).  Process-wide."""
    _check(lib().dsa_debug_pipeline(int(stop_after_tiles), int(wait_ns)))
