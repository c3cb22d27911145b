"""Seeded synthetic inputs for the DSA indexer / IndexShare / sparse-attention path.

This module only draws random numbers and lays out geometry (positions, key ranges).  It
holds none of the method's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it: the oracle always reads the very bytes the kernels read.

Workload shapes (the five standard workloads of the path):

* ``tiny``        T=256 prefill, 4 layers F S S S, 4 index heads x 64 (RoPE on the last
                  16 dims, theta 1e4), top-k 32, 4 attention heads.
* ``prefill_4k``  T=4096 prefill, 8 layers F F F S S S F S, 32 x 128 (last 64 RoPE,
                  theta 8e6), top-k 2048, 16 attention heads.
* ``long_32k``    T=32768 prefill, 8 layers (F S S S) x 2, 64 x 128, top-k 2048, 64 heads;
                  1 % of key positions get +3/sqrt(d_I) on every index-key dim.
* ``decode_64``   64 sequences, one query each, cached lengths uniform in [8192, 131072],
                  4 layers F S S S, 64 x 128, top-k 2048, 128 heads; the index-key cache
                  is stored already rotated.
* ``chunk_1m``    4096 queries at positions 1,044,480 ... 1,048,575 over a 1,048,576-key
                  causal prefix, 8 layers (F S S S) x 2, 64 x 128, top-k 2048, 64 heads.

Value distributions: index q/k and attention q/kv are N(0,1)/sqrt(d) rounded to bf16
(``attn_scale='unit'`` gives N(0,1) attention inputs instead); head weights are N(0,1)
float32.  Layer l draws from seed ``seed + 17 * l``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

FULL = "full"
SHARED = "shared"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" | "decode" | "chunk"
    n_q: int
    layers: tuple
    n_heads_idx: int          # H_I
    head_dim_idx: int         # d_I
    rope_dim: int
    theta: float
    topk: int
    n_heads: int              # H (attention)
    d_qk: int = 576
    d_v: int = 512
    key_bias_frac: float = 0.0
    n_seqs: int = 0           # decode
    len_lo: int = 0           # decode
    len_hi: int = 0           # decode
    chunk_pos0: int = 0       # chunk
    chunk_keys: int = 0       # chunk
    rope_k: bool = True

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_qk)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


F, S = FULL, SHARED
WORKLOADS = {
    "tiny": Workload("tiny", "prefill", 256, (F, S, S, S), 4, 64, 16, 1e4, 32, 4),
    "prefill_4k": Workload("prefill_4k", "prefill", 4096, (F, F, F, S, S, S, F, S), 32, 128, 64,
                           8e6, 2048, 16),
    "long_32k": Workload("long_32k", "prefill", 32768, (F, S, S, S) * 2, 64, 128, 64, 8e6, 2048,
                         64, key_bias_frac=0.01),
    "decode_64": Workload("decode_64", "decode", 64, (F, S, S, S), 64, 128, 64, 8e6, 2048, 128,
                          n_seqs=64, len_lo=8192, len_hi=131072, rope_k=False),
    "chunk_1m": Workload("chunk_1m", "chunk", 4096, (F, S, S, S) * 2, 64, 128, 64, 8e6, 2048, 64,
                         chunk_pos0=1044480, chunk_keys=1048576),
}


@dataclasses.dataclass
class Geometry:
    """Positions and per-query key ranges (all int32 numpy arrays)."""
    n_kv: int
    q_pos: np.ndarray
    k_pos: np.ndarray
    ks: np.ndarray
    ke: np.ndarray

    @property
    def max_len(self) -> int:
        return int((self.ke - self.ks).max()) if self.ks.size else 0

    @property
    def max_pos(self) -> int:
        return int(max(self.q_pos.max(initial=0), self.k_pos.max(initial=0))) + 1


def geometry(w: Workload, seed: int = 1234) -> Geometry:
    """Causal key ranges: each query sees every key up to and including its own position."""
    if w.kind == "prefill":
        T = w.n_q
        pos = np.arange(T, dtype=np.int32)
        return Geometry(T, pos.copy(), pos.copy(), np.zeros(T, np.int32), pos + 1)
    if w.kind == "chunk":
        n_kv = w.chunk_keys
        q_pos = (w.chunk_pos0 + np.arange(w.n_q)).astype(np.int32)
        return Geometry(n_kv, q_pos, np.arange(n_kv, dtype=np.int32),
                        np.zeros(w.n_q, np.int32), (q_pos + 1).astype(np.int32))
    if w.kind == "decode":
        rng = np.random.default_rng(seed)
        lens = rng.integers(w.len_lo, w.len_hi + 1, size=w.n_seqs).astype(np.int64)
        off = np.concatenate([[0], np.cumsum(lens)[:-1]])
        n_kv = int(lens.sum())
        k_pos = (np.arange(n_kv) - np.repeat(off, lens)).astype(np.int32)
        return Geometry(n_kv, (lens - 1).astype(np.int32), k_pos,
                        off.astype(np.int32), (off + lens).astype(np.int32))
    raise ValueError(w.kind)


def mtp_geometry(w: Workload, steps: int, seed: int = 1234) -> list:
    """Batched decode with multi-step MTP drafting: sequence b holds lens[b] cached rows plus
    room for the steps' draft rows; at step s its query sits at position lens[b] - 1 + s and
    sees keys [off_b, off_b + lens[b] + s).  Returns one Geometry per step (same key cache)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(w.len_lo, w.len_hi + 1, size=w.n_seqs).astype(np.int64)
    span = lens + steps - 1
    off = np.concatenate([[0], np.cumsum(span)[:-1]])
    n_kv = int(span.sum())
    k_pos = (np.arange(n_kv) - np.repeat(off, span)).astype(np.int32)
    return [Geometry(n_kv, (lens - 1 + s).astype(np.int32), k_pos, off.astype(np.int32),
                     (off + lens + s).astype(np.int32)) for s in range(steps)]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def layer_inputs(w: Workload, geo: Geometry, layer: int, seed: int = 1234, device="cpu",
                 attn_scale: str = "config", with_attn: bool = True) -> dict:
    """Tensors of one layer.  Full layers also get the indexer inputs.

    attn_scale: 'config' -> q/kv ~ N(0,1)/sqrt(576);  'unit' -> N(0,1).
    """
    g = _gen(device, seed + 17 * layer)
    out = {}
    if w.layers[layer] == FULL:
        d = w.head_dim_idx
        out["q_idx"] = _normal_bf16((w.n_q, w.n_heads_idx, d), 1.0 / math.sqrt(d), g, device)
        k = torch.randn((geo.n_kv, d), generator=g, device=device, dtype=torch.float32) / math.sqrt(d)
        if w.key_bias_frac > 0.0:
            n_b = max(1, int(round(w.key_bias_frac * geo.n_kv)))
            rows = torch.randperm(geo.n_kv, generator=g, device=device)[:n_b]
            k[rows] += 3.0 / math.sqrt(d)
        out["k_idx"] = k.to(torch.bfloat16)
        out["w"] = torch.randn((w.n_q, w.n_heads_idx), generator=g, device=device, dtype=torch.float32)
    if with_attn:
        std = 1.0 if attn_scale == "unit" else 1.0 / math.sqrt(w.d_qk)
        out["q"] = _normal_bf16((w.n_q, w.n_heads, w.d_qk), std, g, device)
        out["kv"] = _normal_bf16((geo.n_kv, w.d_qk), std, g, device)
    return out


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a bf16/float32 tensor (for the oracle)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def sample_rows(n_q: int, n: int, topk: int, seed: int = 99) -> np.ndarray:
    """Stratified query rows: first, last, rows around t = topk, and a seeded spread."""
    if n >= n_q:
        return np.arange(n_q)
    fixed = {0, 1, n_q - 1, n_q - 2}
    for t in (topk - 2, topk - 1, topk, topk + 1):
        if 0 <= t < n_q:
            fixed.add(t)
    rng = np.random.default_rng(seed)
    rest = rng.choice(n_q, size=max(0, n - len(fixed)), replace=False)
    return np.array(sorted(fixed | set(int(r) for r in rest)))[:max(n, len(fixed))]
