"""Benchmark of the IndexShare DSA hot path on one GB300 (or N independent replicas).

One step = one `indexshare_layers_forward` over the 8-layer T=4096 prefill workload
(indexer_types F F F S S S F S, 32 index heads x 128 with the last 64 dims RoPE'd at
theta 8e6, top-k 2048, 16 attention heads of 576/512): 4 lightning-indexer + fused top-k
passes and 8 sparse-attention passes, every step of the path in libdsa's kernels.

Prints one JSON line.  `value` = query tokens per second (whole job, inputs resident in
HBM), `e2e` = the same through the C ABI with every input copied from pinned host memory
and every layer output copied back inside the timed region.  `roofline` describes the
dominant kernel (sparse attention); `cpu_baseline` times the float64 CPU oracle on a
bounded sample of the same workload.  `--impl reference` times only that oracle.

Timing: W warm-up steps, then K steps each bracketed by CUDA events on the launching
stream; L2 is flushed (a 512 MiB write) between timed steps, outside the events.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "prefill_4k"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--mtp-steps", type=int, default=0,
                    help="decode workloads: also time multi-step MTP drafting with IndexShare (indexer at step 0, "
                         "later steps reuse its indices) and report it under 'mtp'")
    ap.add_argument("--proj", action="store_true",
                    help="also time the indexer's input projections (wq_b, wk + k_norm, weights_proj) for the "
                         "workload's query rows, hidden width 6144 and query latent 2048, under 'proj'")
    ap.add_argument("--bwd", action="store_true",
                    help="also time the sparse-attention backward (dq, dkv) of the first layer for a seeded "
                         "upstream gradient, under 'bwd'")
    ap.add_argument("--paged", action="store_true",
                    help="decode workloads: also time the paged-cache indexer and attention (128-row pages, "
                         "shuffled) against the contiguous calls on the same data, under 'paged'")
    ap.add_argument("--only", choices=["attn", "indexer"], default=None,
                    help="run just one kernel call of the workload (for profiler captures); prints nothing")
    return ap.parse_args()


# --------------------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank float over all ranks (identity for a single process)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = max(mx, float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- workload
def build_inputs(w, geo, device, n_layers=None):
    from dsa_indexer_cross_gb300 import synth
    layers = []
    for l in range(len(w.layers) if n_layers is None else n_layers):
        L = synth.layer_inputs(w, geo, l, device=device)
        L["out"] = torch.empty((w.n_q, w.n_heads, w.d_v), dtype=torch.bfloat16, device=device)
        L["lse"] = torch.empty((w.n_q, w.n_heads), dtype=torch.float32, device=device)
        layers.append(L)
    return layers


def roofline_numbers(w, geo):
    """Algorithmic work of one launch of each kernel (definitions in the design notes)."""
    L = (geo.ke - geo.ks).astype(np.int64)
    rows = np.minimum(L, w.topk).sum()                       # selected rows per layer
    pairs = L.sum()                                          # causal (query, key) pairs
    attn_gathered = rows * w.d_qk * 2 + w.n_q * w.n_heads * (w.d_qk + w.d_v) * 2 + w.n_q * w.topk * 4
    attn_flops = 2.0 * rows * w.n_heads * (w.d_qk + w.d_v)
    idx_flops_causal = 2.0 * pairs * w.n_heads_idx * w.head_dim_idx
    # rows whose prefix is no longer than k select all of it; only the others need scores
    idx_flops = 2.0 * L[L > w.topk].sum() * w.n_heads_idx * w.head_dim_idx
    idx_bytes = (w.n_q * w.n_heads_idx * w.head_dim_idx * 2 + geo.n_kv * w.head_dim_idx * 2 + w.n_q * w.n_heads_idx * 4
                 + w.n_q * w.topk * 4)
    attn_min_bytes = (w.n_q * w.n_heads * w.d_qk * 2 + geo.n_kv * w.d_qk * 2 + w.n_q * w.topk * 4
                      + w.n_q * w.n_heads * (w.d_v * 2 + 4))
    return dict(attn_gathered=float(attn_gathered), attn_flops=attn_flops, idx_flops=idx_flops,
                idx_flops_causal=idx_flops_causal, idx_bytes=float(idx_bytes), attn_min_bytes=float(attn_min_bytes),
                rows=int(rows), pairs=int(pairs))


# DRAM bytes (read + write) of one sparse_attn_kernel launch, per workload, from an ncu capture
# of the current kernel (profiles/sparse_attn_<workload>.md); workloads not listed report None.
ATTN_TRAFFIC_BYTES = {"prefill_4k": 112.24e6, "chunk_1m": 8.671e9}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------------------- oracle timing
def time_oracle(w, geo, layers_host, budget_s: float, max_rows: int = 512):
    """Run the float64 oracle over all layers on growing row samples until ~budget_s of work."""
    from dsa_indexer_cross_gb300 import synth
    from oracle import dsa_oracle as O
    rng = np.random.default_rng(7)
    n = 4
    spent, done_rows = 0.0, 0
    while True:
        rows = np.sort(rng.choice(w.n_q, size=min(n, w.n_q), replace=False))
        t0 = time.perf_counter()
        O.layers_forward(w.layers, layers_host, geo.q_pos, geo.k_pos, geo.ks, geo.ke, w.rope_dim, w.theta, w.topk,
                         w.softmax_scale, rows=rows)
        dt = time.perf_counter() - t0
        spent += dt
        done_rows += len(rows)
        if spent >= budget_s or n >= max_rows:
            break
        n = min(max_rows, max(n * 2, int(n * budget_s / max(dt, 1e-3) * 0.5)))
    return done_rows / spent, done_rows, spent


def host_layers(layers):
    from dsa_indexer_cross_gb300 import synth
    out = []
    for L in layers:
        H = {k: synth.to_f64(v) for k, v in L.items() if k in ("q_idx", "k_idx", "w", "q", "kv")}
        out.append(H)
    return out


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from dsa_indexer_cross_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    geo = synth.geometry(w)
    layers = [synth.layer_inputs(w, geo, l, device="cpu") for l in range(len(w.layers))]
    hl = host_layers(layers)
    from oracle import dsa_oracle as O
    rows_per_step = 8
    rng = np.random.default_rng(11)
    times = []
    for s in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(w.n_q, size=rows_per_step, replace=False))
        t0 = time.perf_counter()
        O.layers_forward(w.layers, hl, geo.q_pos, geo.k_pos, geo.ks, geo.ke, w.rope_dim, w.theta, w.topk,
                         w.softmax_scale, rows=rows)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = rows_per_step / sec
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": "indexer+top-k and sparse-attn query-tokens/sec", "value": value,
            "unit": "query_tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded Gaussian, bf16 inputs)",
            "config": {"workload": f"{w.name}: T={w.n_q}, {len(w.layers)} layers {''.join(t[0].upper() for t in w.layers)}, "
                                   f"H_I={w.n_heads_idx}x{w.head_dim_idx}, topk={w.topk}, H={w.n_heads}",
                       "sample": f"{rows_per_step} random query rows per step through all layers"},
            "cpu_baseline": {"value": value, "unit": "query_tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{rows_per_step} query rows x {len(w.layers)} layers per step"},
            "e2e": {"value": value, "unit": "query_tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- MTP drafting
def time_mtp(D, synth, w, steps: int, dev, stream, flush, reps: int = 10):
    """Time one draft cycle of `steps` MTP steps (dsa_mtp_indexshare_step: the indexer at step 0,
    attention only at the later steps), one query per sequence per step.  Median over reps,
    L2 flushed before each cycle."""
    geos = synth.mtp_geometry(w, steps)
    g0 = geos[0]
    L0 = synth.layer_inputs(w.replace(layers=("full",)), g0, 0, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    ks, k_pos = t(g0.ks), t(g0.k_pos)
    kes, qps = [t(g.ke) for g in geos], [t(g.q_pos) for g in geos]
    rope = D.dsa_rope_table(w.theta, w.rope_dim, max(g.max_pos for g in geos)).to(dev)
    flags = D.DSA_IDX_ROPE_Q | (D.DSA_IDX_ROPE_K if w.rope_k else 0) | D.DSA_IDX_INDEPENDENT_ROWS
    idesc = D.indexer_desc(w.n_q, g0.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, g0.max_len, flags)
    adesc = D.attn_desc(w.n_q, g0.n_kv, w.n_heads, w.topk, w.softmax_scale)
    ws = torch.empty(D.dsa_layers_workspace_size(idesc, adesc), dtype=torch.uint8, device=dev)
    mtp_idx = torch.empty((w.n_q, w.topk), dtype=torch.int32, device=dev)
    layer = dict(L0)
    layer["out"] = torch.empty((w.n_q, w.n_heads, w.d_v), dtype=torch.bfloat16, device=dev)
    layer["lse"] = torch.empty((w.n_q, w.n_heads), dtype=torch.float32, device=dev)

    def cycle(ev=None):
        for s in range(steps):
            if ev is not None:
                ev[s].record(stream)
            D.dsa_mtp_indexshare_step(idesc, adesc, s, layer, ks, kes[s], qps[s], k_pos, rope, mtp_idx, ws=ws,
                                      stream=stream)
        if ev is not None:
            ev[steps].record(stream)

    cycle()
    torch.cuda.synchronize()
    per_step = [[] for _ in range(steps)]
    for _ in range(reps):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        cycle(ev)
        torch.cuda.synchronize()
        for s in range(steps):
            per_step[s].append(ev[s].elapsed_time(ev[s + 1]))
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set during the MTP cycles")
    step_ms = [statistics.median(x) for x in per_step]
    cyc = sum(step_ms)
    return {"steps": steps, "step_ms": step_ms, "cycle_ms": cyc,
            "draft_tokens_per_s": steps * w.n_q / (cyc / 1e3),
            "note": "indexer at step 0 only; later steps attend with step 0's indices"}


# --------------------------------------------------------------------------- projections
def time_proj(D, w, dev, stream, flush, tc_peak, d_hidden: int = 6144, d_q: int = 2048, reps: int = 20):
    """Median time of dsa_indexer_projections for the workload's query rows (synthetic weights),
    against the bf16 peak on its FLOPs: 2 T (H_I d_I d_q + d_I d_h + H_I d_h)."""
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    T, H, d = w.n_q, w.n_heads_idx, w.head_dim_idx
    rn = lambda *s: torch.randn(s, generator=g, device=dev, dtype=torch.float32)
    x = (rn(T, d_hidden) * 0.5).to(torch.bfloat16)
    ql = (rn(T, d_q) * 0.5).to(torch.bfloat16)
    wq = (rn(H * d, d_q) / math.sqrt(d_q)).to(torch.bfloat16)
    wk = (rn(d, d_hidden) / math.sqrt(d_hidden)).to(torch.bfloat16)
    wp = (rn(H, d_hidden) / math.sqrt(d_hidden)).to(torch.bfloat16)
    gamma, beta = torch.ones(d, device=dev), torch.zeros(d, device=dev)
    q_idx = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    k_idx = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    wo = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    desc = D.ProjDesc(T, d_hidden, d_q, H, d, 1e-6)
    call = lambda: D.dsa_indexer_projections(desc, x, ql, wq, wk, gamma, beta, wp, q_idx, k_idx, wo, ws=ws,
                                             stream=stream)
    call()
    ms = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set by the projections")
    m = statistics.median(ms)
    flops = 2.0 * T * (H * d * d_q + d * d_hidden + H * d_hidden)
    return {"d_hidden": d_hidden, "d_q": d_q, "ms": m, "tflops": flops / (m / 1e3) / 1e12,
            "frac_of_bf16_peak": flops / (m / 1e3) / 1e12 / tc_peak,
            "note": "synthetic weights; widths assumed (the pages give none)"}


# --------------------------------------------------------------------------- backward
def time_bwd(D, w, adesc, L0, idx, ks, attn_ms, flops_fwd, dev, stream, flush, tc_peak, reps: int = 5):
    """Median time of dsa_sparse_attn_backward on one layer (the forward's own out and lse, a
    seeded d_out), L2 flushed before each call.  FLOPs: 2.5x the forward's (S and dP recomputed,
    then dQ, dS^T Q and P^T dO)."""
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    d_out = torch.randn(L0["out"].shape, generator=g, device=dev).to(torch.bfloat16)
    dq = torch.empty((w.n_q, w.n_heads, w.d_qk), dtype=torch.float32, device=dev)
    dkv = torch.empty((adesc.n_kv, w.d_qk), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    D.dsa_sparse_attn(adesc, L0["q"], L0["kv"], idx, ks, L0["out"], L0["lse"], stream=stream)
    call = lambda: D.dsa_sparse_attn_backward(adesc, L0["q"], L0["kv"], idx, ks, L0["out"], L0["lse"], d_out, dq, dkv,
                                              ws=ws, stream=stream)
    call()
    ms = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set by the backward")
    m = statistics.median(ms)
    flops = 2.5 * flops_fwd
    return {"ms": m, "forward_ms": attn_ms, "flops": flops, "tflops": flops / (m / 1e3) / 1e12,
            "frac_of_bf16_peak": flops / (m / 1e3) / 1e12 / tc_peak,
            "kernel": "sparse_attn_bwd_kernel (bf16 warp-level MMAs, dkv by 16-byte atomics)"}


# --------------------------------------------------------------------------- paged caches
def time_paged(D, synth, w, geo, L0, idx_full, attn_ms_contig, idx_ms_contig, dev, stream, flush, reps: int = 20,
               seed: int = 3):
    """The same decode layer with its index-key and latent caches in shuffled 128-row pages behind a
    block table: median time of dsa_indexer_topk_paged and dsa_sparse_attn_paged (L2 flushed
    before each call), beside the contiguous calls' times."""
    P = D.DSA_PAGE_ROWS
    lens = (geo.ke - geo.ks).astype(np.int64)
    n_pp = (lens + P - 1) // P
    n_pages = int(n_pp.sum())
    perm = np.random.default_rng(seed).permutation(n_pages)
    bt = np.full((lens.size, int(n_pp.max())), -1, dtype=np.int32)
    phys = np.zeros(int(lens.sum()), dtype=np.int64)
    k = 0
    for t, L in enumerate(lens):
        bt[t, :n_pp[t]] = perm[k:k + n_pp[t]]
        k += n_pp[t]
        j = np.arange(L)
        phys[geo.ks[t] + j] = bt[t, j // P].astype(np.int64) * P + j % P
    phys_t = torch.from_numpy(phys).to(dev)
    k_cache = torch.zeros((n_pages * P, w.head_dim_idx), dtype=torch.bfloat16, device=dev)
    kv_cache = torch.zeros((n_pages * P, w.d_qk), dtype=torch.bfloat16, device=dev)
    k_cache[phys_t] = L0["k_idx"]
    kv_cache[phys_t] = L0["kv"]
    bt_d = torch.from_numpy(bt).to(dev)
    sl_d = torch.from_numpy(lens.astype(np.int32)).to(dev)
    pages = D.paged_cache(bt_d, sl_d, n_pages)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(dev)
    q_pos = torch.from_numpy(geo.q_pos).to(dev)
    flags = D.DSA_IDX_ROPE_Q | D.DSA_IDX_INDEPENDENT_ROWS
    idesc = D.indexer_desc(w.n_q, n_pages * P, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len, flags)
    adesc = D.attn_desc(w.n_q, n_pages * P, w.n_heads, w.topk, w.softmax_scale)
    idx = torch.empty((w.n_q, w.topk), dtype=torch.int32, device=dev)
    out = torch.empty((w.n_q, w.n_heads, w.d_v), dtype=torch.bfloat16, device=dev)
    iws = torch.empty(D.dsa_indexer_workspace_size(idesc), dtype=torch.uint8, device=dev)
    aws = torch.empty(D.dsa_sparse_attn_workspace_size(adesc), dtype=torch.uint8, device=dev)

    def timed(fn):
        fn()
        ms = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.median(ms)

    i_ms = timed(lambda: D.dsa_indexer_topk_paged(idesc, L0["q_idx"], k_cache, L0["w"], q_pos, pages, rope, idx, None,
                                                  ws=iws, stream=stream))
    if D.dsa_workspace_status(iws) != 0:
        raise RuntimeError("device status set by the paged indexer")
    same = bool(torch.equal(idx, idx_full))
    a_ms = timed(lambda: D.dsa_sparse_attn_paged(adesc, L0["q"], kv_cache, idx, pages, out, None, ws=aws,
                                                 stream=stream))
    if D.dsa_workspace_status(aws) != 0:
        raise RuntimeError("device status set by the paged attention")
    return {"page_rows": P, "n_pages": n_pages, "indexer_ms": i_ms, "attn_ms": a_ms,
            "contiguous_indexer_ms": idx_ms_contig, "contiguous_attn_ms": attn_ms_contig,
            "indices_equal_contiguous": same}


# --------------------------------------------------------------------------- native arm
def run_native(args):
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws_n, "nccl")
    from dsa_indexer_cross_gb300.build import build
    build()
    import dsa_indexer_cross_gb300 as D
    from dsa_indexer_cross_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    geo = synth.geometry(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q_pos, k_pos, ks, ke = t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke)
    # a profiler capture (--only) needs the first layer alone
    layers = build_inputs(w, geo, dev, n_layers=1 if args.only is not None else None)
    cache = D.IndexCache(w.layers, w.n_q, w.topk, device=dev)
    flags = D.DSA_IDX_ROPE_Q | (D.DSA_IDX_ROPE_K if w.rope_k else 0)
    if w.kind == "decode":
        flags |= D.DSA_IDX_INDEPENDENT_ROWS
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len, flags)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(dev)
    ws = torch.empty(D.dsa_layers_workspace_size(idesc, adesc), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def step():
        D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache, ws=ws,
                                    stream=stream)

    if args.only is not None:
        # one indexer pass to produce real indices, then the requested kernel once
        L0 = layers[0]
        idx0 = cache.buffers[0]
        iws = torch.empty(D.dsa_indexer_workspace_size(idesc), dtype=torch.uint8, device=dev)
        D.dsa_indexer_topk(idesc, L0["q_idx"], L0["k_idx"], L0["w"], q_pos, k_pos, ks, ke, rope, idx0, None, ws=iws,
                           stream=stream)
        if args.only == "attn":
            D.dsa_sparse_attn(adesc, L0["q"], L0["kv"], idx0, ks, L0["out"], L0["lse"], stream=stream)
        else:
            D.dsa_indexer_topk(idesc, L0["q_idx"], L0["k_idx"], L0["w"], q_pos, k_pos, ks, ke, rope, idx0, None,
                               ws=iws, stream=stream)
        torch.cuda.synchronize()
        return 0

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set during warm-up")

    # ---------------- timed steps (device-resident inputs)
    barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = [a.elapsed_time(b) for a, b in evs]
    ms_step = max_over_ranks(sum(ms) / len(ms), dev)
    value = ws_n * w.n_q / (ms_step / 1e3)

    # ---------------- per-kernel timing of the dominant kernel (sparse attention) and the indexer
    idx_full = cache.buffers[0]
    attn_ws = torch.empty(D.dsa_sparse_attn_workspace_size(adesc), dtype=torch.uint8, device=dev)
    idx_ws = torch.empty(D.dsa_indexer_workspace_size(idesc), dtype=torch.uint8, device=dev)
    L0 = layers[0]

    def time_call(fn, n):
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        fn()
        for a, b in e:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in e)

    attn_ms = time_call(lambda: D.dsa_sparse_attn(adesc, L0["q"], L0["kv"], idx_full, ks, L0["out"], L0["lse"],
                                                  ws=attn_ws, stream=stream), 20)
    idx_ms = time_call(lambda: D.dsa_indexer_topk(idesc, L0["q_idx"], L0["k_idx"], L0["w"], q_pos, k_pos, ks, ke, rope,
                                                  idx_full, None, ws=idx_ws, stream=stream), 20)

    # ---------------- per-phase split of the indexer call (CUDA events between its launches,
    # recorded only in this separate loop); median over 20 calls, L2 flushed before each
    D.dsa_profile_enable(True)
    phases = []
    try:
        for _ in range(20):
            flush.zero_()
            D.dsa_indexer_topk(idesc, L0["q_idx"], L0["k_idx"], L0["w"], q_pos, k_pos, ks, ke, rope, idx_full, None,
                               ws=idx_ws, stream=stream)
            phases.append(D.dsa_profile_indexer_last())
    finally:
        D.dsa_profile_enable(False)
    phase_ms = [statistics.median(p[i] for p in phases) for i in range(4)]

    # ---------------- end to end through the C ABI from pinned host buffers: every layer's
    # inputs are uploaded and every layer's output downloaded inside the timed region, with
    # the library's host pipeline overlapping the transfers of one layer with the kernels of
    # another
    from dsa_indexer_cross_gb300.pipeline import HostLayerPipeline
    in_keys = ("q_idx", "k_idx", "w", "q", "kv")
    host_in = [{k: v.cpu().pin_memory() for k, v in L.items() if k in in_keys} for L in layers]
    host_out = [torch.empty(L["out"].shape, dtype=L["out"].dtype).pin_memory() for L in layers]
    h2d = sum(v.numel() * v.element_size() for H in host_in for v in H.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out)
    pipe = HostLayerPipeline(idesc, adesc, w.layers, host_in, dev)

    def e2e_step():
        pipe.forward(host_in, host_out, ks, ke, q_pos, k_pos, rope, stream=stream)

    e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(max(3, args.steps // 2))]
    for a, b in e2e_ev:
        a.record(stream)
        e2e_step()
        b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev) / len(e2e_ev), dev)
    if D.dsa_workspace_status(pipe.iws) != 0 or D.dsa_workspace_status(pipe.aws) != 0:
        raise RuntimeError("device status set during the end-to-end steps")
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set during the timed region")

    hbm, tc_burst, tc_sus, peak_kind = peaks()
    R = roofline_numbers(w, geo)
    hbm_bound_attn = geo.n_kv * w.d_qk * 2 > (64 << 20)   # one layer's latent cache well beyond L2
    attn_gbs = R["attn_gathered"] / (attn_ms / 1e3) / 1e9
    attn_strict_tflops = R["attn_flops"] / (attn_ms / 1e3) / 1e12
    idx_tflops = R["idx_flops"] / (idx_ms / 1e3) / 1e12
    idx_gbs = R["idx_bytes"] / (idx_ms / 1e3) / 1e9
    score_tflops = R["idx_flops"] / (phase_ms[2] / 1e3) / 1e12
    gpu_launches = sum((3 if t == "full" else 0) + 2 for t in w.layers) + 2 * sum(t == "full" for t in w.layers)

    line = {
        "metric": "indexer+top-k and sparse-attn query-tokens/sec",
        "value": value, "unit": "query_tokens/s", "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (fp32 accumulate)", "data": "synthetic (seeded Gaussian, bf16)",
        "config": {"workload": f"{w.name}: {w.n_q} queries ({w.kind}, {geo.n_kv} keys), {len(w.layers)} layers "
                               f"{''.join(t[0].upper() for t in w.layers)}, H_I={w.n_heads_idx}x{w.head_dim_idx} "
                               f"(rope {w.rope_dim}, theta {w.theta:g}), topk={w.topk}, H={w.n_heads} 576/512",
                   "l2": "flushed between timed steps (512 MiB write outside the events)",
                   "parallelism": "replicas" if ws_n > 1 else "single GPU"},
        "e2e": {"value": ws_n * w.n_q / (e2e_ms / 1e3), "unit": "query_tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": gpu_launches * args.steps,
        # While one layer's latent cache is L2-resident (prefill_4k, long_32k) the binding
        # roofline of the attention is the tensor one: selected (query, head, row) triples x
        # (576 + 512) x 2 FLOPs.  A cache far larger than L2 (chunk_1m, decode_64) makes it the
        # HBM one: every token gathers its own rows (the per-token gather bytes).  Both framings
        # and the minimum HBM bytes (inputs once + outputs) are given either way.
        "roofline": dict(({"bound": "hbm", "achieved": attn_gbs, "peak": hbm, "unit": "GB/s",
                           "frac": attn_gbs / hbm, "peak_kind": peak_kind + " (HBM copy)"}
                          if hbm_bound_attn else
                          {"bound": "tensor", "achieved": attn_strict_tflops, "peak": tc_burst, "unit": "TFLOP/s",
                           "frac": attn_strict_tflops / tc_burst, "peak_kind": peak_kind + " (bf16 burst)"}),
                     kernel="sparse_attn_kernel", traffic=ATTN_TRAFFIC_BYTES.get(w.name),
                     tensor_tflops=attn_strict_tflops, tensor_frac=attn_strict_tflops / tc_burst,
                     algorithmic_flops_per_launch=R["attn_flops"], ms_per_launch=attn_ms,
                     **{
                        "min_hbm_bytes_per_launch": R["attn_min_bytes"],
                        "min_hbm_frac": R["attn_min_bytes"] / (attn_ms / 1e3) / 1e9 / hbm,
                        "per_token_gather_bytes_per_launch": R["attn_gathered"], "per_token_gather_gbs": attn_gbs,
                        # the gather framing of the roofline (each token reads its own rows from HBM);
                        # above 1 means rows were reused from L2 / shared memory across tokens
                        "per_token_gather_frac_of_hbm": attn_gbs / hbm}),
        # decode scores 64 flop per byte of index keys: bound by HBM, not by the tensor cores
        "roofline_indexer": dict(({"bound": "hbm", "achieved": idx_gbs, "peak": hbm, "unit": "GB/s",
                                   "frac": idx_gbs / hbm, "peak_kind": peak_kind + " (HBM copy)"}
                                  if w.kind == "decode" else
                                  {"bound": "tensor", "achieved": idx_tflops, "peak": tc_burst, "unit": "TFLOP/s",
                                   "frac": idx_tflops / tc_burst, "peak_kind": peak_kind + " (bf16 burst)"}),
                                 kernel="indexer call (rope + tcgen05 scores/top-k + select)",
                                 algorithmic_flops_per_launch=R["idx_flops"], algorithmic_bytes_per_launch=R["idx_bytes"],
                                 causal_flops_per_launch=R["idx_flops_causal"], ms_per_launch=idx_ms),
        # the tensor-core score kernel of that call on its own (events between the call's launches)
        "roofline_indexer_kernel": {"kernel": "indexer_kernel (tcgen05 scores + streaming top-k)", "bound": "tensor",
                                    "achieved": score_tflops, "peak": tc_burst, "unit": "TFLOP/s",
                                    "frac": score_tflops / tc_burst, "algorithmic_flops_per_launch": R["idx_flops"],
                                    "ms_per_launch": phase_ms[2], "peak_kind": peak_kind + " (bf16 burst)",
                                    "call_phase_ms": {"rope": phase_ms[0], "ranges": phase_ms[1],
                                                      "scores_topk": phase_ms[2], "select": phase_ms[3]}},
        "clocks": clk.summary(),
    }
    if args.proj:
        line["proj"] = time_proj(D, w, dev, stream, flush, tc_burst)
    if args.bwd:
        line["bwd"] = time_bwd(D, w, adesc, layers[0], idx_full, ks, attn_ms, R["attn_flops"], dev, stream, flush,
                               tc_burst)
    if args.paged and w.kind == "decode":
        line["paged"] = time_paged(D, synth, w, geo, layers[0], idx_full, attn_ms, idx_ms, dev, stream, flush)
    if args.mtp_steps > 0 and w.kind == "decode":
        line["mtp"] = time_mtp(D, synth, w, args.mtp_steps, dev, stream, flush)
    if rank == 0 and not args.no_cpu_baseline:
        hl = host_layers(layers)
        rate, n_rows, spent = time_oracle(w, geo, hl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "query_tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{n_rows} query rows through all {len(w.layers)} layers "
                                          f"({spent:.1f} s of float64 NumPy)"}
    if rank == 0:
        print(json.dumps(line))
    cache.close()
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
