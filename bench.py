"""Benchmark of the IndexShare DSA hot path on one GB300 (or N independent replicas).

Headline workload (the largest one that fits one GPU): ``chunk_1m`` -- 4096 query tokens at
positions 1,044,480 ... 1,048,575 attending a 1,048,576-token causal prefix, 8 layers
(F S S S) x 2, 64 index heads x 128 (last 64 dims RoPE'd at theta 8e6), top-k 2048, 64
attention heads of 576/512.  One step = one ``indexshare_layers_forward`` over the 8 layers:
2 lightning-indexer + streaming top-k passes and 8 sparse-attention passes, every step of
the path in libdsa's kernels.

Prints one JSON line.  ``value`` = query tokens per second (whole job, inputs resident in
HBM), ``e2e`` = the same through the C ABI with every input copied from pinned host memory
and every layer output copied back inside the timed region.  Every kernel launch inside the
timed steps is logged by the library (CUDA events on the launching stream, recorded between
the launches), which gives each kernel's per-launch device time in the same run;
``roofline`` describes the kernel with the largest share of that time, ``roofline_indexer``
/ ``roofline_attn`` the two hot kernels either way.  ``cpu_baseline`` times the float64 CPU
oracle on a bounded sample of query rows.  ``workloads`` repeats the device measurement for
the other workloads (prefill_4k, long_32k, decode_64) with fewer steps.  ``--impl
reference`` times only the oracle.

Timing: W warm-up steps, then K steps each bracketed by CUDA events on the launching stream;
L2 is flushed (a 512 MiB write) between timed steps, outside the events.  nvidia-smi clocks
are sampled every 200 ms over everything that is timed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "chunk_1m"
EXTRA_WORKLOADS = "prefill_4k,long_32k,decode_64"
METRIC = "indexer+top-k and sparse-attn query-tokens/sec"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--extras", default=EXTRA_WORKLOADS,
                    help="comma-separated workloads also measured (device only) under 'workloads'; 'none' (or '') for none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--mtp-steps", type=int, default=0,
                    help="decode workloads: also time multi-step MTP drafting with IndexShare (indexer at step 0, "
                         "later steps reuse its indices) and report it under 'mtp'")
    ap.add_argument("--proj", action="store_true",
                    help="also time the indexer's input projections (wq_b, wk + k_norm, weights_proj) for the "
                         "workload's query rows, hidden width 6144 and query latent 2048, under 'proj'")
    ap.add_argument("--bwd", action="store_true",
                    help="also time the sparse-attention and indexer backward of the first layer for seeded "
                         "upstream gradients, under 'bwd'")
    ap.add_argument("--paged", action="store_true",
                    help="decode workloads: also time the paged-cache indexer and attention (128-row pages, "
                         "shuffled) against the contiguous calls on the same data, under 'paged'")
    ap.add_argument("--only", choices=["attn", "indexer", "indexer_bwd", "attn_bwd"], default=None,
                    help="run just one kernel call of the workload (for profiler captures); prints nothing")
    ap.add_argument("--n-q", type=int, default=0,
                    help="with --only: that many query rows of the workload instead of all (a smaller capture)")
    return ap.parse_args(argv)


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


def build_once(rank: int, world: int) -> None:
    """Compile libdsa.so on rank 0 only; the other ranks wait at a barrier and then load the
    library rank 0 wrote (no two ranks write the same build files)."""
    from dsa_indexer_cross_gb300.build import build
    if rank == 0:
        build()
    if world > 1:
        barrier()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

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
        sm, mx, pw, reasons = [], 0.0, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = max(mx, float(p[2]))
                pw.append(float(p[3]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "sm_mhz_min": min(sm), "power_w_max": max(pw) if pw else None}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


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
    """Algorithmic work of one launch of each hot kernel.

    Attention: every selected (query, row) pair costs 2 (576 + 512) FLOPs per head (the S and
    PV products) and, read per token, 1152 bytes of latent row.  Indexer: every (query, key)
    pair of a row whose prefix is longer than k costs 2 H_I d_I FLOPs (rows with L <= k select
    their whole prefix and are never scored); its compulsory bytes are q, k and w read once
    and the indices written once.
    """
    L = (geo.ke - geo.ks).astype(np.int64)
    rows = np.minimum(L, w.topk).sum()                       # selected rows per layer
    pairs = L.sum()                                          # causal (query, key) pairs
    attn_gathered = rows * w.d_qk * 2 + w.n_q * w.n_heads * (w.d_qk + w.d_v) * 2 + w.n_q * w.topk * 4
    attn_flops = 2.0 * rows * w.n_heads * (w.d_qk + w.d_v)
    idx_flops_causal = 2.0 * pairs * w.n_heads_idx * w.head_dim_idx
    idx_flops = 2.0 * L[L > w.topk].sum() * w.n_heads_idx * w.head_dim_idx
    idx_bytes = (w.n_q * w.n_heads_idx * w.head_dim_idx * 2 + geo.n_kv * w.head_dim_idx * 2 + w.n_q * w.n_heads_idx * 4
                 + w.n_q * w.topk * 4)
    attn_min_bytes = (w.n_q * w.n_heads * w.d_qk * 2 + geo.n_kv * w.d_qk * 2 + w.n_q * w.topk * 4
                      + w.n_q * w.n_heads * (w.d_v * 2 + 4))
    return dict(attn_gathered=float(attn_gathered), attn_flops=attn_flops, idx_flops=idx_flops,
                idx_flops_causal=idx_flops_causal, idx_bytes=float(idx_bytes), attn_min_bytes=float(attn_min_bytes),
                rows=int(rows), pairs=int(pairs))


# DRAM bytes (read + write) of one launch, from an ncu capture, keyed by (kernel, workload):
# (bytes, source file of the kernel, SHA-256 prefix of that file when the counters were taken,
# where the capture is summarised).  A kernel whose source has changed since reports None.
# chunk_1m's indexer was captured on a 608-query slice (152 of the 1024 key streams; a whole
# launch is too long for a full-set capture) and is scaled by the 4096 / 608 units: each
# group streams the same chunks, so the traffic grows with the number of groups.
MEASURED_TRAFFIC = {
    ("indexer", "chunk_1m"): ((1.031415e9 + 0.618000e9) * 4096 / 608, ("indexer.cu", "api.cu"), "ebfe4a38773bb214",
                              "profiles/indexer_chunk_1m.md (608-query slice, scaled by 4096/608)"),
}


def _src_sha(rels) -> str:
    """SHA-256 (first 16 hex digits) over the named csrc files with their whitespace removed:
    the kernel and the host code that plans its launch (buffer sizes change its traffic too);
    a change of layout alone keeps the figure."""
    h = hashlib.sha256()
    for rel in rels:
        with open(os.path.join(ROOT, "dsa_indexer_cross_gb300", "csrc", rel), "rb") as f:
            h.update(re.sub(rb"\s+", b"", f.read()))
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    t = MEASURED_TRAFFIC.get((kernel, workload))
    if t is None:
        return None, "no ncu capture of the current kernel for this workload"
    nbytes, src, sha, where = t
    if _src_sha(src) != sha:
        return None, f"{', '.join(src)} changed since the capture in {where}"
    return nbytes, f"ncu dram__bytes_read.sum + dram__bytes_write.sum, {where}"


# --------------------------------------------------------------------------- oracle inputs
class LazyRows:
    """Row access to a CPU bf16 / fp32 tensor as float64 NumPy, converted on demand, so the
    oracle can read a 1M-row latent cache without a 5 GB float64 copy of every layer."""

    def __init__(self, t: torch.Tensor):
        self.t = t.detach().to("cpu")
        self.shape = tuple(self.t.shape)

    def __getitem__(self, i):
        if isinstance(i, np.ndarray):
            i = torch.from_numpy(np.ascontiguousarray(i.astype(np.int64)))
        elif isinstance(i, (np.integer,)):
            i = int(i)
        return self.t[i].to(torch.float64).numpy()

    def __array__(self, dtype=None, copy=None):
        a = self.t.to(torch.float64).numpy()
        return a if dtype is None else a.astype(dtype, copy=False)


def oracle_layers(layers):
    keys = ("q_idx", "k_idx", "w", "q", "kv")
    return [{k: LazyRows(v) for k, v in L.items() if k in keys} for L in layers]


def time_oracle(w, geo, layers_host, budget_s: float, max_rows: int = 512):
    """Run the float64 oracle over all layers on growing row samples until ~budget_s of work."""
    from oracle import dsa_oracle as O
    rng = np.random.default_rng(7)
    n = 1 if w.kind == "chunk" else 4
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
        n = min(max_rows, max(n * 2, int(n * (budget_s - spent) / max(dt, 1e-3))))
    return done_rows / spent, done_rows, spent


def workload_label(w, geo):
    return (f"{w.name}: {w.n_q} queries ({w.kind}, {geo.n_kv} keys), {len(w.layers)} layers "
            f"{''.join(t[0].upper() for t in w.layers)}, H_I={w.n_heads_idx}x{w.head_dim_idx} "
            f"(rope {w.rope_dim}, theta {w.theta:g}), topk={w.topk}, H={w.n_heads} 576/512")


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from dsa_indexer_cross_gb300 import synth
    from oracle import dsa_oracle as O
    w = synth.WORKLOADS[args.workload]
    geo = synth.geometry(w)
    hl = oracle_layers([synth.layer_inputs(w, geo, l, device="cpu") for l in range(len(w.layers))])
    # the oracle rotates every index key of the prefix per call, so a 1M-key step is one row
    rows_per_step = 1 if w.kind == "chunk" else 8
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
    sample = f"{rows_per_step} random query rows x {len(w.layers)} layers per step"
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "query_tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded Gaussian, bf16 inputs)",
            "config": {"workload": workload_label(w, geo), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "query_tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "query_tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- device measurement
def kernel_stats(log, steps):
    """Per kernel kind: launches, mean and total device ms over the timed steps."""
    out = {}
    for kind, ms in log:
        d = out.setdefault(kind, {"launches": 0, "total_ms": 0.0})
        d["launches"] += 1
        d["total_ms"] += ms
    for d in out.values():
        d["ms_per_launch"] = d["total_ms"] / d["launches"]
    return out


def measure(D, w, steps, warmup, dev, stream, flush, rank=0, world=1, keep=False):
    """Time `steps` layer-loop steps of workload w with device-resident inputs and read every
    launch's device time from the library's launch log.  Returns (result dict, state) where
    state holds the tensors for the end-to-end and oracle legs when keep is set."""
    from dsa_indexer_cross_gb300 import synth
    geo = synth.geometry(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q_pos, k_pos, ks, ke = t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke)
    layers = build_inputs(w, geo, dev)
    cache = D.IndexCache(w.layers, w.n_q, w.topk, device=dev)
    flags = D.DSA_IDX_ROPE_Q | (D.DSA_IDX_ROPE_K if w.rope_k else 0)
    if w.kind == "decode":
        flags |= D.DSA_IDX_INDEPENDENT_ROWS
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len, flags)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(dev)
    ws = torch.empty(D.dsa_layers_workspace_size(idesc, adesc), dtype=torch.uint8, device=dev)

    def step():
        D.indexshare_layers_forward(idesc, adesc, w.layers, layers, ks, ke, q_pos, k_pos, rope, cache, ws=ws,
                                    stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set during warm-up")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    D.dsa_profile_enable(True)
    try:
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        log = D.dsa_profile_read()
    finally:
        D.dsa_profile_enable(False)
    barrier()
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set during the timed steps")
    ms = [a.elapsed_time(b) for a, b in evs]
    ms_step = max_over_ranks(sum(ms) / len(ms), dev)
    timed_s = sum(ms) / 1e3
    ks_ = kernel_stats(log, steps)

    hbm, tc_burst, tc_sus, peak_kind = peaks()
    # a kernel timed inside a loop that runs for seconds is held to the sustained (power-capped)
    # bf16 peak, one timed inside a short loop to the burst peak
    long_loop = timed_s > 1.0
    tc = tc_sus if long_loop else tc_burst
    tc_kind = f"{peak_kind} bf16 {'sustained' if long_loop else 'burst'} ({timed_s:.2f} s timed loop)"
    R = roofline_numbers(w, geo)
    n_full = sum(t_ == "full" for t_ in w.layers)

    a_ms = ks_["attn"]["ms_per_launch"]
    attn_gbs = R["attn_gathered"] / (a_ms / 1e3) / 1e9
    attn_tf = R["attn_flops"] / (a_ms / 1e3) / 1e12
    hbm_bound_attn = geo.n_kv * w.d_qk * 2 > (64 << 20)   # one layer's latent cache well beyond L2
    a_traffic, a_tsrc = traffic_for("attn", w.name)
    roof_attn = dict(({"bound": "hbm", "achieved": attn_gbs, "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm,
                       "peak_kind": peak_kind + " HBM copy"}
                      if hbm_bound_attn else
                      {"bound": "tensor", "achieved": attn_tf, "peak": tc, "unit": "TFLOP/s", "frac": attn_tf / tc,
                       "peak_kind": tc_kind}),
                     kernel="sparse_attn_kernel", launches=ks_["attn"]["launches"], ms_per_launch=a_ms,
                     traffic=a_traffic, traffic_source=a_tsrc, tensor_tflops=attn_tf, tensor_frac_of_burst=attn_tf / tc_burst,
                     algorithmic_flops_per_launch=R["attn_flops"], per_token_gather_bytes_per_launch=R["attn_gathered"],
                     per_token_gather_frac_of_hbm=attn_gbs / hbm, min_hbm_bytes_per_launch=R["attn_min_bytes"],
                     min_hbm_frac=R["attn_min_bytes"] / (a_ms / 1e3) / 1e9 / hbm)

    i_ms = ks_["indexer"]["ms_per_launch"]
    call_kinds = ("rope", "ranges", "indexer", "select")
    call_ms = sum(ks_[k]["total_ms"] for k in call_kinds if k in ks_) / (n_full * steps)
    i_traffic, i_tsrc = traffic_for("indexer", w.name)
    if w.kind == "decode":
        # decode scores 64 flop per byte of index keys: bound by HBM, not by the tensor cores
        ach = R["idx_bytes"] / (i_ms / 1e3) / 1e9
        roof_idx = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                    "peak_kind": peak_kind + " HBM copy", "algorithmic_bytes_per_launch": R["idx_bytes"]}
        call_ach = R["idx_bytes"] / (call_ms / 1e3) / 1e9
        call_roof = {"bound": "hbm", "achieved": call_ach, "peak": hbm, "unit": "GB/s", "frac": call_ach / hbm}
    else:
        ach = R["idx_flops"] / (i_ms / 1e3) / 1e12
        roof_idx = {"bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s", "frac": ach / tc,
                    "peak_kind": tc_kind, "frac_of_burst": ach / tc_burst,
                    "algorithmic_flops_per_launch": R["idx_flops"], "causal_flops_per_launch": R["idx_flops_causal"]}
        call_ach = R["idx_flops"] / (call_ms / 1e3) / 1e12
        call_roof = {"bound": "tensor", "achieved": call_ach, "peak": tc, "unit": "TFLOP/s", "frac": call_ach / tc,
                     "frac_of_burst": call_ach / tc_burst}
    roof_idx.update(kernel="indexer_kernel (tcgen05 scores + streaming top-k)", launches=ks_["indexer"]["launches"],
                    ms_per_launch=i_ms, traffic=i_traffic, traffic_source=i_tsrc)
    call_roof.update(kernel="indexer call (" + " + ".join(k for k in call_kinds if k in ks_) + ")",
                     ms_per_full_layer=call_ms,
                     phase_ms_per_full_layer={k: ks_[k]["total_ms"] / (n_full * steps) for k in call_kinds if k in ks_})

    # the dominant kernel: the largest share of the timed steps' device time
    dom = max(("indexer", "attn"), key=lambda k: ks_[k]["total_ms"])
    roofline = dict(roof_idx if dom == "indexer" else roof_attn)
    res = {
        "value": world * w.n_q / (ms_step / 1e3), "ms_per_step": ms_step, "config": workload_label(w, geo),
        "gpu_launches": len(log), "timed_s": timed_s,
        "kernels": {k: {"launches": v["launches"], "ms_per_launch": v["ms_per_launch"],
                        "share_of_step": v["total_ms"] / sum(ms)} for k, v in ks_.items()},
        "roofline": roofline, "roofline_indexer": roof_idx, "roofline_indexer_call": call_roof,
        "roofline_attn": roof_attn,
    }
    state = None
    if keep:
        state = dict(geo=geo, layers=layers, cache=cache, idesc=idesc, adesc=adesc, rope=rope, ws=ws, q_pos=q_pos,
                     k_pos=k_pos, ks=ks, ke=ke, R=R, attn_ms=a_ms, idx_ms=i_ms, tc=tc)
    else:
        cache.close()
    return res, state


def measure_e2e(D, w, st, steps, dev, stream, world=1):
    """End to end through the C ABI from pinned host buffers: every layer's inputs are uploaded
    and every layer's output downloaded inside the timed region, with the library's host
    pipeline overlapping the transfers of one layer (and of the next pass) with the kernels of
    another."""
    from dsa_indexer_cross_gb300.pipeline import HostLayerPipeline
    in_keys = ("q_idx", "k_idx", "w", "q", "kv")
    host_in = [{k: v.cpu().pin_memory() for k, v in L.items() if k in in_keys} for L in st["layers"]]
    host_out = [torch.empty(L["out"].shape, dtype=L["out"].dtype).pin_memory() for L in st["layers"]]
    h2d = sum(v.numel() * v.element_size() for H in host_in for v in H.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out)
    pipe = HostLayerPipeline(st["idesc"], st["adesc"], w.layers, host_in, dev)

    def e2e_step():
        return pipe.forward(host_in, host_out, st["ks"], st["ke"], st["q_pos"], st["k_pos"], st["rope"], stream=stream)

    e2e_step()
    e2e_step()
    torch.cuda.synchronize()
    # consecutive passes overlap (the next one uploads while this one computes): the time is
    # from the first pass's start on the compute stream to the last pass's last download
    start = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    pipe.up.wait_event(start)
    pipe.down.wait_event(start)
    ends = [e2e_step() for _ in range(steps)]
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(start.elapsed_time(ends[-1]) / steps, dev)
    if D.dsa_workspace_status(pipe.iws) != 0 or D.dsa_workspace_status(pipe.aws) != 0:
        raise RuntimeError("device status set during the end-to-end steps")
    res = {"value": world * w.n_q / (e2e_ms / 1e3), "unit": "query_tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": steps,
           "schedule": "every byte copied inside the timed region; uploads on their own stream, a "
                       "pass's uploads overlap the previous pass's kernels (two device sets), each "
                       "layer's output downloads as soon as its attention ends"}
    del pipe
    return res, host_in


def logged_ms(D, fn, reps, flush, kind):
    """Median device ms of the `kind` launches of fn() over reps calls (L2 flushed before
    each), read from the library's launch log."""
    fn()
    torch.cuda.synchronize()
    D.dsa_profile_enable(True)
    try:
        for _ in range(reps):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        log = D.dsa_profile_read()
    finally:
        D.dsa_profile_enable(False)
    ms = [m for k, m in log if k == kind]
    return statistics.median(ms)
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
    """Median kernel time of dsa_indexer_projections for the workload's query rows (synthetic
    weights), against the bf16 peak on its FLOPs: 2 T (H_I d_I d_q + d_I d_h + H_I d_h)."""
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
    m = logged_ms(D, lambda: D.dsa_indexer_projections(desc, x, ql, wq, wk, gamma, beta, wp, q_idx, k_idx, wo, ws=ws,
                                                       stream=stream), reps, flush, "proj")
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set by the projections")
    flops = 2.0 * T * (H * d * d_q + d * d_hidden + H * d_hidden)
    return {"d_hidden": d_hidden, "d_q": d_q, "ms": m, "tflops": flops / (m / 1e3) / 1e12,
            "frac_of_bf16_peak": flops / (m / 1e3) / 1e12 / tc_peak,
            "note": "synthetic weights; widths assumed (the pages give none); kernel time from the launch log"}


# --------------------------------------------------------------------------- backward
def time_bwd(D, w, st, dev, stream, flush, tc_peak, reps: int = 5):
    """Kernel times of the backward passes on the first layer (seeded upstream gradients), from
    the launch log, L2 flushed before each call.  Attention backward FLOPs: 2.5x the forward's
    (S and dP recomputed, then dQ, dS^T Q and P^T dO).  Indexer backward FLOPs: the scores of
    the selected keys recomputed (2 H_I d_I per pair) plus dq and dk (2 H_I d_I each)."""
    L0, idx, ks, adesc, R = st["layers"][0], st["cache"].buffers[0], st["ks"], st["adesc"], st["R"]
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    d_out = torch.randn(L0["out"].shape, generator=g, device=dev).to(torch.bfloat16)
    dq = torch.empty((w.n_q, w.n_heads, w.d_qk), dtype=torch.float32, device=dev)
    dkv = torch.empty((adesc.n_kv, w.d_qk), dtype=torch.float32, device=dev)
    ws = torch.zeros(D.dsa_sparse_attn_backward_workspace_size(adesc), dtype=torch.uint8, device=dev)
    tc = ws.numel() > 256   # the tcgen05 walks need more than the status words
    D.dsa_sparse_attn(adesc, L0["q"], L0["kv"], idx, ks, L0["out"], L0["lse"], stream=stream)
    m = logged_ms(D, lambda: D.dsa_sparse_attn_backward(adesc, L0["q"], L0["kv"], idx, ks, L0["out"], L0["lse"], d_out,
                                                        dq, dkv, ws=ws, stream=stream), reps, flush, "attn_bwd")
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set by the backward")
    flops = 2.5 * R["attn_flops"]
    out = {"attn": {"ms": m, "forward_ms": st["attn_ms"], "flops": flops, "tflops": flops / (m / 1e3) / 1e12,
                    "frac_of_bf16_peak": flops / (m / 1e3) / 1e12 / tc_peak,
                    "kernel": ("attn_bwd_tc_kernel (tcgen05" if tc else "sparse_attn_bwd_kernel (mma.sync") +
                              "; kernel time from the launch log, dkv cleared before it)"}}
    if hasattr(D, "dsa_indexer_backward"):
        out["indexer"] = time_indexer_bwd(D, w, st, dev, stream, flush, tc_peak, reps)
    return out


def time_indexer_bwd(D, w, st, dev, stream, flush, tc_peak, reps: int = 5):
    """Kernel time of dsa_indexer_backward on the first layer's index inputs and selected keys
    (seeded upstream gradient), from the launch log, L2 flushed before each call.  FLOPs: three
    products per selected (query, key) pair, 2 H_I d_I each (scores recomputed, dq, dk)."""
    L0, idx, R = st["layers"][0], st["cache"].buffers[0], st["R"]
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    d_score = torch.randn((w.n_q, w.topk), generator=g, device=dev)
    dq = torch.empty((w.n_q, w.n_heads_idx, w.head_dim_idx), dtype=torch.float32, device=dev)
    dk = torch.empty((st["geo"].n_kv, w.head_dim_idx), dtype=torch.float32, device=dev)
    dw = torch.empty((w.n_q, w.n_heads_idx), dtype=torch.float32, device=dev)
    desc = st["idesc"]
    ws = torch.empty(D.dsa_indexer_backward_workspace_size(desc), dtype=torch.uint8, device=dev)
    m = logged_ms(D, lambda: D.dsa_indexer_backward(desc, L0["q_idx"], L0["k_idx"], L0["w"], st["q_pos"], st["k_pos"],
                                                    st["ks"], st["ke"], st["rope"], idx, d_score, dq, dk, dw, ws=ws,
                                                    stream=stream), reps, flush, "indexer_bwd")
    if D.dsa_workspace_status(ws) != 0:
        raise RuntimeError("device status set by the indexer backward")
    flops = 3 * 2.0 * R["rows"] * w.n_heads_idx * w.head_dim_idx
    return {"ms": m, "flops": flops, "tflops": flops / (m / 1e3) / 1e12,
            "frac_of_bf16_peak": flops / (m / 1e3) / 1e12 / tc_peak,
            "kernel": "indexer_bwd_kernel + RoPE transpose passes (launch log; dk and dw cleared before)"}


# --------------------------------------------------------------------------- paged caches
def time_paged(D, synth, w, geo, L0, idx_full, attn_ms_contig, idx_ms_contig, dev, stream, flush, reps: int = 20,
               seed: int = 3):
    """The same decode layer with its index-key and latent caches in shuffled 128-row pages behind a
    block table: median kernel times (launch log) of the paged indexer and attention kernels (L2
    flushed before each call), beside the contiguous kernels' times."""
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

    i_ms = logged_ms(D, lambda: D.dsa_indexer_topk_paged(idesc, L0["q_idx"], k_cache, L0["w"], q_pos, pages, rope, idx,
                                                         None, ws=iws, stream=stream), reps, flush, "indexer")
    if D.dsa_workspace_status(iws) != 0:
        raise RuntimeError("device status set by the paged indexer")
    same = bool(torch.equal(idx, idx_full))
    a_ms = logged_ms(D, lambda: D.dsa_sparse_attn_paged(adesc, L0["q"], kv_cache, idx, pages, out, None, ws=aws,
                                                        stream=stream), reps, flush, "attn")
    if D.dsa_workspace_status(aws) != 0:
        raise RuntimeError("device status set by the paged attention")
    return {"page_rows": P, "n_pages": n_pages, "indexer_ms": i_ms, "attn_ms": a_ms,
            "contiguous_indexer_ms": idx_ms_contig, "contiguous_attn_ms": attn_ms_contig,
            "indices_equal_contiguous": same}


# --------------------------------------------------------------------------- native arm
def run_only(D, w, args, dev, stream):
    """One indexer pass (real indices) then the requested kernel once, first layer only: the
    command a profiler capture wraps."""
    from dsa_indexer_cross_gb300 import synth
    geo = synth.geometry(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q_pos, k_pos, ks, ke = t(geo.q_pos), t(geo.k_pos), t(geo.ks), t(geo.ke)
    L0 = build_inputs(w, geo, dev, n_layers=1)[0]
    flags = D.DSA_IDX_ROPE_Q | (D.DSA_IDX_ROPE_K if w.rope_k else 0)
    if w.kind == "decode":
        flags |= D.DSA_IDX_INDEPENDENT_ROWS
    idesc = D.indexer_desc(w.n_q, geo.n_kv, w.n_heads_idx, w.head_dim_idx, w.rope_dim, w.topk, geo.max_len, flags)
    adesc = D.attn_desc(w.n_q, geo.n_kv, w.n_heads, w.topk, w.softmax_scale)
    rope = D.dsa_rope_table(w.theta, w.rope_dim, geo.max_pos).to(dev)
    idx0 = torch.empty((w.n_q, w.topk), dtype=torch.int32, device=dev)
    iws = torch.empty(D.dsa_indexer_workspace_size(idesc), dtype=torch.uint8, device=dev)
    call_idx = lambda: D.dsa_indexer_topk(idesc, L0["q_idx"], L0["k_idx"], L0["w"], q_pos, k_pos, ks, ke, rope, idx0,
                                          None, ws=iws, stream=stream)
    call_idx()
    if args.only == "attn":
        D.dsa_sparse_attn(adesc, L0["q"], L0["kv"], idx0, ks, L0["out"], L0["lse"], stream=stream)
    elif args.only == "attn_bwd":
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        D.dsa_sparse_attn(adesc, L0["q"], L0["kv"], idx0, ks, L0["out"], L0["lse"], stream=stream)
        d_out = torch.randn(L0["out"].shape, generator=g, device=dev).to(torch.bfloat16)
        dq = torch.empty((w.n_q, w.n_heads, w.d_qk), dtype=torch.float32, device=dev)
        dkv = torch.empty((geo.n_kv, w.d_qk), dtype=torch.float32, device=dev)
        D.dsa_sparse_attn_backward(adesc, L0["q"], L0["kv"], idx0, ks, L0["out"], L0["lse"], d_out, dq, dkv,
                                   stream=stream)
    elif args.only == "indexer_bwd":
        g = torch.Generator(device=dev)
        g.manual_seed(9)
        d_score = torch.randn((w.n_q, w.topk), generator=g, device=dev)
        dq = torch.empty((w.n_q, w.n_heads_idx, w.head_dim_idx), dtype=torch.float32, device=dev)
        dk = torch.empty((geo.n_kv, w.head_dim_idx), dtype=torch.float32, device=dev)
        dw = torch.empty((w.n_q, w.n_heads_idx), dtype=torch.float32, device=dev)
        D.dsa_indexer_backward(idesc, L0["q_idx"], L0["k_idx"], L0["w"], q_pos, k_pos, ks, ke, rope, idx0, d_score, dq,
                               dk, dw, stream=stream)
    else:
        call_idx()
    torch.cuda.synchronize()
    return 0


def run_native(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    build_once(rank, world)
    import dsa_indexer_cross_gb300 as D
    from dsa_indexer_cross_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(dev)
    if args.only is not None:
        if args.n_q > 0:
            w = w.replace(n_q=args.n_q)
        return run_only(D, w, args, dev, stream)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    hbm, tc_burst, tc_sus, peak_kind = peaks()

    with ClockSampler(local) as clk:
        res, st = measure(D, w, args.steps, args.warmup, dev, stream, flush, rank, world, keep=True)
        e2e, host_in = (None, None) if args.no_e2e else measure_e2e(D, w, st, max(3, args.steps // 2), dev, stream,
                                                                      world)
    line = {
        "metric": METRIC, "value": res["value"], "unit": "query_tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)", "data": "synthetic (seeded Gaussian, bf16)",
        "config": {"workload": res["config"],
                   "l2": "flushed between timed steps (512 MiB write outside the events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "e2e": e2e,
        "gpu_launches": res["gpu_launches"],
        "roofline": res["roofline"],
        "roofline_indexer": res["roofline_indexer"],
        "roofline_indexer_call": res["roofline_indexer_call"],
        "roofline_attn": res["roofline_attn"],
        "kernels": res["kernels"],
        "clocks": clk.summary(),
    }
    if args.proj:
        line["proj"] = time_proj(D, w, dev, stream, flush, tc_burst)
    if args.bwd:
        line["bwd"] = time_bwd(D, w, st, dev, stream, flush, tc_burst)
    if args.paged and w.kind == "decode":
        line["paged"] = time_paged(D, synth, w, st["geo"], st["layers"][0], st["cache"].buffers[0], st["attn_ms"],
                                   st["idx_ms"], dev, stream, flush)
    if args.mtp_steps > 0 and w.kind == "decode":
        line["mtp"] = time_mtp(D, synth, w, args.mtp_steps, dev, stream, flush)
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle reads the pinned host copies the end-to-end leg made (or fresh ones)
        src = host_in if host_in is not None else [{k: v.cpu() for k, v in L.items()} for L in st["layers"]]
        rate, n_rows, spent = time_oracle(w, st["geo"], oracle_layers(src), args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "query_tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{n_rows} query rows through all {len(w.layers)} layers "
                                          f"({spent:.1f} s of float64 NumPy)"}
    st["cache"].close()
    del st, host_in
    torch.cuda.empty_cache()

    # the other workloads, device-resident, fewer steps
    extras = [x for x in args.extras.split(",") if x and x not in (args.workload, "none")]
    if extras:
        line["workloads"] = {}
        with ClockSampler(local) as clk2:
            for name in extras:
                wx = synth.WORKLOADS[name]
                try:
                    r, _ = measure(D, wx, max(3, args.steps // 2), args.warmup, dev, stream, flush, rank, world)
                except Exception as exc:   # keep the headline line; say what failed
                    line["workloads"][name] = {"error": f"{type(exc).__name__}: {exc}"}
                    torch.cuda.empty_cache()
                    continue
                line["workloads"][name] = {
                    "value": r["value"], "ms_per_step": r["ms_per_step"], "config": r["config"],
                    "gpu_launches": r["gpu_launches"], "roofline": r["roofline"],
                    "roofline_indexer": r["roofline_indexer"], "roofline_indexer_call": r["roofline_indexer_call"],
                    "roofline_attn": r["roofline_attn"], "kernels": r["kernels"]}
                torch.cuda.empty_cache()
        line["workloads_clocks"] = clk2.summary()
    if rank == 0:
        print(json.dumps(line))
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
