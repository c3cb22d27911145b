// Host side of the C ABI declared in include/dsa.h: argument checks, workspace layout,
// tensor maps, the IndexShare donor schedule and index cache, and the layer loop.
// Nothing here computes a result on the host; every step of the path runs in a kernel.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/dsa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

namespace {

thread_local std::string g_err;

dsa_status fail(dsa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

dsa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device properties
struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

DevInfo dev_info() {
  static std::mutex mu;
  static std::vector<DevInfo> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DevInfo{};
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1);
  DevInfo& d = cache[dev];
  if (d.sms == 0) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
  }
  return d;
}

dsa_status check_device() {
  const DevInfo d = dev_info();
  if (d.sms == 0) return fail(DSA_ERR_UNSUPPORTED, "no CUDA device is available");
  if (d.major != 10 || d.minor != 3)
    return fail(DSA_ERR_UNSUPPORTED, "libdsa is built for sm_103a; the current device is sm_%d%d", d.major, d.minor);
  return DSA_OK;
}

// ------------------------------------------------------------------ phase profiling
// Five events per device bracket the four phases of an indexer call while profiling is on.
std::atomic<int> g_profile{0};
struct PhaseEvents {
  cudaEvent_t ev[5];
  bool created = false;
  bool recorded = false;
};
PhaseEvents g_phase[64];
std::mutex g_phase_mu;

// The current device's events, created on first use; nullptr when profiling is off or the
// events cannot be created.
PhaseEvents* phase_events() {
  if (!g_profile.load(std::memory_order_relaxed)) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_phase_mu);
  PhaseEvents& p = g_phase[dev];
  if (!p.created) {
    for (int i = 0; i < 5; ++i) {
      if (cudaEventCreate(&p.ev[i]) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
      }
    }
    p.created = true;
  }
  return &p;
}

// ------------------------------------------------------------------ pipeline test hook
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<int> g_stop_after{-1};

// ------------------------------------------------------------------ launch log
// Per device: a fixed ring of event pairs, created on first use and kept; records are
// appended while profiling is on and read back (after their events complete) by
// dsa_profile_read.  A full log drops further records and says so.
constexpr int kLogCap = 8192;
struct LaunchLog {
  cudaEvent_t ev[kLogCap][2];
  int kind[kLogCap];
  int n_created = 0;   // event pairs created so far
  int n = 0;           // records in the log
  bool dropped = false;
};
LaunchLog* g_log[64] = {};
std::mutex g_log_mu;

LaunchLog* launch_log(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  if (!g_log[dev]) g_log[dev] = new (std::nothrow) LaunchLog;
  return g_log[dev];
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows][inner], 128-byte swizzled boxes of {64, box_rows}.
dsa_status tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return DSA_OK;
}

// Latent cache [rows][576] bf16 viewed as (64 dims, rows, 9 blocks of 64 dims): one box
// {64, 64, 9} is a whole 64-row tile, landing in shared memory as nine 64-row x 128-byte
// blocks (128-byte swizzle), the layout the attention kernel reads.  One copy per tile keeps
// the TMA unit far busier than nine per-block copies.
dsa_status tmap_kv_tiles(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {64, rows, 9};
  cuuint64_t strides[2] = {576 * 2, 64 * 2};
  cuuint32_t box[3] = {64, 64, 9};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled (latent tiles) failed (%d)", static_cast<int>(r));
  return DSA_OK;
}

// ------------------------------------------------------------------ indexer plan
bool supported_heads(int h) { return h == 4 || h == 8 || h == 16 || h == 32 || h == 64; }

struct IndexerLayout {
  IndexerPlan plan{};
  size_t off_q = 0, off_k = 0, off_rr = 0, off_gr = 0, off_units = 0, off_cnt = 0, off_edge = 0,
         off_key = 0, off_idx = 0, total = 0;
};

dsa_status check_indexer_desc(const dsa_indexer_desc* d) {
  if (!d) return fail(DSA_ERR_ARG, "indexer descriptor is NULL");
  if (d->n_q < 0 || d->n_kv < 0) return fail(DSA_ERR_ARG, "n_q and n_kv must be >= 0");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(DSA_ERR_UNSUPPORTED, "index head_dim %d: supported values are 64 and 128", d->head_dim);
  if (!supported_heads(d->n_heads))
    return fail(DSA_ERR_UNSUPPORTED, "index n_heads %d: supported values are 4, 8, 16, 32, 64", d->n_heads);
  if (d->rope_dim < 0 || d->rope_dim > d->head_dim || (d->rope_dim & 1))
    return fail(DSA_ERR_ARG, "rope_dim %d must be even and within [0, head_dim]", d->rope_dim);
  if (d->topk < 1 || d->topk > 2048) return fail(DSA_ERR_UNSUPPORTED, "topk %d: supported range is 1..2048", d->topk);
  if (d->n_q > 0 && (d->max_len < 1 || d->max_len > d->n_kv))
    return fail(DSA_ERR_ARG, "max_len %d must lie in [1, n_kv=%d]", d->max_len, d->n_kv);
  if (d->flags & ~(DSA_IDX_ROPE_Q | DSA_IDX_ROPE_K | DSA_IDX_INDEPENDENT_ROWS))
    return fail(DSA_ERR_ARG, "unknown indexer flags 0x%x", d->flags);
  if (static_cast<long long>(d->n_q) * d->n_heads > 0x7FFFFFFFLL)
    return fail(DSA_ERR_SHAPE, "n_q * n_heads exceeds the int32 range");
  return DSA_OK;
}

IndexerLayout indexer_layout(const dsa_indexer_desc* d, int sms) {
  IndexerLayout L;
  IndexerPlan& p = L.plan;
  const bool indep = (d->flags & DSA_IDX_INDEPENDENT_ROWS) != 0;
  p.n_heads = d->n_heads;
  p.head_dim = d->head_dim;
  p.topk = d->topk;
  // G rows share a key stream: N = G * H_I <= 256 MMA columns, at most 16 rows (the score ring
  // of a unit holds one tile's scores of every row); independent rows fill only 64 columns
  p.group = indep ? (d->n_heads >= 64 ? 1 : 64 / d->n_heads) : std::min(256 / d->n_heads, 16);
  // independent rows have ranges of unequal length (decode), whose empty (group, chunk) slots
  // would leave CTAs idle: the kernel walks a dense list of the units that hold keys.  Shared-
  // prefix groups leave few slots empty and walk every pair in a computed order.
  p.unit_list = indep;
  p.n_groups = (d->n_q + p.group - 1) / p.group;
  const long long max_len = d->max_len > 0 ? d->max_len : 1;
  // keys one group's union of row ranges can span: a row's own range for prefill-like rows
  // (the rows of a group share their prefix), G separate ranges for independent rows
  long long span = max_len;
  if (indep && p.group > 1) span = std::min<long long>(static_cast<long long>(p.group) * max_len, std::max(d->n_kv, 1));
  long long chunk;
  if (p.n_groups >= 4LL * sms) {
    chunk = span;
  } else {
    chunk = (span * p.n_groups + 4LL * sms - 1) / (4LL * sms);
    if (chunk < 4096) chunk = 4096;
  }
  if (chunk > 262144) chunk = 262144;
  if (chunk < (span + 63) / 64) chunk = (span + 63) / 64;     // the final select reads <= 64 chunks
  chunk = (chunk + 127) / 128 * 128;
  p.chunk = static_cast<int>(chunk);
  p.n_chunks = static_cast<int>((span + chunk - 1) / chunk);
  // candidates per (row, chunk), in kSub sub-buffers: room for every key of the chunk, up to 64K
  // entries (chunks of more keys).  Rows longer than kDirectMax keys in the chunk are filtered by
  // the streaming threshold, which keeps about k (1 + ln(chunk / k)) keys with an exact
  // threshold (12K of a 256K chunk at k = 2048) and some 40 % more with its 1/16-octave histogram
  // bins, and the unit's end compacts them to those at or above the final threshold; the room
  // is for the keys kept before the threshold has risen.  A sub-buffer that fills anyway (scores
  // rising along the keys) is cut back to its top-k by its warp, a pass that holds up the whole
  // CTA: with 16K entries for 32K-key chunks and 32K for 256K-key chunks, ~44 K and ~7.5 K
  // cut-backs a call took long_32k's indexer to 21.0 ms and chunk_1m's to 65.3 ms, against
  // 11.1 and 51.4 ms with none.
  // A filtered sub-buffer is cut back once it holds more than cap / kSub - 32 entries: 128
  // entries beyond the chunk's keys keep a chunk that fits from ever reaching that mark
  // (decode's 13824-key chunks with cap = 13824 did, 0.27 -> 0.35 ms).
  const long long span_keys = std::min<long long>(chunk, span);
  const long long room = std::min<long long>(span_keys, 65536) + (span_keys > kDirectMax ? 128 : 0);
  p.cap = static_cast<int>((room + 127) / 128 * 128);
  const long long units = static_cast<long long>(p.n_groups) * p.n_chunks;
  p.grid = static_cast<int>(units < sms ? units : sms);
  if (p.grid < 1) p.grid = 1;

  size_t off = kAlign;  // header
  const bool rq = (d->flags & DSA_IDX_ROPE_Q) && d->rope_dim > 0;
  const bool rk = (d->flags & DSA_IDX_ROPE_K) && d->rope_dim > 0;
  L.off_q = off;
  if (rq) off += align_up(static_cast<size_t>(d->n_q) * d->n_heads * d->head_dim * 2);
  L.off_k = off;
  if (rk) off += align_up(static_cast<size_t>(d->n_kv) * d->head_dim * 2);
  L.off_rr = off;
  off += align_up(static_cast<size_t>(d->n_q) * 8);
  L.off_gr = off;
  off += align_up(static_cast<size_t>(p.n_groups) * 8);
  L.off_units = off;
  if (p.unit_list) off += align_up(static_cast<size_t>(p.n_groups) * p.n_chunks * 8);
  const size_t slots = static_cast<size_t>(d->n_q) * p.n_chunks;
  L.off_cnt = off;
  off += align_up(slots * kSub * 4);
  L.off_edge = off;
  off += align_up(slots * 4);
  L.off_key = off;
  off += align_up(slots * p.cap * 4);
  L.off_idx = off;
  off += align_up(slots * p.cap * 4);
  L.total = off;
  return L;
}

// pg (paged key cache): ks is NULL (every range starts at logical key 0), ke = seq_len, and
// k_idx is the page array itself.
dsa_status run_indexer(const dsa_indexer_desc* d, const void* q_idx, const void* k_idx, const float* w,
                       const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                       const float* rope_cs, int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws,
                       size_t ws_bytes, cudaStream_t st, bool clear_status, const PagedRows* pg = nullptr) {
  dsa_status s = check_indexer_desc(d);
  if (s != DSA_OK) return s;
  if (d->n_q == 0) return DSA_OK;
  const bool rq = (d->flags & DSA_IDX_ROPE_Q) && d->rope_dim > 0;
  const bool rk = (d->flags & DSA_IDX_ROPE_K) && d->rope_dim > 0;
  if (!q_idx || !k_idx || !w || (!ks && !pg) || !ke || !idx_out || !ws)
    return fail(DSA_ERR_ARG, "q_idx, k_idx, w, ks, ke, idx_out and ws must be non-NULL");
  if ((rq && !q_pos) || (rk && !k_pos) || ((rq || rk) && (!rope_cs || rope_n_pos < 1)))
    return fail(DSA_ERR_ARG, "RoPE requested but q_pos/k_pos/rope_cs/rope_n_pos missing");
  if (!aligned16(q_idx) || !aligned16(k_idx)) return fail(DSA_ERR_ARG, "q_idx and k_idx must be 16-byte aligned");
  if (rope_cs && !aligned16(rope_cs)) return fail(DSA_ERR_ARG, "rope_cs must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSA_ERR_ARG, "workspace must be 256-byte aligned");
  if ((s = check_device()) != DSA_OK) return s;
  const DevInfo di = dev_info();
  const IndexerLayout L = indexer_layout(d, di.sms);
  if (ws_bytes < L.total)
    return fail(DSA_ERR_WORKSPACE, "indexer workspace too small: %zu < %zu bytes", ws_bytes, L.total);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(base);
  cudaError_t e;
  if (clear_status && (e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  const void* qr = q_idx;
  const void* kr = k_idx;
  PhaseEvents* pe = phase_events();
  if (pe) (void)cudaEventRecord(pe->ev[0], st);
  if (rq) {
    const int ps = prof_begin(kProfRope, st);
    e = launch_rope_rows(q_idx, base + L.off_q, q_pos, static_cast<int64_t>(d->n_q) * d->n_heads, d->n_heads,
                         d->head_dim, d->rope_dim, rope_cs, rope_n_pos, status, st);
    prof_end(ps, st);
    if (e != cudaSuccess) return cuda_fail(e, "index q RoPE");
    qr = base + L.off_q;
  }
  if (rk && d->n_kv > 0) {
    const int ps = prof_begin(kProfRope, st);
    e = launch_rope_rows(k_idx, base + L.off_k, k_pos, d->n_kv, 1, d->head_dim, d->rope_dim, rope_cs, rope_n_pos,
                         status, st);
    prof_end(ps, st);
    if (e != cudaSuccess) return cuda_fail(e, "index k RoPE");
    kr = base + L.off_k;
  }
  const IndexerPlan& p = L.plan;
  int2* rr = reinterpret_cast<int2*>(base + L.off_rr);
  int2* gr = reinterpret_cast<int2*>(base + L.off_gr);
  if (pe) (void)cudaEventRecord(pe->ev[1], st);
  // rows whose whole range fits in k keep every key; without requested scores they need no scoring
  const int trivial_len = score_out ? 0 : d->topk;
  // paged: logical keys run up to max_pages pages, whatever the physical page count
  const int range_limit = pg ? static_cast<int>(std::min<long long>(static_cast<long long>(pg->max_pages) * kPageRows,
                                                                   0x7FFFFFFF))
                             : d->n_kv;
  int ps = prof_begin(kProfRanges, st);
  e = launch_ranges(ks, ke, d->n_q, p.group, range_limit, d->max_len, trivial_len,
                    static_cast<long long>(p.n_chunks) * p.chunk, rr, gr, status, st);
  prof_end(ps, st);
  if (e != cudaSuccess) return cuda_fail(e, "key ranges");
  if (pe) (void)cudaEventRecord(pe->ev[2], st);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + L.off_cnt);
  uint32_t* edge = reinterpret_cast<uint32_t*>(base + L.off_edge);
  int2* units = reinterpret_cast<int2*>(base + L.off_units);
  uint32_t* ck = reinterpret_cast<uint32_t*>(base + L.off_key);
  int32_t* ci = reinterpret_cast<int32_t*>(base + L.off_idx);
  if (d->n_kv > 0) {
    // the rotated copies hold only the 64-dim blocks with rotary dims; the blocks before
    // them are read from the inputs (same shape and box)
    CUtensorMap tq, tk, tqi, tki;
    const uint64_t q_rows = static_cast<uint64_t>(d->n_q) * d->n_heads;
    const uint32_t q_box = static_cast<uint32_t>(p.group * d->n_heads);
    if ((s = tmap_bf16(&tq, qr, d->head_dim, q_rows, q_box)) != DSA_OK) return s;
    if ((s = tmap_bf16(&tqi, q_idx, d->head_dim, q_rows, q_box)) != DSA_OK) return s;
    if ((s = tmap_bf16(&tk, kr, d->head_dim, d->n_kv, 128)) != DSA_OK) return s;
    if ((s = tmap_bf16(&tki, k_idx, d->head_dim, d->n_kv, 128)) != DSA_OK) return s;
    const int q_split = rq ? rope_split_blocks(d->head_dim, d->rope_dim) : 0;
    const int k_split = rk ? rope_split_blocks(d->head_dim, d->rope_dim) : 0;
    if (p.unit_list) {
      // the units that hold keys, densely (a chunk past a group's range is left out and its
      // rows' counts are zeroed)
      ps = prof_begin(kProfRanges, st);
      e = launch_units(gr, p.n_groups, p.n_chunks, p.chunk, p.group, d->n_q, units, cnt, edge, st);
      prof_end(ps, st);
      if (e != cudaSuccess) return cuda_fail(e, "unit list");
    }
    ps = prof_begin(kProfIndexer, st);
    e = launch_indexer(p, tq, tk, tqi, tki, q_split, k_split, pg ? *pg : PagedRows{}, w, d->n_q, rr, gr, trivial_len,
                       ck, ci, cnt, edge, p.unit_list ? units : nullptr, status, pipeline_debug(), st);
    prof_end(ps, st);
    if (e != cudaSuccess) return cuda_fail(e, "indexer kernel");
  } else {
    if ((e = cudaMemsetAsync(cnt, 0, static_cast<size_t>(d->n_q) * p.n_chunks * kSub * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(edge, 0, static_cast<size_t>(d->n_q) * p.n_chunks * 4, st)) != cudaSuccess)
      return cuda_fail(e, "clear counts");
  }
  if (pe) (void)cudaEventRecord(pe->ev[3], st);
  ps = prof_begin(kProfSelect, st);
  e = launch_select(d->n_q, p.n_chunks, p.cap, d->topk, trivial_len, d->max_len, rr, edge, ck, ci, cnt, idx_out, score_out,
                    status, st);
  prof_end(ps, st);
  if (e != cudaSuccess) return cuda_fail(e, "top-k select");
  if (pe) {
    (void)cudaEventRecord(pe->ev[4], st);
    pe->recorded = true;
  }
  return DSA_OK;
}

// ------------------------------------------------------------------ sparse attention
dsa_status check_attn_desc(const dsa_attn_desc* d) {
  if (!d) return fail(DSA_ERR_ARG, "attention descriptor is NULL");
  if (d->n_q < 0 || d->n_kv < 0) return fail(DSA_ERR_ARG, "n_q and n_kv must be >= 0");
  if (d->d_qk != 576 || d->d_v != 512)
    return fail(DSA_ERR_UNSUPPORTED, "d_qk/d_v %d/%d: this library supports 576/512", d->d_qk, d->d_v);
  if (d->n_heads < 1 || d->n_heads > 128) return fail(DSA_ERR_UNSUPPORTED, "n_heads %d outside 1..128", d->n_heads);
  if (d->topk < 1) return fail(DSA_ERR_ARG, "topk must be >= 1");
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale))
    return fail(DSA_ERR_ARG, "softmax_scale must be positive and finite");
  if (d->flags != 0) return fail(DSA_ERR_ARG, "attention flags must be 0");
  return DSA_OK;
}

size_t attn_ws_bytes(const dsa_attn_desc* d) {
  return kAlign + align_up(sparse_attn_ws_bytes(d->n_q, d->n_heads, d->n_kv, d->topk));
}

// status: device status header (first two words: bits, bad-index count); row_nt: n_q int32.
// pg (paged latent cache): ks is unused, offsets map through the block table.
// reuse_prepass: the workspace already holds the walk's pre-pass results for these index rows
// (the previous call on it used the same idx, ks and shape: IndexShare's shared layers).
dsa_status run_attn(const dsa_attn_desc* d, const void* q, const void* kv, const int32_t* idx, const int32_t* ks,
                    void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t st, bool clear_status,
                    uint32_t* status_override = nullptr, const PagedRows* pg = nullptr, bool reuse_prepass = false) {
  dsa_status s = check_attn_desc(d);
  if (s != DSA_OK) return s;
  if (d->n_q == 0) return DSA_OK;
  if (!q || !kv || !idx || (!ks && !pg) || !out || !ws)
    return fail(DSA_ERR_ARG, "q, kv, idx, ks, out and ws must be non-NULL");
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return fail(DSA_ERR_ARG, "q, kv and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSA_ERR_ARG, "workspace must be 256-byte aligned");
  if ((s = check_device()) != DSA_OK) return s;
  const size_t need = attn_ws_bytes(d);
  if (ws_bytes < need) return fail(DSA_ERR_WORKSPACE, "attention workspace too small: %zu < %zu bytes", ws_bytes, need);
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaError_t e;
  if (clear_status && (e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  uint32_t* status = status_override ? status_override : reinterpret_cast<uint32_t*>(base);
  // tensor maps: q as (token, head) rows; kv as whole 64-row tiles (block-dense walk) or as
  // single rows for four-row gathers (gather walk)
  CUtensorMap tkv, tq;
  std::memset(&tkv, 0, sizeof(tkv));
  std::memset(&tq, 0, sizeof(tq));
  if (!pg && sparse_attn_dense_heads(d->n_heads, d->n_kv, d->topk)) {
    if (d->n_kv > 0) s = tmap_kv_tiles(&tkv, kv, d->n_kv);   // an empty cache gives every block an empty range
  } else if (d->n_kv > 0) {
    s = tmap_bf16(&tkv, kv, 576, d->n_kv, 1);
  } else {
    // an empty cache has no row for the map; every slot is then masked, and the gathers that
    // still run read the first row of q instead (any 576-wide row in bounds will do)
    s = tmap_bf16(&tkv, q, 576, 1, 1);
  }
  if (s != DSA_OK) return s;
  if ((s = tmap_bf16(&tq, q, 576, static_cast<uint64_t>(d->n_q) * d->n_heads,
                     static_cast<uint32_t>(sparse_attn_q_box_rows(d->n_heads, d->n_kv, d->topk, pg != nullptr)))) != DSA_OK)
    return s;
  e = launch_sparse_attn(tkv, tq, d->n_q, d->n_kv, d->n_heads, d->topk, d->softmax_scale, kv, idx, ks,
                         pg ? *pg : PagedRows{}, out, lse, status,
                         base + kAlign, st, reuse_prepass);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention kernel");
  return DSA_OK;
}

}  // namespace

int device_sm_count() { return dev_info().sms; }

PipelineDebug pipeline_debug() {
  PipelineDebug d;
  d.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  d.stop_after_tiles = g_stop_after.load(std::memory_order_relaxed);
  return d;
}

int prof_begin(int kind, cudaStream_t st) {
  if (!g_profile.load(std::memory_order_relaxed)) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(g_log_mu);
  LaunchLog* L = launch_log(dev);
  if (!L) return -1;
  if (L->n >= kLogCap) {
    L->dropped = true;
    return -1;
  }
  const int i = L->n;
  if (i >= L->n_created) {
    if (cudaEventCreate(&L->ev[i][0]) != cudaSuccess) return ((void)cudaGetLastError(), -1);
    if (cudaEventCreate(&L->ev[i][1]) != cudaSuccess) {
      cudaEventDestroy(L->ev[i][0]);
      return ((void)cudaGetLastError(), -1);
    }
    L->n_created = i + 1;
  }
  if (cudaEventRecord(L->ev[i][0], st) != cudaSuccess) return ((void)cudaGetLastError(), -1);
  L->kind[i] = kind;
  L->n = i + 1;
  return i;
}

void prof_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(g_log_mu);
  LaunchLog* L = launch_log(dev);
  if (!L || slot >= L->n) return;
  if (cudaEventRecord(L->ev[slot][1], st) != cudaSuccess) (void)cudaGetLastError();
}

dsa_status indexer_workspace_bytes(const dsa_indexer_desc* d, size_t* bytes) {
  dsa_status s = check_indexer_desc(d);
  if (s != DSA_OK) return s;
  const DevInfo di = dev_info();
  *bytes = indexer_layout(d, di.sms > 0 ? di.sms : 148).total;
  return DSA_OK;
}

dsa_status indexer_run(const dsa_indexer_desc* d, const void* q_idx, const void* k_idx, const float* w,
                       const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                       const float* rope_cs, int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws,
                       size_t ws_bytes, cudaStream_t st) {
  return run_indexer(d, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, rope_n_pos, idx_out, score_out, ws, ws_bytes,
                     st, true);
}

dsa_status set_error(dsa_status s, const char* msg) { return fail(s, "%s", msg); }

}  // namespace dsa

// ====================================================================== C ABI
using namespace dsa;

struct dsa_index_cache {
  std::vector<uint8_t> types;
  std::vector<int32_t> donors;
  std::vector<int32_t*> buffers;
  int32_t n_q = 0, topk = 0;
};

extern "C" {

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_ARG: return "DSA_ERR_ARG";
    case DSA_ERR_SHAPE: return "DSA_ERR_SHAPE";
    case DSA_ERR_NO_DONOR: return "DSA_ERR_NO_DONOR";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_last_error(void) { return g_err.c_str(); }

dsa_status dsa_donor_table(int32_t n_layers, const uint8_t* types, int32_t* donors) {
  if (!types || !donors || n_layers < 1) return fail(DSA_ERR_ARG, "donor table: NULL array or n_layers < 1");
  int32_t last_full = -1;
  for (int32_t l = 0; l < n_layers; ++l) {
    if (types[l] == DSA_LAYER_FULL) {
      last_full = l;
      donors[l] = l;
    } else if (types[l] == DSA_LAYER_SHARED) {
      if (last_full < 0) return fail(DSA_ERR_NO_DONOR, "layer %d is shared but no full layer precedes it", l);
      donors[l] = last_full;
    } else {
      return fail(DSA_ERR_ARG, "layer %d: indexer type %u is neither shared (0) nor full (1)", l, types[l]);
    }
  }
  return DSA_OK;
}

dsa_status dsa_rope_table(double theta, int32_t rope_dim, int32_t n_pos, float* host_out) {
  if (!host_out || rope_dim < 0 || (rope_dim & 1) || n_pos < 1 || !(theta > 0.0))
    return fail(DSA_ERR_ARG, "rope table: bad theta/rope_dim/n_pos or NULL output");
  const int half = rope_dim / 2;
  std::vector<double> inv(half);
  for (int i = 0; i < half; ++i) inv[i] = std::pow(theta, -2.0 * i / rope_dim);
  for (int64_t p = 0; p < n_pos; ++p) {
    float* row = host_out + p * rope_dim;
    for (int i = 0; i < half; ++i) {
      const double a = static_cast<double>(p) * inv[i];
      row[2 * i] = static_cast<float>(std::cos(a));
      row[2 * i + 1] = static_cast<float>(std::sin(a));
    }
  }
  return DSA_OK;
}

dsa_status dsa_indexer_workspace_size(const dsa_indexer_desc* desc, size_t* bytes) {
  dsa_status s = check_indexer_desc(desc);
  if (s != DSA_OK) return s;
  if (!bytes) return fail(DSA_ERR_ARG, "bytes is NULL");
  const DevInfo di = dev_info();
  *bytes = indexer_layout(desc, di.sms > 0 ? di.sms : 148).total;
  return DSA_OK;
}

dsa_status dsa_indexer_topk(const dsa_indexer_desc* desc, const void* q_idx, const void* k_idx, const float* w,
                            const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                            const float* rope_cs, int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws,
                            size_t ws_bytes, void* stream) {
  return run_indexer(desc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, rope_n_pos, idx_out, score_out, ws,
                     ws_bytes, static_cast<cudaStream_t>(stream), true);
}

dsa_status dsa_sparse_attn_workspace_size(const dsa_attn_desc* desc, size_t* bytes) {
  dsa_status s = check_attn_desc(desc);
  if (s != DSA_OK) return s;
  if (!bytes) return fail(DSA_ERR_ARG, "bytes is NULL");
  *bytes = attn_ws_bytes(desc);
  return DSA_OK;
}

dsa_status dsa_sparse_attn(const dsa_attn_desc* desc, const void* q, const void* kv, const int32_t* idx,
                           const int32_t* ks, void* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return run_attn(desc, q, kv, idx, ks, out, lse, ws, ws_bytes, static_cast<cudaStream_t>(stream), true);
}

dsa_status dsa_index_cache_create(int32_t n_layers, const uint8_t* types, int32_t n_q, int32_t topk,
                                  int32_t* const* idx_buffers, dsa_index_cache** cache_out) {
  if (!cache_out) return fail(DSA_ERR_ARG, "cache_out is NULL");
  *cache_out = nullptr;
  if (!idx_buffers || n_q < 0 || topk < 1) return fail(DSA_ERR_ARG, "index cache: NULL buffers or bad n_q/topk");
  std::vector<int32_t> donors(n_layers > 0 ? n_layers : 0);
  dsa_status s = dsa_donor_table(n_layers, types, donors.data());
  if (s != DSA_OK) return s;
  for (int32_t l = 0; l < n_layers; ++l)
    if (types[l] == DSA_LAYER_FULL && !idx_buffers[l])
      return fail(DSA_ERR_ARG, "index cache: full layer %d has no index buffer", l);
  auto* c = new (std::nothrow) dsa_index_cache;
  if (!c) return fail(DSA_ERR_ARG, "index cache: out of host memory");
  c->types.assign(types, types + n_layers);
  c->donors = donors;
  c->buffers.assign(idx_buffers, idx_buffers + n_layers);
  c->n_q = n_q;
  c->topk = topk;
  *cache_out = c;
  return DSA_OK;
}

dsa_status dsa_index_cache_donor(const dsa_index_cache* c, int32_t layer, int32_t* donor) {
  if (!c || !donor) return fail(DSA_ERR_ARG, "index cache or donor is NULL");
  if (layer < 0 || layer >= static_cast<int32_t>(c->donors.size()))
    return fail(DSA_ERR_ARG, "layer %d outside [0, %zu)", layer, c->donors.size());
  *donor = c->donors[layer];
  return DSA_OK;
}

int32_t* dsa_index_cache_indices(const dsa_index_cache* c, int32_t layer) {
  if (!c || layer < 0 || layer >= static_cast<int32_t>(c->donors.size())) {
    fail(DSA_ERR_ARG, "index cache NULL or layer %d out of range", layer);
    return nullptr;
  }
  return c->buffers[c->donors[layer]];
}

void dsa_index_cache_destroy(dsa_index_cache* c) { delete c; }

dsa_status dsa_layers_workspace_size(const dsa_indexer_desc* idx_desc, const dsa_attn_desc* attn_desc, size_t* bytes) {
  size_t a = 0, b = 0;
  dsa_status s = dsa_indexer_workspace_size(idx_desc, &a);
  if (s != DSA_OK) return s;
  if ((s = dsa_sparse_attn_workspace_size(attn_desc, &b)) != DSA_OK) return s;
  *bytes = a + b;
  return DSA_OK;
}

dsa_status indexshare_layers_forward(const dsa_indexer_desc* idx_desc, const dsa_attn_desc* attn_desc,
                                     int32_t n_layers, const uint8_t* indexer_types, const dsa_layer_io* io,
                                     const int32_t* ks, const int32_t* ke, const int32_t* q_pos,
                                     const int32_t* k_pos, const float* rope_cs, int32_t rope_n_pos,
                                     dsa_index_cache* cache, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_indexer_desc(idx_desc);
  if (s != DSA_OK) return s;
  if ((s = check_attn_desc(attn_desc)) != DSA_OK) return s;
  if (!io || !cache || !indexer_types || !ws) return fail(DSA_ERR_ARG, "layer_io, cache, indexer_types and ws must be non-NULL");
  if (n_layers != static_cast<int32_t>(cache->types.size()))
    return fail(DSA_ERR_SHAPE, "n_layers %d differs from the cache's %zu", n_layers, cache->types.size());
  for (int32_t l = 0; l < n_layers; ++l)
    if (indexer_types[l] != cache->types[l])
      return fail(DSA_ERR_SHAPE, "indexer_types[%d] differs from the array the cache was built with", l);
  if (idx_desc->n_q != attn_desc->n_q || idx_desc->topk != attn_desc->topk || idx_desc->n_kv != attn_desc->n_kv)
    return fail(DSA_ERR_SHAPE, "indexer and attention descriptors disagree on n_q, n_kv or topk");
  if (cache->n_q != idx_desc->n_q || cache->topk != idx_desc->topk)
    return fail(DSA_ERR_SHAPE, "cache built for n_q=%d topk=%d", cache->n_q, cache->topk);
  size_t need = 0;
  if ((s = dsa_layers_workspace_size(idx_desc, attn_desc, &need)) != DSA_OK) return s;
  if (ws_bytes < need) return fail(DSA_ERR_WORKSPACE, "layer workspace too small: %zu < %zu bytes", ws_bytes, need);
  for (int32_t l = 0; l < n_layers; ++l) {
    if (!io[l].q || !io[l].kv || !io[l].out) return fail(DSA_ERR_ARG, "layer %d: q, kv and out must be non-NULL", l);
    if (cache->types[l] == DSA_LAYER_FULL && (!io[l].q_idx || !io[l].k_idx || !io[l].w))
      return fail(DSA_ERR_ARG, "full layer %d: q_idx, k_idx and w must be non-NULL", l);
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  size_t idx_ws = 0;
  dsa_indexer_workspace_size(idx_desc, &idx_ws);
  uint8_t* attn_ws = static_cast<uint8_t*>(ws) + idx_ws;
  if ((s = check_device()) != DSA_OK) return s;
  cudaError_t e;
  if ((e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  const int32_t* prev_idx = nullptr;   // index rows whose attention pre-pass the workspace holds
  for (int32_t l = 0; l < n_layers; ++l) {
    if (cache->types[l] == DSA_LAYER_FULL) {
      s = run_indexer(idx_desc, io[l].q_idx, io[l].k_idx, io[l].w, q_pos, k_pos, ks, ke, rope_cs, rope_n_pos,
                      cache->buffers[l], nullptr, ws, idx_ws, st, false);
      if (s != DSA_OK) return s;
    }
    // a shared layer reading the same index rows as the layer before reuses its pre-pass
    const int32_t* idx_l = cache->buffers[cache->donors[l]];
    s = run_attn(attn_desc, io[l].q, io[l].kv, idx_l, ks, io[l].out, io[l].lse, attn_ws, ws_bytes - idx_ws, st, false,
                 static_cast<uint32_t*>(ws), nullptr, idx_l == prev_idx);
    if (s != DSA_OK) return s;
    prev_idx = idx_l;
  }
  return DSA_OK;
}

dsa_status dsa_mtp_indexshare_step(const dsa_indexer_desc* idx_desc, const dsa_attn_desc* attn_desc, int32_t step,
                                   const dsa_layer_io* io, const int32_t* ks, const int32_t* ke,
                                   const int32_t* q_pos, const int32_t* k_pos, const float* rope_cs,
                                   int32_t rope_n_pos, int32_t* mtp_idx, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_indexer_desc(idx_desc);
  if (s != DSA_OK) return s;
  if ((s = check_attn_desc(attn_desc)) != DSA_OK) return s;
  if (step < 0) return fail(DSA_ERR_ARG, "MTP step %d must be >= 0", step);
  if (!io || !mtp_idx || !ws) return fail(DSA_ERR_ARG, "layer_io, mtp_idx and ws must be non-NULL");
  if (idx_desc->n_q != attn_desc->n_q || idx_desc->topk != attn_desc->topk)
    return fail(DSA_ERR_SHAPE, "indexer and attention descriptors disagree on n_q or topk");
  if (!io->q || !io->kv || !io->out) return fail(DSA_ERR_ARG, "q, kv and out must be non-NULL");
  if (step == 0 && (!io->q_idx || !io->k_idx || !io->w))
    return fail(DSA_ERR_ARG, "MTP step 0 runs the indexer: q_idx, k_idx and w must be non-NULL");
  size_t need = 0;
  if ((s = dsa_layers_workspace_size(idx_desc, attn_desc, &need)) != DSA_OK) return s;
  if (ws_bytes < need) return fail(DSA_ERR_WORKSPACE, "MTP workspace too small: %zu < %zu bytes", ws_bytes, need);
  if ((s = check_device()) != DSA_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  size_t idx_ws = 0;
  dsa_indexer_workspace_size(idx_desc, &idx_ws);
  cudaError_t e;
  if ((e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  if (step == 0) {
    s = run_indexer(idx_desc, io->q_idx, io->k_idx, io->w, q_pos, k_pos, ks, ke, rope_cs, rope_n_pos, mtp_idx,
                    nullptr, ws, idx_ws, st, false);
    if (s != DSA_OK) return s;
  }
  return run_attn(attn_desc, io->q, io->kv, mtp_idx, ks, io->out, io->lse, static_cast<uint8_t*>(ws) + idx_ws,
                  ws_bytes - idx_ws, st, false, static_cast<uint32_t*>(ws));
}

namespace {
dsa_status check_pages(const dsa_paged_cache* pc, int32_t n_kv, PagedRows* pg) {
  if (!pc || !pc->block_table || !pc->seq_len) return fail(DSA_ERR_ARG, "paged cache: block_table and seq_len must be non-NULL");
  if (pc->page_rows != kPageRows)
    return fail(DSA_ERR_UNSUPPORTED, "page_rows %d: this library supports %d-row pages", pc->page_rows, kPageRows);
  if (pc->max_pages < 1 || pc->n_pages < 1) return fail(DSA_ERR_ARG, "max_pages and n_pages must be >= 1");
  if (static_cast<long long>(pc->n_pages) * kPageRows != n_kv)
    return fail(DSA_ERR_SHAPE, "n_kv %d must equal n_pages * page_rows = %lld", n_kv,
                static_cast<long long>(pc->n_pages) * kPageRows);
  pg->block_table = pc->block_table;
  pg->seq_len = pc->seq_len;
  pg->max_pages = pc->max_pages;
  pg->n_pages = pc->n_pages;
  return DSA_OK;
}
}  // namespace

dsa_status dsa_indexer_topk_paged(const dsa_indexer_desc* desc, const void* q_idx, const void* k_cache, const float* w,
                                  const int32_t* q_pos, const dsa_paged_cache* pages, const float* rope_cs,
                                  int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws, size_t ws_bytes,
                                  void* stream) {
  dsa_status s = check_indexer_desc(desc);
  if (s != DSA_OK) return s;
  PagedRows pg;
  if ((s = check_pages(pages, desc->n_kv, &pg)) != DSA_OK) return s;
  if (!(desc->flags & DSA_IDX_INDEPENDENT_ROWS) || (desc->flags & DSA_IDX_ROPE_K))
    return fail(DSA_ERR_ARG, "a paged key cache needs DSA_IDX_INDEPENDENT_ROWS and a pre-rotated cache (no DSA_IDX_ROPE_K)");
  if (desc->n_heads != 64)
    return fail(DSA_ERR_UNSUPPORTED, "paged key cache: %d index heads (one row per key stream needs 64)", desc->n_heads);
  if (static_cast<long long>(desc->max_len) > static_cast<long long>(pages->max_pages) * kPageRows)
    return fail(DSA_ERR_ARG, "max_len %d exceeds max_pages * page_rows", desc->max_len);
  return run_indexer(desc, q_idx, k_cache, w, q_pos, nullptr, nullptr, pages->seq_len, rope_cs, rope_n_pos, idx_out,
                     score_out, ws, ws_bytes, static_cast<cudaStream_t>(stream), true, &pg);
}

dsa_status dsa_sparse_attn_paged(const dsa_attn_desc* desc, const void* q, const void* kv_cache, const int32_t* idx,
                                 const dsa_paged_cache* pages, void* out, float* lse, void* ws, size_t ws_bytes,
                                 void* stream) {
  dsa_status s = check_attn_desc(desc);
  if (s != DSA_OK) return s;
  PagedRows pg;
  if ((s = check_pages(pages, desc->n_kv, &pg)) != DSA_OK) return s;
  return run_attn(desc, q, kv_cache, idx, nullptr, out, lse, ws, ws_bytes, static_cast<cudaStream_t>(stream), true,
                  nullptr, &pg);
}

dsa_status dsa_indexer_projections(const dsa_proj_desc* d, const void* x, const void* q_latent, const void* wq_b,
                                   const void* wk, const float* k_norm_w, const float* k_norm_b,
                                   const void* weights_proj, void* q_idx, void* k_idx, float* w, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (!d) return fail(DSA_ERR_ARG, "projection descriptor is NULL");
  if (d->n_tokens < 0) return fail(DSA_ERR_ARG, "n_tokens must be >= 0");
  if (d->d_hidden <= 0 || d->d_hidden % 64 || d->d_q <= 0 || d->d_q % 64)
    return fail(DSA_ERR_UNSUPPORTED, "d_hidden %d / d_q %d must be positive multiples of 64", d->d_hidden, d->d_q);
  if (!supported_heads(d->n_heads)) return fail(DSA_ERR_UNSUPPORTED, "index n_heads %d", d->n_heads);
  if (d->head_dim != 64 && d->head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "index head_dim %d", d->head_dim);
  if (!(d->ln_eps >= 0.f) || !std::isfinite(d->ln_eps)) return fail(DSA_ERR_ARG, "ln_eps must be finite and >= 0");
  if (!x || !q_latent || !wq_b || !wk || !k_norm_w || !k_norm_b || !weights_proj || !q_idx || !k_idx || !w || !ws)
    return fail(DSA_ERR_ARG, "every tensor and ws must be non-NULL");
  if (!aligned16(x) || !aligned16(q_latent) || !aligned16(wq_b) || !aligned16(wk) || !aligned16(weights_proj) ||
      !aligned16(q_idx) || !aligned16(k_idx))
    return fail(DSA_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSA_ERR_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < kAlign) return fail(DSA_ERR_WORKSPACE, "projection workspace too small: %zu < %zu bytes", ws_bytes, kAlign);
  if (d->n_tokens == 0) return DSA_OK;
  dsa_status s;
  if ((s = check_device()) != DSA_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  const int nq = d->n_heads * d->head_dim;
  const int nw_box = std::max(32, (d->n_heads + 31) / 32 * 32);   // head-weight rows in the key tile
  const uint64_t T = static_cast<uint64_t>(d->n_tokens);
  // the key + head-weight units (d_hidden / 64 K blocks each) go first, the shorter query
  // units after them, so the last round of the persistent grid is made of short units
  CUtensorMap ta[2], tb[2], tb2;
  if ((s = tmap_bf16(&ta[0], x, d->d_hidden, T, 128)) != DSA_OK) return s;
  if ((s = tmap_bf16(&tb[0], wk, d->d_hidden, d->head_dim, d->head_dim)) != DSA_OK) return s;
  if ((s = tmap_bf16(&tb2, weights_proj, d->d_hidden, d->n_heads, nw_box)) != DSA_OK) return s;
  if ((s = tmap_bf16(&ta[1], q_latent, d->d_q, T, 128)) != DSA_OK) return s;
  if ((s = tmap_bf16(&tb[1], wq_b, d->d_q, nq, 256)) != DSA_OK) return s;
  ProjJobs J{};
  J.n_jobs = 2;
  J.job[0] = ProjJob{d->head_dim, d->d_hidden, d->head_dim + nw_box, kProjEpiLayerNormF32, k_idx, k_norm_w, k_norm_b,
                     d->ln_eps, w, d->n_heads};
  J.job[1] = ProjJob{nq, d->d_q, 256, kProjEpiBf16, q_idx, nullptr, nullptr, 0.f, nullptr, 0};
  const int m_tiles = (d->n_tokens + 127) / 128;
  J.first_unit[0] = 0;
  J.first_unit[1] = m_tiles;
  J.first_unit[2] = m_tiles + m_tiles * (nq / 256);
  const int ps = prof_begin(kProfProj, st);
  e = launch_projections(ta, tb, tb2, J, d->n_tokens, static_cast<uint32_t*>(ws), st);
  prof_end(ps, st);
  if (e != cudaSuccess) return cuda_fail(e, "projection kernel");
  return DSA_OK;
}

namespace {
// The tcgen05 backward reads q and d_out in boxes of 64 (token, head) rows: it takes every
// shape with at least 64 of them; smaller ones take the per-token kernel.
bool attn_bwd_tc(const dsa_attn_desc* d) { return static_cast<long long>(d->n_q) * d->n_heads >= kDenseCols; }

// Backward workspace: the status header, then (tcgen05) D = d_out . out per (token, head) and
// the walk's pre-pass arrays (block-dense: key ranges and selection bitmasks; gather: 64-slot
// tiles per token).
size_t attn_bwd_ws_bytes(const dsa_attn_desc* d) {
  if (!attn_bwd_tc(d)) return kAlign;
  const size_t walk = sparse_attn_dense_heads(d->n_heads, d->n_kv, d->topk)
                          ? sparse_attn_ws_bytes(d->n_q, d->n_heads, d->n_kv, d->topk)
                          : static_cast<size_t>(d->n_q) * sizeof(int32_t);
  return kAlign + align_up(sparse_attn_bwd_dense_delta_bytes(d->n_q, d->n_heads)) + align_up(walk);
}
}  // namespace

dsa_status dsa_sparse_attn_backward_workspace_size(const dsa_attn_desc* desc, size_t* bytes) {
  dsa_status s = check_attn_desc(desc);
  if (s != DSA_OK) return s;
  if (!bytes) return fail(DSA_ERR_ARG, "bytes is NULL");
  *bytes = attn_bwd_ws_bytes(desc);
  return DSA_OK;
}

dsa_status dsa_sparse_attn_backward(const dsa_attn_desc* desc, const void* q, const void* kv, const int32_t* idx,
                                    const int32_t* ks, const void* out, const float* lse, const void* d_out,
                                    float* dq, float* dkv, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_attn_desc(desc);
  if (s != DSA_OK) return s;
  if (!q || !kv || !idx || !ks || !out || !lse || !d_out || !dq || !dkv || !ws)
    return fail(DSA_ERR_ARG, "every tensor and ws must be non-NULL");
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(d_out) || !aligned16(dq) || !aligned16(dkv))
    return fail(DSA_ERR_ARG, "q, kv, out, d_out, dq and dkv must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSA_ERR_ARG, "workspace must be 256-byte aligned");
  const size_t need = attn_bwd_ws_bytes(desc);
  if (ws_bytes < need) return fail(DSA_ERR_WORKSPACE, "backward workspace too small: %zu < %zu bytes", ws_bytes, need);
  if ((s = check_device()) != DSA_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  if (desc->n_kv > 0 &&
      (e = cudaMemsetAsync(dkv, 0, static_cast<size_t>(desc->n_kv) * 576 * sizeof(float), st)) != cudaSuccess)
    return cuda_fail(e, "clear dkv");
  if (desc->n_q == 0) return DSA_OK;
  uint32_t* status = static_cast<uint32_t*>(ws);
  if (attn_bwd_tc(desc)) {
    // tcgen05: q and d_out as 64-row boxes; block-dense walk: kv as whole 64-row tiles
    CUtensorMap tq, tdo;
    const uint64_t rows = static_cast<uint64_t>(desc->n_q) * desc->n_heads;
    if ((s = tmap_bf16(&tq, q, 576, rows, kDenseCols)) != DSA_OK) return s;
    if ((s = tmap_bf16(&tdo, d_out, 512, rows, kDenseCols)) != DSA_OK) return s;
    uint8_t* base = static_cast<uint8_t*>(ws);
    float* delta = reinterpret_cast<float*>(base + kAlign);
    void* scratch = base + kAlign + align_up(sparse_attn_bwd_dense_delta_bytes(desc->n_q, desc->n_heads));
    const int hd = sparse_attn_dense_heads(desc->n_heads, desc->n_kv, desc->topk);
    if (hd) {
      CUtensorMap tkv;
      std::memset(&tkv, 0, sizeof(tkv));
      if (desc->n_kv > 0 && (s = tmap_kv_tiles(&tkv, kv, desc->n_kv)) != DSA_OK) return s;
      e = launch_sparse_attn_bwd_dense(hd, tkv, tq, tdo, desc->n_q, desc->n_kv, desc->topk, desc->softmax_scale, idx,
                                       ks, out, lse, d_out, dq, dkv, status, delta, scratch, st);
      if (e != cudaSuccess) return cuda_fail(e, "sparse attention backward (block-dense)");
    } else {
      e = launch_sparse_attn_bwd_gather(tq, tdo, desc->n_q, desc->n_kv, desc->n_heads, desc->topk, desc->softmax_scale,
                                        kv, idx, ks, out, lse, d_out, dq, dkv, status, delta,
                                        static_cast<int32_t*>(scratch), st);
      if (e != cudaSuccess) return cuda_fail(e, "sparse attention backward (gather)");
    }
    return DSA_OK;
  }
  const int ps = prof_begin(kProfAttnBwd, st);
  e = launch_sparse_attn_bwd(desc->n_q, desc->n_kv, desc->n_heads, desc->topk, desc->softmax_scale, q, kv, idx, ks, out,
                             lse, d_out, dq, dkv, status, st);
  prof_end(ps, st);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention backward");
  return DSA_OK;
}

namespace {
struct IndexerBwdLayout {
  size_t off_q = 0, off_k = 0, total = 0;
};
IndexerBwdLayout indexer_bwd_layout(const dsa_indexer_desc* d) {
  IndexerBwdLayout L;
  size_t off = kAlign;   // status header
  const bool rq = (d->flags & DSA_IDX_ROPE_Q) && d->rope_dim > 0;
  const bool rk = (d->flags & DSA_IDX_ROPE_K) && d->rope_dim > 0;
  L.off_q = off;
  if (rq) off += align_up(static_cast<size_t>(d->n_q) * d->n_heads * d->head_dim * 2);
  L.off_k = off;
  if (rk) off += align_up(static_cast<size_t>(d->n_kv) * d->head_dim * 2);
  L.total = off;
  return L;
}
dsa_status check_indexer_bwd_desc(const dsa_indexer_desc* d) {
  dsa_status s = check_indexer_desc(d);
  if (s != DSA_OK) return s;
  if (d->head_dim != 128)
    return fail(DSA_ERR_UNSUPPORTED, "indexer backward: head_dim %d, supported value is 128", d->head_dim);
  if (d->flags & DSA_IDX_INDEPENDENT_ROWS)
    return fail(DSA_ERR_UNSUPPORTED, "indexer backward: independent rows are not supported");
  return DSA_OK;
}
}  // namespace

dsa_status dsa_indexer_backward_workspace_size(const dsa_indexer_desc* desc, size_t* bytes) {
  if (!bytes) return fail(DSA_ERR_ARG, "bytes is NULL");
  dsa_status s = check_indexer_bwd_desc(desc);
  if (s != DSA_OK) return s;
  *bytes = indexer_bwd_layout(desc).total;
  return DSA_OK;
}

dsa_status dsa_indexer_backward(const dsa_indexer_desc* desc, const void* q_idx, const void* k_idx, const float* w,
                                const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                                const float* rope_cs, int32_t rope_n_pos, const int32_t* idx, const float* d_score,
                                float* dq_idx, float* dk_idx, float* dw, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_indexer_bwd_desc(desc);
  if (s != DSA_OK) return s;
  const dsa_indexer_desc* d = desc;
  const bool rq = (d->flags & DSA_IDX_ROPE_Q) && d->rope_dim > 0;
  const bool rk = (d->flags & DSA_IDX_ROPE_K) && d->rope_dim > 0;
  if (!q_idx || !k_idx || !w || !ks || !ke || !idx || !d_score || !dq_idx || !dk_idx || !dw || !ws)
    return fail(DSA_ERR_ARG, "q_idx, k_idx, w, ks, ke, idx, d_score, dq_idx, dk_idx, dw and ws must be non-NULL");
  if ((rq && !q_pos) || (rk && !k_pos) || ((rq || rk) && (!rope_cs || rope_n_pos < 1)))
    return fail(DSA_ERR_ARG, "RoPE requested but q_pos/k_pos/rope_cs/rope_n_pos missing");
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(dq_idx) || !aligned16(dk_idx))
    return fail(DSA_ERR_ARG, "q_idx, k_idx, w, dq_idx and dk_idx must be 16-byte aligned");
  if (rope_cs && !aligned16(rope_cs)) return fail(DSA_ERR_ARG, "rope_cs must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSA_ERR_ARG, "workspace must be 256-byte aligned");
  if ((s = check_device()) != DSA_OK) return s;
  const IndexerBwdLayout L = indexer_bwd_layout(d);
  if (ws_bytes < L.total)
    return fail(DSA_ERR_WORKSPACE, "indexer backward workspace too small: %zu < %zu bytes", ws_bytes, L.total);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(base);
  cudaError_t e;
  if ((e = cudaMemsetAsync(ws, 0, kAlign, st)) != cudaSuccess) return cuda_fail(e, "clear status");
  if (d->n_kv > 0 &&
      (e = cudaMemsetAsync(dk_idx, 0, static_cast<size_t>(d->n_kv) * d->head_dim * sizeof(float), st)) != cudaSuccess)
    return cuda_fail(e, "clear dk_idx");
  if (d->n_q == 0) return DSA_OK;
  if ((e = cudaMemsetAsync(dw, 0, static_cast<size_t>(d->n_q) * d->n_heads * sizeof(float), st)) != cudaSuccess)
    return cuda_fail(e, "clear dw");
  const void* qr = q_idx;
  const void* kr = k_idx;
  const int ps = prof_begin(kProfIndexerBwd, st);
  if (rq) {
    e = launch_rope_rows(q_idx, base + L.off_q, q_pos, static_cast<int64_t>(d->n_q) * d->n_heads, d->n_heads,
                         d->head_dim, d->rope_dim, rope_cs, rope_n_pos, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "index q RoPE");
    qr = base + L.off_q;
  }
  if (rk && d->n_kv > 0) {
    e = launch_rope_rows(k_idx, base + L.off_k, k_pos, d->n_kv, 1, d->head_dim, d->rope_dim, rope_cs, rope_n_pos,
                         status, st);
    if (e != cudaSuccess) return cuda_fail(e, "index k RoPE");
    kr = base + L.off_k;
  }
  const int q_split = rq ? rope_split_blocks(d->head_dim, d->rope_dim) : 0;
  const int k_split = rk ? rope_split_blocks(d->head_dim, d->rope_dim) : 0;
  const DevInfo di = dev_info();
  e = launch_indexer_bwd(d->n_q, d->n_kv, d->n_heads, d->head_dim, d->topk, qr, q_idx, kr, k_idx, q_split, k_split, w,
                         ks, ke, idx, d_score, dq_idx, dk_idx, dw, di.sms > 0 ? di.sms : 148, status, pipeline_debug(),
                         st);
  if (e != cudaSuccess) return cuda_fail(e, "indexer backward");
  if (rq) {
    e = launch_rope_rows_transpose_f32(dq_idx, q_pos, static_cast<int64_t>(d->n_q) * d->n_heads, d->n_heads,
                                       d->head_dim, d->rope_dim, rope_cs, rope_n_pos, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "dq RoPE transpose");
  }
  if (rk && d->n_kv > 0) {
    e = launch_rope_rows_transpose_f32(dk_idx, k_pos, d->n_kv, 1, d->head_dim, d->rope_dim, rope_cs, rope_n_pos, status,
                                       st);
    if (e != cudaSuccess) return cuda_fail(e, "dk RoPE transpose");
  }
  prof_end(ps, st);
  return DSA_OK;
}

dsa_status dsa_workspace_status(const void* ws, void* stream, uint32_t* device_bits) {
  if (!ws) return fail(DSA_ERR_ARG, "workspace is NULL");
  WsHeader h{};
  cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "read workspace status");
  if (device_bits) *device_bits = h.status;
  if (h.status & DEV_ERR_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a device pipeline wait ran past its bound");
  if (h.status) return fail(DSA_ERR_DEVICE, "device status 0x%x (%u bad indices)", h.status, h.bad_count);
  return DSA_OK;
}

dsa_status dsa_debug_pipeline(int32_t stop_after_tiles, uint64_t wait_ns) {
  if (stop_after_tiles < -1) return fail(DSA_ERR_ARG, "stop_after_tiles must be >= -1");
  g_stop_after.store(stop_after_tiles, std::memory_order_relaxed);
  g_wait_ns.store(wait_ns == 0 ? 2000000000ull : static_cast<unsigned long long>(wait_ns), std::memory_order_relaxed);
  return DSA_OK;
}

dsa_status dsa_profile_enable(int32_t on) {
  if (on) {
    // a new measurement starts with an empty launch log on every device
    std::lock_guard<std::mutex> lock(g_log_mu);
    for (LaunchLog* L : g_log)
      if (L) {
        L->n = 0;
        L->dropped = false;
      }
  }
  g_profile.store(on ? 1 : 0, std::memory_order_relaxed);
  return DSA_OK;
}

dsa_status dsa_profile_read(dsa_profile_record* out, int32_t cap, int32_t* n) {
  if (!n || cap < 0 || (cap > 0 && !out)) return fail(DSA_ERR_ARG, "n must be non-NULL and out must hold cap records");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_log_mu);
  LaunchLog* L = (dev >= 0 && dev < 64) ? g_log[dev] : nullptr;
  const int have = L ? L->n : 0;
  *n = have;
  for (int i = 0; i < have && i < cap; ++i) {
    if ((e = cudaEventSynchronize(L->ev[i][1])) != cudaSuccess) return cuda_fail(e, "launch log events");
    float t = 0.f;
    if ((e = cudaEventElapsedTime(&t, L->ev[i][0], L->ev[i][1])) != cudaSuccess) return cuda_fail(e, "launch log events");
    out[i].kind = L->kind[i];
    out[i].ms = t;
  }
  if (L && L->dropped) return fail(DSA_ERR_WORKSPACE, "launch log full: records after the first %d were dropped", kLogCap);
  return DSA_OK;
}

dsa_status dsa_profile_indexer_last(float* ms, int32_t n) {
  if (!ms || n < 1) return fail(DSA_ERR_ARG, "ms must be non-NULL and n >= 1");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device %d out of range", dev);
  PhaseEvents* p = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_phase_mu);
    if (g_phase[dev].created && g_phase[dev].recorded) p = &g_phase[dev];
  }
  if (!p) return fail(DSA_ERR_UNSUPPORTED, "no profiled indexer call on device %d", dev);
  if ((e = cudaEventSynchronize(p->ev[4])) != cudaSuccess) return cuda_fail(e, "profile events");
  for (int i = 0; i < 4 && i < n; ++i) {
    float t = 0.f;
    if ((e = cudaEventElapsedTime(&t, p->ev[i], p->ev[i + 1])) != cudaSuccess) return cuda_fail(e, "profile events");
    ms[i] = t;
  }
  return DSA_OK;
}

}  // extern "C"
