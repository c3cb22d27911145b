// Lightning-indexer score contraction on tcgen05 with a fused streaming causal top-k.
//
//   s[t, j] = sum_h w[t, h] * max(0, q[t, h] . k[j])            (q, k already rotated)
//
// ("GLM-5.2 IndexShare" explainer, section 1: the indexer scores the prefix tokens of each
// query and keeps the top-k positions; the weighted ReLU head sum with one shared key head
// follows "GLM-5/5.1/5.2 DSA + LoRA enablement", indexer RoPE half-swap commit.)
//
// Tiling.  A work unit is (group of G consecutive query rows, chunk of the group's key
// range).  The MMA puts 128 KEYS in M and the G*H_I (query, head) pairs of the group in
// N (<= 256), so one key tile is one tcgen05.mma chain of d_I/16 instructions:
//     S^T[key, (g, h)] = K_tile[key, :] . Q_group[(g, h), :]
// into one of two TMEM accumulators.
//
// Candidates.  Every (row, chunk) has kSub sub-buffers of cap / kSub (order-preserving score
// key, key index) entries, one per TMEM lane quarter (keys j with (j - chunk start) % 128 in
// [32 q, 32 q + 32)), each in key order; launch_select later picks each row's exact top-k from
// them.  A row keeps a key only if its score is at or above the row's threshold tau: minus
// infinity for rows of at most direct_max keys in the chunk (every key is kept), else the lower
// edge of the bin of a log-spaced score histogram that holds the row's k-th largest kept
// score -- every key below that edge has at least k kept keys above it.  The expected number
// kept over N keys is about k (1 + ln(N/k)).
//
// Warp roles (no role waits on a CTA-wide barrier inside the tile loop):
//   warp 0            TMA producer: Q of the unit once, K tiles through a STAGES-deep ring;
//   warp 1            MMA issuer (owns TMEM);
//   warp 2            threshold warp: keeps raising each filtered query's tau from its
//                     histogram while the unit runs; histograms and taus are double-buffered
//                     by unit parity;
//   warp 3            idle (completes warpgroup 0, which gives registers to the head-sum warps);
//   warps 4..         NE = 4 or 8 head-sum warps: a warp owns one TMEM lane quarter (32 keys)
//                     and half or all of the group's queries; it reduces the heads of each
//                     query with the head weights held in registers (ReLU * w with packed fp32
//                     FMAs), keeps the keys at or above the query's tau in its own sub-buffer
//                     (no other warp writes there) and counts them in the query's histogram.
//                     A sub-buffer that could overflow (scores that keep rising along the
//                     keys) is cut back by its warp to exactly its top-k, which still holds
//                     every key of the row's top-k that lies in it.
// The score matrix is never written anywhere.
#include <cuda_bf16.h>

#include <cstddef>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int kKeyTile = 128;
constexpr int kBins = 256;        // value-linear bins of a warp's cut-back
constexpr int kBoundary = 64;     // boundary-bin entries ranked directly by a warp
constexpr int kLoadsInFlight = 16;
constexpr int kLog2Span = 5;      // each sign's half of the threshold histogram covers 2^kLog2Span
constexpr int kLowExp = 127 - 16; // octaves of |score| from 2^-16 (smaller magnitudes share a bin)

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Per head-sum warp scratch of a cut-back: histogram bins, then the boundary bin's entries.  (In
// global memory instead, the call into the cut-back made the compiler keep the head-sum state
// in local memory and halved the kernel's speed.)
struct WarpScratch {
  uint32_t hist[kBins];
  uint32_t bkey[kBoundary];
  int32_t bidx[kBoundary];
  int bc[4];
};

template <int HI, int DI, int G>
struct Cfg {
  static constexpr int N = G * HI;                       // MMA N: (query, head) pairs
  static constexpr int KB = DI / 64;                     // 128-byte K blocks per row
  static constexpr int Q_BYTES = N * DI * 2;
  static constexpr int K_STAGE_BYTES = kKeyTile * DI * 2;
  // head-sum warps: one per TMEM lane quarter per half; with several queries per group the
  // queries (and their TMEM columns) are split between two halves
  static constexpr int HALVES = G >= 2 && N >= 128 ? 2 : 1;
  static constexpr int NE = 4 * HALVES;
  static constexpr int GH = G / HALVES;                  // queries per half
  static constexpr int NH = N / HALVES;                  // TMEM columns per half
  // warpgroup 0: producer, MMA, threshold and one idle warp; then NE / 4 head-sum warpgroups
  static constexpr int THREADS = 32 * (4 + NE);
  // With two head-sum warpgroups (384 threads, 168 registers a thread at launch) warpgroup 0
  // hands registers to the head-sum warps, which keep all NH head weights of their queries in
  // registers: 128 * REG_LOW + 256 * REG_HIGH stays within the 384 * 168 the block holds.
  static constexpr bool REG_SPLIT = NE == 8;
  static constexpr int REG_LAUNCH = 168, REG_LOW = 56, REG_HIGH = 224;
  static_assert(!REG_SPLIT || 128 * REG_LOW + 256 * REG_HIGH <= THREADS * REG_LAUNCH, "register split");
  // threshold histograms: NB bins per query per unit parity (32 KB in all for G >= 4); bins
  // [0, NBH) hold negative scores and [NBH, NB) positive ones, each half log-spaced over
  // 2^kLog2Span octaves of |score| (a row whose k-th largest score is negative -- head weights
  // of mostly one sign -- still gets a rising threshold)
  static constexpr int NB = 4096 / G < 1024 ? 4096 / G : 1024;
  static constexpr int NBH = NB / 2;
  static constexpr int SHIFT = 23 + kLog2Span - ilog2(NBH);  // key bits below the bin index
  // key >> SHIFT of +2^-16 and of -2^(2^kLog2Span - 16): the lowest bin of each half
  static constexpr uint32_t BASE_POS = (0x80000000u | (static_cast<uint32_t>(kLowExp) << 23)) >> SHIFT;
  static constexpr uint32_t BASE_NEG =
      (~(0x80000000u | (static_cast<uint32_t>(kLowExp + (1 << kLog2Span)) << 23))) >> SHIFT;
  static constexpr int SMEM_MAX = 232448;                // dynamic + static per CTA
  static constexpr int STATIC_EST = 1024 + 2 * G * NB * 4 + 4 * G * 4 + NE * static_cast<int>(sizeof(WarpScratch));
  static constexpr int AVAIL = SMEM_MAX - STATIC_EST - 1024 - Q_BYTES;
  static constexpr int STAGES_FIT = AVAIL / K_STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int DYN_SMEM = 1024 + Q_BYTES + STAGES * K_STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = (2 * N <= 32) ? 32 : (2 * N <= 64) ? 64 : (2 * N <= 128) ? 128 : (2 * N <= 256) ? 256 : 512;
  static_assert(N % 64 == 0 && N >= 64 && N <= 256, "MMA N");
  static_assert(NH % 32 == 0 && NH <= 128, "head-sum reads 32 columns at a time, weights in registers");
  static_assert(GH * HI == NH, "a half holds whole queries");
  static_assert(G <= 16, "the threshold warp keeps one query per lane, at most 16");
  static_assert(STAGES >= 2, "shared memory");
  static_assert(SHIFT + ilog2(NBH) == 23 + kLog2Span, "NB / 2 bins span 2^kLog2Span octaves");
  static_assert(kLowExp + (1 << kLog2Span) < 255, "histogram range within the float exponents");
};

// Threshold-histogram bin of a score key under Cfg C's map (monotone non-decreasing in the key):
// negative scores below -2^(2^kLog2Span - 16) share bin 0, negative magnitudes under 2^-16 share
// bin NBH - 1, positive scores under 2^-16 (and +0) share bin NBH, scores above the span the
// top bin.  bin_edge_key(b) is the smallest key of bin b.
template <class C>
__device__ __forceinline__ int hist_bin(uint32_t key) {
  const int hi = static_cast<int>(key >> C::SHIFT);
  int b = (key & 0x80000000u) ? hi - static_cast<int>(C::BASE_POS) : hi - static_cast<int>(C::BASE_NEG);
  b = b < 0 ? 0 : (b >= C::NBH ? C::NBH - 1 : b);
  return (key & 0x80000000u) ? C::NBH + b : b;
}
template <class C>
__device__ __forceinline__ uint32_t bin_edge_key(int b) {
  if (b >= C::NBH + 1) return static_cast<uint32_t>(b - C::NBH + static_cast<int>(C::BASE_POS)) << C::SHIFT;
  if (b == C::NBH) return 0x80000000u;
  return b > 0 ? static_cast<uint32_t>(b + static_cast<int>(C::BASE_NEG)) << C::SHIFT : 0u;
}


template <int G, int NB, int NE>
struct Shared {
  uint64_t k_full[6], k_empty[6];
  uint64_t q_full, q_empty;
  uint64_t t_full[2], t_empty[2];
  uint64_t u_done[2], u_ready[2];  // per unit parity: head-sum warps done / histograms reset
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t tau[2][G];              // per unit parity and query: threshold key (0: keep every key)
  uint32_t hist[2][G][NB];         // threshold histograms of the filtered queries
  WarpScratch ws[NE];              // cut-back scratch of each head-sum warp
};

struct UnitInfo {
  int group, chunk, kbeg, kend, n_tiles;
};

// A query's key range within a unit and whether it is scored (rows of at most trivial_len
// keys are left to the select pass) and filtered (longer than direct_max keys).
struct QueryRange {
  int a, b;
  bool live, filtered;
};
__device__ __forceinline__ QueryRange query_range(const int2* row_range, int t, int n_q, const UnitInfo& ui,
                                                  int trivial_len, int direct_max) {
  QueryRange r;
  int2 rr = make_int2(0, 0);
  if (t < n_q) rr = row_range[t];
  r.live = t < n_q && rr.y - rr.x > trivial_len;
  r.a = max(rr.x, ui.kbeg);
  r.b = r.live ? min(rr.y, ui.kend) : r.a;
  if (r.b < r.a) r.b = r.a;
  r.filtered = r.b - r.a > direct_max;
  return r;
}

// Warp-uniform bounded wait (every lane polls; the result is agreed across the warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t* status, unsigned long long limit_ns) {
  const bool ok = mbar_wait_for(bar, parity, abort_flag, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ warp-level top-k helpers
// A top-k warp works on one candidate buffer at a time (keys[], idxs[] of n entries in the
// workspace, sorted by key index).  Entry e is held by lane e % 32; passes over a buffer keep
// kLoadsInFlight loads per lane in flight.

// Histogram increment aggregated over the lanes that hit the same bin (bin -1: none).
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, int bin) {
  const uint32_t peers = __match_any_sync(0xffffffffu, bin);
  if (bin >= 0 && static_cast<int>(threadIdx.x & 31u) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

// Bin of a key under a value-linear map of [fmin, fmax] onto kBins bins; monotone
// non-decreasing in the key, so a higher bin never holds a smaller score.
struct BinMap {
  float fmin, scale;
  __device__ __forceinline__ BinMap(uint32_t kmin, uint32_t kmax) {
    fmin = key_float(kmin);
    const float span = key_float(kmax) - fmin;
    scale = span > 0.f && span < 3.0e38f ? static_cast<float>(kBins) / span : 0.f;
  }
  __device__ __forceinline__ int operator()(uint32_t key) const {
    const float y = (key_float(key) - fmin) * scale;
    return y >= static_cast<float>(kBins - 1) ? kBins - 1 : (y > 0.f ? static_cast<int>(y) : 0);
  }
};

// The bin b holding the need-th largest entry (bins visited from the top): returns b, the
// entries in bins above b and the entries in b.  Lane l owns bins [16 l, 16 l + 16).
struct Boundary {
  int b, above, hb;
};
__device__ __forceinline__ Boundary warp_boundary(const uint32_t* hist, int need) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = kBins / 32;
  int h[kPer], s = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    h[j] = static_cast<int>(hist[lane * kPer + j]);
    s += h[j];
  }
  int x = s;   // inclusive suffix sum over lanes >= this one
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += y;
  }
  int c = x - s;
  int fb = -1, fa = 0, fh = 0;
#pragma unroll
  for (int j = kPer - 1; j >= 0; --j) {
    if (c < need && need <= c + h[j]) {
      fb = lane * kPer + j;
      fa = c;
      fh = h[j];
    }
    c += h[j];
  }
  const uint32_t m = __ballot_sync(0xffffffffu, fb >= 0);
  const int src = m ? __ffs(m) - 1 : 0;
  Boundary r;
  r.b = __shfl_sync(0xffffffffu, fb, src);
  r.above = __shfl_sync(0xffffffffu, fa, src);
  r.hb = __shfl_sync(0xffffffffu, fh, src);
  return r;
}

// Calls f(valid, key, idx) for every entry of the buffer, all lanes together (f may use warp
// collectives); with kWithIdx false, idx is not loaded (0).
template <bool kWithIdx, class F>
__device__ __forceinline__ void warp_for_each(const uint32_t* keys, const int32_t* idxs, int n, F&& f) {
  const int lane = threadIdx.x & 31;
  for (int e0 = 0; e0 < n; e0 += 32 * kLoadsInFlight) {
    uint32_t k[kLoadsInFlight];
    int32_t ix[kLoadsInFlight];
#pragma unroll
    for (int u = 0; u < kLoadsInFlight; ++u) {
      const int e = e0 + u * 32 + lane;
      k[u] = e < n ? keys[e] : 0u;
      ix[u] = (kWithIdx && e < n) ? idxs[e] : 0;
    }
#pragma unroll
    for (int u = 0; u < kLoadsInFlight; ++u) f(e0 + u * 32 + lane < n, k[u], ix[u]);
  }
}

// Exact threshold (v, cut): exactly K entries satisfy key > v || (key == v && idx <= cut),
// the top-K by key with ties to the lower index.  One histogram pass finds the boundary bin;
// its entries (normally a handful) are gathered and ranked directly; a crowded boundary bin
// (many equal or nearly equal scores) falls back to radix passes over the whole buffer.
__device__ void warp_exact_threshold(const uint32_t* keys, const int32_t* idxs, int n, int K, uint32_t kmin,
                                     uint32_t kmax, WarpScratch& ws, int* bc, uint32_t& v, uint32_t& cut) {
  const int lane = threadIdx.x & 31;
  const BinMap bin(kmin, kmax);
  for (int i = lane; i < kBins; i += 32) ws.hist[i] = 0u;
  __syncwarp();
  warp_for_each<false>(keys, idxs, n, [&](bool ok, uint32_t key, int32_t) { warp_hist_add(ws.hist, ok ? bin(key) : -1); });
  __syncwarp();
  const Boundary bd = warp_boundary(ws.hist, K);
  if (bd.hb <= kBoundary) {
    int got = 0;
    warp_for_each<true>(keys, idxs, n, [&](bool ok, uint32_t key, int32_t idx) {
      const bool in = ok && bin(key) == bd.b;
      const uint32_t m = __ballot_sync(0xffffffffu, in);
      if (in) {
        const int p = got + __popc(m & ((1u << lane) - 1u));
        ws.bkey[p] = key;
        ws.bidx[p] = idx;
      }
      got += __popc(m);
    });
    __syncwarp();
    const int need = K - bd.above;   // 1 <= need <= hb
    uint32_t fv = 0, fc = 0;
    bool found = false;
    for (int i = lane; i < bd.hb; i += 32) {
      const uint32_t ki = ws.bkey[i];
      const int32_t ii = ws.bidx[i];
      int rank = 0;
      for (int j = 0; j < bd.hb; ++j) rank += (ws.bkey[j] > ki || (ws.bkey[j] == ki && ws.bidx[j] < ii)) ? 1 : 0;
      if (rank == need - 1) {
        fv = ki;
        fc = static_cast<uint32_t>(ii);
        found = true;
      }
    }
    const uint32_t m = __ballot_sync(0xffffffffu, found);
    const int src = m ? __ffs(m) - 1 : 0;
    v = __shfl_sync(0xffffffffu, fv, src);
    cut = __shfl_sync(0xffffffffu, fc, src);
    __syncwarp();
    return;
  }
  __syncwarp();
  auto fe = [&](auto&& f) {
    warp_for_each<true>(keys, idxs, n, [&](bool ok, uint32_t key, int32_t idx) {
      if (ok) f(key, idx);
    });
  };
  radix_threshold<32>([] { __syncwarp(); }, fe, lane, K, ws.hist, bc, v, cut);
}

// Stable in-place compaction of the buffer to the entries `keep` selects; returns the count
// and the smallest / largest kept key (warp-uniform).
template <class Keep>
__device__ __forceinline__ int warp_compact(uint32_t* keys, int32_t* idxs, int n, const Keep& keep, uint32_t& kmin,
                                            uint32_t& kmax) {
  const int lane = threadIdx.x & 31;
  int written = 0;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int e0 = 0; e0 < n; e0 += 32 * kLoadsInFlight) {
    uint32_t k[kLoadsInFlight];
    int32_t ix[kLoadsInFlight];
#pragma unroll
    for (int u = 0; u < kLoadsInFlight; ++u) {
      const int e = e0 + u * 32 + lane;
      k[u] = e < n ? keys[e] : 0u;
      ix[u] = e < n ? idxs[e] : 0;
    }
    __syncwarp();   // every lane's loads of this batch before any store into it
#pragma unroll
    for (int u = 0; u < kLoadsInFlight; ++u) {
      const bool kp = e0 + u * 32 + lane < n && keep(k[u], ix[u]);
      const uint32_t m = __ballot_sync(0xffffffffu, kp);
      if (kp) {
        const int p = written + __popc(m & ((1u << lane) - 1u));
        keys[p] = k[u];
        idxs[p] = ix[u];
        mn = min(mn, k[u]);
        mx = max(mx, k[u]);
      }
      written += __popc(m);
    }
  }
  __syncwarp();
  kmin = __reduce_min_sync(0xffffffffu, mn);
  kmax = __reduce_max_sync(0xffffffffu, mx);
  return written;
}

// Cut a candidate buffer back to exactly its top-K (ties to the lower index), keeping the
// survivors in key order; returns the count and updates [kmin, kmax] to the kept keys.  Kept
// out of line: it runs only when scores keep rising along the keys.
__device__ __noinline__ int warp_cut_to_topk(uint32_t* keys, int32_t* idxs, int n, int K, WarpScratch& ws) {
  // extremes of the buffer's keys
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int e = static_cast<int>(threadIdx.x & 31u); e < n; e += 32) {
    const uint32_t kk = keys[e];
    kmin = min(kmin, kk);
    kmax = max(kmax, kk);
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  uint32_t v = 0, cut = 0;
  warp_exact_threshold(keys, idxs, n, K, kmin, kmax, ws, ws.bc, v, cut);
  return warp_compact(keys, idxs, n, [&](uint32_t key, int32_t idx) { return topk_keep(key, idx, v, cut); }, kmin,
                      kmax);
}

// Drops the entries below key tq from the buffer (in place, order kept); returns the count.
__device__ __noinline__ int warp_drop_below(uint32_t* keys, int32_t* idxs, int n, uint32_t tq) {
  uint32_t kmin = 0u, kmax = 0u;
  return warp_compact(keys, idxs, n, [&](uint32_t key, int32_t) { return key >= tq; }, kmin, kmax);
}

// ------------------------------------------------------------------ the kernel
struct IndexerArgs {
  const float* w;
  int n_q;
  const int2* row_range;
  const int2* group_range;
  int n_groups, n_chunks, chunk_len, cap, topk, trivial_len;
  int direct_max;               // rows with at most this many keys in a chunk keep every key
  uint32_t* cand_key;
  int32_t* cand_idx;
  uint32_t* cand_cnt;           // [row][chunk][kSub]
  uint32_t* cand_edge;          // per (row, chunk): a key below which no entry can be in the row's top-k (0: none)
  const int2* units;            // the dense unit list (launch_units), n_groups * n_chunks entries, or null
  uint32_t* status;
  unsigned long long wait_ns;   // bound of every pipeline wait
  int stop_after;               // test hook: the producer stops after this many key tiles (< 0: never)
};

// Unit u.  LIST: entry u of the dense list (launch_units: (group, chunk) pairs that hold keys,
// chunk-major, later groups first, then (-1, -1) entries without tiles).  Otherwise the same
// order over every pair, empty ones included: chunk u / n_groups, later (longer) groups first.
template <bool LIST>
__device__ __forceinline__ UnitInfo unit_info(int u, const IndexerArgs& A) {
  UnitInfo ui;
  if constexpr (LIST) {
    const int2 gc = A.units[u];
    ui.group = gc.x;
    ui.chunk = gc.y;
    if (gc.x < 0) {
      ui.kbeg = ui.kend = ui.n_tiles = 0;
      return ui;
    }
  } else {
    ui.chunk = u / A.n_groups;
    ui.group = A.n_groups - 1 - (u - ui.chunk * A.n_groups);
  }
  const int2 gr = A.group_range[ui.group];
  const long long b = static_cast<long long>(gr.x) + static_cast<long long>(ui.chunk) * A.chunk_len;
  const long long e = min(static_cast<long long>(gr.y), b + A.chunk_len);
  ui.kbeg = static_cast<int>(b);
  ui.kend = static_cast<int>(e > b ? e : b);
  ui.n_tiles = e > b ? static_cast<int>((e - b + kKeyTile - 1) / kKeyTile) : 0;
  return ui;
}


// Raise query g's boundary bin while the entries strictly above it number k or more; returns
// the new boundary bin and (in *above) the entries at or above it.  Histogram counts only grow
// while this runs, so a stale read can only stop the climb early.
template <int NB>
__device__ __forceinline__ int climb(const uint32_t* hist, int b, int topk, int* above) {
  const int lane = threadIdx.x & 31;
  // entries at or above b, summed by the whole warp
  int s = 0;
  for (int i = b + lane; i < NB; i += 32) s += static_cast<int>(*reinterpret_cast<const volatile uint32_t*>(&hist[i]));
  s = __reduce_add_sync(0xffffffffu, s);
  while (b < NB - 1) {
    const int h = static_cast<int>(*reinterpret_cast<const volatile uint32_t*>(&hist[b]));
    if (s - h < topk) break;
    s -= h;
    ++b;
  }
  *above = s;
  return b;
}

template <int HI, int DI, int G, bool LIST>
__global__ void __launch_bounds__(Cfg<HI, DI, G>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_q_in, const __grid_constant__ CUtensorMap tmap_k_in,
                   int q_split, int k_split, const PagedRows pg, const IndexerArgs A) {
  using C = Cfg<HI, DI, G>;
  constexpr int N = C::N, KB = C::KB, STAGES = C::STAGES, NE = C::NE, NH = C::NH, NB = C::NB;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared<G, NB, NE> sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::Q_BYTES;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_units = A.n_groups * A.n_chunks;
  uint32_t* status = A.status;
  const int cap4 = A.cap / kSub;
  // k-th unit of this CTA, in "snake" order: forward on even rounds, backward on odd ones,
  // so a CTA that drew a long unit in one round draws a short one in the next.
  auto snake_unit = [&](int k) {
    const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    return k * g + ((k & 1) ? (g - 1 - b) : b);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.t_full[b], 1);
      mbar_init(&sh.t_empty[b], NE);     // one arrive per head-sum warp
      mbar_init(&sh.u_done[b], NE);
      mbar_init(&sh.u_ready[b], 1);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  // both parities start reset: units 0 and 1 may begin at once
  for (int i = threadIdx.x; i < 2 * G * NB; i += blockDim.x) (&sh.hist[0][0][0])[i] = 0u;
  for (int i = threadIdx.x; i < 2 * G; i += blockDim.x) (&sh.tau[0][0])[i] = 0u;
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    mbar_arrive(&sh.u_ready[0]);
    mbar_arrive(&sh.u_ready[1]);
  }
  const uint32_t tmem = sh.tmem_base;
  const unsigned long long wait_ns = A.wait_ns;
  if (warp >= 4) {
    if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::REG_HIGH>();
    // ------------------------------------------------------------------ head-sum warps
    constexpr int GH = C::GH;
    const int hw = warp - 4;
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int half = hw >> 2;                  // queries [half * GH, half * GH + GH)
    const int g0 = half * GH;
    const int row = quarter * 32 + lane;       // key within the tile
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t below = (1u << lane) - 1u;
    uint32_t tile = 0, unit_ord = 0;
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && ok; ++k) {
      const int u = snake_unit(k);
      if (u >= n_units) continue;
      const UnitInfo ui = unit_info<LIST>(u, A);
      if (ui.n_tiles == 0) continue;
      const int par = unit_ord & 1;
      // this unit's histograms and thresholds have been reset
      ok = warp_wait(&sh.u_ready[par], (unit_ord >> 1) & 1, &sh.abort_flag, status, wait_ns);
      if (!ok) break;
      // the head weights of this warp's queries (lane l loads weights l, l + 32, ...) and their
      // key ranges
      const int t0 = ui.group * G + g0;
      float wl[NH / 32];
#pragma unroll
      for (int c = 0; c < NH / 32; ++c) {
        const int i = c * 32 + lane;
        wl[c] = t0 + i / HI < A.n_q ? __ldg(A.w + static_cast<size_t>(t0) * HI + i) : 0.f;
      }
      int qa[GH], qb[GH], cnt[GH];
      bool qf[GH];
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        const QueryRange r = query_range(A.row_range, t0 + g, A.n_q, ui, A.trivial_len, A.direct_max);
        qa[g] = r.a;
        qb[g] = r.b;
        qf[g] = r.filtered;
        cnt[g] = 0;
      }
      // every head weight of the warp's queries stays in registers, in every lane, for the whole
      // unit: read from shared memory per tile, each weight would cost a broadcast load into all
      // 32 lanes of all eight warps, 1024 cycles of load bandwidth per tile, as long as the
      // tile's MMAs
      float wreg[NH];
#pragma unroll
      for (int c = 0; c < NH; ++c) wreg[c] = __shfl_sync(0xffffffffu, wl[c / 32], c % 32);
      // this warp's sub-buffer of each query in this chunk
      size_t sub_off[GH];
#pragma unroll
      for (int g = 0; g < GH; ++g)
        sub_off[g] = ((static_cast<size_t>(t0 + g) * A.n_chunks + ui.chunk) * kSub + quarter) * cap4;
      // partial sums per query (NP / 2 packed pairs): four with 16 or more heads, two below (the
      // half's many queries already give independent chains)
      constexpr int NP = HI >= 16 ? 4 : 2;
      constexpr int NPP = NP / 2;
      // the tiles run in an inner loop with no call in it: a sub-buffer that could overflow on
      // the next tile leaves it, is cut back here, and the tiles go on
      uint32_t full = 0u;
      for (int i = 0;;) {
        for (; i < ui.n_tiles; ++i, ++tile) {
          const int buf = tile & 1;
          ok = warp_wait(&sh.t_full[buf], (tile >> 1) & 1, &sh.abort_flag, status, wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tbase = tmem + t_lane + buf * N + half * NH;
          // thresholds read now (a stale one is lower, which only keeps more), used after the sum
          uint32_t tk[GH];
#pragma unroll
          for (int g = 0; g < GH; ++g) tk[g] = qf[g] ? *reinterpret_cast<volatile uint32_t*>(&sh.tau[par][g0 + g]) : 0u;
          float part[GH][NP];
#pragma unroll
          for (int g = 0; g < GH; ++g)
#pragma unroll
            for (int p = 0; p < NP; ++p) part[g][p] = 0.f;
          // ReLU * w summed into the partial sums of columns [cb, cb + width) of v
          auto reduce = [&](const auto& v, int cb) {
            constexpr int W = sizeof(v) / sizeof(v[0]);
#pragma unroll
            for (int j = 0; j < W; j += 4) {
              const int c = cb + j;
              const int gl = c / HI;   // query within the half (HI is a multiple of 4)
              const int pa = (2 * (c / 4)) % NPP, pb = (2 * (c / 4) + 1) % NPP;
              const float r0 = fmaxf(__uint_as_float(v[j]), 0.f), r1 = fmaxf(__uint_as_float(v[j + 1]), 0.f);
              const float r2 = fmaxf(__uint_as_float(v[j + 2]), 0.f), r3 = fmaxf(__uint_as_float(v[j + 3]), 0.f);
              fma2(part[gl][2 * pa], part[gl][2 * pa + 1], wreg[c], wreg[c + 1], r0, r1);
              fma2(part[gl][2 * pb], part[gl][2 * pb + 1], wreg[c + 2], wreg[c + 3], r2, r3);
            }
          };
          if constexpr (GH >= 4) {
            // four rows per warp (8-row groups): each 16-column TMEM load is in flight while the
            // 16 columns before it are reduced (a wait covers every earlier load, so it follows
            // the reduction it overlaps): prefill_4k 75.6 -> 72.0 us, and no spills
            auto landed = [](uint32_t (&v)[16]) {   // uses of v stay after the wait
              asm volatile("" : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                           "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                           "+r"(v[14]), "+r"(v[15]));
            };
            uint32_t va[16], vb[16];
            tmem_ld16(tbase, va);
            tmem_ld_wait();
            landed(va);
#pragma unroll
            for (int c0 = 0; c0 < NH; c0 += 32) {
              tmem_ld16(tbase + c0 + 16, vb);
              reduce(va, c0);
              tmem_ld_wait();
              landed(vb);
              if (c0 + 32 < NH) tmem_ld16(tbase + c0 + 32, va);
              reduce(vb, c0 + 16);
              if (c0 + 32 < NH) {
                tmem_ld_wait();
                landed(va);
              }
            }
          } else {
            // two rows or fewer per warp: whole 32-column loads measured faster (chunk_1m's 4-row
            // groups: 50.6 ms against 51.4 with the overlapped 16-column form)
#pragma unroll
            for (int c0 = 0; c0 < NH; c0 += 32) {
              uint32_t v[32];
              tmem_ld32(tbase + c0, v);
              tmem_ld_wait();
              reduce(v, c0);
            }
          }
          float accs[GH];   // this lane's key (row of the quarter): its score for every query of the half
#pragma unroll
          for (int g = 0; g < GH; ++g) {
            float sp[NP];
#pragma unroll
            for (int p = 0; p < NP; ++p) sp[p] = part[g][p];
#pragma unroll
            for (int w2 = NP / 2; w2 >= 1; w2 /= 2)
#pragma unroll
              for (int p = 0; p < w2; ++p) sp[p] += sp[p + w2];
            accs[g] = sp[0];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.t_empty[buf]);
          const int j = ui.kbeg + i * kKeyTile + row;
          // every query's keep mask first (independent work), then the stores where one is set
          uint32_t keys[GH], masks[GH], any = 0u;
#pragma unroll
          for (int g = 0; g < GH; ++g) {
            keys[g] = float_key(accs[g]);
            masks[g] = __ballot_sync(0xffffffffu, j >= qa[g] && j < qb[g] && keys[g] >= tk[g]);
            any |= masks[g];
          }
          if (any == 0u) continue;
#pragma unroll
          for (int g = 0; g < GH; ++g) {
            const uint32_t m = masks[g];
            if (m == 0u) continue;
            const bool keep = (m >> lane) & 1u;
            const int p = cnt[g] + __popc(m & below);
            if (keep && p < cap4) {
              A.cand_key[sub_off[g] + p] = keys[g];
              A.cand_idx[sub_off[g] + p] = j;
            }
            if (keep && qf[g]) atomicAdd(&sh.hist[par][g0 + g][hist_bin<C>(keys[g])], 1u);
            cnt[g] += __popc(m);
            full |= (qf[g] && cnt[g] > cap4 - 32) ? 1u << g : 0u;
          }
          if (full != 0u) {   // warp-uniform: masks and counts are the same in every lane
            ++i;
            ++tile;
            break;
          }
        }
        if (full == 0u) break;   // every tile done, or a wait ran out (ok is false)
        __syncwarp();            // this warp's stores are visible to all its lanes
        for (int g = 0; g < GH; ++g) {
          if (!((full >> g) & 1u)) continue;
          // scores rising along the keys: cut the sub-buffer back to exactly its own top-k,
          // which keeps every key of the row's top-k that lies in it
          if (cnt[g] > cap4) {
            if (lane == 0) atomicOr(status, DEV_ERR_OVERFLOW);
            cnt[g] = cap4;
          }
          cnt[g] = warp_cut_to_topk(A.cand_key + sub_off[g], A.cand_idx + sub_off[g], cnt[g], A.topk, sh.ws[hw]);
        }
        full = 0u;
      }
      if (!ok) break;
      // A filtered query's sub-buffer still holds the keys kept while its threshold was lower:
      // drop those below the threshold as it stands now (no higher than the chunk's final edge,
      // so no key of the row's top-k goes), while the buffer is still in L2.  The final select
      // then reads about k entries per chunk instead of k (1 + ln(chunk / k)).
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        const uint32_t tq = qf[g] ? *reinterpret_cast<volatile uint32_t*>(&sh.tau[par][g0 + g]) : 0u;
        if (tq > 0u && cnt[g] > 0)
          cnt[g] = warp_drop_below(A.cand_key + sub_off[g], A.cand_idx + sub_off[g], min(cnt[g], cap4), tq);
      }
      // this warp's count of each of its queries in this chunk
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          const int t = t0 + g;
          if (t < A.n_q)
            A.cand_cnt[(static_cast<size_t>(t) * A.n_chunks + ui.chunk) * kSub + quarter] =
                static_cast<uint32_t>(min(cnt[g], cap4));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.u_done[par]);
      ++unit_ord;
    }
  } else {
    // warpgroup 0
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REG_LOW>();
    if (warp == 0) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_q_in);
        tma_prefetch_desc(&tmap_k_in);
        uint32_t kstage = 0, q_uses = 0;
        bool ok = true;
        for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && ok; ++k) {
          const int u = snake_unit(k);
          if (u >= n_units) continue;
          const UnitInfo ui = unit_info<LIST>(u, A);
          if (ui.n_tiles == 0) continue;
          if (q_uses > 0) ok = mbar_wait_for(&sh.q_empty, (q_uses - 1) & 1, &sh.abort_flag, status, wait_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(&sh.q_full, C::Q_BYTES);
          // 64-dim blocks without rotary dims come from the unrotated input
          for (int b = 0; b < KB; ++b)
            tma_load_2d(sQ + b * N * 128, b < q_split ? &tmap_q_in : &tmap_q, &sh.q_full, b * 64, ui.group * N);
          ++q_uses;
          for (int i = 0; i < ui.n_tiles; ++i, ++kstage) {
            if (A.stop_after >= 0 && kstage >= static_cast<uint32_t>(A.stop_after)) {
              ok = false;   // test hook: stop feeding the pipeline; its waits then run out
              break;
            }
            const int s = kstage % STAGES;
            if (kstage >= STAGES) {
              ok = mbar_wait_for(&sh.k_empty[s], ((kstage / STAGES) - 1) & 1, &sh.abort_flag, status, wait_ns);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(&sh.k_full[s], C::K_STAGE_BYTES);
            uint8_t* dst = sK + s * C::K_STAGE_BYTES;
            // cache row of the tile's first key: contiguous, or its page (one 128-key tile per
            // page; a group is one row in paged mode).  A page outside the cache is flagged and
            // row 0 read instead (the tile's scores are then meaningless, the status says so).
            int krow = ui.kbeg + i * kKeyTile;
            if (pg.block_table) {
              const int lp = krow >> kPageShift;
              const int page = lp < pg.max_pages ? __ldg(pg.block_table + static_cast<size_t>(ui.group) * pg.max_pages + lp) : -1;
              if (page < 0 || page >= pg.n_pages) {
                atomicOr(status, DEV_ERR_BAD_INDEX);
                krow = 0;
              } else {
                krow = page << kPageShift;
              }
            }
            for (int b = 0; b < KB; ++b)
              tma_load_2d(dst + b * kKeyTile * 128, b < k_split ? &tmap_k_in : &tmap_k, &sh.k_full[s], b * 64, krow);
          }
        }
        // let copies still in flight land before the CTA can exit (bounded; normally all done)
        if (q_uses > 0) mbar_drain(&sh.q_full, (q_uses - 1) & 1, 200000000ull);
        for (uint32_t j = kstage > STAGES ? kstage - STAGES : 0; j < kstage; ++j)
          mbar_drain(&sh.k_full[j % STAGES], (j / STAGES) & 1, 200000000ull);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------ MMA issuer
      // The whole warp runs the loop (descriptors stay warp-uniform, built once per tile as a
      // base plus compile-time offsets) and one elected lane issues each instruction: issuing
      // from a single thread with descriptors rebuilt per MMA cost about 110 cycles per MMA,
      // enough to leave the tensor pipe idle a third of the time.
      constexpr uint32_t idesc = idesc_bf16_f32(128, N, 0, 0);
      const uint64_t qd0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_for(bar, parity, &sh.abort_flag, status, wait_ns));
      };
      uint32_t kstage = 0, q_uses = 0, tile = 0;
      bool ok = true;
      for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && ok; ++k) {
        const int u = snake_unit(k);
        if (u >= n_units) continue;
        const UnitInfo ui = unit_info<LIST>(u, A);
        if (ui.n_tiles == 0) continue;
        ok = wait(&sh.q_full, q_uses & 1);
        if (!ok) break;
        ++q_uses;
        for (int i = 0; i < ui.n_tiles; ++i, ++kstage, ++tile) {
          const int s = kstage % STAGES;
          const int buf = tile & 1;
          ok = wait(&sh.k_full[s], (kstage / STAGES) & 1);
          if (ok && tile >= 2) ok = wait(&sh.t_empty[buf], ((tile >> 1) - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd0 = sdesc_sw128(smem_u32(sK + s * C::K_STAGE_BYTES), 16, 1024);
#pragma unroll
          for (int k = 0; k < DI / 16; ++k) {
            const int kb = k >> 2, sub = k & 3;
            umma_bf16_elect(tmem + buf * N, kd0 + static_cast<uint64_t>((kb * kKeyTile * 128 + sub * 32) >> 4),
                            qd0 + static_cast<uint64_t>((kb * N * 128 + sub * 32) >> 4), idesc, k > 0 ? 1u : 0u);
          }
          umma_commit_elect(&sh.k_empty[s]);
          umma_commit_elect(&sh.t_full[buf]);
        }
        if (ok) umma_commit_elect(&sh.q_empty);
      }
      // every MMA issued has completed before TMEM is released
      umma_commit_elect(&sh.mma_done);
      mbar_drain(&sh.mma_done, 0, 200000000ull);
      __syncwarp();
    } else if (warp == 2) {
      // ------------------------------------------------------------------ threshold warp
      uint32_t unit_ord = 0;
      bool ok = true;
      for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && ok; ++k) {
        const int u = snake_unit(k);
        if (u >= n_units) continue;
        const UnitInfo ui = unit_info<LIST>(u, A);
        if (ui.n_tiles == 0) {
          // an empty chunk still tells the final select that it holds no candidates (the
          // unit list has zeroed those counts already and pads with group -1)
          if constexpr (!LIST) {
            for (int e = lane; e < G * kSub; e += 32) {
              const int t = ui.group * G + e / kSub;
              if (t < A.n_q) A.cand_cnt[(static_cast<size_t>(t) * A.n_chunks + ui.chunk) * kSub + (e % kSub)] = 0u;
            }
            for (int g = lane; g < G; g += 32) {
              const int t = ui.group * G + g;
              if (t < A.n_q) A.cand_edge[static_cast<size_t>(t) * A.n_chunks + ui.chunk] = 0u;
            }
          }
          continue;
        }
        const int par = unit_ord & 1;
        // per filtered query (lane g holds query g's state)
        bool filt = false;
        if (lane < G) filt = query_range(A.row_range, ui.group * G + lane, A.n_q, ui, A.trivial_len, A.direct_max).filtered;
        const uint32_t fmask = __ballot_sync(0xffffffffu, filt);
        int bstar = 0, above = 0;   // lane g: query g's boundary bin and entries at or above it
        const uint64_t t0 = globaltimer_ns();
        while (true) {
          const bool done = mbar_try_wait(&sh.u_done[par], (unit_ord >> 1) & 1);
          // raise the threshold of every filtered query (the whole warp sums one histogram)
          for (uint32_t fm = fmask; fm; fm &= fm - 1) {
            const int g = __ffs(fm) - 1;
            const int b0 = __shfl_sync(0xffffffffu, bstar, g);
            int ab = 0;
            const int b = climb<NB>(sh.hist[par][g], b0, A.topk, &ab);
            if (lane == g) {
              bstar = b;
              above = ab;
            }
            if (b != b0 && lane == 0)
              *reinterpret_cast<volatile uint32_t*>(&sh.tau[par][g]) = b > 0 ? bin_edge_key<C>(b) : 0u;
          }
          if (__all_sync(0xffffffffu, done)) break;
          if (sh.abort_flag) {
            ok = false;
            break;
          }
          // the head-sum warps' own bounded waits end a stalled unit (abort flag above); this
          // bound is only a safety net
          if (globaltimer_ns() - t0 > 100ull * wait_ns) {
            if (lane == 0) {
              sh.abort_flag = 1u;
              atomicOr(status, DEV_ERR_TIMEOUT);
            }
            ok = false;
            break;
          }
          // a fresher threshold keeps fewer keys: pauses of 64 ns rather than 256 took chunk_1m's
          // indexer from 66.2 to 65.6 ms, none at all to 69.3 ms (the scans then crowd out the
          // head-sum warps on this warp's scheduler)
          __nanosleep(fmask ? 64 : 2048);
        }
        if (!ok) break;
        // the unit is done: each row's edge in this chunk (the lower edge of its boundary bin
        // when at least k entries lie at or above it: nothing below can make the row's top-k)
        if (lane < G) {
          const int t = ui.group * G + lane;
          if (t < A.n_q)
            A.cand_edge[static_cast<size_t>(t) * A.n_chunks + ui.chunk] =
                filt && bstar > 0 && above >= A.topk ? bin_edge_key<C>(bstar) : 0u;
        }
        // reset this parity for the unit after next, then let its head-sum warps start
        for (int i = lane; i < G * NB; i += 32) (&sh.hist[par][0][0])[i] = 0u;
        if (lane < G) sh.tau[par][lane] = 0u;
        __syncwarp();
        __threadfence_block();
        if (lane == 0) mbar_arrive(&sh.u_ready[par]);
        ++unit_ord;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int HI, int DI, int G, bool LIST>
cudaError_t launch_t(const IndexerPlan& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tqi,
                     const CUtensorMap& tki, int q_split, int k_split, const PagedRows& pg, const IndexerArgs& A,
                     cudaStream_t st) {
  using C = Cfg<HI, DI, G>;
  auto kern = indexer_kernel<HI, DI, G, LIST>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (C::REG_SPLIT) {
      // the head-sum warpgroups' setmaxnreg.inc waits for registers the block must hold from
      // launch: refuse to launch a build whose register count would leave it waiting
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs < C::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    }
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  kern<<<p.grid, C::THREADS, C::DYN_SMEM, st>>>(tq, tk, tqi, tki, q_split, k_split, pg, A);
  return cudaGetLastError();
}

}  // namespace


cudaError_t launch_indexer(const IndexerPlan& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tqi,
                           const CUtensorMap& tki, int q_split, int k_split, const PagedRows& pg, const float* w, int n_q,
                           const int2* row_range, const int2* group_range, int trivial_len, uint32_t* ck, int32_t* ci,
                           uint32_t* cc, uint32_t* ce, const int2* units, uint32_t* status,
                           const PipelineDebug& dbg, cudaStream_t st) {
  if (p.n_groups * p.n_chunks == 0) return cudaSuccess;
  if (pg.block_table && (p.group != 1 || p.chunk % kPageRows != 0)) return cudaErrorInvalidValue;
  IndexerArgs A;
  A.w = w;
  A.n_q = n_q;
  A.row_range = row_range;
  A.group_range = group_range;
  A.n_groups = p.n_groups;
  A.n_chunks = p.n_chunks;
  A.chunk_len = p.chunk;
  A.cap = p.cap;
  A.direct_max = kDirectMax;
  A.topk = p.topk;
  A.trivial_len = trivial_len;
  A.cand_key = ck;
  A.cand_idx = ci;
  A.cand_cnt = cc;
  A.cand_edge = ce;
  A.units = units;
  A.status = status;
  A.wait_ns = dbg.wait_ns;
  A.stop_after = dbg.stop_after_tiles;
  // shared-prefix groups (G = min(256 / H_I, 16)) walk every (group, chunk) pair; independent
  // rows (G = 64 / H_I) read the dense unit list
#define DSA_IDX_CASE(HI_, DI_, G_, LIST_)                                                              \
  if (p.n_heads == HI_ && p.head_dim == DI_ && p.group == G_ && p.unit_list == LIST_)                 \
    return launch_t<HI_, DI_, G_, LIST_>(p, tq, tk, tqi, tki, q_split, k_split, pg, A, st);
  DSA_IDX_CASE(4, 64, 16, false)
  DSA_IDX_CASE(8, 64, 16, false)
  DSA_IDX_CASE(16, 64, 16, false)
  DSA_IDX_CASE(32, 64, 8, false)
  DSA_IDX_CASE(64, 64, 4, false)
  DSA_IDX_CASE(4, 128, 16, false)
  DSA_IDX_CASE(8, 128, 16, false)
  DSA_IDX_CASE(16, 128, 16, false)
  DSA_IDX_CASE(32, 128, 8, false)
  DSA_IDX_CASE(64, 128, 4, false)
  DSA_IDX_CASE(4, 64, 16, true)
  DSA_IDX_CASE(8, 64, 8, true)
  DSA_IDX_CASE(16, 64, 4, true)
  DSA_IDX_CASE(32, 64, 2, true)
  DSA_IDX_CASE(64, 64, 1, true)
  DSA_IDX_CASE(4, 128, 16, true)
  DSA_IDX_CASE(8, 128, 8, true)
  DSA_IDX_CASE(16, 128, 4, true)
  DSA_IDX_CASE(32, 128, 2, true)
  DSA_IDX_CASE(64, 128, 1, true)
#undef DSA_IDX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dsa
