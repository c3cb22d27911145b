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
// A thread of the epilogue owns one key (one TMEM lane) and reduces the heads of every
// query in registers, so the head sum and the ReLU/weight epilogue never leave the SM and
// the score matrix is never written anywhere.
//
// Streaming top-k.  Per (row, chunk) the kernel keeps a candidate buffer of `cap` entries
// (order-preserving score key, key index) in the workspace and a running threshold tau in
// shared memory.  A score is appended only when it beats tau.  When a buffer could
// overflow on the next tile the epilogue threads cut it back to a superset of its top-k (one
// binned pass, exact radix select when the boundary bin is crowded) and raise tau to the
// smallest kept key.  Keys of a unit are visited in increasing index order, so "beats tau" is
// a strict comparison.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (owns TMEM), then the epilogue:
// warps 2..5 (TMEM lane quarters 2, 3, 0, 1), and with several queries per group warps 6..9
// as a second half that takes the other half of the queries (192 or 320 threads).  Q is
// single-buffered per unit, K tiles go through a STAGES-deep ring, S^T is double-buffered in
// TMEM.
#include <cuda_bf16.h>

#include <cstddef>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int kKeyTile = 128;
constexpr int kMaxCap = 4224;    // cap = 2k + 128 with k <= 2048
constexpr int kCutBins = 2048;   // value-linear bins of a cut-back

template <int HI, int DI, int G>
struct Cfg {
  static constexpr int N = G * HI;                       // MMA N: (query, head) pairs
  static constexpr int KB = DI / 64;                     // 128-byte K blocks per row
  static constexpr int Q_BYTES = N * DI * 2;
  static constexpr int K_STAGE_BYTES = kKeyTile * DI * 2;
  static constexpr int SMEM_BUDGET = 232448 - 14336;     // dynamic budget after static smem
  static constexpr int STAGES_FIT = (SMEM_BUDGET - 1024 - Q_BYTES) / K_STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int DYN_SMEM = 1024 + Q_BYTES + STAGES * K_STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = (2 * N <= 32) ? 32 : (2 * N <= 64) ? 64 : (2 * N <= 128) ? 128 : (2 * N <= 256) ? 256 : 512;
  // Epilogue: one warp per TMEM lane quarter per half; with several queries per group the
  // queries (and their TMEM columns) are split between two halves, so two warps share every
  // lane quarter and hide each other's latencies.
  static constexpr int HALVES = G >= 2 && N >= 128 ? 2 : 1;
  static constexpr int EPI = 128 * HALVES;               // epilogue threads
  static constexpr int THREADS = 64 + EPI;
  static constexpr int GH = G / HALVES;                  // queries per half
  static constexpr int NH = N / HALVES;                  // TMEM columns per half
  static_assert(N % 64 == 0 && N >= 64 && N <= 256, "MMA N");
  static_assert(NH % 64 == 0, "epilogue reads 64 columns at a time");
  static_assert(STAGES >= 2, "shared memory");
};

struct Shared {
  alignas(16) float w_s[256];   // read as float4 by the epilogue: keep 16-byte aligned
  alignas(8) int2 rr[64];
  uint64_t k_full[8], k_empty[8];
  uint64_t q_full, q_empty;
  uint64_t t_full[2], t_empty[2];
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t hist[kCutBins];   // cut-back histogram (the radix fallback uses the first 256 bins)
  int bc[4];
  int warp_off[8];
  uint32_t wmin[8], wmax[8];
  uint32_t tau[64];
  int cnt[2][64];        // candidates held per query; [tile parity] so a tile reads one copy and writes the other
  alignas(16) int qcnt[4][64];   // this tile's appends per (TMEM lane quarter, query)
  int epi_abort;
};
static_assert(offsetof(Shared, w_s) % 16 == 0, "float4 access");
static_assert(sizeof(Shared) <= 14336, "static shared memory within the budget the stage count assumes");

// Named barrier over n threads that also returns the OR of a predicate across them.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Candidate store through the global state space.  No "memory" clobber: the compiler may keep
// shared-memory state in registers across it (a generic store could alias shared memory).
// The store stays in program order with the other volatile asm statements (barriers, fences)
// that publish it.
__device__ __forceinline__ void st_global_u32(uint32_t* p, uint32_t v) {
  asm volatile("{\n .reg .u64 ga;\n cvta.to.global.u64 ga, %0;\n st.global.u32 [ga], %1;\n}\n" ::"l"(p), "r"(v));
}

struct UnitInfo {
  int group, chunk, kbeg, kend, n_tiles;
};

__device__ __forceinline__ UnitInfo unit_info(int u, int n_groups, int chunk_len, const int2* group_range) {
  UnitInfo ui;
  ui.chunk = u / n_groups;
  ui.group = n_groups - 1 - (u - ui.chunk * n_groups);  // later (longer) groups first
  const int2 gr = group_range[ui.group];
  const long long b = static_cast<long long>(gr.x) + static_cast<long long>(ui.chunk) * chunk_len;
  const long long e = min(static_cast<long long>(gr.y), b + chunk_len);
  ui.kbeg = static_cast<int>(b);
  ui.kend = static_cast<int>(e > b ? e : b);
  ui.n_tiles = e > b ? static_cast<int>((e - b + kKeyTile - 1) / kKeyTile) : 0;
  return ui;
}

// Cut the candidate buffer of one (row, chunk) back to a superset of its top-K, keeping the
// survivors in their original (key index) order.  Called by the NT epilogue threads together.
//
// The buffer only has to keep every entry that can still be in the final top-K, so the cut
// need not be exact: one histogram of 2048 bins linear in score over the buffer's [min, max]
// finds the bin b holding the K-th largest score, and every entry in bins >= b is kept (at
// least K entries; bins are monotone in score, so everything dropped scores below everything
// kept).  The new threshold is the smallest kept key: a later key at or below it has at least
// K earlier keys at or above it and loses to them (ties go to the lower key index).  When the
// boundary bin is crowded (many equal or nearly equal scores) so that the cut would free less
// than half the headroom, the exact radix select (threshold (v, cut), exactly K kept) runs
// instead.  Returns {threshold key, entries kept}.
struct CutResult {
  uint32_t tau;
  int kept;
};
template <int NT>
__device__ CutResult compact_buffer(uint32_t* keys, int32_t* idxs, int n, int K, int tid, Shared& sh) {
  // Entry tid + NT i is held by thread tid in slot i (coalesced loads and stores); round i
  // is the NT entries [NT i, NT i + NT), so list order = (round, thread) order.
  constexpr int kMaxPer = (kMaxCap + NT - 1) / NT;
  constexpr int NW = NT / 32;
  const int lane = tid & 31, wq = tid >> 5;
  const int rounds = (n + NT - 1) / NT;   // <= kMaxPer
  uint32_t rk[kMaxPer];
  int32_t ri[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int e = tid + i * NT;
    const bool in = e < n;
    rk[i] = in ? keys[e] : 0u;
    ri[i] = in ? idxs[e] : 0;
  }
  auto sync = [] { named_bar_sync(1, NT); };
  auto fe = [&](auto&& f) {
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i)
      if (tid + i * NT < n) f(rk[i], ri[i]);
  };
  // ---- coarse cut: key range, then one histogram pass
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  fe([&](uint32_t key, int32_t) {
    mn = min(mn, key);
    mx = max(mx, key);
  });
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    sh.wmin[wq] = mn;
    sh.wmax[wq] = mx;
  }
  for (int i = tid; i < kCutBins; i += NT) sh.hist[i] = 0u;
  sync();
  uint32_t kmin = sh.wmin[0], kmax = sh.wmax[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    kmin = min(kmin, sh.wmin[w]);
    kmax = max(kmax, sh.wmax[w]);
  }
  const float fmin = key_float(kmin), fmax = key_float(kmax);
  const float span = fmax - fmin;
  const float scale = span > 0.f && span < 3.0e38f ? static_cast<float>(kCutBins) / span : 0.f;
  auto bin_of = [&](uint32_t key) {
    const float y = (key_float(key) - fmin) * scale;
    return y >= static_cast<float>(kCutBins - 1) ? kCutBins - 1 : (y > 0.f ? static_cast<int>(y) : 0);
  };
  fe([&](uint32_t key, int32_t) { atomicAdd(&sh.hist[bin_of(key)], 1u); });
  sync();
  // thread tid owns the kPerT bins [kCutBins - kPerT (tid + 1), kCutBins - kPerT tid), visited
  // from the top
  constexpr int kPerT = kCutBins / NT;
  {
    int h[kPerT], sum = 0;
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
      h[j] = static_cast<int>(sh.hist[kCutBins - 1 - (tid * kPerT + j)]);
      sum += h[j];
    }
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) sh.warp_off[wq] = x;
    sync();
    int c = x - sum;
    for (int w = 0; w < wq; ++w) c += sh.warp_off[w];
    if (c < K && K <= c + sum) {
#pragma unroll
      for (int j = 0; j < kPerT; ++j) {
        if (c < K && K <= c + h[j]) {
          sh.bc[0] = kCutBins - 1 - (tid * kPerT + j);
          sh.bc[1] = c + h[j];   // entries in bins >= the boundary bin
        }
        c += h[j];
      }
    }
    sync();
  }
  const int bb = sh.bc[0], kept_coarse = sh.bc[1];
  const int cap_free = n - kKeyTile;   // the cut is only worth it if it frees half the headroom
  const bool coarse = kept_coarse <= K + (cap_free - K) / 2;
  uint32_t v = 0, cut = 0x7FFFFFFFu;
  if (!coarse) {
    sync();
    radix_threshold<NT>(sync, fe, tid, K, sh.hist, sh.bc, v, cut);
  }
  // ---- stable compaction: per round, a ballot per warp; warp counts of every round go to
  // shared memory (sh.hist is free now), one warp turns them into exclusive offsets in
  // (round, warp) order, and every kept entry lands at its offset + its rank in the ballot
  uint32_t kb[kMaxPer];
  uint32_t kmin_kept = 0xFFFFFFFFu;
  uint32_t* rc = sh.hist;   // [kMaxPer][NW] counts, then offsets
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const bool in = tid + i * NT < n;
    const bool k = in && (coarse ? bin_of(rk[i]) >= bb : topk_keep(rk[i], ri[i], v, cut));
    kb[i] = __ballot_sync(0xffffffffu, k);
    if (k) kmin_kept = min(kmin_kept, rk[i]);
    if (lane == 0 && i < rounds) rc[i * NW + wq] = __popc(kb[i]);
  }
  kmin_kept = __reduce_min_sync(0xffffffffu, kmin_kept);
  if (lane == 0) sh.wmin[wq] = kmin_kept;
  sync();
  if (wq == 0) {
    // exclusive scan of rounds * NW counts in order, 32 lanes x kPer entries
    constexpr int kPer = (kMaxPer * NW + 31) / 32;
    const int m = rounds * NW;
    uint32_t c[kPer], sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = lane * kPer + j;
      c[j] = e < m ? rc[e] : 0u;
      sum += c[j];
    }
    uint32_t x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    uint32_t run = x - sum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = lane * kPer + j;
      if (e < m) rc[e] = run;
      run += c[j];
    }
    if (lane == 31) sh.bc[2] = static_cast<int>(x);   // total kept
  }
  sync();
  const int kept = sh.bc[2];
  uint32_t tau = v;
  if (coarse) {
    tau = sh.wmin[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) tau = min(tau, sh.wmin[w]);
  }
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    if (i < rounds && ((kb[i] >> lane) & 1u)) {
      const int pos = static_cast<int>(rc[i * NW + wq] + __popc(kb[i] & below));
      keys[pos] = rk[i];
      idxs[pos] = ri[i];
    }
  }
  __threadfence_block();
  sync();
  return CutResult{tau, kept};
}

template <int HI, int DI, int G>
__global__ void __launch_bounds__(Cfg<HI, DI, G>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_q_in, const __grid_constant__ CUtensorMap tmap_k_in,
                   int q_split, int k_split, const PagedRows pg,
                   const float* __restrict__ w, int n_q, const int2* __restrict__ row_range,
                   const int2* __restrict__ group_range, int n_groups, int n_chunks, int chunk_len, int cap, int topk,
                   uint32_t* __restrict__ cand_key, int32_t* __restrict__ cand_idx, uint32_t* __restrict__ cand_cnt,
                   uint32_t* status) {
  using C = Cfg<HI, DI, G>;
  constexpr int N = C::N, KB = C::KB, STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::Q_BYTES;
  const int warp = threadIdx.x >> 5;
  const int n_units = n_groups * n_chunks;
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
      mbar_init(&sh.t_empty[b], C::EPI / 32);   // one arrive per epilogue warp
    }
    sh.abort_flag = 0;
    sh.epi_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_lane0()) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_q_in);
      tma_prefetch_desc(&tmap_k_in);
      uint32_t kstage = 0, q_uses = 0;
      bool ok = true;
      for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && ok; ++k) {
        const int u = snake_unit(k);
        if (u >= n_units) continue;
        const UnitInfo ui = unit_info(u, n_groups, chunk_len, group_range);
        if (ui.n_tiles == 0) continue;
        if (q_uses > 0) ok = mbar_wait(&sh.q_empty, (q_uses - 1) & 1, &sh.abort_flag, status);
        if (!ok) break;
        mbar_arrive_expect_tx(&sh.q_full, C::Q_BYTES);
        // 64-dim blocks without rotary dims come from the unrotated input
        for (int b = 0; b < KB; ++b)
          tma_load_2d(sQ + b * N * 128, b < q_split ? &tmap_q_in : &tmap_q, &sh.q_full, b * 64, ui.group * N);
        ++q_uses;
        for (int i = 0; i < ui.n_tiles; ++i, ++kstage) {
          const int s = kstage % STAGES;
          if (kstage >= STAGES) {
            ok = mbar_wait(&sh.k_empty[s], ((kstage / STAGES) - 1) & 1, &sh.abort_flag, status);
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
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_lane0()) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, N, 0, 0);
      uint32_t kstage = 0, q_uses = 0, tile = 0;
      bool ok = true;
      for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && ok; ++k) {
        const int u = snake_unit(k);
        if (u >= n_units) continue;
        const UnitInfo ui = unit_info(u, n_groups, chunk_len, group_range);
        if (ui.n_tiles == 0) continue;
        ok = mbar_wait(&sh.q_full, q_uses & 1, &sh.abort_flag, status);
        if (!ok) break;
        ++q_uses;
        for (int i = 0; i < ui.n_tiles; ++i, ++kstage, ++tile) {
          const int s = kstage % STAGES;
          const int buf = tile & 1;
          ok = mbar_wait(&sh.k_full[s], (kstage / STAGES) & 1, &sh.abort_flag, status);
          if (ok && tile >= 2) ok = mbar_wait(&sh.t_empty[buf], ((tile >> 1) - 1) & 1, &sh.abort_flag, status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sK + s * C::K_STAGE_BYTES);
          const uint32_t b0 = smem_u32(sQ);
#pragma unroll
          for (int k = 0; k < DI / 16; ++k) {
            const int kb = k >> 2, sub = k & 3;
            const uint64_t ad = sdesc_sw128(a0 + kb * kKeyTile * 128 + sub * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + kb * N * 128 + sub * 32, 16, 1024);
            umma_bf16(tmem + buf * N, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
          umma_commit(&sh.k_empty[s]);
          umma_commit(&sh.t_full[buf]);
        }
        if (ok) umma_commit(&sh.q_empty);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    constexpr int EPI = C::EPI, GH = C::GH, NH = C::NH;
    const int tid = threadIdx.x - 64;          // 0 .. EPI - 1
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    const int half = tid / 128;                // queries [half * GH, half * GH + GH)
    const int g0 = half * GH;
    const int lane = threadIdx.x & 31;
    const int row = quarter * 32 + lane;       // key within the tile
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    // A failed (timed-out) wait reaches every epilogue warp through the per-tile
    // barrier-reduction (fast tiles) or through sh.epi_abort, written only before the
    // barrier-reduction and read only after it (slow tiles), so all epilogue warps leave the
    // loops at the same point.
    uint32_t tile = 0;
    bool stop = false;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_units && !stop; ++k) {
      const int u = snake_unit(k);
      if (u >= n_units) continue;
      const UnitInfo ui = unit_info(u, n_groups, chunk_len, group_range);
      const int t0 = ui.group * G;
      // per-unit state
      for (int i = tid; i < N; i += EPI) {
        const int t = t0 + i / HI;
        sh.w_s[i] = t < n_q ? __ldg(w + static_cast<size_t>(t) * HI + (i % HI)) : 0.f;
      }
      if (tid < G) {
        const int t = t0 + tid;
        sh.rr[tid] = t < n_q ? row_range[t] : make_int2(0, 0);
        sh.tau[tid] = 0u;
        sh.cnt[tile & 1][tid] = 0;
      }
      named_bar_sync(1, EPI);
      for (int i = 0; i < ui.n_tiles; ++i, ++tile) {
        const int buf = tile & 1;
        const int tile0 = ui.kbeg + i * kKeyTile;
        // Fast tile: no query's buffer has been cut back yet and none can fill up through
        // this tile (uniform across the CTA).  tau is then still below every key, so every
        // in-range key is appended and its slot is its offset in the range: no ballots, no
        // counts exchanged.  Counts only grow with i, so once a tile is slow the rest are.
        bool fast = true;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int2 rr = sh.rr[g];
          const int a = max(rr.x, ui.kbeg), b = min(rr.y, ui.kend);
          fast = fast && min(b, tile0 + kKeyTile) - a <= cap - kKeyTile;
        }
        bool ok = mbar_wait(&sh.t_full[buf], (tile >> 1) & 1, &sh.abort_flag, status);
        ok = __all_sync(0xffffffffu, ok);
        uint32_t msk[GH];
        uint32_t key[GH];
        float acc[GH];
        if (ok) {
          tc_fence_after();
          // Head sum of this half's queries with NP independent partial sums per query
          // (breaks the dependent FMA chain), TMEM read 64 columns per wait.
          constexpr int NP = HI >= 16 ? 4 : 1;
          float part[GH][NP];
#pragma unroll
          for (int g = 0; g < GH; ++g)
#pragma unroll
            for (int p = 0; p < NP; ++p) part[g][p] = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < NH; c0 += 64) {
            const int cc = half * NH + c0;   // TMEM column of this chunk
            uint32_t v[64];
            tmem_ld32(tmem + t_lane + buf * N + cc, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tmem + t_lane + buf * N + cc + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              const float4 wv = *reinterpret_cast<const float4*>(&sh.w_s[cc + j]);
              const float r0 = fmaxf(__uint_as_float(v[j]), 0.f), r1 = fmaxf(__uint_as_float(v[j + 1]), 0.f);
              const float r2 = fmaxf(__uint_as_float(v[j + 2]), 0.f), r3 = fmaxf(__uint_as_float(v[j + 3]), 0.f);
              const int gl = (c0 + j) / HI;   // query within the half
              if constexpr (NP == 4) {
                // columns cc+j .. cc+j+3 feed partial sums 0..3 of query gl: two packed FMAs
                fma2(part[gl][0], part[gl][1], wv.x, wv.y, r0, r1);
                fma2(part[gl][2], part[gl][3], wv.z, wv.w, r2, r3);
              } else {
                const float wj[4] = {wv.x, wv.y, wv.z, wv.w}, rj[4] = {r0, r1, r2, r3};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float& acc_e = part[(c0 + j + e) / HI][0];
                  acc_e = fmaf(wj[e], rj[e], acc_e);
                }
              }
            }
          }
#pragma unroll
          for (int g = 0; g < GH; ++g) {
            if constexpr (NP == 4) acc[g] = (part[g][0] + part[g][1]) + (part[g][2] + part[g][3]);
            else acc[g] = part[g][0];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.t_empty[buf]);
          if (fast) {
            // every in-range key is appended: key j of query g goes to slot j - a_g
            const int j = tile0 + row;
            const size_t rowbase = (static_cast<size_t>(t0) * n_chunks + ui.chunk) * cap;
#pragma unroll
            for (int gl = 0; gl < GH; ++gl) {
              const int g = g0 + gl;
              const int2 rr = sh.rr[g];
              const int a = max(rr.x, ui.kbeg), b = min(rr.y, ui.kend);
              if (j >= a && j < b) {
                const size_t off = rowbase + static_cast<size_t>(g) * n_chunks * cap + (j - a);
                st_global_u32(cand_key + off, float_key(acc[gl]));
                st_global_u32(reinterpret_cast<uint32_t*>(cand_idx) + off, static_cast<uint32_t>(j));
              }
            }
            if (tid < G) {
              const int2 rr = sh.rr[tid];
              const int a = max(rr.x, ui.kbeg), b = min(rr.y, ui.kend);
              sh.cnt[(tile & 1) ^ 1][tid] = max(0, min(b, tile0 + kKeyTile) - a);
            }
          }
        }
        if (fast) {
          // one barrier-reduction per tile carries a timed-out wait to every epilogue warp
          if (bar_red_or(1, EPI, !ok)) {
            stop = true;
            break;
          }
          continue;
        }
        if (ok) {
          // append candidates that beat the running threshold, in key order: per query the
          // four lane quarters publish their counts, then each writes after the lower ones
          const int j = tile0 + row;
#pragma unroll
          for (int gl = 0; gl < GH; ++gl) {
            const int g = g0 + gl;
            const int2 rr = sh.rr[g];
            key[gl] = float_key(acc[gl]);
            msk[gl] = __ballot_sync(0xffffffffu, j >= rr.x && j < rr.y && j < ui.kend && key[gl] > sh.tau[g]);
          }
          if (lane == 0) {
#pragma unroll
            for (int gl = 0; gl < GH; ++gl) sh.qcnt[quarter][g0 + gl] = __popc(msk[gl]);
          }
        }
        named_bar_sync(1, EPI);                               // X: per-quarter counts published
        const int cur = tile & 1, nxt = cur ^ 1;
        bool need = false;
        if (ok) {
          const int j = tile0 + row;
          // every query's write offset first (shared loads only), then the global stores
          int pos[GH];
#pragma unroll
          for (int gl = 0; gl < GH; ++gl) pos[gl] = sh.cnt[cur][g0 + gl] + __popc(msk[gl] & ((1u << lane) - 1u));
          for (int q = 0; q < quarter; ++q) {
#pragma unroll
            for (int gl = 0; gl < GH; ++gl) pos[gl] += sh.qcnt[q][g0 + gl];
          }
          int tot = 0;
          if (tid < G) tot = (sh.qcnt[0][tid] + sh.qcnt[1][tid]) + (sh.qcnt[2][tid] + sh.qcnt[3][tid]);
          const size_t rowbase = (static_cast<size_t>(t0) * n_chunks + ui.chunk) * cap;
#pragma unroll
          for (int gl = 0; gl < GH; ++gl) {
            if (((msk[gl] >> lane) & 1u) && pos[gl] < cap) {
              const size_t off = rowbase + static_cast<size_t>(g0 + gl) * n_chunks * cap + pos[gl];
              st_global_u32(cand_key + off, key[gl]);
              st_global_u32(reinterpret_cast<uint32_t*>(cand_idx) + off, static_cast<uint32_t>(j));
            }
          }
          if (tid < G) {
            const int n = sh.cnt[cur][tid] + tot;
            sh.cnt[nxt][tid] = n;
            need = n > cap - kKeyTile;                      // could overflow on the next tile
          }
        }
        // Y: one barrier-reduction decides whether anything beyond the appends is needed (a
        // cut-back or an abort).  The abort flag is written before it and read only in the
        // slow path, between it and one more barrier, so all epilogue warps branch alike.
        if (!ok && lane == 0) sh.epi_abort = 1;
        if (bar_red_or(1, EPI, need || !ok)) {
          stop = sh.epi_abort != 0;
          named_bar_sync(1, EPI);
          if (stop) break;
#pragma unroll 1
          for (int g = 0; g < G; ++g) {
            const int n = sh.cnt[nxt][g];
            if (n > cap - kKeyTile) {
              const size_t off = (static_cast<size_t>(t0 + g) * n_chunks + ui.chunk) * cap;
              __threadfence_block();
              const CutResult cr = compact_buffer<EPI>(cand_key + off, cand_idx + off, n, topk, tid, sh);
              if (tid == 0) {
                sh.tau[g] = cr.tau;
                sh.cnt[nxt][g] = cr.kept;
              }
              named_bar_sync(1, EPI);
            }
          }
        }
      }
      if (stop) break;
      if (tid < G && t0 + tid < n_q)
        cand_cnt[static_cast<size_t>(t0 + tid) * n_chunks + ui.chunk] =
            static_cast<uint32_t>(min(sh.cnt[tile & 1][tid], cap));
      named_bar_sync(1, EPI);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int HI, int DI, int G>
cudaError_t launch_t(const IndexerPlan& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tqi,
                     const CUtensorMap& tki, int q_split, int k_split, const PagedRows& pg, const float* w, int n_q,
                     const int2* row_range, const int2* group_range, uint32_t* ck, int32_t* ci, uint32_t* cc,
                     uint32_t* status, cudaStream_t st) {
  using C = Cfg<HI, DI, G>;
  auto kern = indexer_kernel<HI, DI, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<p.grid, C::THREADS, C::DYN_SMEM, st>>>(tq, tk, tqi, tki, q_split, k_split, pg, w, n_q, row_range, group_range,
                                             p.n_groups, p.n_chunks,
                                             p.chunk, p.cap, p.topk, ck, ci, cc, status);
  return cudaGetLastError();
}

}  // namespace


cudaError_t launch_indexer(const IndexerPlan& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tqi,
                           const CUtensorMap& tki, int q_split, int k_split, const PagedRows& pg, const float* w, int n_q,
                           const int2* row_range, const int2* group_range, uint32_t* ck, int32_t* ci, uint32_t* cc,
                           uint32_t* status, cudaStream_t st) {
  if (p.n_groups * p.n_chunks == 0) return cudaSuccess;
  if (pg.block_table && (p.group != 1 || p.chunk % kPageRows != 0)) return cudaErrorInvalidValue;
#define DSA_IDX_CASE(HI_, DI_, G_)                                                                      \
  if (p.n_heads == HI_ && p.head_dim == DI_ && p.group == G_)                                           \
    return launch_t<HI_, DI_, G_>(p, tq, tk, tqi, tki, q_split, k_split, pg, w, n_q, row_range, group_range, ck, ci, cc, \
                                  status, st);
  DSA_IDX_CASE(4, 64, 64)
  DSA_IDX_CASE(8, 64, 32)
  DSA_IDX_CASE(16, 64, 16)
  DSA_IDX_CASE(32, 64, 8)
  DSA_IDX_CASE(64, 64, 4)
  DSA_IDX_CASE(4, 128, 64)
  DSA_IDX_CASE(8, 128, 32)
  DSA_IDX_CASE(16, 128, 16)
  DSA_IDX_CASE(32, 128, 8)
  DSA_IDX_CASE(64, 128, 4)
  DSA_IDX_CASE(4, 64, 16)
  DSA_IDX_CASE(8, 64, 8)
  DSA_IDX_CASE(16, 64, 4)
  DSA_IDX_CASE(32, 64, 2)
  DSA_IDX_CASE(64, 64, 1)
  DSA_IDX_CASE(4, 128, 16)
  DSA_IDX_CASE(8, 128, 8)
  DSA_IDX_CASE(16, 128, 4)
  DSA_IDX_CASE(32, 128, 2)
  DSA_IDX_CASE(64, 128, 1)
#undef DSA_IDX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dsa
