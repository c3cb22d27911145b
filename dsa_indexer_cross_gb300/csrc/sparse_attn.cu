// MLA-absorbed sparse attention over the selected latent rows, on tcgen05.
//
//   o[t, h] = sum_{j in I_t} softmax_j(tau * q[t, h] . kv[ks_t + j]) * kv[ks_t + j, :512]
//
// ("GLM-5.2 IndexShare" explainer, section 1 and "What is actually shared?": every layer
// runs its own attention over the selected positions; the 576 = 512 latent + 64 rope key
// and the 512-d value follow "GLM-5/5.1/5.2 DSA + LoRA enablement", qk_rope_head_dim
// commit.)  All heads of a token read the same selected rows.
//
// Formulation.  A CTA owns a work item of HB "columns" (query, head pairs) and walks rows
// of the latent cache in tiles of 64.  HB (16..64) is too small for the M side of the tensor
// core, so both products run transposed, with the latent rows on M:
//     S^T[r, c]  = Rows[r, :576] . Q[c, :576]            M = 64 rows,   N = HB, K = 576
//     O^T[d, c] += Rows[:, d]^T  . P^T[r, c]             M = 128 dims,  N = HB, K = 64
// A tile is stored once in shared memory as nine 64-dim blocks in the 128-byte-swizzled
// layout, read as a K-major operand by the first product and as an MN-major operand by the
// second, so each row is brought on chip once per item.  Two tiles are in flight, each slot set
// with one full/empty barrier pair; block-dense tiles arrive as one 3-D TMA box (one copy of
// 72 KB keeps the TMA unit much busier than nine 8 KB copies).  P^T of tile g (bf16, MN-major)
// is written into that tile's rope block, which the first product no longer needs once S^T is
// complete.  S^T is double-buffered in TMEM; O^T (512 x HB fp32) stays in TMEM for the whole
// item.
//
// Two ways to walk the rows (template parameter HD):
//   HD == 0  "gather": item = (token, block of HB heads); the tile holds the token's next
//            64 selected rows, fetched with cp.async (an empty slot reads zeros and is
//            masked); a paged cache maps each offset through the token's block table
//            (template parameter PAGED).
//   HD  > 0  "block-dense": item = HB / HD consecutive tokens with all HD heads; the tile is
//            64 CONSECUTIVE latent rows of the block's key range, fetched by TMA, and a
//            per-(token, row) selection bitmask built from the index rows masks S^T.  Used
//            when the selections are dense (short prefixes, k close to the prefix length):
//            every row is then fetched once per block instead of once per token.
// Both compute exactly the same sums; only unselected (masked) entries are skipped.
//
// Online softmax (base 2): the per-column max in use lives in shared memory and changes only
// when a score exceeds it by more than 8 (a factor 256); one barrier-reduction per tile
// detects that, and only then are the tile's column maxima exchanged and O^T and the running
// sums rescaled (exact either way).  A softmax warp reads its 16 rows of S^T with the 16x256b
// TMEM shape, so each thread holds two rows and HB/4 columns; running sums stay in registers
// and are reduced once per item.
//
// Warp roles: warps 0-1 load Q and the rows (Q as nine 64-dim TMA boxes; the rows as one
// 3-D TMA box per tile in block-dense mode, or with cp.async in the gather walk); warp 2 issues the S^T products; warps 3-6 (and 8-11 in
// the block-dense walk) run the softmax and the epilogue; warp 7 owns TMEM and issues the PV
// products (256 threads, 384 block-dense).  With the two products issued from separate
// warps, PV(g) goes out as soon as P(g) exists instead of queueing behind S^T(g+1), whose
// blocks may still be in flight.  Persistent CTAs.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kRows = 64;          // latent rows per tile
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kKB = kDqk / 64;     // 64-dim blocks per tile (the last one holds the rope dims)
constexpr int kBlkBytes = kRows * 128;         // one block: 64 rows x 128 B
constexpr int kSlots = 2 * kKB;                // two tiles in flight
constexpr int kProd = 64;                      // warps 0-1
// Gather walk: every 64-dim block of a tile comes through cp.async (the load/store unit).
// Four-row TMA gathers for some of the blocks were slower: the TMA unit takes ~37 cycles per
// gather, and moving the last of them to cp.async cut the walk's time by a quarter (1M-key
// chunk) to a third (32K prefill).
constexpr int kCpBlocks = 9;
// Warps 0-1 load, warp 2 issues S^T, warps 3-6 (and, block-dense, 8-11) run the softmax,
// warp 7 owns TMEM and issues PV.
constexpr int kMaskBytes = kDenseMaskBytes;    // selection bitmask budget (block-dense)

template <int HB, int HD>
struct ACfg {
  static constexpr bool DENSE = HD > 0;
  static constexpr int B = DENSE ? HB / HD : 1;                        // tokens per item
  static constexpr int MAXR = DENSE ? (kMaskBytes * 8 / B) / 64 * 64 : 0;  // longest key range
  static constexpr int Q_BYTES = HB * kDqk * 2;
  static constexpr int M_BYTES = DENSE ? kMaskBytes : 0;
  static constexpr int DYN_SMEM = 1024 + kSlots * kBlkBytes + Q_BYTES + M_BYTES;
  static constexpr uint32_t TMEM_COLS = 6 * HB <= 128 ? 128 : 6 * HB <= 256 ? 256 : 512;
  static constexpr int O_COL = 0;
  static constexpr int S_COL = 4 * HB;
  static constexpr int SW = DENSE ? 8 : 4;                             // softmax warps (2 or 1 per lane quarter)
  static constexpr int SOFT = 32 * SW;
  static constexpr int THREADS = kProd + 32 + SOFT + 32;
  static constexpr int CW = HB / (SW / 4);                             // columns per softmax warp
  static constexpr int NR = CW / 8;                                    // 16x256b repetitions per warp
  static_assert(HB % 16 == 0 && HB <= 64, "columns");
  static_assert(CW % 16 == 0, "the epilogue reads 16-column groups");
  static_assert(!DENSE || HB % HD == 0, "whole tokens per dense item");
  static_assert(HB * kRows * 2 <= kBlkBytes, "P^T must fit in the rope block");
};

// Per-column softmax state lives in shared memory (uniform across the softmax threads).
struct AShared {
  uint64_t full[2], empty[2];   // per tile slot set (nine 64-dim blocks)
  uint64_t q_full, q_empty, s_full[2], s_empty[2], p_full, o_done[2], o_free;   // o_done[g & 1]: PV(g) complete
  uint64_t mma_done;            // both MMA warps' last commits: nothing of theirs in flight
  uint32_t tmem_base, abort_flag, soft_abort;
  uint32_t prod_ok;
  alignas(16) float red[4][64];
  alignas(16) float m_used[64];
  alignas(16) float l_run[64];
  alignas(16) float alpha[64];
};
static_assert(ACfg<64, 0>::DYN_SMEM + sizeof(AShared) <= 232448, "HB=64 must fit in shared memory");
static_assert(ACfg<64, 16>::DYN_SMEM + sizeof(AShared) <= 232448, "block-dense must fit in shared memory");

__device__ __forceinline__ int slot_of(uint32_t g, int kb) { return static_cast<int>(g & 1u) * kKB + kb; }

// 16 consecutive floats of shared memory into registers (four 16-byte loads issued together).
__device__ __forceinline__ void load_row16(float (&r)[16], const float* p) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = *reinterpret_cast<const float4*>(p + 4 * i);
    r[4 * i] = v.x;
    r[4 * i + 1] = v.y;
    r[4 * i + 2] = v.z;
    r[4 * i + 3] = v.w;
  }
}
// Store through the explicit shared state space (the compiler then knows it cannot alias the
// shared-memory loads around it).
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// 2^x by the hardware approximation (ex2.approx.ftz.f32; relative error far below the bf16
// rounding that P goes through next); exp2(-inf) = +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Gather walk split over several CTAs per (token, head block) (few tokens, long selections:
// decode): split s of n walks the token's tiles [s T / n, (s + 1) T / n) and writes its output
// normalised by its own running sum, in fp32, with its log-sum-exp; a combine pass merges the
// splits.  n == 1: no split, the kernel writes out and lse itself.
struct SplitOut {
  int n;
  float* o;      // [n][n_q * H][512]
  float* lse;    // [n][n_q * H]
};

// Work item description shared by all roles.
struct Item {
  int t0;        // gather: the token; block-dense: first token of the block
  int hb;        // gather: head block; block-dense: 0
  int nt;        // tiles of 64 rows
  int lo;        // block-dense: first latent row of the block's range
  int i0;        // gather: first tile of the split
  int split;     // gather: split index
};

template <int HB, int HD>
__device__ __forceinline__ Item item_info(int item, int n_hb, int n_split, const int32_t* row_nt,
                                          const int2* block_range) {
  Item it{};
  if constexpr (HD == 0) {
    const int per_tok = n_hb * n_split;
    it.t0 = item / per_tok;
    const int r = item - it.t0 * per_tok;
    it.hb = r / n_split;
    it.split = r - it.hb * n_split;
    const int T = __ldg(row_nt + it.t0);
    it.i0 = (it.split * T) / n_split;
    it.nt = ((it.split + 1) * T) / n_split - it.i0;
    it.lo = 0;
  } else {
    it.t0 = item * (HB / HD);
    it.hb = 0;
    const int2 r = block_range[item];
    it.lo = r.x;
    it.nt = r.y > r.x ? (r.y - r.x + kRows - 1) / kRows : 0;
  }
  return it;
}

// Where one token's selection offsets live: rows kst + j of a contiguous cache, or (PAGED)
// through the token's block-table row, offsets valid below lim.  Built once per work item so
// the per-slot mapping touches no further per-token state; the cache kind is a template
// parameter, so the contiguous kernel carries no trace of paging.
struct TokenRows {
  long long kst;
  const int32_t* bt;
  int lim;
};
template <bool PAGED>
__device__ __forceinline__ TokenRows token_rows(const PagedRows& pg, const int32_t* ks, int t) {
  TokenRows r{};
  if constexpr (PAGED) {
    r.bt = pg.block_table + static_cast<size_t>(t) * pg.max_pages;
    r.lim = min(__ldg(pg.seq_len + t), pg.max_pages << kPageShift);
  } else {
    r.kst = __ldg(ks + t);
  }
  return r;
}
// Latent row of selection offset j: -1 for an empty slot (j < 0), -2 for an offset or page
// outside the cache.
template <bool PAGED>
__device__ __forceinline__ long long latent_row(const TokenRows& tr, const PagedRows& pg, int n_kv, int j) {
  if (j < 0) return -1;
  if constexpr (PAGED) {
    if (j >= tr.lim) return -2;
    const int page = __ldg(tr.bt + (j >> kPageShift));
    if (page < 0 || page >= pg.n_pages) return -2;
    return (static_cast<long long>(page) << kPageShift) + (j & (kPageRows - 1));
  } else {
    const long long row = tr.kst + j;
    return row >= 0 && row < n_kv ? row : -2;
  }
}

template <int HB, int HD, bool PAGED>
__global__ void __launch_bounds__(ACfg<HB, HD>::THREADS, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tmap_kv, const __grid_constant__ CUtensorMap tmap_q,
                       const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx,
                       const int32_t* __restrict__ ks, const PagedRows pg, const int32_t* __restrict__ row_nt,
                       const int2* __restrict__ block_range, const uint32_t* __restrict__ block_mask,
                       uint16_t* __restrict__ out, float* __restrict__ lse, int n_q, int n_kv, int H, int topk,
                       float scale_log2, uint32_t* status, uint32_t* bad_count, unsigned long long wait_ns,
                       int stop_after, const SplitOut split) {
  using C = ACfg<HB, HD>;
  constexpr bool DENSE = C::DENSE;
  constexpr int B = C::B;
  constexpr int NR = C::NR;
  extern __shared__ uint8_t smem_raw[];
  __shared__ AShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sT = smem;                                   // kSlots blocks of 64 rows x 128 B
  uint8_t* sQ = smem + kSlots * kBlkBytes;              // HB x 576, 9 blocks of HB x 128 B
  uint32_t* sMask = reinterpret_cast<uint32_t*>(sQ + C::Q_BYTES);   // block-dense: B x MAXR bits
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_hb = DENSE ? 1 : (H + HB - 1) / HB;
  const int n_split = DENSE ? 1 : split.n;
  const int n_items = DENSE ? (n_q + B - 1) / B : n_q * n_hb * n_split;
  // k-th item of this CTA in "snake" order (forward on even rounds, backward on odd ones):
  // causal items grow with their index, so alternating directions balances the CTAs.  The
  // block-dense walk takes its items from the last (largest) down, so that the partial last
  // round holds the smallest ones.  Past the end: n_items.
  auto snake_item = [&](int k) {
    const int gdim = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    const int r = k * gdim + ((k & 1) ? (gdim - 1 - b) : b);
    if constexpr (DENSE) return r < n_items ? n_items - 1 - r : n_items;
    return r;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.full[s], DENSE || kCpBlocks == 0 ? 1 : 1 + kProd);   // + the cp.async arrivals
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_empty[b], C::SW);   // one arrive per softmax warp
    }
    mbar_init(&sh.p_full, C::SW);
    mbar_init(&sh.o_done[0], 1);
    mbar_init(&sh.o_done[1], 1);
    mbar_init(&sh.o_free, C::SW);
    mbar_init(&sh.mma_done, 2);
    sh.abort_flag = 0;
    sh.soft_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 7) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp < 2) {
    // ---------------------------------------------------------------- Q and the rows (TMA)
    // Thread 0 does every wait and arms every barrier, then publishes the outcome in
    // sh.prod_ok between two named barriers (id 2), so the two producer warps always stop at
    // the same point and no copy is issued before its barrier expects the bytes.
    const int tid = threadIdx.x;
    uint32_t g = 0, it = 0;
    bool ok = true;
    auto sync_ok = [&](bool mine) -> bool {
      if (tid == 0) sh.prod_ok = mine ? 1u : 0u;
      named_bar_sync(2, kProd);
      const bool r = sh.prod_ok != 0;
      named_bar_sync(2, kProd);
      return r;
    };
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && ok; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      const Item I = item_info<HB, HD>(item, n_hb, n_split, row_nt, block_range);
      if (I.nt == 0) continue;
      bool w_ok = true;
      if (tid == 0) {
        if (it > 0) w_ok = mbar_wait_for(&sh.q_empty, (it - 1) & 1, &sh.abort_flag, status, wait_ns);
        if (w_ok) {
          // the item's HB consecutive (token, head) rows of q, as nine boxes of HB x 64 dims;
          // rows past the end of q read as zeros, and columns past the last head are never stored
          const int qrow = I.t0 * H + (DENSE ? 0 : I.hb * HB);
          mbar_arrive_expect_tx(&sh.q_full, C::Q_BYTES);
#pragma unroll 1
          for (int kb = 0; kb < kKB; ++kb) tma_load_2d(sQ + kb * (HB * 128), &tmap_q, &sh.q_full, kb * 64, qrow);
        }
      }
      ok = sync_ok(w_ok);
      if (!ok) break;
      if constexpr (DENSE) {
        // one thread streams the block's consecutive latent rows, one whole 64-row tile (nine
        // 64-dim blocks, one 3-D box) per copy as soon as its slot set is released
        if (tid == 0) {
          for (int i = 0; i < I.nt && ok; ++i, ++g) {
            const int s = g & 1;
            if (stop_after >= 0 && g >= static_cast<uint32_t>(stop_after)) {
              ok = false;   // test hook: stop feeding the pipeline; the waits behind it run out
              break;
            }
            if (g >= 2) {
              ok = mbar_wait_for(&sh.empty[s], ((g >> 1) - 1) & 1, &sh.abort_flag, status, wait_ns);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(&sh.full[s], kKB * kBlkBytes);
            tma_load_3d(sT + slot_of(g, 0) * kBlkBytes, &tmap_kv, &sh.full[s], 0, I.lo + i * kRows, 0);
          }
        }
        ok = sync_ok(ok);
      } else {
        // A tile is 64 selected rows x 9 blocks of 64 dims, copied with cp.async: thread tid
        // copies 16-byte chunk tid % 8 of rows tid / 8 + 8 m (m < 8) in every block, so a warp
        // reads four whole 128-byte row segments per instruction.  Row indices are read before
        // the slot set is released.  A slot without a selection (-1) reads zeros and is masked
        // by the softmax.
        static_assert(kCpBlocks == kKB, "the gather walk copies whole rows with cp.async");
        const int t = I.t0;
        const int32_t* irow = idx + static_cast<size_t>(t) * topk;
        const TokenRows trow = token_rows<PAGED>(pg, ks, t);
        // the index of a slot (-1 past topk), then its latent row (-1: none, flagged if invalid)
        auto index_of = [&](int slot) -> int { return slot < topk ? __ldg(irow + slot) : -1; };
        auto row_of = [&](int j, bool count_bad) -> int {
          long long row;
          bool v, bad;
          if constexpr (PAGED) {
            row = latent_row<true>(trow, pg, n_kv, j);
            v = row >= 0;
            bad = row == -2;
          } else {
            row = trow.kst + j;
            v = j >= 0 && row >= 0 && row < n_kv;
            bad = j >= 0 && !v;
          }
          if (count_bad && bad) {
            atomicOr(status, DEV_ERR_BAD_INDEX);
            atomicAdd(bad_count, 1u);
          }
          return v ? static_cast<int>(row) : -1;
        };
        // each tile's indices are loaded one tile ahead, so their latency hides behind the
        // previous tile's slot wait and copies
        int jn[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) jn[m] = index_of(I.i0 * kRows + (tid >> 3) + 8 * m);
        for (int i = 0; i < I.nt; ++i, ++g) {
          int crow[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) crow[m] = row_of(jn[m], (tid & 7) == 0);
          if (i + 1 < I.nt) {
#pragma unroll
            for (int m = 0; m < 8; ++m) jn[m] = index_of((I.i0 + i + 1) * kRows + (tid >> 3) + 8 * m);
          }
          // test hook: stop feeding the pipeline; the waits behind it run out
          w_ok = stop_after < 0 || g < static_cast<uint32_t>(stop_after);
          if (tid == 0 && w_ok) {
            if (g >= 2) w_ok = mbar_wait_for(&sh.empty[g & 1], ((g >> 1) - 1) & 1, &sh.abort_flag, status, wait_ns);
            if (w_ok) mbar_arrive(&sh.full[g & 1]);
          }
          ok = sync_ok(w_ok);
          if (!ok) break;
          uint8_t* tile = sT + slot_of(g, 0) * kBlkBytes;
          const int ch = tid & 7;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const int r = (tid >> 3) + 8 * m;
            const uint16_t* src = kv + static_cast<size_t>(crow[m] >= 0 ? crow[m] : 0) * kDqk + ch * 8;
#pragma unroll
            for (int b = 0; b < kKB; ++b)
              cp_async_16_zfill(smem_u32(tile + b * kBlkBytes + sw128(r, ch)), src + b * 64, crow[m] >= 0);
          }
          cp_async_mbar_arrive(&sh.full[g & 1]);
        }
      }
      ++it;
    }
    // let every copy this CTA started land before its shared memory can be released
    // (bounded; after a normal run everything has landed already)
    if constexpr (!DENSE && kCpBlocks > 0) cp_async_wait<0>();
    if (tid == 0) {
      if (it > 0) mbar_drain(&sh.q_full, (it - 1) & 1, 200000000ull);
      for (uint32_t j = g > 2 ? g - 2 : 0; j < g; ++j) mbar_drain(&sh.full[j & 1], (j >> 1) & 1, 200000000ull);
    }
  } else if ((warp >= 3 && warp < 7) || warp >= 8) {
    // ---------------------------------------------------------------- softmax + epilogue
    constexpr int kSoft = C::SOFT;
    const int tid = warp < 7 ? static_cast<int>(threadIdx.x) - 96 : 128 + static_cast<int>(threadIdx.x) - 256;
    const int qd = warp & 3;               // TMEM lane quarter
    const int c_off = warp >= 8 ? C::CW : 0;   // this warp's columns: [c_off, c_off + CW)
    const int r0 = qd * 16 + (lane >> 2);  // S^T rows held: r0 and r0 + 8
    const int cq = 2 * (lane & 3);         // column pair within each group of 8 columns
    const uint32_t t_lane = static_cast<uint32_t>(qd * 32) << 16;
    // A failed (timed-out) wait is published through sh.soft_abort, written only before a
    // named barrier and read right after it; the next write can only happen after a later
    // barrier, so all softmax warps always leave the loops at the same point.
    uint32_t g = 0, it = 0;
    bool stop = false;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && !stop; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      const Item I = item_info<HB, HD>(item, n_hb, n_split, row_nt, block_range);
      // column c -> (token, head)
      auto col_token = [&](int c) { return DENSE ? I.t0 + c / (DENSE ? HD : 1) : I.t0; };
      auto col_head = [&](int c) { return DENSE ? c % (DENSE ? HD : 1) : I.hb * HB + c; };
      auto col_ok = [&](int c) { return col_token(c) < n_q && col_head(c) < H; };
      if (I.nt == 0) {
        if (n_split > 1) {
          // an empty split: weight zero in the combine
          const size_t pbase = static_cast<size_t>(I.split) * n_q * H;
          for (int e = tid; e < HB * kDv; e += kSoft) {
            const int c = e / kDv;
            if (col_ok(c))
              split.o[(pbase + static_cast<size_t>(col_token(c)) * H + col_head(c)) * kDv + (e - c * kDv)] = 0.f;
          }
          if (tid < HB && col_ok(tid)) split.lse[pbase + static_cast<size_t>(col_token(tid)) * H + col_head(tid)] = -INFINITY;
          continue;
        }
        for (int e = tid; e < HB * kDv; e += kSoft) {
          const int c = e / kDv;
          if (col_ok(c))
            out[(static_cast<size_t>(col_token(c)) * H + col_head(c)) * kDv + (e - c * kDv)] = 0;
        }
        if (lse && tid < HB && col_ok(tid))
          lse[static_cast<size_t>(col_token(tid)) * H + col_head(tid)] = -INFINITY;
        continue;
      }
      // Column max in shared memory (read by all softmax threads); the running sums of this
      // thread's two rows stay in registers and are reduced across rows once per item.
      if (tid < HB) sh.m_used[tid] = -INFINITY;
      float lp[2 * NR];
#pragma unroll
      for (int c = 0; c < 2 * NR; ++c) lp[c] = 0.f;
      const int32_t* irow = idx + static_cast<size_t>(I.t0) * topk;
      if constexpr (DENSE) {
        // the item's selection bitmask over its key range, built by the pre-pass: one
        // round of 16-byte loads into shared memory
        constexpr int kVec = kMaskBytes / 16;
        const int4* gm = reinterpret_cast<const int4*>(block_mask) + static_cast<size_t>(item) * kVec;
        int4 mv[(kVec + kSoft - 1) / kSoft];
#pragma unroll
        for (int u = 0; u < (kVec + kSoft - 1) / kSoft; ++u) {
          const int e = tid + u * kSoft;
          if (e < kVec) mv[u] = __ldg(gm + e);
        }
#pragma unroll
        for (int u = 0; u < (kVec + kSoft - 1) / kSoft; ++u) {
          const int e = tid + u * kSoft;
          if (e < kVec) reinterpret_cast<int4*>(sMask)[e] = mv[u];
        }
      }
      named_bar_sync(1, kSoft);
      TokenRows trow{};
      if constexpr (!DENSE) trow = token_rows<PAGED>(pg, ks, I.t0);
      for (int i = 0; i < I.nt; ++i, ++g) {
        const int sb = g & 1;
        bool rv0 = false, rv1 = false;   // gather: rows r0 / r0 + 8 hold a valid selection
        if constexpr (!DENSE) {
          const int s0 = (I.i0 + i) * kRows + r0, s1 = s0 + 8;
          const int j0 = s0 < topk ? __ldg(irow + s0) : -1;
          const int j1 = s1 < topk ? __ldg(irow + s1) : -1;
          if constexpr (PAGED) {
            rv0 = latent_row<true>(trow, pg, n_kv, j0) >= 0;
            rv1 = latent_row<true>(trow, pg, n_kv, j1) >= 0;
          } else {
            const long long kst = trow.kst;
            rv0 = j0 >= 0 && kst + j0 >= 0 && kst + j0 < n_kv;
            rv1 = j1 >= 0 && kst + j1 >= 0 && kst + j1 < n_kv;
          }
        }
        bool ok = mbar_wait_for(&sh.s_full[sb], (g >> 1) & 1, &sh.abort_flag, status, wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        float sc[4 * NR];   // [4k + j]: j = 0,1 row r0 columns 8k+cq, +1;  j = 2,3 row r0 + 8
        bool need = false;
        if (ok) {
          tc_fence_after();
          uint32_t v[4 * NR];
          tmem_ld_16x256b<NR>(tmem + t_lane + C::S_COL + sb * HB + c_off, v);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.s_empty[sb]);
#pragma unroll
          for (int kk = 0; kk < NR; ++kk) {
            const float2 mu = *reinterpret_cast<const float2*>(&sh.m_used[c_off + 8 * kk + cq]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = c_off + 8 * kk + cq + (j & 1);
              bool valid;
              if constexpr (DENSE) {
                const int r = r0 + ((j & 2) ? 8 : 0);
                const uint2 mw = *reinterpret_cast<const uint2*>(
                    &sMask[(c / (DENSE ? HD : 1)) * (C::MAXR / 32) + i * (kRows / 32)]);
                valid = (((r < 32 ? mw.x : mw.y) >> (r & 31)) & 1u) != 0u;
              } else {
                valid = (j & 2) ? rv1 : rv0;
              }
              const float x = valid ? __uint_as_float(v[4 * kk + j]) * scale_log2 : -INFINITY;
              sc[4 * kk + j] = x;
              need |= x > ((j & 1) ? mu.y : mu.x) + 8.f;   // only a max that grew by > 2^8 forces a rescale
            }
          }
        }
        // One barrier-reduction per tile decides whether the slow path runs.  The abort
        // flag is written before it and read only inside the slow path, between two more
        // barriers, so every softmax warp takes the same branch.
        if (!ok && lane == 0) sh.soft_abort = 1;
        if (bar_red_or(1, kSoft, need || !ok)) {
          if (ok) {
#pragma unroll
            for (int kk = 0; kk < NR; ++kk) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float x = fmaxf(sc[4 * kk + e], sc[4 * kk + 2 + e]);
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
                if (lane < 4) sh.red[qd][c_off + 8 * kk + cq + e] = x;
              }
            }
            // O^T may only be rescaled once the previous tile's PV has finished
            if (i > 0) {
              ok = mbar_wait_for(&sh.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1, &sh.abort_flag, status, wait_ns);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok && lane == 0) sh.soft_abort = 1;
            }
          }
          named_bar_sync(1, kSoft);
          stop = sh.soft_abort != 0;
          if (!stop && tid < HB) {
            const int c = tid;
            const float m = fmaxf(fmaxf(sh.red[0][c], sh.red[1][c]), fmaxf(sh.red[2][c], sh.red[3][c]));
            float a = 1.f;
            if (m > sh.m_used[c] + 8.f) {
              a = exp2f(sh.m_used[c] - m);         // 0 when the old max is -inf
              sh.m_used[c] = m;
            }
            sh.alpha[c] = a;
          }
          named_bar_sync(1, kSoft);
          if (stop) break;
          tc_fence_after();
          bool any = false;
#pragma unroll
          for (int kk = 0; kk < NR; ++kk) {
            const float2 a = *reinterpret_cast<const float2*>(&sh.alpha[c_off + 8 * kk + cq]);
            lp[2 * kk] *= a.x;
            lp[2 * kk + 1] *= a.y;
          }
#pragma unroll
          for (int c0 = 0; c0 < HB; c0 += 16) {
            float ar[16];
            load_row16(ar, &sh.alpha[c0]);
#pragma unroll
            for (int c = 0; c < 16; ++c) any |= ar[c] != 1.f;
          }
          if (any && i > 0) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
#pragma unroll
              for (int hw = 0; hw < C::CW / 16; ++hw) {
                const int hh = c_off / 16 + hw;
                uint32_t o[16];
                tmem_ld16(tmem + t_lane + C::O_COL + b * HB + hh * 16, o);
                tmem_ld_wait();
                float ar[16];
                load_row16(ar, &sh.alpha[hh * 16]);
#pragma unroll
                for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * ar[h]);
                tmem_st16(tmem + t_lane + C::O_COL + b * HB + hh * 16, o);
              }
            }
            tmem_st_wait();
          }
        }
        // P = exp2(s - m) in bf16, written MN-major (row-by-row, 64 columns per 128 B) into
        // this tile's rope block as the B operand of the second product; the running sums
        // add the same rounded values the tensor core multiplies.
        const uint32_t p_base = smem_u32(sT + slot_of(g, kKB - 1) * kBlkBytes);
#pragma unroll
        for (int kk = 0; kk < NR; ++kk) {
          // a column whose max is still -inf has only masked (-inf) entries so far: subtract 0
          // there so that exp2(-inf) = 0 instead of exp2(NaN)
          float2 mu = *reinterpret_cast<const float2*>(&sh.m_used[c_off + 8 * kk + cq]);
          mu.x = mu.x == -INFINITY ? 0.f : mu.x;
          mu.y = mu.y == -INFINITY ? 0.f : mu.y;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = r0 + 8 * h;
            const float p0 = ex2_approx(sc[4 * kk + 2 * h] - mu.x);
            const float p1 = ex2_approx(sc[4 * kk + 2 * h + 1] - mu.y);
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            const int chunk = c_off / 8 + kk;   // 8-column (16-byte) chunk of the 64-column row
            st_shared_u32(p_base + r * 128 + ((chunk ^ (r & 7)) << 4) + cq * 2, *reinterpret_cast<const uint32_t*>(&pb));
            lp[2 * kk] += __low2float(pb);
            lp[2 * kk + 1] += __high2float(pb);
          }
        }
        // P(g) goes out without waiting for PV(g - 1): PV(g) queues behind it in the tensor
        // pipe anyway.  PV completions are signalled on o_done[g & 1]; S^T(g) complete implies
        // tile g was loaded, hence PV(g - 2) and everything before it finished, so a wait for
        // PV(g - 1) on o_done[(g - 1) & 1] at parity ((g - 1) >> 1) & 1 is exact.
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_full);
      }
      if (stop) break;
      // item end: column sums over the 64 rows, then O^T / l -> out
#pragma unroll
      for (int kk = 0; kk < NR; ++kk) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = lp[2 * kk + e];
          x += __shfl_xor_sync(0xffffffffu, x, 4);
          x += __shfl_xor_sync(0xffffffffu, x, 8);
          x += __shfl_xor_sync(0xffffffffu, x, 16);
          if (lane < 4) sh.red[qd][c_off + 8 * kk + cq + e] = x;
        }
      }
      bool ok = mbar_wait_for(&sh.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1, &sh.abort_flag, status, wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) sh.soft_abort = 1;
      named_bar_sync(1, kSoft);
      stop = sh.soft_abort != 0;
      if (tid < HB) sh.l_run[tid] = (sh.red[0][tid] + sh.red[1][tid]) + (sh.red[2][tid] + sh.red[3][tid]);
      named_bar_sync(1, kSoft);
      if (stop) break;
      tc_fence_after();
      // Column c is output row row0 + c in both walks (block-dense: HD == H, so the block's
      // (token, head) rows are consecutive; gather: the head block of one token); this thread
      // writes dimension b*128 + qd*32 + lane of every valid column of its column range.
      {
        const long long row0 = static_cast<long long>(I.t0) * H + (DENSE ? 0 : I.hb * HB);
        const int n_cols = DENSE ? min(HB, (n_q - I.t0) * H) : min(HB, H - I.hb * HB);
        uint16_t* obase = out + row0 * kDv + qd * 32 + lane;
#pragma unroll
        for (int hw = 0; hw < C::CW / 16; ++hw) {
          const int hh = c_off / 16 + hw;
          float inv[16];
          load_row16(inv, &sh.l_run[hh * 16]);
#pragma unroll
          for (int h = 0; h < 16; ++h) inv[h] = inv[h] > 0.f ? 1.f / inv[h] : 0.f;
          uint32_t o[4][16];
#pragma unroll
          for (int b = 0; b < 4; ++b) tmem_ld16(tmem + t_lane + C::O_COL + b * HB + hh * 16, o[b]);
          tmem_ld_wait();
#pragma unroll
          if (n_split > 1) {
            // this split's output, fp32, normalised by its own sum
            float* pbase = split.o + (static_cast<size_t>(I.split) * n_q * H + row0) * kDv + qd * 32 + lane;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              const int c = hh * 16 + h;
              if (c < n_cols) {
#pragma unroll
                for (int b = 0; b < 4; ++b)
                  pbase[static_cast<long long>(c) * kDv + b * 128] = __uint_as_float(o[b][h]) * inv[h];
              }
            }
            continue;
          }
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const int c = hh * 16 + h;
            if (c < n_cols) {
              uint16_t* orow = obase + static_cast<long long>(c) * kDv;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const __nv_bfloat16 ob = __float2bfloat16_rn(__uint_as_float(o[b][h]) * inv[h]);
                orow[b * 128] = *reinterpret_cast<const uint16_t*>(&ob);
              }
            }
          }
        }
      }
      if (tid < HB && col_ok(tid)) {
        const float lv = sh.l_run[tid];
        const float lval = lv > 0.f ? (sh.m_used[tid] + log2f(lv)) * 0.69314718055994531f : -INFINITY;
        const size_t r = static_cast<size_t>(col_token(tid)) * H + col_head(tid);
        if (n_split > 1) {
          split.lse[static_cast<size_t>(I.split) * n_q * H + r] = lval;
        } else if (lse) {
          lse[r] = lval;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.o_free);
      named_bar_sync(1, kSoft);                                 // per-column state and mask may be reset now
      ++it;
    }
  } else {
    // ---------------------------------------------------------------- MMA issuers
    // Warp 2 issues S^T, warp 7 issues PV.  Each whole warp runs its loop, so every
    // descriptor is warp-uniform and built as a per-tile base plus compile-time offsets; one
    // elected lane issues each instruction.  A commit tracks the MMAs of its own warp.
    constexpr uint32_t id_qk = idesc_bf16_f32(64, HB, 0, 0);
    constexpr uint32_t id_pv = idesc_bf16_f32(128, HB, 1, 1);
    const uint32_t st0 = smem_u32(sT);
    uint32_t g = 0, it = 0;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_for(bar, parity, &sh.abort_flag, status, wait_ns));
    };
    const bool qk_warp = warp == 2;
    const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);       // Q: B operand of S^T, K-major
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && ok; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      const Item I = item_info<HB, HD>(item, n_hb, n_split, row_nt, block_range);
      if (I.nt == 0) continue;
      if (qk_warp) {
        // S^T(g) = tile . Q^T once the whole tile has landed
        ok = wait(&sh.q_full, it & 1);
        for (int i = 0; i < I.nt && ok; ++i, ++g) {
          const int sb = g & 1;
          if (g >= 2 && !(ok = wait(&sh.s_empty[sb], ((g >> 1) - 1) & 1))) break;
          if (!(ok = wait(&sh.full[g & 1], (g >> 1) & 1))) break;
          if constexpr (!DENSE && kCpBlocks > 0) fence_proxy_async_smem();   // cp.async-written blocks
          tc_fence_after();
          const uint64_t da = sdesc_sw128(st0 + (g & 1u) * (kKB * kBlkBytes), 16, 1024);
          const uint32_t d_s = tmem + C::S_COL + sb * HB;
#pragma unroll
          for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
            for (int sub = 0; sub < 4; ++sub)
              umma_bf16_elect(d_s, da + static_cast<uint64_t>((kb * kBlkBytes + sub * 32) >> 4),
                              dq0 + static_cast<uint64_t>((kb * HB * 128 + sub * 32) >> 4), id_qk, (kb | sub) ? 1u : 0u);
          }
          umma_commit_elect(&sh.s_full[sb]);
        }
        if (ok) umma_commit_elect(&sh.q_empty);          // Q may be replaced once these finish
      } else {
        // O^T += V^T P^T: A = the tile's value blocks (MN-major, 64-dim blocks one slot
        // apart), B = P^T in the rope block (MN-major)
        for (int i = 0; i < I.nt && ok; ++i, ++g) {
          ok = wait(&sh.p_full, g & 1);
          if constexpr (!DENSE && kCpBlocks > 0) fence_proxy_async_smem();   // V blocks written by cp.async
          if (ok && i == 0 && it > 0) ok = wait(&sh.o_free, (it - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = st0 + (g & 1u) * (kKB * kBlkBytes);
          const uint64_t dv = sdesc_sw128(tb, kBlkBytes, 1024);
          const uint64_t dp = sdesc_sw128(tb + (kKB - 1) * kBlkBytes, kBlkBytes, 1024);
          const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int kq = 0; kq < kRows / 16; ++kq)
              umma_bf16_elect(tmem + C::O_COL + b * HB, dv + static_cast<uint64_t>((2 * b * kBlkBytes + kq * 2048) >> 4),
                              dp + static_cast<uint64_t>((kq * 2048) >> 4), id_pv, kq > 0 ? 1u : acc0);
          }
          umma_commit_elect(&sh.empty[g & 1]);    // the tile (whose rope block also held P^T) may be refilled
          umma_commit_elect(&sh.o_done[g & 1]);
        }
      }
      ++it;
    }
    // every MMA this warp issued has completed before TMEM is released
    umma_commit_elect(&sh.mma_done);
    mbar_drain(&sh.mma_done, 0, 200000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 7) tmem_dealloc(tmem, C::TMEM_COLS);
}

// row_nt[t] = number of 64-slot tiles up to the last slot holding an index >= 0.
__global__ void __launch_bounds__(256) row_tiles_kernel(const int32_t* __restrict__ idx, int n_q, int topk,
                                                        int32_t* __restrict__ row_nt) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= n_q) return;
  const int32_t* irow = idx + static_cast<size_t>(t) * topk;
  int last = -1;
  for (int s = lane; s < topk; s += 32)
    if (__ldg(irow + s) >= 0) last = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
  if (lane == 0) row_nt[t] = (last + kRows) / kRows;
}

// Pre-pass of the block-dense walk, one CTA per block of B tokens:
//   block_range[b] = [min, max + 1) of the in-range latent rows the block's tokens select
//                    ((0, 0) when none);
//   block_mask[b]  = for each token, bit o of its MAXR-bit row is set when row min + o is one of
//                    its selections (the layout the attention kernel copies into shared memory).
// Index slots outside [0, n_kv) are counted in the status words (they are skipped).
template <int B, int MAXR>
__global__ void __launch_bounds__(256) block_mask_kernel(const int32_t* __restrict__ idx,
                                                         const int32_t* __restrict__ ks, int n_q, int n_kv,
                                                         int topk, int2* __restrict__ block_range,
                                                         uint32_t* __restrict__ block_mask, uint32_t* status,
                                                         uint32_t* bad_count) {
  constexpr int kRowWords = MAXR / 32;
  constexpr int kWords = B * kRowWords;
  __shared__ long long kst[B];
  __shared__ int red_lo[8], red_hi[8];
  __shared__ alignas(16) uint32_t mask[kWords];
  const int blk = blockIdx.x;
  const int t0 = blk * B;
  const int nt = min(B, n_q - t0);
  for (int i = threadIdx.x; i < nt; i += blockDim.x) kst[i] = __ldg(ks + t0 + i);
  for (int i = threadIdx.x; i < kWords; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  const int32_t* base = idx + static_cast<size_t>(t0) * topk;
  const int total = nt * topk;
  const bool vec = (topk & 3) == 0 && (reinterpret_cast<uintptr_t>(base) & 15) == 0;
  // pass 1: the range (and the bad-index count)
  int lo = 0x7FFFFFFF, hi = -1;
  auto take = [&](int j, int b) {
    const long long row = kst[b] + j;
    if (j >= 0) {
      if (row >= 0 && row < n_kv) {
        lo = min(lo, static_cast<int>(row));
        hi = max(hi, static_cast<int>(row));
      } else {
        atomicOr(status, DEV_ERR_BAD_INDEX);
        atomicAdd(bad_count, 1u);
      }
    }
  };
  if (vec) {
    for (int e = threadIdx.x * 4; e < total; e += blockDim.x * 4) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(base + e));
      const int b = e / topk;        // the four entries belong to one token (topk % 4 == 0)
      take(v.x, b);
      take(v.y, b);
      take(v.z, b);
      take(v.w, b);
    }
  } else {
    for (int e = threadIdx.x; e < total; e += blockDim.x) take(__ldg(base + e), e / topk);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red_lo[w] = lo;
    red_hi[w] = hi;
  }
  __syncthreads();
  lo = red_lo[0];
  hi = red_hi[0];
  for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) {
    lo = min(lo, red_lo[i]);
    hi = max(hi, red_hi[i]);
  }
  if (threadIdx.x == 0) block_range[blk] = hi >= lo ? make_int2(lo, hi + 1) : make_int2(0, 0);
  // pass 2: the bits, relative to lo (hi - lo < n_kv <= MAXR)
  auto mark = [&](int j, int b) {
    const long long row = kst[b] + j;
    if (j >= 0 && row >= 0 && row < n_kv) {
      const int o = static_cast<int>(row) - lo;
      atomicOr(&mask[b * kRowWords + (o >> 5)], 1u << (o & 31));
    }
  };
  if (hi >= lo) {
    if (vec) {
      for (int e = threadIdx.x * 4; e < total; e += blockDim.x * 4) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(base + e));
        const int b = e / topk;
        mark(v.x, b);
        mark(v.y, b);
        mark(v.z, b);
        mark(v.w, b);
      }
    } else {
      for (int e = threadIdx.x; e < total; e += blockDim.x) mark(__ldg(base + e), e / topk);
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(block_mask + static_cast<size_t>(blk) * kWords);
  for (int i = threadIdx.x; i < kWords / 4; i += blockDim.x) dst[i] = reinterpret_cast<const uint4*>(mask)[i];
}

// Merge of the gather walk's splits: per (token, head) row, out = sum_s w_s o_s / sum_s w_s
// with w_s = exp(lse_s - max lse), lse = max + log(sum w_s); a row whose splits are all empty
// gets zeros and -inf.  One warp per row.
__global__ void __launch_bounds__(256) split_combine_kernel(const float* __restrict__ po, const float* __restrict__ plse,
                                                            int n_split, long long n_rows, uint16_t* __restrict__ out,
                                                            float* __restrict__ lse) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  float m = -INFINITY;
  for (int s = 0; s < n_split; ++s) m = fmaxf(m, __ldg(plse + s * n_rows + row));
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float den = 0.f;
  if (m > -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float ls = __ldg(plse + s * n_rows + row);
      const float w = ls > -INFINITY ? __expf(ls - m) : 0.f;
      den += w;
      const float4* src = reinterpret_cast<const float4*>(po + (s * n_rows + row) * kDv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = __ldg(src + lane + 32 * i);
        acc[4 * i] += w * v.x;
        acc[4 * i + 1] += w * v.y;
        acc[4 * i + 2] += w * v.z;
        acc[4 * i + 3] += w * v.w;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(out + row * kDv);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * i] * inv, acc[4 * i + 1] * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
    dst[lane + 32 * i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
  if (lse && lane == 0) lse[row] = den > 0.f ? m + __logf(den) : -INFINITY;
}

template <int HB, int HD, bool PAGED = false>
cudaError_t launch_cfg(const CUtensorMap& tmap, const CUtensorMap& tmap_q, int n_q, int n_kv, int H, int topk,
                       float scale, const void* kv, const int32_t* idx, const int32_t* ks, const PagedRows& pg,
                       const int32_t* row_nt,
                       const int2* block_range, const uint32_t* block_mask, void* out, float* lse, uint32_t* status,
                       cudaStream_t st, const SplitOut& split = SplitOut{1, nullptr, nullptr}) {
  using C = ACfg<HB, HD>;
  auto kern = sparse_attn_kernel<HB, HD, PAGED>;
  cudaError_t e = smem_attr_once<sparse_attn_kernel<HB, HD, PAGED>>(C::DYN_SMEM);
  if (e != cudaSuccess) return e;
  const int n_items = C::DENSE ? (n_q + C::B - 1) / C::B : n_q * ((H + HB - 1) / HB) * split.n;
  const int grid = n_items < device_sm_count() ? n_items : device_sm_count();
  const PipelineDebug dbg = pipeline_debug();
  const int ps = prof_begin(kProfAttn, st);
  kern<<<grid, C::THREADS, C::DYN_SMEM, st>>>(tmap, tmap_q, static_cast<const uint16_t*>(kv), idx, ks, pg, row_nt,
                                            block_range, block_mask,
                                            static_cast<uint16_t*>(out), lse, n_q, n_kv, H, topk,
                                            scale * 1.4426950408889634f, status, status + 1, dbg.wait_ns,
                                            dbg.stop_after_tiles, split);
  e = cudaGetLastError();
  if (e == cudaSuccess && !C::DENSE && split.n > 1) {
    // merge the splits (inside the same launch-log entry: one attention call)
    const long long rows = static_cast<long long>(n_q) * H;
    split_combine_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(split.o, split.lse, split.n, rows,
                                                                               static_cast<uint16_t*>(out), lse);
    e = cudaGetLastError();
  }
  prof_end(ps, st);
  return e;
}


}  // namespace

int sparse_attn_dense_heads(int n_heads, int n_kv, int topk) {
  // block-dense walk pays off when each row of the block's key range is selected by
  // several of the block's tokens; it needs the whole range to fit the selection mask.
  // Returns n_heads: the walk takes all heads of a token (HD == H, which the kernel's output
  // row mapping relies on).
  if (n_heads != 1 && n_heads != 2 && n_heads != 4 && n_heads != 8 && n_heads != 16) return 0;
  const int B = kDenseCols / n_heads;
  const int maxr = (kMaskBytes * 8 / B) / 64 * 64;
  if (n_kv > maxr) return 0;
  if (2LL * B * topk < n_kv) return 0;
  return n_heads;
}

namespace {

// Block-dense scratch: per token block its key range (int2), then (16-byte aligned) its
// selection bitmask of kMaskBytes.
size_t dense_mask_offset(int n_blk) { return (static_cast<size_t>(n_blk) * sizeof(int2) + 15) & ~size_t(15); }

template <int HD>
cudaError_t launch_dense(const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q, int n_q, int n_kv, int n_heads,
                         int topk, float scale, const int32_t* idx, const int32_t* ks, void* out, float* lse,
                         uint32_t* status, void* scratch, cudaStream_t st, bool reuse_prepass) {
  const DenseScratch ds = dense_scratch(scratch, n_q, HD);
  if (!reuse_prepass) {
    const int ps = prof_begin(kProfAttnPrep, st);
    cudaError_t e = launch_block_mask(HD, idx, ks, n_q, n_kv, topk, ds, status, st);
    prof_end(ps, st);
    if (e != cudaSuccess) return e;
  }
  return launch_cfg<kDenseCols, HD>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, nullptr, idx, ks, PagedRows{},
                                    nullptr, ds.block_range, ds.block_mask, out,
                                    lse, status, st);
}

template <int HD>
cudaError_t launch_mask_t(const int32_t* idx, const int32_t* ks, int n_q, int n_kv, int topk, const DenseScratch& ds,
                          uint32_t* status, cudaStream_t st) {
  using C = ACfg<kDenseCols, HD>;
  static_assert(C::B * (C::MAXR / 32) * 4 == kMaskBytes, "one bitmask per block fills the budget exactly");
  const int n_blk = (n_q + C::B - 1) / C::B;
  block_mask_kernel<C::B, C::MAXR><<<n_blk, 256, 0, st>>>(idx, ks, n_q, n_kv, topk, ds.block_range, ds.block_mask,
                                                          status, status + 1);
  return cudaGetLastError();
}

}  // namespace

namespace {
// Gather walk, contiguous or paged cache (separate instantiations).
template <int HB>
cudaError_t launch_gather(const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q, int n_q, int n_kv, int n_heads,
                          int topk, float scale, const void* kv, const int32_t* idx, const int32_t* ks,
                          const PagedRows& pg, const int32_t* row_nt, void* out, float* lse, uint32_t* status,
                          const SplitOut& split, cudaStream_t st) {
  if (pg.block_table)
    return launch_cfg<HB, 0, true>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, kv, idx, ks, pg, row_nt, nullptr,
                                   nullptr, out, lse, status, st, split);
  return launch_cfg<HB, 0, false>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, kv, idx, ks, pg, row_nt, nullptr,
                                  nullptr, out, lse, status, st, split);
}

// Splits of each (token, head block) in the gather walk: when the items leave SMs idle, as many
// as still fit one round of the persistent CTAs (a second round repeats each split's fixed
// costs -- q, the pipeline fill, its fp32 output -- for no gain), each split keeping at least
// four 64-row tiles, at most eight.
int gather_splits(int n_q, int n_heads, int topk) {
  const int hb = n_heads <= 16 ? 16 : n_heads <= 32 ? 32 : 64;
  const long long items = static_cast<long long>(n_q) * ((n_heads + hb - 1) / hb);
  const int sms = device_sm_count();
  if (items <= 0 || 2 * items > sms) return 1;
  int ns = static_cast<int>(sms / items);
  const int tiles = (topk + kRows - 1) / kRows;
  ns = std::min(ns, std::max(1, tiles / 4));
  return std::max(1, std::min(ns, 8));
}

// Gather-walk scratch: row_nt (n_q int32), then for splits the per-split fp32 outputs and
// log-sum-exps.
size_t gather_split_offset(int n_q) { return (static_cast<size_t>(n_q) * sizeof(int32_t) + 15) & ~size_t(15); }
size_t gather_ws_bytes(int n_q, int n_heads, int topk) {
  const int ns = gather_splits(n_q, n_heads, topk);
  size_t b = gather_split_offset(n_q);
  if (ns > 1) b += static_cast<size_t>(ns) * n_q * n_heads * (kDv + 1) * sizeof(float);
  return b;
}
}  // namespace

cudaError_t launch_row_tiles(const int32_t* idx, int n_q, int topk, int32_t* row_nt, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  row_tiles_kernel<<<(n_q + 7) / 8, 256, 0, st>>>(idx, n_q, topk, row_nt);
  return cudaGetLastError();
}

DenseScratch dense_scratch(void* scratch, int n_q, int hd) {
  const int b = kDenseCols / hd;
  const int n_blk = (n_q + b - 1) / b;
  DenseScratch ds;
  ds.block_range = static_cast<int2*>(scratch);
  ds.block_mask = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scratch) + dense_mask_offset(n_blk));
  return ds;
}

cudaError_t launch_block_mask(int hd, const int32_t* idx, const int32_t* ks, int n_q, int n_kv, int topk,
                              const DenseScratch& ds, uint32_t* status, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  switch (hd) {
    case 1: return launch_mask_t<1>(idx, ks, n_q, n_kv, topk, ds, status, st);
    case 2: return launch_mask_t<2>(idx, ks, n_q, n_kv, topk, ds, status, st);
    case 4: return launch_mask_t<4>(idx, ks, n_q, n_kv, topk, ds, status, st);
    case 8: return launch_mask_t<8>(idx, ks, n_q, n_kv, topk, ds, status, st);
    case 16: return launch_mask_t<16>(idx, ks, n_q, n_kv, topk, ds, status, st);
    default: return cudaErrorInvalidValue;
  }
}

size_t sparse_attn_ws_bytes(int n_q, int n_heads, int n_kv, int topk) {
  // the gather walk's needs always (a paged cache takes it whatever the shape), the
  // block-dense walk's when that applies
  size_t b = gather_ws_bytes(n_q, n_heads, topk);
  const int hd = sparse_attn_dense_heads(n_heads, n_kv, topk);
  if (hd) {
    const int n_blk = (n_q + kDenseCols / hd - 1) / (kDenseCols / hd);
    b = std::max(b, dense_mask_offset(n_blk) + static_cast<size_t>(n_blk) * kMaskBytes);
  }
  return b;
}

int sparse_attn_q_box_rows(int n_heads, int n_kv, int topk, bool paged) {
  if (!paged && sparse_attn_dense_heads(n_heads, n_kv, topk)) return kDenseCols;
  return n_heads <= 16 ? 16 : n_heads <= 32 ? 32 : 64;
}

cudaError_t launch_sparse_attn(const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q, int n_q, int n_kv, int n_heads,
                               int topk, float scale, const void* kv, const int32_t* idx, const int32_t* ks,
                               const PagedRows& pg, void* out, float* lse, uint32_t* status, void* scratch,
                               cudaStream_t st, bool reuse_prepass) {
  if (n_q <= 0) return cudaSuccess;
  const int hd = pg.block_table ? 0 : sparse_attn_dense_heads(n_heads, n_kv, topk);   // paged: gather walk
  if (hd) {
    switch (hd) {
      case 1: return launch_dense<1>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, idx, ks, out, lse, status, scratch, st, reuse_prepass);
      case 2: return launch_dense<2>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, idx, ks, out, lse, status, scratch, st, reuse_prepass);
      case 4: return launch_dense<4>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, idx, ks, out, lse, status, scratch, st, reuse_prepass);
      case 8: return launch_dense<8>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, idx, ks, out, lse, status, scratch, st, reuse_prepass);
      default: return launch_dense<16>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, idx, ks, out, lse, status, scratch, st, reuse_prepass);
    }
  }
  int32_t* row_nt = static_cast<int32_t*>(scratch);
  if (!reuse_prepass) {
    const int ps = prof_begin(kProfAttnPrep, st);
    row_tiles_kernel<<<(n_q + 7) / 8, 256, 0, st>>>(idx, n_q, topk, row_nt);
    prof_end(ps, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  SplitOut split{gather_splits(n_q, n_heads, topk), nullptr, nullptr};
  if (split.n > 1) {
    split.o = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + gather_split_offset(n_q));
    split.lse = split.o + static_cast<size_t>(split.n) * n_q * n_heads * kDv;
  }
  switch (sparse_attn_q_box_rows(n_heads, n_kv, topk, pg.block_table != nullptr)) {
    case 16: return launch_gather<16>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, kv, idx, ks, pg, row_nt, out,
                                      lse, status, split, st);
    case 32: return launch_gather<32>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, kv, idx, ks, pg, row_nt, out,
                                      lse, status, split, st);
    default: return launch_gather<64>(tmap_kv, tmap_q, n_q, n_kv, n_heads, topk, scale, kv, idx, ks, pg, row_nt, out,
                                      lse, status, split, st);
  }
}

}  // namespace dsa
