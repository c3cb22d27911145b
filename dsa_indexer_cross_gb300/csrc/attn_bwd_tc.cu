// Backward of the MLA-absorbed sparse attention on tcgen05: the block-dense walk and the gather
// walk (one token's selected rows per item).
//
// The same gradients as the per-token kernel (attn_bwd.cu): for column c = (token, head) and a
// selected latent row j,
//   p = exp(tau q_c . kv_j - lse_c),  dp = d_o_c . kv_j[:512],  ds' = tau p (dp - D_c),
//   dq_c += ds' kv_j,  dkv_j += ds' q_c + p d_o_c (first 512 dims),
// with D_c = d_o_c . o_c from the forward's output.  ("GLM-5/5.1/5.2 DSA + LoRA enablement",
// Megatron-Bridge pull request #15, names a backward for the fused sparse-MLA kernel without
// defining it; this is the exact gradient of the forward.)
//
// Work item = the forward's block-dense item: 64 columns (64 / H consecutive tokens with all
// H heads) and the union of their key ranges, walked in tiles of 64 consecutive latent rows
// (one 72 KB 3-D TMA box) with the per-(token, row) selection bitmask of the pre-pass.  Per
// tile, with the rows on the M side wherever the columns are too few for it:
//   [S^T | dP^T] [64 rows x 128] = Rows . [Q | dO]^T   M = 64, N = 128, K = 512, then
//   S^T += Rows[:, 512:] . Q[:, 512:]^T                 (the rope block, N = 64)
//   softmax warps: P and dS' per (row, col), bf16, into two 8 KB blocks laid out [row][col]
//   dQ^T [576 dims x 64 cols] += Rows^T . dS'^T         M = 128 per dim chunk, K = 64 rows
//   dKV^T piece [128 dims x 64 rows] = Q^T . dS' (+ dO^T . P)   K = 64 cols
// q and d_out sit in shared memory interleaved by 64-dim block, so each block's K-major
// [q; d_out] operand feeds S^T and dP^T in one N = 128 MMA; the same blocks are the MN-major A
// operands of the pieces.  The [row][col] blocks are read as the MN-major B of dQ^T and as the
// K-major B of the pieces (the same bytes).  576 dims are five 128-dim chunks, the last one
// starting at dim 448 (its first 64 lanes repeat chunk 3 and are ignored), so no operand reads
// past its tile.  dQ^T (320 TMEM columns) accumulates over the item and is written once.  The
// five pieces of a tile go to three 64-column TMEM slots: the spare columns and S^T's and
// dP^T's, free from the softmax's read until the next tile's S^T (which waits for the drains of
// the pieces parked there; the tile's last piece takes the spare slot, so that wait ends one
// piece early).  Each piece is drained by eight warps with fp32 reductions into dkv, the item's
// 64 columns summed first.  These products read two operands of 2-6 KB from shared memory per
// 16-deep step, so the tensor core runs near its rate only on the N = 128 S^T | dP^T step; and
// the reductions (147 KB a tile) run close to the L2's reduction throughput.  TMEM: S^T 64 +
// dP^T 64 + dQ^T 320 + spare 64 = 512 columns; shared memory: q 72 KB + d_out 64 KB + tile
// 72 KB + P and dS' 16 KB.
//
// Warp roles (576 threads): warp 0 loads (TMA); warp 1 owns TMEM, takes every wait of the
// products and has its lane 0 issue them; warps 2-7, 16 and 17 drain the pieces and dQ^T (two
// per TMEM lane quarter); warps 8-15 run the softmax (two per lane quarter, 32 columns each).
// Every wait is bounded; a timeout sets the CTA's abort flag and the device status, and every
// role then leaves its loop.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kR = 64;                      // latent rows per tile
constexpr int kC = kDenseCols;              // columns per item
constexpr int kDqk = 576, kDv = 512;
constexpr int kQB = kDqk / 64, kVB = kDv / 64;
constexpr int kBlk = 64 * 128;              // one 64 x 128-byte block
constexpr int kMaskWords = kDenseMaskBytes / 4;
static_assert(kC == 64, "the [row][col] blocks hold 64 columns in one 128-byte row");

constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kColKV = 448, kTmemCols = 512;
// dKV^T piece slots (64 columns each): the spare columns, then S^T's and dP^T's, which are free
// from the softmax's read of a tile until the next tile's S^T
__device__ __forceinline__ uint32_t kv_slot_col(int slot) { return slot == 0 ? kColKV : slot == 1 ? kColS : kColDP; }
// Slot of a tile's piece m: the last piece goes to the spare slot, so the next tile's S^T waits
// only for the drain of the fourth
__device__ __forceinline__ int piece_slot(int m) { return m == 0 || m == 3 ? 1 : m == 1 ? 2 : 0; }

// q and d_out interleaved by 64-dim block: [q block kb | d_out block kb] for kb < 8, then q's
// rope block, so one N = 128 K-major operand per block feeds S^T and dP^T together
constexpr int kOffQD = 0;
constexpr int kOffR = kOffQD + (kQB + kVB) * kBlk;
constexpr int kOffP = kOffR + kQB * kBlk;
constexpr int kOffDS = kOffP + kBlk;
constexpr int kDynSmem = 1024 + kOffDS + kBlk;   // + alignment slack for the 1024-byte swizzle atoms

constexpr int kThreads = 576;
constexpr int kSoftWarps = 8, kDrainWarps = 8;

struct BShared {
  int rows[3][kR];   // gather walk: latent row of each slot of the tile (-1: none), three tiles deep
  uint32_t rows_tag[3];   // the tile whose row list each slot holds (published after the list)
  uint64_t q_full, q_empty, full, empty, s_full, s_empty, p_full;
  uint64_t kv_full[3], kv_empty[3], dq_full, dq_empty, mma_done;
  uint32_t tmem_base, abort_flag;
};
static_assert(kDynSmem + sizeof(BShared) <= 232448, "backward tile set must fit in shared memory");

// byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled block of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// first dim of 128-dim chunk m (the last chunk overlaps the previous one by 64 dims)
__device__ __forceinline__ constexpr int chunk_dim0(int m) { return m < 4 ? 128 * m : 448; }

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// D = d_out . out per (token, head) row, one warp per row (bf16 inputs, fp32 sum).
__global__ void __launch_bounds__(256) attn_bwd_delta_kernel(const uint16_t* __restrict__ out,
                                                             const uint16_t* __restrict__ dout, long long n_rows,
                                                             float* __restrict__ delta) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  const uint4* o4 = reinterpret_cast<const uint4*>(out + row * kDv);
  const uint4* d4 = reinterpret_cast<const uint4*>(dout + row * kDv);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kDv / 8 / 32; ++i) {
    const uint4 a = __ldg(o4 + lane + 32 * i), b = __ldg(d4 + lane + 32 * i);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __bfloat1622float2(a2[k]), y = __bfloat1622float2(b2[k]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

struct BwdArgs {
  const int2* block_range;      // block-dense walk: the items' key ranges and selection bitmasks
  const uint32_t* block_mask;
  const uint16_t* kv;           // gather walk: the latent cache, selections, row starts and
  const int32_t* idx;           // 64-slot tiles per token
  const int32_t* ks;
  const int32_t* row_nt;
  const float* lse;
  const float* delta;           // D = d_out . out per (token, head)
  float* dq;
  float* dkv;
  int n_q, n_kv, H, topk;
  float scale, scale_log2;
  uint32_t* status;             // [0] bits, [1] bad-index count
  unsigned long long wait_ns;
  int stop_after;               // test hook: the load warp stops after this many tiles (< 0: never)
};

// HD > 0: block-dense walk over items of 64 / HD tokens x HD heads (HD == H).  HD == 0: gather
// walk, item = (token, 64-head block), the tile = the token's next 64 selected rows, fetched by
// the load warp with cp.async.
template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_kv, const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_do, const int2* __restrict__ block_range,
                       const uint32_t* __restrict__ block_mask, const uint16_t* __restrict__ kv,
                       const int32_t* __restrict__ idx, const int32_t* __restrict__ ks,
                       const int32_t* __restrict__ row_nt, const float* __restrict__ lse,
                       const float* __restrict__ delta, float* __restrict__ dq, float* __restrict__ dkv, int n_q,
                       int n_kv, int H, int topk, float scale, float scale_log2, uint32_t* status,
                       unsigned long long wait_ns, int stop_after) {
  // (separate __restrict__ parameters: passing them in one struct cost 4% on the block-dense walk)
  constexpr bool GATHER = HD == 0;
  constexpr int B = GATHER ? 1 : kC / (GATHER ? 1 : HD);          // tokens per item
  constexpr int RW = kDenseMaskBytes * 8 / B / 32;                 // mask words per token
  const int n_hb = GATHER ? (H + kC - 1) / kC : 1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQD = smem + kOffQD;
  uint8_t* sR = smem + kOffR;
  uint8_t* sP = smem + kOffP;
  uint8_t* sDS = smem + kOffDS;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = GATHER ? n_q * n_hb : (n_q + B - 1) / B;
  // k-th item of this CTA: causal items grow with their index, so the walk takes them from the
  // last (largest) down, alternating directions across the CTAs each round; the partial last
  // round then holds the smallest items.  Past the end: n_items.
  auto snake_item = [&](int k) {
    const int gdim = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    const int r = k * gdim + ((k & 1) ? (gdim - 1 - b) : b);
    return r < n_items ? n_items - 1 - r : n_items;
  };
  // tiles of an item; block-dense: lo = its first latent row
  auto item_tiles = [&](int item, int& lo) {
    if constexpr (GATHER) {
      lo = 0;
      return __ldg(row_nt + item / n_hb);
    } else {
      const int2 r = __ldg(block_range + item);
      lo = r.x;
      return r.y > r.x ? (r.y - r.x + kR - 1) / kR : 0;
    }
  };
  // the item's first (token, head) row of q / d_out / dq and its number of real columns
  auto item_row0 = [&](int item) -> long long {
    if constexpr (GATHER) return static_cast<long long>(item / n_hb) * H + (item % n_hb) * kC;
    else return static_cast<long long>(item) * kC;
  };
  auto item_cols = [&](int item) -> int {
    if constexpr (GATHER) return min(kC, H - (item % n_hb) * kC);
    else return min(kC, (n_q - item * B) * HD);
  };

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    mbar_init(&sh.full, GATHER ? 1 + 32 : 1);   // gather: + the load warp's cp.async arrivals
    mbar_init(&sh.empty, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.s_empty, kSoftWarps);
    mbar_init(&sh.p_full, kSoftWarps);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      mbar_init(&sh.kv_empty[s], kDrainWarps);
    }
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_empty, kDrainWarps);
    mbar_init(&sh.mma_done, 1);
    for (int i = 0; i < 3 * kR; ++i) sh.rows[i / kR][i % kR] = -1;
    for (int i = 0; i < 3; ++i) sh.rows_tag[i] = 0xFFFFFFFFu;
    sh.abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  // Gather walk: wait (bounded) until the row list of tile g is published; its products are
  // complete by then in every caller, so this only orders the list's shared-memory writes.
  auto wait_rows = [&](uint32_t g) -> bool {
    const volatile uint32_t* tag = &sh.rows_tag[g % 3];
    if (*tag != g) {
      const uint64_t t0 = globaltimer_ns();
      while (*tag != g) {
        if (sh.abort_flag) return false;
        if (globaltimer_ns() - t0 > wait_ns) {
          sh.abort_flag = 1u;
          atomicOr(status, DEV_ERR_TIMEOUT);
          return false;
        }
      }
    }
    __threadfence_block();
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ loads
    // Lane 0 takes every wait and issues the TMA copies (q and d_out; block-dense: the tile);
    // the gather walk's tile rows come through cp.async from all 32 lanes.
    uint32_t g = 0, it = 0;
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && ok; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      int lo;
      const int nt = item_tiles(item, lo);
      if (nt == 0) continue;
      bool w_ok = true;
      if (lane == 0) {
        if (it > 0) w_ok = mbar_wait_for(&sh.q_empty, (it - 1) & 1, &sh.abort_flag, status, wait_ns);
        if (w_ok) {
          // the item's 64 (token, head) rows of q and d_out; rows past the end read as zeros
          const int qrow = static_cast<int>(item_row0(item));
          mbar_arrive_expect_tx(&sh.q_full, (kQB + kVB) * kBlk);
#pragma unroll 1
          for (int kb = 0; kb < kQB; ++kb) tma_load_2d(sQD + 2 * kb * kBlk, &tmap_q, &sh.q_full, kb * 64, qrow);
#pragma unroll 1
          for (int kb = 0; kb < kVB; ++kb)
            tma_load_2d(sQD + (2 * kb + 1) * kBlk, &tmap_do, &sh.q_full, kb * 64, qrow);
        }
      }
      ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!ok) break;
      if constexpr (GATHER) {
        // lane l copies 16-byte chunk l % 8 of slots l / 8 + 4 m (m < 16) in all nine blocks;
        // a slot without a selection (-1, or past topk) reads zeros and is masked
        const int t = item / n_hb;
        const int32_t* irow = idx + static_cast<size_t>(t) * topk;
        const long long kst = __ldg(ks + t);
        const int ch = lane & 7;
        for (int i = 0; i < nt; ++i, ++g) {
          int crow[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const int slot = i * kR + (lane >> 3) + 4 * m;
            const int j = slot < topk ? __ldg(irow + slot) : -1;
            const long long row = kst + j;
            const bool v = j >= 0 && row >= 0 && row < n_kv;
            if (j >= 0 && !v && ch == 0) {
              atomicOr(status, DEV_ERR_BAD_INDEX);
              atomicAdd(status + 1, 1u);
            }
            crow[m] = v ? static_cast<int>(row) : -1;
          }
          // test hook: stop feeding the pipeline; the waits behind it run out
          if (stop_after >= 0 && g >= static_cast<uint32_t>(stop_after)) w_ok = false;
          if (lane == 0 && g > 0 && w_ok)
            w_ok = mbar_wait_for(&sh.empty, (g - 1) & 1, &sh.abort_flag, status, wait_ns);
          ok = __shfl_sync(0xffffffffu, w_ok, 0);
          if (!ok) break;
          // the tile's row list (three tiles deep: the drains of tile g - 3 finished before the
          // products of tile g - 1, which released this slot)
          if (ch == 0) {
#pragma unroll
            for (int m = 0; m < 16; ++m) sh.rows[g % 3][(lane >> 3) + 4 * m] = crow[m];
          }
          __syncwarp();
          if (lane == 0) {
            __threadfence_block();
            *reinterpret_cast<volatile uint32_t*>(&sh.rows_tag[g % 3]) = g;
            mbar_arrive(&sh.full);
          }
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const int r = (lane >> 3) + 4 * m;
            const uint16_t* rowp = kv + static_cast<size_t>(crow[m] >= 0 ? crow[m] : 0) * kDqk + ch * 8;
#pragma unroll
            for (int b = 0; b < kQB; ++b)
              cp_async_16_zfill(smem_u32(sR + b * kBlk + sw128(r, ch)), rowp + b * 64, crow[m] >= 0);
          }
          cp_async_mbar_arrive(&sh.full);
        }
      } else {
        if (lane == 0) {
          for (int i = 0; i < nt; ++i, ++g) {
            if (stop_after >= 0 && g >= static_cast<uint32_t>(stop_after)) {
              w_ok = false;   // test hook: stop feeding the pipeline; the waits behind it run out
              break;
            }
            if (g > 0 && !(w_ok = mbar_wait_for(&sh.empty, (g - 1) & 1, &sh.abort_flag, status, wait_ns))) break;
            mbar_arrive_expect_tx(&sh.full, kQB * kBlk);
            tma_load_3d(sR, &tmap_kv, &sh.full, 0, lo + i * kR, 0);
          }
        }
        g = __shfl_sync(0xffffffffu, g, 0);
        ok = __shfl_sync(0xffffffffu, w_ok, 0);
      }
      ++it;
    }
    // copies in flight land before the CTA's shared memory is released
    if constexpr (GATHER) cp_async_wait<0>();
    if (lane == 0) {
      if (it > 0) mbar_drain(&sh.q_full, (it - 1) & 1, 200000000ull);
      if (g > 0) mbar_drain(&sh.full, (g - 1) & 1, 200000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp takes every wait; lane 0 alone issues the MMAs and their commits (the
    // descriptors are bases plus compile-time offsets, so issuing costs little more than the
    // instruction itself).
    constexpr uint32_t id_sd = idesc_bf16_f32(64, 2 * kC, 0, 0);   // S^T and dP^T together
    constexpr uint32_t id_s = idesc_bf16_f32(64, kC, 0, 0);        // S^T alone (rope block)
    constexpr uint32_t id_dq = idesc_bf16_f32(128, kC, 1, 1);
    constexpr uint32_t id_kv = idesc_bf16_f32(128, kR, 1, 0);
    const uint64_t dR_k = sdesc_sw128(smem_u32(sR), 16, 1024);             // rows, K-major (A of S^T, dP^T)
    const uint64_t dQD_k = sdesc_sw128(smem_u32(sQD), 16, 1024);           // [q; d_out], K-major (B)
    const uint64_t dR_mn = sdesc_sw128(smem_u32(sR), kBlk, 1024);          // rows^T, MN-major (A of dQ^T)
    const uint64_t dDS_mn = sdesc_sw128(smem_u32(sDS), kBlk, 1024);        // dS'^T, MN-major (B of dQ^T)
    const uint64_t dQ_mn = sdesc_sw128(smem_u32(sQD), 2 * kBlk, 1024);     // q^T, MN-major (A of dKV^T)
    const uint64_t dO_mn = sdesc_sw128(smem_u32(sQD + kBlk), 2 * kBlk, 1024);   // d_out^T (A of dKV^T)
    const uint64_t dDS_k = sdesc_sw128(smem_u32(sDS), 16, 1024);           // dS', K-major (B of dKV^T)
    const uint64_t dP_k = sdesc_sw128(smem_u32(sP), 16, 1024);             // P, K-major (B of dKV^T)
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_for(bar, parity, &sh.abort_flag, status, wait_ns));
    };
    uint32_t g = 0, it = 0;
    uint32_t su[3] = {0u, 0u, 0u};   // uses of each piece slot so far
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && ok; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      int lo;
      const int nt = item_tiles(item, lo);
      if (nt == 0) continue;
      if (!(ok = wait(&sh.q_full, it & 1))) break;
      for (int i = 0; i < nt && ok; ++i, ++g) {
        if (!(ok = wait(&sh.full, g & 1))) break;
        if constexpr (GATHER) fence_proxy_async_smem();   // the tile was written by cp.async
        if (g > 0 && !(ok = wait(&sh.s_empty, (g - 1) & 1))) break;
        // S^T and dP^T's columns held pieces of the previous tile: wait for their drains
        if (su[1] > 0 && !(ok = wait(&sh.kv_empty[1], (su[1] - 1) & 1))) break;
        if (su[2] > 0 && !(ok = wait(&sh.kv_empty[2], (su[2] - 1) & 1))) break;
        tc_fence_after();
        if (lane == 0) {
          // S^T | dP^T = Rows [q | d_out]^T over the eight value blocks, then S^T += the rope block
#pragma unroll
          for (int kb = 0; kb < kVB; ++kb) {
#pragma unroll
            for (int sub = 0; sub < 4; ++sub)
              umma_bf16(tmem + kColS, dR_k + static_cast<uint64_t>((kb * kBlk + sub * 32) >> 4),
                        dQD_k + static_cast<uint64_t>((2 * kb * kBlk + sub * 32) >> 4), id_sd, (kb | sub) ? 1u : 0u);
          }
#pragma unroll
          for (int sub = 0; sub < 4; ++sub)
            umma_bf16(tmem + kColS, dR_k + static_cast<uint64_t>((kVB * kBlk + sub * 32) >> 4),
                      dQD_k + static_cast<uint64_t>((2 * kVB * kBlk + sub * 32) >> 4), id_s, 1u);
          umma_commit(&sh.s_full);
        }
        __syncwarp();
        if (!(ok = wait(&sh.p_full, g & 1))) break;
        if (i == 0 && it > 0 && !(ok = wait(&sh.dq_empty, (it - 1) & 1))) break;
        tc_fence_after();
        if (lane == 0) {
          // dQ^T += Rows^T dS'^T, five 128-dim chunks, K = the tile's 64 rows
#pragma unroll
          for (int m = 0; m < 5; ++m) {
#pragma unroll
            for (int kq = 0; kq < kR / 16; ++kq)
              umma_bf16(tmem + kColDQ + m * kC,
                        dR_mn + static_cast<uint64_t>(((chunk_dim0(m) / 64) * kBlk + kq * 2048) >> 4),
                        dDS_mn + static_cast<uint64_t>((kq * 2048) >> 4), id_dq, (i > 0 || kq > 0) ? 1u : 0u);
          }
          umma_commit(&sh.empty);                  // the tile may be refilled
          if (i == nt - 1) umma_commit(&sh.dq_full);
        }
        __syncwarp();
        // dKV^T pieces: dims chunk m x the tile's 64 rows, K = the item's 64 columns
#pragma unroll
        for (int m = 0; m < 5 && ok; ++m) {
          const int slot = piece_slot(m);
          if (su[slot] > 0 && !(ok = wait(&sh.kv_empty[slot], (su[slot] - 1) & 1))) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t d_kv = tmem + kv_slot_col(slot);
            const uint32_t a_off = static_cast<uint32_t>((chunk_dim0(m) / 64) * 2 * kBlk);
#pragma unroll
            for (int kq = 0; kq < kC / 16; ++kq)
              umma_bf16(d_kv, dQ_mn + static_cast<uint64_t>((a_off + kq * 2048) >> 4),
                        dDS_k + static_cast<uint64_t>((kq * 32) >> 4), id_kv, kq > 0 ? 1u : 0u);
            if (m < 4) {
#pragma unroll
              for (int kq = 0; kq < kC / 16; ++kq)
                umma_bf16(d_kv, dO_mn + static_cast<uint64_t>((a_off + kq * 2048) >> 4),
                          dP_k + static_cast<uint64_t>((kq * 32) >> 4), id_kv, 1u);
            }
            umma_commit(&sh.kv_full[slot]);
          }
          __syncwarp();
          ++su[slot];
        }
      }
      if (ok && lane == 0) umma_commit(&sh.q_empty);   // q and d_out may be replaced once these finish
      __syncwarp();
      ++it;
    }
    // every MMA issued here has completed before TMEM is released
    if (lane == 0) umma_commit(&sh.mma_done);
    __syncwarp();
    mbar_drain(&sh.mma_done, 0, 200000000ull);
  } else if ((warp >= 2 && warp < 8) || warp >= 16) {
    // ------------------------------------------------------------------ drains: dKV^T pieces, dQ^T
    // two warps per TMEM lane quarter: set 0 (warps 4-7) takes the first half of every piece's
    // rows and of dQ^T's columns, set 1 (warps 2, 3, 16, 17) the second half
    const int qd = warp & 3;
    const int set = (warp >= 4 && warp < 8) ? 0 : 1;
    const int drain_id = set * 4 + qd;
    const uint32_t t_lane = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t g = 0, it = 0;
    uint32_t su[3] = {0u, 0u, 0u};   // uses of each piece slot so far
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && ok; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      int lo;
      const int nt = item_tiles(item, lo);
      const int n_cols = item_cols(item);   // columns of real (token, head) rows
      float* dq_item = dq + static_cast<size_t>(item_row0(item)) * kDqk;
      if (nt == 0) {
        // nothing selected: zero gradients for the item's rows of dq
        for (int e = drain_id * 32 + lane; e < n_cols * kDqk; e += kDrainWarps * 32) dq_item[e] = 0.f;
        continue;
      }
      for (int i = 0; i < nt && ok; ++i, ++g) {
        // rows of the tile some column selects (the others add nothing to dkv); gather: read
        // from the tile's row list once its first piece is complete (below)
        uint32_t any_lo = 0u, any_hi = 0u;
        int my_row = -1;
        if constexpr (!GATHER) {
          for (int b = lane; b < B; b += 32) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(block_mask + static_cast<size_t>(item) * kMaskWords +
                                                                 b * RW + 2 * i));
            any_lo |= w.x;
            any_hi |= w.y;
          }
          any_lo = __reduce_or_sync(0xffffffffu, any_lo);
          any_hi = __reduce_or_sync(0xffffffffu, any_hi);
        }
        const long long row0 = static_cast<long long>(lo) + static_cast<long long>(i) * kR;
#pragma unroll
        for (int m = 0; m < 5; ++m) {
          const int slot = piece_slot(m);
          ok = __all_sync(0xffffffffu,
                          mbar_wait_for(&sh.kv_full[slot], su[slot] & 1, &sh.abort_flag, status, wait_ns));
          if (!ok) break;
          ++su[slot];
          tc_fence_after();
          if constexpr (GATHER) {
            if (m == 0) {
              // this warp's 32 slots of the tile, lane j holding slot 32 set + j
              ok = __all_sync(0xffffffffu, wait_rows(g));
              if (!ok) break;
              my_row = sh.rows[g % 3][32 * set + lane];
              const uint32_t bits = __ballot_sync(0xffffffffu, my_row >= 0);
              any_lo = set ? 0u : bits;
              any_hi = set ? bits : 0u;
            }
          }
          const bool mine = m < 4 || qd >= 2;     // chunk 4's first 64 lanes repeat chunk 3
          uint32_t v[32];
          if (mine) {
            tmem_ld32(tmem + t_lane + kv_slot_col(slot) + set * 32, v);
            tmem_ld_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.kv_empty[slot]);
          if (mine) {
            const uint32_t any = set ? any_hi : any_lo;
            if constexpr (GATHER) {
              float* col = dkv + chunk_dim0(m) + 32 * qd + lane;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int row = __shfl_sync(0xffffffffu, my_row, j);
                if ((any >> j) & 1u) red_add_f32(col + static_cast<size_t>(row) * kDqk, __uint_as_float(v[j]));
              }
            } else {
              float* col = dkv + (row0 + 32 * set) * kDqk + chunk_dim0(m) + 32 * qd + lane;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if ((any >> j) & 1u) red_add_f32(col + static_cast<size_t>(j) * kDqk, __uint_as_float(v[j]));
            }
          }
        }
      }
      if (!ok) break;
      // the item's dQ^T, written once: lane = dim, TMEM column = (token, head) column
      ok = __all_sync(0xffffffffu, mbar_wait_for(&sh.dq_full, it & 1, &sh.abort_flag, status, wait_ns));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int m = 0; m < 5; ++m) {
        if (m == 4 && qd < 2) continue;
        const int d = chunk_dim0(m) + 32 * qd + lane;
        uint32_t v[32];
        tmem_ld32(tmem + t_lane + kColDQ + m * kC + set * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = set * 32 + j;
          if (c < n_cols) dq_item[static_cast<size_t>(c) * kDqk + d] = __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.dq_empty);
      ++it;
    }
  } else if (warp >= 8 && warp < 16) {
    // ------------------------------------------------------------------ softmax: P and dS'
    const int qd = warp & 3;                  // TMEM lane quarter
    const int c_off = warp >= 12 ? 32 : 0;    // this warp's 32 columns
    const int r0 = qd * 16 + (lane >> 2);     // S^T rows held: r0 and r0 + 8
    const int cq = 2 * (lane & 3);            // column pair within each group of 8
    const uint32_t t_lane = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t p_base = smem_u32(sP), ds_base = smem_u32(sDS);
    uint32_t g = 0;
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items && ok; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      int lo;
      const int nt = item_tiles(item, lo);
      if (nt == 0) continue;
      // this thread's eight columns: c = c_off + 8 kk + cq + e
      float l2[8], dd[8];
      const int n_cols = item_cols(item);
      const long long qrow0 = item_row0(item);
      uint32_t col_ok = 0u;   // gather: columns of real heads (the others belong to other tokens)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = c_off + 8 * kk + cq + e;
          const bool real = c < n_cols;
          const size_t row = static_cast<size_t>(qrow0 + c);
          l2[2 * kk + e] = real ? __ldg(lse + row) * 1.4426950408889634f : 0.f;
          dd[2 * kk + e] = real ? __ldg(delta + row) : 0.f;
          col_ok |= (real ? 1u : 0u) << (2 * kk + e);
        }
      }
      const uint32_t* mrow = GATHER ? nullptr : block_mask + static_cast<size_t>(item) * kMaskWords;
      for (int i = 0; i < nt; ++i, ++g) {
        // selection bits of rows r0 and r0 + 8 for each column's token (e = 0, 1 share a token
        // unless there is one head); gather: all columns share the token
        uint2 mw[4][2];
        if constexpr (!GATHER) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              if (e == 0 || HD == 1) {
                const int b = (c_off + 8 * kk + cq + e) / (GATHER ? 1 : HD);
                mw[kk][e] = __ldg(reinterpret_cast<const uint2*>(mrow + b * RW + 2 * i));
              } else {
                mw[kk][e] = mw[kk][0];
              }
            }
          }
        }
        ok = __all_sync(0xffffffffu, mbar_wait_for(&sh.s_full, g & 1, &sh.abort_flag, status, wait_ns));
        if (!ok) break;
        tc_fence_after();
        bool rsel[2] = {false, false};   // gather: slots r0 and r0 + 8 hold a selection
        if constexpr (GATHER) {
          ok = __all_sync(0xffffffffu, wait_rows(g));
          if (!ok) break;
          rsel[0] = sh.rows[g % 3][r0] >= 0;
          rsel[1] = sh.rows[g % 3][r0 + 8] >= 0;
        }
        uint32_t vs[16], vd[16];
        tmem_ld_16x256b<4>(tmem + t_lane + kColS + c_off, vs);
        tmem_ld_16x256b<4>(tmem + t_lane + kColDP + c_off, vd);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.s_empty);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int chunk = c_off / 8 + kk;   // 16-byte chunk of the 128-byte [row] line
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = r0 + 8 * hh;
            float p[2], ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              bool sel;
              if constexpr (GATHER) {
                sel = rsel[hh] && ((col_ok >> (2 * kk + e)) & 1u);
              } else {
                const uint2 w = mw[kk][e];
                sel = (((r < 32 ? w.x : w.y) >> (r & 31)) & 1u) != 0u;
              }
              const float s = __uint_as_float(vs[4 * kk + 2 * hh + e]);
              const float dp = __uint_as_float(vd[4 * kk + 2 * hh + e]);
              p[e] = sel ? ex2_approx(s * scale_log2 - l2[2 * kk + e]) : 0.f;
              ds[e] = sel ? scale * p[e] * (dp - dd[2 * kk + e]) : 0.f;
            }
            const uint32_t off = static_cast<uint32_t>(r * 128 + ((chunk ^ (r & 7)) << 4) + cq * 2);
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p[0], p[1]);
            const __nv_bfloat162 db = __floats2bfloat162_rn(ds[0], ds[1]);
            st_shared_u32(p_base + off, *reinterpret_cast<const uint32_t*>(&pb));
            st_shared_u32(ds_base + off, *reinterpret_cast<const uint32_t*>(&db));
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_full);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q, const CUtensorMap& tmap_do,
                      const BwdArgs& A, cudaStream_t st) {
  cudaError_t e = smem_attr_once<attn_bwd_tc_kernel<HD>>(kDynSmem);
  if (e != cudaSuccess) return e;
  const int n_items = HD == 0 ? A.n_q * ((A.H + kC - 1) / kC) : (A.n_q + kC / (HD ? HD : 1) - 1) / (kC / (HD ? HD : 1));
  const int grid = n_items < device_sm_count() ? n_items : device_sm_count();
  attn_bwd_tc_kernel<HD><<<grid, kThreads, kDynSmem, st>>>(
      tmap_kv, tmap_q, tmap_do, A.block_range, A.block_mask, A.kv, A.idx, A.ks, A.row_nt, A.lse, A.delta, A.dq, A.dkv,
      A.n_q, A.n_kv, A.H, A.topk, A.scale, A.scale_log2, A.status, A.wait_ns, A.stop_after);
  return cudaGetLastError();
}

BwdArgs bwd_args(int n_q, int n_kv, int H, int topk, float scale, const float* lse, const float* delta, float* dq,
                 float* dkv, uint32_t* status) {
  BwdArgs A{};
  A.lse = lse;
  A.delta = delta;
  A.dq = dq;
  A.dkv = dkv;
  A.n_q = n_q;
  A.n_kv = n_kv;
  A.H = H;
  A.topk = topk;
  A.scale = scale;
  A.scale_log2 = scale * 1.4426950408889634f;
  A.status = status;
  const PipelineDebug dbg = pipeline_debug();
  A.wait_ns = dbg.wait_ns;
  A.stop_after = dbg.stop_after_tiles;
  return A;
}

cudaError_t launch_delta(const void* out, const void* dout, long long n_rows, float* delta, cudaStream_t st) {
  attn_bwd_delta_kernel<<<static_cast<unsigned>((n_rows + 7) / 8), 256, 0, st>>>(
      static_cast<const uint16_t*>(out), static_cast<const uint16_t*>(dout), n_rows, delta);
  return cudaGetLastError();
}

}  // namespace

size_t sparse_attn_bwd_dense_delta_bytes(int n_q, int n_heads) {
  return static_cast<size_t>(n_q) * static_cast<size_t>(n_heads) * sizeof(float);
}

cudaError_t launch_sparse_attn_bwd_dense(int hd, const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q,
                                         const CUtensorMap& tmap_do, int n_q, int n_kv, int topk, float scale,
                                         const int32_t* idx, const int32_t* ks, const void* out, const float* lse,
                                         const void* dout, float* dq, float* dkv, uint32_t* status, float* delta,
                                         void* scratch, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  const DenseScratch ds = dense_scratch(scratch, n_q, hd);
  int ps = prof_begin(kProfAttnPrep, st);
  cudaError_t e = launch_delta(out, dout, static_cast<long long>(n_q) * hd, delta, st);
  if (e == cudaSuccess) e = launch_block_mask(hd, idx, ks, n_q, n_kv, topk, ds, status, st);
  prof_end(ps, st);
  if (e != cudaSuccess) return e;
  BwdArgs A = bwd_args(n_q, n_kv, hd, topk, scale, lse, delta, dq, dkv, status);
  A.block_range = ds.block_range;
  A.block_mask = ds.block_mask;
  ps = prof_begin(kProfAttnBwd, st);
  switch (hd) {
    case 1: e = launch_hd<1>(tmap_kv, tmap_q, tmap_do, A, st); break;
    case 2: e = launch_hd<2>(tmap_kv, tmap_q, tmap_do, A, st); break;
    case 4: e = launch_hd<4>(tmap_kv, tmap_q, tmap_do, A, st); break;
    case 8: e = launch_hd<8>(tmap_kv, tmap_q, tmap_do, A, st); break;
    case 16: e = launch_hd<16>(tmap_kv, tmap_q, tmap_do, A, st); break;
    default: e = cudaErrorInvalidValue;
  }
  prof_end(ps, st);
  return e;
}

cudaError_t launch_sparse_attn_bwd_gather(const CUtensorMap& tmap_q, const CUtensorMap& tmap_do, int n_q, int n_kv,
                                          int n_heads, int topk, float scale, const void* kv, const int32_t* idx,
                                          const int32_t* ks, const void* out, const float* lse, const void* dout,
                                          float* dq, float* dkv, uint32_t* status, float* delta, int32_t* row_nt,
                                          cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  int ps = prof_begin(kProfAttnPrep, st);
  cudaError_t e = launch_delta(out, dout, static_cast<long long>(n_q) * n_heads, delta, st);
  if (e == cudaSuccess) e = launch_row_tiles(idx, n_q, topk, row_nt, st);
  prof_end(ps, st);
  if (e != cudaSuccess) return e;
  BwdArgs A = bwd_args(n_q, n_kv, n_heads, topk, scale, lse, delta, dq, dkv, status);
  A.kv = static_cast<const uint16_t*>(kv);
  A.idx = idx;
  A.ks = ks;
  A.row_nt = row_nt;
  ps = prof_begin(kProfAttnBwd, st);
  e = launch_hd<0>(tmap_q, tmap_q, tmap_do, A, st);   // the gather walk reads no tile map of kv
  prof_end(ps, st);
  return e;
}

}  // namespace dsa
