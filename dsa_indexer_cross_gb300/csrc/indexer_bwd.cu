// Lightning-indexer backward on tcgen05: gradients of the selected scores.
//
// For query t, selected slot n (key row j = ks_t + idx[t, n]) and upstream g = d_score[t, n]:
//     x[h]   = q~[t, h] . k~[j]
//     dw[t, h]      += g max(0, x[h])
//     dq~[t, h, :]  += g w[t, h] [x[h] > 0] k~[j, :]
//     dk~[j, :]     += sum_h g w[t, h] [x[h] > 0] q~[t, h, :]
// then dq = R(q_pos)^T dq~ and dk = R(k_pos)^T dk~ through the index RoPE (a separate pass).
// ("GLM-5/5.1/5.2 DSA + LoRA enablement": the commit vendoring the fused lighting_indexer
// "with fwd/bwd" names this backward; it is the derivative of the score of "GLM-5.2
// IndexShare", section 1.)
//
// A CTA takes one query at a time (persistent, queries strided over the grid) and walks its
// selected keys in tiles of 128.  With G[j, h] = g_j w[h] [x[j, h] > 0] (bf16) three products
// per tile run on the tensor core, all from tiles that are already in shared memory:
//     X[j, h]   = K[j, :] . Q[h, :]      M = 128 keys, N = 64 heads, K = d    (A, B K-major)
//     dK[j, :]  = G[j, :] . Q[:, :]      M = 128 keys, N = d, K = 64 heads     (A K-major, B MN-major)
//       or its transpose dK^T = Q^T G^T  M = d, N = 128 keys                     (A MN-major, B K-major)
//     dQ^T[:, h] += K[:, :]^T . G[:, h]  M = d, N = 64 heads, K = 128 keys     (A, B MN-major)
// Heads are padded to 64 with zero rows of Q and zero weights (so G is one 128-byte row per
// key).  X and dK are double-buffered in TMEM, dQ^T accumulates over the query's tiles (two
// buffers, one per query parity).  The epilogue reads X, keeps the per-head dw sums in
// registers, writes G into shared memory in the 128-byte-swizzled layout, and adds dK into dk~
// with fp32 reductions, in one of two forms chosen per call (template parameter TR, below).
// Rows selected by several queries receive several adds: the order, and the last bits of dk,
// vary between runs.  dq~ is written once per query.
//
// Warp roles (256 threads): warps 0-1 gather Q, w and the selected key rows with cp.async
// (zero-filled where a slot is empty); warp 2 issues X; warp 3 owns TMEM and issues dK and
// dQ^T; warps 4-7 run the epilogue, one TMEM lane quarter each.  Every wait is bounded.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kBKeys = 128;                 // selected keys per tile
constexpr int kHP = 64;                     // heads padded to one 128-byte bf16 row
constexpr int kBD = 128;                    // index head dim
constexpr int kStagesB = 3;                 // key tiles in flight
constexpr int kQBytes = kHP * kBD * 2;      // 16 KB: two 64-dim blocks of [64 heads][128 B]
constexpr int kKBytes = kBKeys * kBD * 2;   // 32 KB: two 64-dim blocks of [128 keys][128 B]
constexpr int kGBytes = kBKeys * kHP * 2;   // 16 KB: [128 keys][64 heads]
constexpr int kBwdThreads = 256;
constexpr int kProdThreads = 64;
constexpr uint32_t kXCol = 0, kDkCol = 128, kDqCol = 384;   // TMEM: X 2x64, dK 2x128, dQ^T 2x64
constexpr int kBwdDynSmem = 1024 + 2 * kQBytes + kStagesB * kKBytes + 2 * kGBytes;

struct BwdShared {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kStagesB], k_empty[kStagesB];
  uint64_t x_full[2], x_empty[2], g_full[2], g_empty[2], dk_full[2], dk_empty[2], dq_full[2], dq_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort_flag;
  alignas(16) float w[2][kHP];   // head weights of the query in each Q slot (0 past n_heads)
  int32_t idx[2][2048];           // the query's selected offsets, per Q slot
  float ds[2][2048];              // and their upstream gradients
};

struct BwdArgs {
  const uint16_t* q_rot;   // rotated q (64-dim blocks from q_split on), [n_q][H][128]
  const uint16_t* q_in;    // unrotated q (blocks before q_split)
  const uint16_t* k_rot;
  const uint16_t* k_in;
  int q_split, k_split;
  const float* w;          // [n_q][H]
  const int32_t* ks;
  const int32_t* ke;
  const int32_t* idx;      // [n_q][topk]
  const float* d_score;    // [n_q][topk]
  float* dq;               // [n_q][H][128]: dq~ (written)
  float* dk;               // [n_kv][128]: dk~ (accumulated)
  float* dw;               // [n_q][H] (accumulated, zeroed before)
  int n_q, n_kv, n_heads, topk;
  uint32_t* status;
  unsigned long long wait_ns;
};

__device__ __forceinline__ uint32_t sw128b(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Selected slots of query t: min(topk, ke_t - ks_t); none for an empty range or one outside
// [0, n_kv) (the producer flags those).
__device__ __forceinline__ bool range_ok(const int32_t* ks, const int32_t* ke, int n_kv, int t) {
  const int a = __ldg(ks + t), b = __ldg(ke + t);
  return a >= 0 && b <= n_kv && a <= b;
}
__device__ __forceinline__ int row_slots(const int32_t* ks, const int32_t* ke, int n_kv, int topk, int t) {
  if (!range_ok(ks, ke, n_kv, t)) return 0;
  const int len = __ldg(ke + t) - __ldg(ks + t);
  return len <= 0 ? 0 : min(topk, len);
}

__device__ __forceinline__ bool warp_all_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              uint32_t* status, unsigned long long limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait_for(bar, parity, abort_flag, status, limit_ns));
}

// TR: dK computed transposed (dK^T, a TMEM lane per dim) and added with 128-byte scalar
// reductions per key row; else dK (a TMEM lane per key) added with 16-byte reductions, one
// key row per thread.  The first wins when few queries share a key row (long caches), the
// second when many do (a short causal prefix, whose rows every query reduces into at once).
template <bool TR>
__global__ void __launch_bounds__(kBwdThreads, 1)
    indexer_bwd_kernel(const uint16_t* __restrict__ q_rot, const uint16_t* __restrict__ q_in,
                       const uint16_t* __restrict__ k_rot, const uint16_t* __restrict__ k_in, int q_split,
                       int k_split, const float* __restrict__ w, const int32_t* __restrict__ ks,
                       const int32_t* __restrict__ ke, const int32_t* __restrict__ idx,
                       const float* __restrict__ d_score, float* __restrict__ dq, float* __restrict__ dk,
                       float* __restrict__ dw, int n_q, int n_kv, int n_heads, int topk, uint32_t* status,
                       unsigned long long wait_ns) {
  // (separate __restrict__ parameters rather than one struct of them)
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // 2 slots
  uint8_t* sK = sQ + 2 * kQBytes;                       // kStagesB slots
  uint8_t* sG = sK + kStagesB * kKBytes;                // 2 slots
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.q_full[b], kProdThreads);
      mbar_init(&sh.q_empty[b], 2);   // both MMA warps read Q
      mbar_init(&sh.x_full[b], 1);
      mbar_init(&sh.x_empty[b], 4);
      mbar_init(&sh.g_full[b], 4);
      mbar_init(&sh.g_empty[b], 1);
      mbar_init(&sh.dk_full[b], 1);
      mbar_init(&sh.dk_empty[b], 4);
      mbar_init(&sh.dq_full[b], 1);
      mbar_init(&sh.dq_empty[b], 4);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&sh.k_full[s], kProdThreads);
      mbar_init(&sh.k_empty[s], 2);   // X (warp 2) and dQ^T (warp 3) read the K tile
    }
    mbar_init(&sh.mma_done, 2);
    sh.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 3) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp < 2) {
    // ------------------------------------------------------------------ producers (cp.async)
    const int tid = threadIdx.x;   // 0 .. 63
    uint32_t T = 0, qc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_q && ok; t += gridDim.x) {
      if (tid == 0 && !range_ok(ks, ke, n_kv, t)) atomicOr(status, DEV_ERR_RANGE);
      const int kt = row_slots(ks, ke, n_kv, topk, t);
      if (kt == 0) continue;
      const int nt = (kt + kBKeys - 1) / kBKeys;
      const int qs = qc & 1;
      if (qc >= 2 && !(ok = mbar_wait_for(&sh.q_empty[qs], ((qc >> 1) - 1) & 1, &sh.abort_flag, status, wait_ns)))
        break;
      // Q rows (heads past n_heads land as zeros) and the head weights
      uint8_t* q_dst = sQ + qs * kQBytes;
      for (int c = tid; c < kHP * 16; c += kProdThreads) {
        const int h = c >> 4, ch = c & 15, blk = ch >> 3;
        const bool valid = h < n_heads;
        const uint16_t* src = (blk < q_split ? q_in : q_rot) +
                              (static_cast<size_t>(t) * n_heads + (valid ? h : 0)) * kBD + ch * 8;
        cp_async_16_zfill(smem_u32(q_dst + blk * (kQBytes / 2) + sw128b(h, ch & 7)), src, valid);
      }
      if (tid < kHP / 4) {
        const bool valid = tid * 4 < n_heads;
        cp_async_16_zfill(smem_u32(&sh.w[qs][tid * 4]), w + static_cast<size_t>(t) * n_heads + (valid ? tid * 4 : 0),
                          valid);
      }
      // the query's selected offsets and upstream gradients, staged once (both roles read them
      // per tile; from global memory each read was a full memory latency)
      for (int n = tid; n < kt; n += kProdThreads) {
        cp_async_4(smem_u32(&sh.idx[qs][n]), idx + static_cast<size_t>(t) * topk + n);
        cp_async_4(smem_u32(&sh.ds[qs][n]), d_score + static_cast<size_t>(t) * topk + n);
      }
      cp_async_mbar_arrive(&sh.q_full[qs]);
      const int len = __ldg(ke + t) - __ldg(ks + t);
      const int ks_t = __ldg(ks + t);
      // the offsets staged by all producer threads have landed
      if (!(ok = mbar_wait_for(&sh.q_full[qs], (qc >> 1) & 1, &sh.abort_flag, status, wait_ns))) break;
      for (int i = 0; i < nt && ok; ++i, ++T) {
        const int s = T % kStagesB;
        if (T >= kStagesB &&
            !(ok = mbar_wait_for(&sh.k_empty[s], ((T / kStagesB) - 1) & 1, &sh.abort_flag, status, wait_ns)))
          break;
        uint8_t* k_dst = sK + s * kKBytes;
        const int ch = tid & 15, blk = ch >> 3;
        const uint16_t* kb = blk < k_split ? k_in : k_rot;
#pragma unroll 4
        for (int m = 0; m < kBKeys / 4; ++m) {
          const int key = (tid >> 4) + 4 * m;
          const int n = i * kBKeys + key;
          int j = n < kt ? sh.idx[qs][n] : -1;
          if (j >= len) {
            if (ch == 0) atomicOr(status, DEV_ERR_BAD_INDEX);
            j = -1;
          }
          const bool valid = j >= 0;
          const uint16_t* src = kb + static_cast<size_t>(valid ? ks_t + j : 0) * kBD + ch * 8;
          cp_async_16_zfill(smem_u32(k_dst + blk * (kKBytes / 2) + sw128b(key, ch & 7)), src, valid);
        }
        cp_async_mbar_arrive(&sh.k_full[s]);
      }
      ++qc;
    }
    cp_async_wait<0>();   // every copy has landed before the CTA can exit
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 2 issues X for each tile as soon as its keys have landed; warp 3 (which owns TMEM)
    // issues dK and dQ^T as soon as the tile's G is written.  Issued from one warp, dK of tile i
    // queued behind X of tile i + 1 and so behind that tile's gather; and the K stages, released
    // after dQ^T, held the gather back in turn.
    constexpr uint32_t id_x = idesc_bf16_f32(128, kHP, 0, 0);
    constexpr uint32_t id_dk = TR ? idesc_bf16_f32(kBD, kBKeys, 1, 0)    // dK^T: M = d, N = keys
                                  : idesc_bf16_f32(kBKeys, kBD, 0, 1);   // dK: M = keys, N = d
    constexpr uint32_t id_dq = idesc_bf16_f32(128, kHP, 1, 1);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_for(bar, parity, &sh.abort_flag, status, wait_ns));
    };
    uint32_t T = 0, qc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_q && ok; t += gridDim.x) {
      const int kt = row_slots(ks, ke, n_kv, topk, t);
      if (kt == 0) continue;
      const int nt = (kt + kBKeys - 1) / kBKeys;
      const int qs = qc & 1;
      if (!(ok = wait(&sh.q_full[qs], (qc >> 1) & 1))) break;
      const uint32_t q_addr = smem_u32(sQ + qs * kQBytes);
      for (int i = 0; i < nt && ok; ++i, ++T) {
        const int s = T % kStagesB, b = T & 1;
        const uint32_t k_addr = smem_u32(sK + s * kKBytes);
        if (warp == 2) {
          // X = K Q^T
          if (!(ok = wait(&sh.k_full[s], (T / kStagesB) & 1))) break;
          if (T >= 2 && !(ok = wait(&sh.x_empty[b], ((T >> 1) - 1) & 1))) break;
          fence_proxy_async_smem();   // cp.async-written tiles
          tc_fence_after();
          const uint64_t da = sdesc_sw128(k_addr, 16, 1024);
          const uint64_t db = sdesc_sw128(q_addr, 16, 1024);
#pragma unroll
          for (int k = 0; k < kBD / 16; ++k) {
            const int kb = k >> 2, sub = k & 3;
            umma_bf16_elect(tmem + kXCol + b * kHP, da + static_cast<uint64_t>((kb * (kKBytes / 2) + sub * 32) >> 4),
                            db + static_cast<uint64_t>((kb * (kQBytes / 2) + sub * 32) >> 4), id_x, k > 0 ? 1u : 0u);
          }
          umma_commit_elect(&sh.x_full[b]);
          umma_commit_elect(&sh.k_empty[s]);   // this warp's read of the tile
        } else {
          if (!(ok = wait(&sh.g_full[b], (T >> 1) & 1))) break;
          if (T >= 2 && !(ok = wait(&sh.dk_empty[b], ((T >> 1) - 1) & 1))) break;
          if (i == 0 && qc >= 2 && !(ok = wait(&sh.dq_empty[qs], ((qc >> 1) - 1) & 1))) break;
          fence_proxy_async_smem();   // G written with generic stores
          tc_fence_after();
          const uint32_t g_addr = smem_u32(sG + b * kGBytes);
          // TR: dK^T = Q^T G^T (A = Q, MN-major over d: 64-dim blocks 8 KB apart; B = G, K-major
          // over heads); else dK = G Q (A = G, B = Q, the same descriptors); 16 heads per step
          const uint64_t dq_mn = sdesc_sw128(q_addr, kQBytes / 2, 1024);
          const uint64_t dg_k = sdesc_sw128(g_addr, 16, 1024);
#pragma unroll
          for (int k = 0; k < kHP / 16; ++k) {
            const uint64_t qk = dq_mn + static_cast<uint64_t>((k * 16 * 128) >> 4);
            const uint64_t gk = dg_k + static_cast<uint64_t>((k * 32) >> 4);
            umma_bf16_elect(tmem + kDkCol + b * kBKeys, TR ? qk : gk, TR ? gk : qk, id_dk, k > 0 ? 1u : 0u);
          }
          umma_commit_elect(&sh.dk_full[b]);
          // dQ^T += K^T G: A = K tile (MN-major over d: 64-dim blocks 16 KB apart), B = G (MN-major
          // over heads); 16 keys (2 KB of rows) per step
          const uint64_t dka = sdesc_sw128(k_addr, kKBytes / 2, 1024);
          const uint64_t dgb = sdesc_sw128(g_addr, kGBytes, 1024);
#pragma unroll
          for (int k = 0; k < kBKeys / 16; ++k)
            umma_bf16_elect(tmem + kDqCol + qs * kHP, dka + static_cast<uint64_t>((k * 16 * 128) >> 4),
                            dgb + static_cast<uint64_t>((k * 16 * 128) >> 4), id_dq, (i > 0 || k > 0) ? 1u : 0u);
          umma_commit_elect(&sh.k_empty[s]);   // this warp's read of the tile
          umma_commit_elect(&sh.g_empty[b]);
        }
      }
      if (!ok) break;
      if (warp == 3) umma_commit_elect(&sh.dq_full[qs]);
      umma_commit_elect(&sh.q_empty[qs]);
      ++qc;
    }
    // every product this warp issued has completed before TMEM is released
    umma_commit_elect(&sh.mma_done);
    mbar_drain(&sh.mma_done, 0, 200000000ull);
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int e = warp - 4;                                  // TMEM lane quarter
    const uint32_t t_lane = static_cast<uint32_t>(e * 32) << 16;
    const int row = e * 32 + lane;                           // key within the tile / dim of dQ^T
    uint32_t T = 0, qc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_q && ok; t += gridDim.x) {
      const int kt = row_slots(ks, ke, n_kv, topk, t);
      if (kt == 0) {
        // nothing selected: dq~ is zero (dw was cleared before the launch)
        float* dq_t = dq + static_cast<size_t>(t) * n_heads * kBD;
        for (int i = threadIdx.x - 128; i < n_heads * kBD; i += 128) dq_t[i] = 0.f;
        continue;
      }
      const int nt = (kt + kBKeys - 1) / kBKeys;
      const int qs = qc & 1;
      const int len = __ldg(ke + t) - __ldg(ks + t);
      const int ks_t = __ldg(ks + t);
      if (!(ok = warp_all_wait(&sh.q_full[qs], (qc >> 1) & 1, &sh.abort_flag, status, wait_ns))) break;
      float dwacc[kHP];
#pragma unroll
      for (int h = 0; h < kHP; ++h) dwacc[h] = 0.f;
      for (int i = 0; i < nt && ok; ++i, ++T) {
        const int b = T & 1;
        const int n = i * kBKeys + row;
        int j = n < kt ? sh.idx[qs][n] : -1;
        if (j >= len) j = -1;   // flagged by the producer
        const float g = j >= 0 ? sh.ds[qs][n] : 0.f;
        if (!(ok = warp_all_wait(&sh.x_full[b], (T >> 1) & 1, &sh.abort_flag, status, wait_ns))) break;
        tc_fence_after();
        uint32_t xv[kHP];
        tmem_ld32(tmem + t_lane + kXCol + b * kHP, *reinterpret_cast<uint32_t(*)[32]>(&xv[0]));
        tmem_ld32(tmem + t_lane + kXCol + b * kHP + 32, *reinterpret_cast<uint32_t(*)[32]>(&xv[32]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.x_empty[b]);
        // dw sums and G = g w [x > 0] (bf16, 8 heads per 16-byte chunk)
        uint32_t gp[kHP / 2];
#pragma unroll
        for (int h = 0; h < kHP; h += 4) {
          const float4 wv = *reinterpret_cast<const float4*>(&sh.w[qs][h]);
          const float x0 = __uint_as_float(xv[h]), x1 = __uint_as_float(xv[h + 1]);
          const float x2 = __uint_as_float(xv[h + 2]), x3 = __uint_as_float(xv[h + 3]);
          dwacc[h] = fmaf(g, fmaxf(x0, 0.f), dwacc[h]);
          dwacc[h + 1] = fmaf(g, fmaxf(x1, 0.f), dwacc[h + 1]);
          dwacc[h + 2] = fmaf(g, fmaxf(x2, 0.f), dwacc[h + 2]);
          dwacc[h + 3] = fmaf(g, fmaxf(x3, 0.f), dwacc[h + 3]);
          gp[h / 2] = pack_bf16x2(x0 > 0.f ? g * wv.x : 0.f, x1 > 0.f ? g * wv.y : 0.f);
          gp[h / 2 + 1] = pack_bf16x2(x2 > 0.f ? g * wv.z : 0.f, x3 > 0.f ? g * wv.w : 0.f);
        }
        if (T >= 2 && !(ok = warp_all_wait(&sh.g_empty[b], ((T >> 1) - 1) & 1, &sh.abort_flag, status, wait_ns)))
          break;
        uint8_t* g_row = sG + b * kGBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(g_row + sw128b(row, c)) =
              make_uint4(gp[4 * c], gp[4 * c + 1], gp[4 * c + 2], gp[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.g_full[b]);
        // dK^T into dk~: this thread is dim `row` of the tile's 128 keys (TMEM columns); per chunk
        // of 32 keys lane c looks up key c's row (-1 when it adds nothing: no selection, or
        // g = 0) and the warp takes them by shuffle, so no shared-memory read sits between two
        // reductions
        if (!(ok = warp_all_wait(&sh.dk_full[b], (T >> 1) & 1, &sh.abort_flag, status, wait_ns))) break;
        tc_fence_after();
        if constexpr (TR) {
          float* dk_dim = dk + row;
#pragma unroll 1
          for (int c0 = 0; c0 < kBKeys; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + t_lane + kDkCol + b * kBKeys + c0, v);
            const int nk = i * kBKeys + c0 + lane;
            const int jk = nk < kt ? sh.idx[qs][nk] : -1;
            const int kr = (jk >= 0 && jk < len && sh.ds[qs][nk] != 0.f) ? ks_t + jk : -1;
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int r = __shfl_sync(0xffffffffu, kr, c);
              if (r >= 0) red_add_f32(dk_dim + static_cast<size_t>(r) * kBD, __uint_as_float(v[c]));
            }
          }
        } else {
          // this thread's key row (`row` = key), 16 bytes a reduction
          float* dk_row = dk + static_cast<size_t>(j >= 0 ? ks_t + j : 0) * kBD;
          const bool add = j >= 0 && g != 0.f;
#pragma unroll
          for (int c0 = 0; c0 < kBD; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + t_lane + kDkCol + b * kBD + c0, v);
            tmem_ld_wait();
            if (add) {
#pragma unroll
              for (int q = 0; q < 32; q += 4)
                red_add_v4(dk_row + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                           __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.dk_empty[b]);
      }
      if (!ok) break;
      // dw: reduce-scatter the 64 per-lane sums over the warp (each lane ends with two heads),
      // then one atomic add per head and warp
      int h0 = 0;
#pragma unroll
      for (int half = kHP / 2, o = 16; o >= 1; half >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i2 = 0; i2 < half; ++i2) {
          const float send = up ? dwacc[i2] : dwacc[i2 + half];
          const float keep = up ? dwacc[i2 + half] : dwacc[i2];
          dwacc[i2] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (up) h0 += half;
      }
      float* dw_t = dw + static_cast<size_t>(t) * n_heads;
      if (h0 < n_heads) atomicAdd(dw_t + h0, dwacc[0]);
      if (h0 + 1 < n_heads) atomicAdd(dw_t + h0 + 1, dwacc[1]);
      // dq~: lane = dim, columns = heads
      if (!(ok = warp_all_wait(&sh.dq_full[qs], (qc >> 1) & 1, &sh.abort_flag, status, wait_ns))) break;
      tc_fence_after();
      float* dq_t = dq + static_cast<size_t>(t) * n_heads * kBD;
#pragma unroll
      for (int c0 = 0; c0 < kHP; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + t_lane + kDqCol + qs * kHP + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (c0 + q < n_heads) dq_t[static_cast<size_t>(c0 + q) * kBD + row] = __uint_as_float(v[q]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.dq_empty[qs]);
      ++qc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 3) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_indexer_bwd(int n_q, int n_kv, int n_heads, int head_dim, int topk, const void* q_rot,
                               const void* q_in, const void* k_rot, const void* k_in, int q_split, int k_split,
                               const float* w, const int32_t* ks, const int32_t* ke, const int32_t* idx,
                               const float* d_score, float* dq, float* dk, float* dw, int grid, uint32_t* status,
                               const PipelineDebug& dbg, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  if (head_dim != kBD || n_heads < 1 || n_heads > kHP || n_heads % 4 || grid < 1) return cudaErrorInvalidValue;
  cudaError_t e = smem_attr_once<indexer_bwd_kernel<true>>(kBwdDynSmem);
  if (e == cudaSuccess) e = smem_attr_once<indexer_bwd_kernel<false>>(kBwdDynSmem);
  if (e != cudaSuccess) return e;
  BwdArgs A;
  A.q_rot = static_cast<const uint16_t*>(q_rot);
  A.q_in = static_cast<const uint16_t*>(q_in);
  A.k_rot = static_cast<const uint16_t*>(k_rot);
  A.k_in = static_cast<const uint16_t*>(k_in);
  A.q_split = q_split;
  A.k_split = k_split;
  A.w = w;
  A.ks = ks;
  A.ke = ke;
  A.idx = idx;
  A.d_score = d_score;
  A.dq = dq;
  A.dk = dk;
  A.dw = dw;
  A.n_q = n_q;
  A.n_kv = n_kv;
  A.n_heads = n_heads;
  A.topk = topk;
  A.status = status;
  A.wait_ns = dbg.wait_ns;
  // the transposed dK form unless many queries share each key row (about 64 or more
  // selections per row on average: a short prefix)
  const bool tr = static_cast<long long>(n_q) * topk <= 64LL * (n_kv > 0 ? n_kv : 1);
  const int g = grid < n_q ? grid : n_q;
  auto kern = tr ? indexer_bwd_kernel<true> : indexer_bwd_kernel<false>;
  kern<<<g, kBwdThreads, kBwdDynSmem, st>>>(A.q_rot, A.q_in, A.k_rot, A.k_in, A.q_split, A.k_split, A.w, A.ks, A.ke,
                                           A.idx, A.d_score, A.dq, A.dk, A.dw, A.n_q, A.n_kv, A.n_heads, A.topk,
                                           A.status, A.wait_ns);
  return cudaGetLastError();
}

}  // namespace dsa
