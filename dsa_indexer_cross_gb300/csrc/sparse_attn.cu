// MLA-absorbed sparse attention over gathered latent rows, on tcgen05.
//
//   o[t, h] = sum_{j in I_t} softmax_j(tau * q[t, h] . kv[ks_t + j]) * kv[ks_t + j, :512]
//
// ("GLM-5.2 IndexShare" explainer, section 1 and "What is actually shared?": every layer
// runs its own attention over the selected positions; the 576 = 512 latent + 64 rope key
// and the 512-d value follow "GLM-5/5.1/5.2 DSA + LoRA enablement", qk_rope_head_dim
// commit.)  All heads of a token read the same selected rows.
//
// Formulation.  A CTA owns (token t, block of HB heads) and walks the token's index row in
// tiles of 64 selected rows.  Because HB (16 or 32) is too small for the M side of the
// tensor core, both products run transposed, with the gathered rows on M:
//     S^T[r, h]  = Rows[r, :576] . Q[h, :576]            M = 64 rows,   N = HB, K = 576
//     O^T[d, h] += Rows[:, d]^T  . P^T[r, h]             M = 128 dims,  N = HB, K = 64
// The gathered tile is stored once in shared memory in the 128-byte-swizzled layout and
// read as a K-major operand by the first product and as an MN-major operand by the
// second, so each row is fetched from memory exactly once.  S^T is double-buffered in
// TMEM; O^T (512 x HB fp32) stays in TMEM for the whole token.
//
// Online softmax (base 2): per head the running max m and sum l live in registers of the
// softmax warps; a tile whose max exceeds the max in use by more than 8 (a factor 256)
// triggers a rescale of O^T in TMEM, otherwise the old max is kept (exact either way).
//
// Warp roles (288 threads): warps 0-3 gather rows with cp.async (zero-fill for unused or
// out-of-range slots); warps 4-7 run the softmax and the epilogue; warp 8 owns TMEM and
// issues the MMAs from one thread.  The CTA is persistent over (token, head block) items.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kRows = 64;          // selected rows per tile
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kChunks = kDqk / 8;  // 16-byte chunks per latent row
constexpr int kStages = 2;
constexpr int kProd = 128;
constexpr int kSoft = 128;
constexpr int kThreads = kProd + kSoft + 32;
constexpr int kTileBytes = kRows * kDqk * 2;   // 72 KB

template <int HB>
struct ACfg {
  static constexpr int Q_BYTES = HB * kDqk * 2;
  static constexpr int P_BYTES = HB * kRows * 2;
  static constexpr int DYN_SMEM = 1024 + kStages * kTileBytes + Q_BYTES + P_BYTES;
  static constexpr uint32_t TMEM_COLS = 6 * HB <= 128 ? 128 : 256;
  static constexpr int O_COL = 0;
  static constexpr int S_COL = 4 * HB;
};

struct AShared {
  uint64_t full[kStages], empty[kStages];
  uint64_t q_empty, s_full[2], s_empty[2], p_full, o_done, o_free;
  uint32_t tmem_base, abort_flag, soft_abort;
  float red[4][32];
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int HB>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx,
                       const int32_t* __restrict__ ks, const int32_t* __restrict__ row_nt, uint16_t* __restrict__ out,
                       float* __restrict__ lse, int n_q, int n_kv, int H, int topk, float scale_log2,
                       uint32_t* status, uint32_t* bad_count) {
  using C = ACfg<HB>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ AShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sT = smem;                                   // kStages tiles
  uint8_t* sQ = smem + kStages * kTileBytes;            // HB x 576, 9 blocks of HB x 128 B
  uint8_t* sP = sQ + C::Q_BYTES;                        // P^T: HB x 64, K-major
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_hb = (H + HB - 1) / HB;
  const int n_items = n_q * n_hb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], kProd);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_empty[b], kSoft);
    }
    mbar_init(&sh.p_full, kSoft);
    mbar_init(&sh.o_done, 1);
    mbar_init(&sh.o_free, kSoft);
    sh.abort_flag = 0;
    sh.soft_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp < 4) {
    // ---------------------------------------------------------------- gather producers
    const int tid = threadIdx.x;
    uint32_t g = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int t = item / n_hb, hb = item - t * n_hb;
      const int nt = __ldg(row_nt + t);
      if (nt == 0) continue;
      if (it > 0) ok = mbar_wait(&sh.q_empty, (it - 1) & 1, &sh.abort_flag, status);
      if (!ok) break;
      // Q block: HB heads x 72 chunks
      for (int c = tid; c < HB * kChunks; c += kProd) {
        const int h = c / kChunks, ch = c - h * kChunks;
        const int head = hb * HB + h;
        const bool v = head < H;
        const uint16_t* src = q + (static_cast<size_t>(t) * H + (v ? head : 0)) * kDqk + ch * 8;
        cp_async_16_zfill(smem_u32(sQ + (ch >> 3) * (HB * 128) + sw128(h, ch & 7)), src, v);
      }
      const int kst = __ldg(ks + t);
      const int32_t* irow = idx + static_cast<size_t>(t) * topk;
      for (int i = 0; i < nt; ++i, ++g) {
        const int s = g % kStages;
        if (g >= kStages) {
          ok = mbar_wait(&sh.empty[s], ((g / kStages) - 1) & 1, &sh.abort_flag, status);
          if (!ok) break;
        }
        uint8_t* dst = sT + s * kTileBytes;
        for (int c = tid; c < kRows * kChunks; c += kProd) {
          const int r = c / kChunks, ch = c - r * kChunks;
          const int slot = i * kRows + r;
          const int j = slot < topk ? __ldg(irow + slot) : -1;
          const long long row = static_cast<long long>(kst) + j;
          const bool v = j >= 0 && row < n_kv && row >= 0;
          if (ch == 0 && j >= 0 && !v) {
            atomicOr(status, DEV_ERR_BAD_INDEX);
            atomicAdd(bad_count, 1u);
          }
          const uint16_t* src = kv + (v ? row : 0) * kDqk + ch * 8;
          cp_async_16_zfill(smem_u32(dst + (ch >> 3) * (kRows * 128) + sw128(r, ch & 7)), src, v);
        }
        cp_async_mbar_arrive(&sh.full[s]);
      }
      ++it;
    }
    cp_async_wait<0>();
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int tid = threadIdx.x - kProd;   // 0..127
    const int qd = warp & 3;               // TMEM lane quarter
    const int r = qd * 16 + lane;          // S^T row owned (lanes 0..15 of the quarter)
    const bool row_lane = lane < 16;
    const uint32_t t_lane = static_cast<uint32_t>(qd * 32) << 16;
    // A failed (timed-out) wait is published through sh.soft_abort, written only before a
    // named barrier and read right after it; the next write can only happen after a later
    // barrier, so the four softmax warps always leave the loops at the same point.
    uint32_t g = 0, it = 0;
    bool stop = false;
    for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
      const int t = item / n_hb, hb = item - t * n_hb;
      const int nt = __ldg(row_nt + t);
      if (nt == 0) {
        for (int e = tid; e < HB * kDv; e += kSoft) {
          const int h = e / kDv, head = hb * HB + h;
          if (head < H) out[(static_cast<size_t>(t) * H + head) * kDv + (e - h * kDv)] = 0;
        }
        if (lse && tid < HB && hb * HB + tid < H) lse[static_cast<size_t>(t) * H + hb * HB + tid] = -INFINITY;
        continue;
      }
      const int kst = __ldg(ks + t);
      const int32_t* irow = idx + static_cast<size_t>(t) * topk;
      float m_used[HB], l_run[HB];
#pragma unroll
      for (int h = 0; h < HB; ++h) {
        m_used[h] = -INFINITY;
        l_run[h] = 0.f;
      }
      for (int i = 0; i < nt; ++i, ++g) {
        const int sb = g & 1;
        bool ok = mbar_wait(&sh.s_full[sb], (g >> 1) & 1, &sh.abort_flag, status);
        ok = __all_sync(0xffffffffu, ok);
        float sc[HB];
        bool valid = false;
        if (ok) {
          tc_fence_after();
          uint32_t raw[HB];
          if constexpr (HB == 16) {
            uint32_t v16[16];
            tmem_ld16(tmem + t_lane + C::S_COL + sb * HB, v16);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 16; ++h) raw[h] = v16[h];
          } else {
            uint32_t v32[32];
            tmem_ld32(tmem + t_lane + C::S_COL + sb * HB, v32);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) raw[h] = v32[h];
          }
          tc_fence_before();
          mbar_arrive(&sh.s_empty[sb]);
          const int slot = i * kRows + r;
          const int j = (row_lane && slot < topk) ? __ldg(irow + slot) : -1;
          const long long row = static_cast<long long>(kst) + j;
          valid = row_lane && j >= 0 && row >= 0 && row < n_kv;
#pragma unroll
          for (int h = 0; h < HB; ++h) sc[h] = valid ? __uint_as_float(raw[h]) * scale_log2 : -INFINITY;
          // tile max per head over the 64 rows
#pragma unroll
          for (int h = 0; h < HB; ++h) {
            float x = sc[h];
            x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
            x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
            x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
            x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
            if (lane == 0) sh.red[qd][h] = x;
          }
          // the previous tile's PV must be done before P is overwritten or O^T rescaled
          if (g > 0) {
            ok = mbar_wait(&sh.o_done, (g - 1) & 1, &sh.abort_flag, status);
            ok = __all_sync(0xffffffffu, ok);
          }
        }
        if (!ok && lane == 0) sh.soft_abort = 1;
        named_bar_sync(1, kSoft);
        stop = sh.soft_abort != 0;
        float alpha[HB];
        float ps[HB];
        if (!stop) {
          tc_fence_after();
          bool rescale = false;
#pragma unroll
          for (int h = 0; h < HB; ++h) {
            const float m = fmaxf(fmaxf(sh.red[0][h], sh.red[1][h]), fmaxf(sh.red[2][h], sh.red[3][h]));
            alpha[h] = 1.f;
            if (m > m_used[h] + 8.f) {
              alpha[h] = exp2f(m_used[h] - m);   // 0 when m_used = -inf
              m_used[h] = m;
              rescale = true;
            }
          }
          if (rescale && i > 0) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
#pragma unroll
              for (int hh = 0; hh < HB / 16; ++hh) {
                uint32_t o[16];
                tmem_ld16(tmem + t_lane + C::O_COL + b * HB + hh * 16, o);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[hh * 16 + h]);
                tmem_st16(tmem + t_lane + C::O_COL + b * HB + hh * 16, o);
              }
            }
            tmem_st_wait();
          }
          // P = exp2(s - m) in bf16, written as the K-major B operand of the second product
#pragma unroll
          for (int h = 0; h < HB; ++h) {
            const float p = valid ? exp2f(sc[h] - m_used[h]) : 0.f;
            const __nv_bfloat16 pb = __float2bfloat16_rn(p);
            ps[h] = __bfloat162float(pb);
            if (row_lane) {
              const uint32_t off = (h >> 3) * 1024 + (h & 7) * 128 + ((((r >> 3) ^ (h & 7)) & 7) << 4) + (r & 7) * 2;
              *reinterpret_cast<__nv_bfloat16*>(sP + off) = pb;
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&sh.p_full);
        }
        named_bar_sync(1, kSoft);      // everyone has read red[] (max) and soft_abort
        if (stop) break;
        // row sums per head
#pragma unroll
        for (int h = 0; h < HB; ++h) {
          float x = ps[h];
          x += __shfl_xor_sync(0xffffffffu, x, 8);
          x += __shfl_xor_sync(0xffffffffu, x, 4);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          if (lane == 0) sh.red[qd][h] = x;
        }
        named_bar_sync(1, kSoft);
#pragma unroll
        for (int h = 0; h < HB; ++h)
          l_run[h] = l_run[h] * alpha[h] + ((sh.red[0][h] + sh.red[1][h]) + (sh.red[2][h] + sh.red[3][h]));
        named_bar_sync(1, kSoft);      // red[] free for the next tile
      }
      if (stop) break;
      // epilogue: O^T / l -> out
      bool ok = mbar_wait(&sh.o_done, (g - 1) & 1, &sh.abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) sh.soft_abort = 1;
      named_bar_sync(1, kSoft);
      stop = sh.soft_abort != 0;
      named_bar_sync(1, kSoft);
      if (stop) break;
      tc_fence_after();
      float inv[HB];
#pragma unroll
      for (int h = 0; h < HB; ++h) inv[h] = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
#pragma unroll
        for (int hh = 0; hh < HB / 16; ++hh) {
          uint32_t o[16];
          tmem_ld16(tmem + t_lane + C::O_COL + b * HB + hh * 16, o);
          tmem_ld_wait();
          const int d = b * 128 + qd * 32 + lane;
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const int head = hb * HB + hh * 16 + h;
            if (head < H) {
              const __nv_bfloat16 ob = __float2bfloat16_rn(__uint_as_float(o[h]) * inv[hh * 16 + h]);
              out[(static_cast<size_t>(t) * H + head) * kDv + d] = *reinterpret_cast<const uint16_t*>(&ob);
            }
          }
        }
      }
      if (lse && tid < HB && hb * HB + tid < H) {
        float mv = 0.f, lv = 0.f;
#pragma unroll
        for (int h = 0; h < HB; ++h)
          if (h == tid) {
            mv = m_used[h];
            lv = l_run[h];
          }
        lse[static_cast<size_t>(t) * H + hb * HB + tid] = lv > 0.f ? (mv + log2f(lv)) * 0.69314718055994531f : -INFINITY;
      }
      tc_fence_before();
      mbar_arrive(&sh.o_free);
      ++it;
    }
  } else {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(64, HB, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, HB, 1, 0);
      const uint32_t sq = smem_u32(sQ), sp = smem_u32(sP), st0 = smem_u32(sT);
      uint32_t g = 0, it = 0;
      bool ok = true;
      auto issue_qk = [&](uint32_t gq) -> bool {
        const int s = gq % kStages, sb = gq & 1;
        if (!mbar_wait(&sh.full[s], (gq / kStages) & 1, &sh.abort_flag, status)) return false;
        if (gq >= 2 && !mbar_wait(&sh.s_empty[sb], ((gq >> 1) - 1) & 1, &sh.abort_flag, status)) return false;
        tc_fence_after();
        const uint32_t a0 = st0 + s * kTileBytes;
#pragma unroll 4
        for (int k = 0; k < kDqk / 16; ++k) {
          const int kb = k >> 2, sub = k & 3;
          umma_bf16(tmem + C::S_COL + sb * HB, sdesc_sw128(a0 + kb * (kRows * 128) + sub * 32, 16, 1024),
                    sdesc_sw128(sq + kb * (HB * 128) + sub * 32, 16, 1024), id_qk, k > 0 ? 1u : 0u);
        }
        umma_commit(&sh.s_full[sb]);
        return true;
      };
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int t = item / n_hb;
        const int nt = __ldg(row_nt + t);
        if (nt == 0) continue;
        ok = issue_qk(g);
        for (int i = 0; i < nt && ok; ++i, ++g) {
          if (i + 1 < nt) ok = issue_qk(g + 1);
          else umma_commit(&sh.q_empty);
          if (!ok) break;
          ok = mbar_wait(&sh.p_full, g & 1, &sh.abort_flag, status);
          if (ok && i == 0 && it > 0) ok = mbar_wait(&sh.o_free, (it - 1) & 1, &sh.abort_flag, status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = st0 + (g % kStages) * kTileBytes;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int k = 0; k < kRows / 16; ++k) {
              umma_bf16(tmem + C::O_COL + b * HB, sdesc_sw128(a0 + (2 * b) * (kRows * 128) + k * 2048, kRows * 128, 1024),
                        sdesc_sw128(sp + k * 32, 16, 1024), id_pv, (i > 0 || k > 0) ? 1u : 0u);
            }
          }
          umma_commit(&sh.empty[g % kStages]);
          umma_commit(&sh.o_done);
        }
        ++it;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) tmem_dealloc(tmem, C::TMEM_COLS);
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

template <int HB>
cudaError_t launch_hb(int n_q, int n_kv, int H, int topk, float scale, const void* q, const void* kv,
                      const int32_t* idx, const int32_t* ks, const int32_t* row_nt, void* out, float* lse,
                      uint32_t* status, cudaStream_t st) {
  using C = ACfg<HB>;
  auto kern = sparse_attn_kernel<HB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
  if (e != cudaSuccess) return e;
  const int n_items = n_q * ((H + HB - 1) / HB);
  const int grid = n_items < device_sm_count() ? n_items : device_sm_count();
  kern<<<grid, kThreads, C::DYN_SMEM, st>>>(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(kv), idx, ks,
                                            row_nt, static_cast<uint16_t*>(out), lse, n_q, n_kv, H, topk,
                                            scale * 1.4426950408889634f, status, status + 1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_attn(int n_q, int n_kv, int n_heads, int topk, float scale, const void* q, const void* kv,
                               const int32_t* idx, const int32_t* ks, void* out, float* lse, uint32_t* status,
                               int32_t* row_nt, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  row_tiles_kernel<<<(n_q + 7) / 8, 256, 0, st>>>(idx, n_q, topk, row_nt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (n_heads <= 16) return launch_hb<16>(n_q, n_kv, n_heads, topk, scale, q, kv, idx, ks, row_nt, out, lse, status, st);
  return launch_hb<32>(n_q, n_kv, n_heads, topk, scale, q, kv, idx, ks, row_nt, out, lse, status, st);
}

}  // namespace dsa
