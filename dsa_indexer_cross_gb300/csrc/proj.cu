// Projections upstream of the lightning indexer, on the tensor cores.
//
// "GLM-5/5.1/5.2 DSA + LoRA enablement" (Megatron-Bridge pull request; the indexer RoPE
// half-swap commit) names the indexer's weights: wq_b (index queries), wk (the shared index
// key), k_norm (a LayerNorm with weight and bias, applied to the key before RoPE) and
// weights_proj (one scalar per index head).  For one full layer:
//   q_idx[t] = q_latent[t] . wq_b^T          -> [H_I * d_I] bf16
//   k_idx[t] = LayerNorm(x[t] . wk^T)        -> [d_I] bf16 (affine k_norm weight / bias)
//   w[t]     = x[t] . weights_proj^T         -> [H_I] fp32
// Every output is a GEMM over the token rows, so one persistent kernel walks the units (job,
// 128-token tile, N tile) of two jobs: the query projection, and the key and head-weight
// projections together (wk's rows and weights_proj's rows stacked in one weight tile, so both
// read the activations once).  TMA streams 64-wide K blocks of the activations and of the
// weight rows into a four-stage ring, one thread issues tcgen05.mma (M = 128 tokens, N <= 256,
// K = 16) into a double-buffered TMEM accumulator, and four epilogue warps (thread = token row
// = TMEM lane) convert and store; a key row is whole in one tile (N >= d_I), so the LayerNorm
// happens in registers.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kPM = 128;                                  // tokens per tile (MMA M)
constexpr int kPThreads = 192;                            // TMA warp, MMA warp, 4 epilogue warps
constexpr int kPStages = 4;
constexpr int kPMaxN = 256;
constexpr int kPABytes = kPM * 128;                       // one 64-wide K block of 128 token rows
constexpr int kPStageBytes = kPABytes + kPMaxN * 128;     // + up to 256 weight rows
constexpr int kPDynSmem = 1024 + kPStages * kPStageBytes;

struct ProjShared {
  uint64_t full[kPStages], empty[kPStages];
  uint64_t t_full[2], t_empty[2];
  uint32_t tmem_base;
  uint32_t abort_flag;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Which job (output matrix) and which tiles unit u covers.
struct PUnit {
  int job, m0, n0;
};
__device__ __forceinline__ PUnit punit(const ProjJobs& J, int u, int m_tiles) {
  int job = 0;
  while (job + 1 < J.n_jobs && u >= J.first_unit[job + 1]) ++job;
  const int r = u - J.first_unit[job];
  const int nt = r / m_tiles;
  return PUnit{job, (r - nt * m_tiles) * kPM, nt * J.job[job].n_tile};
}

__global__ void __launch_bounds__(kPThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
                const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1,
                const __grid_constant__ CUtensorMap tb_2, const ProjJobs J, int n_tokens, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ ProjShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int m_tiles = (n_tokens + kPM - 1) / kPM;
  const int n_units = J.first_unit[J.n_jobs];
  auto maps = [&](int job, const CUtensorMap*& a, const CUtensorMap*& b) {
    a = job == 0 ? &ta0 : &ta1;
    b = job == 0 ? &tb0 : &tb1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.t_full[b], 1);
      mbar_init(&sh.t_empty[b], 4);   // one arrive per epilogue warp
    }
    sh.abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 2 * kPMaxN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_lane0()) {
      uint32_t st = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const PUnit p = punit(J, u, m_tiles);
        const ProjJob& jb = J.job[p.job];
        const CUtensorMap *ma, *mb;
        maps(p.job, ma, mb);
        const uint32_t bytes = kPABytes + jb.n_tile * 128;
        for (int kb = 0; kb < jb.k / 64; ++kb, ++st) {
          const int s = st % kPStages;
          if (st >= kPStages && !(ok = mbar_wait(&sh.empty[s], ((st / kPStages) - 1) & 1, &sh.abort_flag, status)))
            break;
          uint8_t* a = smem + s * kPStageBytes;
          mbar_arrive_expect_tx(&sh.full[s], bytes);
          tma_load_2d(a, ma, &sh.full[s], kb * 64, p.m0);                 // rows past n_tokens read zeros
          tma_load_2d(a + kPABytes, mb, &sh.full[s], kb * 64, p.n0);      // rows past the matrix read zeros
          if (jb.epi == kProjEpiLayerNormF32)                             // the stacked second matrix
            tma_load_2d(a + kPABytes + jb.n_total * 128, &tb_2, &sh.full[s], kb * 64, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_lane0()) {
      uint32_t st = 0, tile = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++tile) {
        const PUnit p = punit(J, u, m_tiles);
        const ProjJob& jb = J.job[p.job];
        const uint32_t idesc = idesc_bf16_f32(kPM, jb.n_tile, 0, 0);
        const int buf = tile & 1;
        if (tile >= 2 && !(ok = mbar_wait(&sh.t_empty[buf], ((tile >> 1) - 1) & 1, &sh.abort_flag, status))) break;
        for (int kb = 0; kb < jb.k / 64; ++kb, ++st) {
          const int s = st % kPStages;
          if (!(ok = mbar_wait(&sh.full[s], (st / kPStages) & 1, &sh.abort_flag, status))) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * kPStageBytes);
#pragma unroll
          for (int sub = 0; sub < 4; ++sub) {
            const uint64_t ad = sdesc_sw128(a0 + sub * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(a0 + kPABytes + sub * 32, 16, 1024);
            umma_bf16(tmem + buf * kPMaxN, ad, bd, idesc, (kb | sub) ? 1u : 0u);
          }
          umma_commit(&sh.empty[s]);
        }
        if (ok) umma_commit(&sh.t_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int lane = threadIdx.x & 31;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t tile = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++tile) {
      const PUnit p = punit(J, u, m_tiles);
      const ProjJob& jb = J.job[p.job];
      const int buf = tile & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&sh.t_full[buf], (tile >> 1) & 1, &sh.abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      const int token = p.m0 + quarter * 32 + lane;
      const bool live = token < n_tokens;
      const uint32_t tcol = tmem + t_lane + buf * kPMaxN;
      if (jb.epi == kProjEpiLayerNormF32) {
        // mean, then the centred sum of squares, then the normalised, scaled, shifted row
        float sum = 0.f;
        for (int c0 = 0; c0 < jb.n_total; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tcol + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) sum += __uint_as_float(v[i]);
        }
        const float mean = sum / static_cast<float>(jb.n_total);
        float ss = 0.f;
        for (int c0 = 0; c0 < jb.n_total; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tcol + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float d = __uint_as_float(v[i]) - mean;
            ss = fmaf(d, d, ss);
          }
        }
        const float rstd = rsqrtf(ss / static_cast<float>(jb.n_total) + jb.eps);
        for (int c0 = 0; c0 < jb.n_total; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tcol + c0, v);
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float y0 = fmaf((__uint_as_float(v[i]) - mean) * rstd, __ldg(jb.gamma + c0 + i), __ldg(jb.beta + c0 + i));
            const float y1 = fmaf((__uint_as_float(v[i + 1]) - mean) * rstd, __ldg(jb.gamma + c0 + i + 1),
                                  __ldg(jb.beta + c0 + i + 1));
            o[i / 2] = pack_bf16x2(y0, y1);
          }
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(jb.out) +
                                                  static_cast<size_t>(token) * jb.n_total + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        }
        // the stacked head-weight columns: fp32, possibly fewer than 32 (H_I < 32)
        for (int c0 = jb.n_total; c0 < jb.n_total + jb.n2; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tcol + c0, v);
          tmem_ld_wait();
          if (!live) continue;
          float* dst = jb.out2 + static_cast<size_t>(token) * jb.n2 + (c0 - jb.n_total);
          const int n = min(32, jb.n_total + jb.n2 - c0);
          for (int i = 0; i < n; ++i) dst[i] = __uint_as_float(v[i]);
        }
      } else {
        for (int c0 = 0; c0 < jb.n_tile; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tcol + c0, v);
          tmem_ld_wait();
          const int col = p.n0 + c0;
          if (!live || col >= jb.n_total) continue;
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) o[i / 2] = pack_bf16x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(jb.out) +
                                                static_cast<size_t>(token) * jb.n_total + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.t_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * kPMaxN);
}

}  // namespace

cudaError_t launch_projections(const CUtensorMap* ta, const CUtensorMap* tb, const CUtensorMap& tb2,
                               const ProjJobs& J, int n_tokens, uint32_t* status, cudaStream_t st) {
  if (n_tokens <= 0 || J.first_unit[J.n_jobs] <= 0) return cudaSuccess;
  if (J.n_jobs != 2) return cudaErrorInvalidValue;
  for (int j = 0; j < J.n_jobs; ++j) {
    const ProjJob& jb = J.job[j];
    if (jb.k <= 0 || jb.k % 64 || jb.n_tile < 32 || jb.n_tile > kPMaxN || jb.n_tile % 32 ||
        (jb.epi == kProjEpiLayerNormF32 && (jb.n_total % 32 || jb.n_tile < jb.n_total + jb.n2)))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = smem_attr_once<proj_kernel>(kPDynSmem);
  if (e != cudaSuccess) return e;
  const int units = J.first_unit[J.n_jobs];
  const int grid = units < device_sm_count() ? units : device_sm_count();
  proj_kernel<<<grid, kPThreads, kPDynSmem, st>>>(ta[0], tb[0], ta[1], tb[1], tb2, J, n_tokens, status);
  return cudaGetLastError();
}

}  // namespace dsa
