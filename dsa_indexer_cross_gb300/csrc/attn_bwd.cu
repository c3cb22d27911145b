// Backward of the MLA-absorbed sparse attention: gradients of q and of the latent rows.
//
// The forward (sparse_attn.cu) computes, for token t, head h and the selected rows j,
//   s_j = tau q . kv_j,   p_j = exp(s_j - lse),   o = sum_j p_j kv_j[:512].
// Given the upstream d_o, with D = d_o . o (from the forward's own output):
//   dp_j = d_o . kv_j[:512],   ds_j = p_j (dp_j - D),
//   dq   = tau sum_j ds_j kv_j,
//   dkv_j += tau ds_j q + p_j d_o (first 512 dims), summed over every (token, head) selecting j.
// The training pages only name the backward kernels; this is the exact gradient of the forward.
//
// First version, on the CUDA cores: one CTA per (token, block of 16 heads); q, d_o and a chunk
// of 16 selected rows are staged in shared memory as fp32 (rows padded to an odd stride so
// that 16 rows read at one dim fall in 16 banks); P and dS of the chunk are computed one
// (head, row) pair per thread; dq stays in registers; dkv is scattered with fp32 atomic adds
// (rows are shared by many tokens).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kBH = 16;                  // heads per CTA
constexpr int kBR = 16;                  // selected rows per chunk
constexpr int kBThreads = kBH * kBR;     // 256
constexpr int kDq = 576, kDvB = 512;
constexpr int kQS = kDq + 1;             // padded fp32 row strides
constexpr int kOS = kDvB + 1;
constexpr int kPer = kDq / kBR;          // 36 dims per thread in the dq / dkv phases

struct BwdSmem {
  float q[kBH * kQS];
  float dout[kBH * kOS];
  float kv[kBR * kQS];
  float p[kBH][kBR + 1];
  float ds[kBH][kBR + 1];
  float dsum[kBH];
  float lse[kBH];
  long long row[kBR];
};

__device__ __forceinline__ float bf(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }

__global__ void __launch_bounds__(kBThreads) sparse_attn_bwd_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ ks, const uint16_t* __restrict__ out, const float* __restrict__ lse,
    const uint16_t* __restrict__ dout, float* __restrict__ dq, float* __restrict__ dkv, int n_kv, int H, int topk,
    float scale, uint32_t* status, uint32_t* bad_count) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem& S = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int t = blockIdx.x;
  const int h0 = blockIdx.y * kBH;
  const int tid = threadIdx.x;
  // ---- stage q and d_o of the block's heads (zeros past the last head), lse and D = d_o . o
  for (int e = tid; e < kBH * kDq; e += kBThreads) {
    const int h = e / kDq, d = e - h * kDq;
    S.q[h * kQS + d] = h0 + h < H ? bf(__ldg(q + (static_cast<size_t>(t) * H + h0 + h) * kDq + d)) : 0.f;
  }
  for (int e = tid; e < kBH * kDvB; e += kBThreads) {
    const int h = e / kDvB, d = e - h * kDvB;
    S.dout[h * kOS + d] = h0 + h < H ? bf(__ldg(dout + (static_cast<size_t>(t) * H + h0 + h) * kDvB + d)) : 0.f;
  }
  {
    // D: thread (h = tid / 16, part = tid % 16) sums 32 dims, then 16 lanes reduce
    const int h = tid / kBR, part = tid % kBR;
    float acc = 0.f;
    if (h0 + h < H) {
      const size_t o0 = (static_cast<size_t>(t) * H + h0 + h) * kDvB;
      for (int d = part; d < kDvB; d += kBR) acc = fmaf(bf(__ldg(dout + o0 + d)), bf(__ldg(out + o0 + d)), acc);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (part == 0) {
      S.dsum[h] = acc;
      S.lse[h] = h0 + h < H ? __ldg(lse + static_cast<size_t>(t) * H + h0 + h) : 0.f;
    }
  }
  __syncthreads();
  const long long kst = __ldg(ks + t);
  const int32_t* irow = idx + static_cast<size_t>(t) * topk;
  // dq accumulators: head hq = tid / 16, dims dd = tid % 16 + 16 m
  const int hq = tid / kBR, dd = tid % kBR;
  float acc[kPer];
#pragma unroll
  for (int m = 0; m < kPer; ++m) acc[m] = 0.f;
  const int n_chunks = (topk + kBR - 1) / kBR;
  for (int c = 0; c < n_chunks; ++c) {
    if (tid < kBR) {
      const int slot = c * kBR + tid;
      const int j = slot < topk ? __ldg(irow + slot) : -1;
      long long row = -1;
      if (j >= 0) {
        row = kst + j;
        if (row < 0 || row >= n_kv) {
          if (blockIdx.y == 0) {
            atomicOr(status, DEV_ERR_BAD_INDEX);
            atomicAdd(bad_count, 1u);
          }
          row = -1;
        }
      }
      S.row[tid] = row;
    }
    __syncthreads();
    bool any = false;
#pragma unroll
    for (int r = 0; r < kBR; ++r) any |= S.row[r] >= 0;
    if (!any) {   // uniform: nothing selected in this chunk (the tail of a short row)
      __syncthreads();
      continue;
    }
    for (int e = tid; e < kBR * kDq; e += kBThreads) {
      const int r = e / kDq, d = e - r * kDq;
      const long long row = S.row[r];
      S.kv[r * kQS + d] = row >= 0 ? bf(__ldg(kv + static_cast<size_t>(row) * kDq + d)) : 0.f;
    }
    __syncthreads();
    {
      // P and dS: thread (h = tid / 16, r = tid % 16)
      const int h = tid / kBR, r = tid % kBR;
      float s = 0.f, dp = 0.f;
      const float* qh = S.q + h * kQS;
      const float* oh = S.dout + h * kOS;
      const float* kr = S.kv + r * kQS;
      for (int d = 0; d < kDvB; ++d) {
        s = fmaf(qh[d], kr[d], s);
        dp = fmaf(oh[d], kr[d], dp);
      }
      for (int d = kDvB; d < kDq; ++d) s = fmaf(qh[d], kr[d], s);
      const bool live = S.row[r] >= 0 && h0 + h < H;
      const float p = live ? expf(scale * s - S.lse[h]) : 0.f;
      S.p[h][r] = p;
      S.ds[h][r] = p * (dp - S.dsum[h]);
    }
    __syncthreads();
    // dq += scale * dS . kv_chunk
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int d = dd + kBR * m;
      float a = 0.f;
#pragma unroll
      for (int r = 0; r < kBR; ++r) a = fmaf(S.ds[hq][r], S.kv[r * kQS + d], a);
      acc[m] = fmaf(scale, a, acc[m]);
    }
    {
      // dkv_r += scale * dS^T q + P^T d_o: thread (row r = tid / 16, dims tid % 16 + 16 m)
      const int r = tid / kBR;
      const long long row = S.row[r];
      if (row >= 0) {
        float* dst = dkv + static_cast<size_t>(row) * kDq;
        for (int m = 0; m < kPer; ++m) {
          const int d = dd + kBR * m;
          float a = 0.f, b = 0.f;
#pragma unroll
          for (int h = 0; h < kBH; ++h) {
            a = fmaf(S.ds[h][r], S.q[h * kQS + d], a);
            if (d < kDvB) b = fmaf(S.p[h][r], S.dout[h * kOS + d], b);
          }
          atomicAdd(dst + d, fmaf(scale, a, b));
        }
      }
    }
    __syncthreads();
  }
  if (h0 + hq < H) {
    float* dst = dq + (static_cast<size_t>(t) * H + h0 + hq) * kDq;
#pragma unroll
    for (int m = 0; m < kPer; ++m) dst[dd + kBR * m] = acc[m];
  }
}

}  // namespace

cudaError_t launch_sparse_attn_bwd(int n_q, int n_kv, int n_heads, int topk, float scale, const void* q,
                                   const void* kv, const int32_t* idx, const int32_t* ks, const void* out,
                                   const float* lse, const void* dout, float* dq, float* dkv, uint32_t* status,
                                   cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(BwdSmem));
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n_q, (n_heads + kBH - 1) / kBH);
  sparse_attn_bwd_kernel<<<grid, kBThreads, smem, st>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(kv), idx, ks, static_cast<const uint16_t*>(out),
      lse, static_cast<const uint16_t*>(dout), dq, dkv, n_kv, n_heads, topk, scale, status, status + 1);
  return cudaGetLastError();
}

}  // namespace dsa
