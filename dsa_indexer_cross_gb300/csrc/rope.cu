// RoPE pre-pass of the index heads and the per-row / per-group key-range plan.
//
// Index RoPE rotates the LAST `rope` dims of every index head ("GLM-5/5.1/5.2 DSA + LoRA
// enablement", indexer RoPE half-swap commit), pairing dim (d - r + i) with dim
// (d - r/2 + i).  cos/sin come from a float32 table evaluated in float64 on the host; the
// rotation runs in float32 and is rounded to bf16 (round-to-nearest-even), the precision
// the tensor-core contraction consumes.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Vector path: (d - rope) % 8 == 0 and (rope / 2) % 8 == 0.  One thread per unit of 8
// copied elements or of 8 rotated pairs.  Only dims [d0, d) are written, d0 = the start of
// the first 64-dim block holding rotary dims: the score kernel reads the blocks before it
// straight from the unrotated input.
__global__ void __launch_bounds__(256) rope_rows_vec(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                                                     const int32_t* __restrict__ pos, int64_t n_rows,
                                                     int rows_per_pos, int d, int rope, const float* __restrict__ cs,
                                                     int n_pos, uint32_t* status) {
  const int d0 = (d - rope) / 64 * 64;
  const int copy_units = (d - rope - d0) >> 3;
  const int half = rope >> 1;
  const int units = copy_units + (half >> 3);
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_rows * units) return;
  const int64_t row = gid / units;
  const int u = static_cast<int>(gid - row * units);
  const uint16_t* src = in + row * d;
  uint16_t* dst = out + row * d;
  if (u < copy_units) {
    *reinterpret_cast<uint4*>(dst + d0 + u * 8) = __ldg(reinterpret_cast<const uint4*>(src + d0 + u * 8));
    return;
  }
  const int i0 = (u - copy_units) * 8;
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(src + (d - rope) + i0));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(src + (d - half) + i0));
  const int p = __ldg(pos + row / rows_per_pos);
  if (p < 0 || p >= n_pos) {
    atomicOr(status, DEV_ERR_BAD_INDEX);
    *reinterpret_cast<uint4*>(dst + (d - rope) + i0) = a;
    *reinterpret_cast<uint4*>(dst + (d - half) + i0) = b;
    return;
  }
  const float4* t = reinterpret_cast<const float4*>(cs + (static_cast<int64_t>(p) * half + i0) * 2);
  float c[8], s[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = __ldg(t + q);
    c[2 * q] = v.x;
    s[2 * q] = v.y;
    c[2 * q + 1] = v.z;
    s[2 * q + 1] = v.w;
  }
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
  uint32_t ya[4], yb[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float x1l = bf_lo(av[q]), x1h = bf_hi(av[q]);
    const float x2l = bf_lo(bv[q]), x2h = bf_hi(bv[q]);
    const float cl = c[2 * q], sl = s[2 * q], ch = c[2 * q + 1], sh = s[2 * q + 1];
    ya[q] = pack_bf2(x1l * cl - x2l * sl, x1h * ch - x2h * sh);
    yb[q] = pack_bf2(x2l * cl + x1l * sl, x2h * ch + x1h * sh);
  }
  *reinterpret_cast<uint4*>(dst + (d - rope) + i0) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
  *reinterpret_cast<uint4*>(dst + (d - half) + i0) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
}

// Scalar path for any even rope: one thread per element of dims [d0, d - r/2) (d0 as above).
__global__ void __launch_bounds__(256) rope_rows_scalar(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                                                        const int32_t* __restrict__ pos, int64_t n_rows,
                                                        int rows_per_pos, int d, int rope,
                                                        const float* __restrict__ cs, int n_pos, uint32_t* status) {
  const int half = rope >> 1;
  const int d0 = (d - rope) / 64 * 64;
  const int per_row = d - half - d0;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_rows * per_row) return;
  const int64_t row = gid / per_row;
  const int e = d0 + static_cast<int>(gid - row * per_row);
  const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(in) + row * d;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out) + row * d;
  if (e < d - rope) {
    dst[e] = src[e];
    return;
  }
  const int i = e - (d - rope);
  const float x1 = __bfloat162float(src[d - rope + i]);
  const float x2 = __bfloat162float(src[d - half + i]);
  const int p = pos[row / rows_per_pos];
  if (p < 0 || p >= n_pos) {
    atomicOr(status, DEV_ERR_BAD_INDEX);
    dst[d - rope + i] = src[d - rope + i];
    dst[d - half + i] = src[d - half + i];
    return;
  }
  const float c = cs[(static_cast<int64_t>(p) * half + i) * 2];
  const float s = cs[(static_cast<int64_t>(p) * half + i) * 2 + 1];
  dst[d - rope + i] = __float2bfloat16_rn(x1 * c - x2 * s);
  dst[d - half + i] = __float2bfloat16_rn(x2 * c + x1 * s);
}

// One thread per row; blocks of 256 rows hold whole groups (group divides 256), and each
// group's union of non-trivial ranges is gathered with shared-memory atomics.
__global__ void __launch_bounds__(256) ranges_kernel(const int32_t* __restrict__ ks, const int32_t* __restrict__ ke,
                                                     int n_q, int group, int n_kv, int max_len, int trivial_len,
                                                     long long span_limit, int2* row_range, int2* group_range,
                                                     uint32_t* status) {
  __shared__ int s_lo[256], s_hi[256];
  const int per_block = 256 / group;
  if (static_cast<int>(threadIdx.x) < per_block) {
    s_lo[threadIdx.x] = 0x7FFFFFFF;
    s_hi[threadIdx.x] = 0;
  }
  __syncthreads();
  const int t = blockIdx.x * 256 + threadIdx.x;
  if (t < n_q) {
    const int a = ks ? __ldg(ks + t) : 0, b = __ldg(ke + t);
    int2 r = make_int2(0, 0);
    if (a < 0 || b < a || b > n_kv || b - a > max_len) {
      atomicOr(status, DEV_ERR_RANGE);
    } else if (b > a) {
      r = make_int2(a, b);
      if (b - a > trivial_len) {
        atomicMin(&s_lo[threadIdx.x / group], a);
        atomicMax(&s_hi[threadIdx.x / group], b);
      }
    }
    row_range[t] = r;
  }
  __syncthreads();
  const int g = blockIdx.x * per_block + static_cast<int>(threadIdx.x);
  if (static_cast<int>(threadIdx.x) < per_block && g * group < n_q) {
    const int lo = s_lo[threadIdx.x];
    int hi = s_hi[threadIdx.x];
    if (lo < hi && static_cast<long long>(hi) - lo > span_limit) {
      atomicOr(status, DEV_ERR_RANGE);   // rows of one group further apart than the plan covers
      hi = static_cast<int>(lo + span_limit);
    }
    group_range[g] = lo < hi ? make_int2(lo, hi) : make_int2(0, 0);
  }
}

// Transposed rotation on fp32 rows in place: one thread per rotated pair.
__global__ void __launch_bounds__(256) rope_rows_transpose_f32(float* __restrict__ x, const int32_t* __restrict__ pos,
                                                               int64_t n_rows, int rows_per_pos, int d, int rope,
                                                               const float* __restrict__ cs, int n_pos,
                                                               uint32_t* status) {
  const int half = rope >> 1;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_rows * half) return;
  const int64_t row = gid / half;
  const int i = static_cast<int>(gid - row * half);
  const int p = __ldg(pos + row / rows_per_pos);
  if (p < 0 || p >= n_pos) {
    atomicOr(status, DEV_ERR_BAD_INDEX);
    return;
  }
  const float c = __ldg(cs + (static_cast<int64_t>(p) * half + i) * 2);
  const float s = __ldg(cs + (static_cast<int64_t>(p) * half + i) * 2 + 1);
  float* r = x + row * d;
  const float a = r[d - rope + i], b = r[d - half + i];
  r[d - rope + i] = a * c + b * s;
  r[d - half + i] = b * c - a * s;
}

// Dense unit list, one block of 1024 threads: for every chunk c (outer) the groups whose
// range reaches into chunk c, last group first, compacted with a block scan; the list's tail,
// up to n_groups * n_chunks entries, holds (-1, -1).
__global__ void __launch_bounds__(1024) units_kernel(const int2* __restrict__ group_range, int n_groups, int n_chunks,
                                                     int chunk_len, int group, int n_q, int2* __restrict__ units,
                                                     uint32_t* __restrict__ cand_cnt, uint32_t* __restrict__ cand_edge) {
  __shared__ int wsum[32];
  __shared__ int base;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) base = 0;
  __syncthreads();
  for (int c = 0; c < n_chunks; ++c) {
    for (int g0 = 0; g0 < n_groups; g0 += 1024) {
      const int gi = g0 + tid;                  // position in "last group first" order
      const int g = n_groups - 1 - gi;
      int has = 0;
      if (gi < n_groups) {
        const int2 gr = group_range[g];
        const long long b = static_cast<long long>(gr.x) + static_cast<long long>(c) * chunk_len;
        has = b < gr.y ? 1 : 0;
        if (!has) {
          // an empty (group, chunk): its rows' counts and edges read as empty
          for (int r = 0; r < group; ++r) {
            const int t = g * group + r;
            if (t >= n_q) break;
            const size_t rc = static_cast<size_t>(t) * n_chunks + c;
            for (int q = 0; q < kSub; ++q) cand_cnt[rc * kSub + q] = 0u;
            cand_edge[rc] = 0u;
          }
        }
      }
      int x = has;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (lane == 31) wsum[w] = x;
      __syncthreads();
      int before = 0, all = 0;
      for (int i = 0; i < 32; ++i) {
        before += i < w ? wsum[i] : 0;
        all += wsum[i];
      }
      if (has) units[base + before + x - 1] = make_int2(g, c);
      __syncthreads();
      if (tid == 0) base += all;
      __syncthreads();
    }
  }
  const int total = n_groups * n_chunks;
  for (int i = base + tid; i < total; i += 1024) units[i] = make_int2(-1, -1);
}

}  // namespace

cudaError_t launch_rope_rows(const void* in, void* out, const int32_t* pos, int64_t n_rows, int rows_per_pos, int d,
                             int rope, const float* cs, int n_pos, uint32_t* status, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const int half = rope / 2;
  if ((d - rope) % 8 == 0 && half % 8 == 0) {
    const int64_t total = n_rows * ((d - rope) / 8 + half / 8);
    const int64_t blocks = (total + 255) / 256;
    rope_rows_vec<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint16_t*>(in),
                                                                 static_cast<uint16_t*>(out), pos, n_rows,
                                                                 rows_per_pos, d, rope, cs, n_pos, status);
  } else {
    const int64_t total = n_rows * (d - half);
    const int64_t blocks = (total + 255) / 256;
    rope_rows_scalar<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint16_t*>(in),
                                                                    static_cast<uint16_t*>(out), pos, n_rows,
                                                                    rows_per_pos, d, rope, cs, n_pos, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_ranges(const int32_t* ks, const int32_t* ke, int n_q, int group, int n_kv, int max_len,
                          int trivial_len, long long span_limit, int2* row_range, int2* group_range,
                          uint32_t* status, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  if (group < 1 || 256 % group != 0) return cudaErrorInvalidValue;
  ranges_kernel<<<(n_q + 255) / 256, 256, 0, st>>>(ks, ke, n_q, group, n_kv, max_len, trivial_len, span_limit, row_range,
                                                   group_range, status);
  return cudaGetLastError();
}

cudaError_t launch_rope_rows_transpose_f32(float* x, const int32_t* pos, int64_t n_rows, int rows_per_pos, int d,
                                           int rope, const float* cs, int n_pos, uint32_t* status, cudaStream_t st) {
  if (n_rows <= 0 || rope <= 0) return cudaSuccess;
  const int64_t total = n_rows * (rope / 2);
  rope_rows_transpose_f32<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(x, pos, n_rows, rows_per_pos, d,
                                                                                       rope, cs, n_pos, status);
  return cudaGetLastError();
}

cudaError_t launch_units(const int2* group_range, int n_groups, int n_chunks, int chunk_len, int group, int n_q,
                         int2* units, uint32_t* cand_cnt, uint32_t* cand_edge, cudaStream_t st) {
  if (n_groups <= 0 || n_chunks <= 0) return cudaSuccess;
  units_kernel<<<1, 1024, 0, st>>>(group_range, n_groups, n_chunks, chunk_len, group, n_q, units, cand_cnt, cand_edge);
  return cudaGetLastError();
}

}  // namespace dsa
