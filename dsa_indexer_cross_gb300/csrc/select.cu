// Final exact top-k of every query row from the indexer's per-chunk candidate buffers.
//
// Row t keeps k_t = min(topk, ke_t - ks_t) keys: the largest scores, ties to the lower key
// index.  They are written as offsets j - ks_t in ascending order, then -1 up to width
// topk ("GLM-5/5.1/5.2 DSA + LoRA enablement", commit capping top-k at the sequence length
// and padding back with -1).  Candidates are (order-preserving score key, absolute key
// index) pairs; every chunk buffer holds a superset of that chunk's top-k.
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kMaxTopk = 2048;

__global__ void __launch_bounds__(kSelThreads) select_kernel(int n_chunks, int cap, int topk,
                                                             const int2* __restrict__ row_range,
                                                             const uint32_t* __restrict__ cand_key,
                                                             const int32_t* __restrict__ cand_idx,
                                                             const uint32_t* __restrict__ cand_cnt,
                                                             int32_t* __restrict__ idx_out, float* score_out,
                                                             uint32_t* status) {
  __shared__ uint32_t hist[256];
  __shared__ int bc[4];
  __shared__ int sel_n;
  __shared__ int32_t sel_idx[kMaxTopk];
  __shared__ uint32_t sel_key[kMaxTopk];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int2 r = row_range[t];
  int kt = min(topk, r.y - r.x);
  const size_t base = static_cast<size_t>(t) * n_chunks * cap;
  const uint32_t* cnt_row = cand_cnt + static_cast<size_t>(t) * n_chunks;
  int total = 0;
  for (int c = 0; c < n_chunks; ++c) total += min(static_cast<int>(cnt_row[c]), cap);
  if (total < kt) {
    if (tid == 0) atomicOr(status, DEV_ERR_OVERFLOW);
    kt = total;
  }
  auto fe = [&](auto&& f) {
    for (int c = 0; c < n_chunks; ++c) {
      const int n = min(static_cast<int>(cnt_row[c]), cap);
      const uint32_t* kp = cand_key + base + static_cast<size_t>(c) * cap;
      const int32_t* ip = cand_idx + base + static_cast<size_t>(c) * cap;
      for (int e = tid; e < n; e += kSelThreads) f(__ldg(kp + e), __ldg(ip + e));
    }
  };
  uint32_t v = 0, cut = 0x7FFFFFFFu;
  const bool take_all = total <= kt;
  if (kt > 0 && !take_all) {
    radix_threshold<kSelThreads>([] { __syncthreads(); }, fe, tid, kt, hist, bc, v, cut);
  }
  if (tid == 0) sel_n = 0;
  __syncthreads();
  if (kt > 0) {
    fe([&](uint32_t key, int32_t idx) {
      if (take_all || topk_keep(key, idx, v, cut)) {
        const int p = atomicAdd(&sel_n, 1);
        if (p < kMaxTopk) {
          sel_idx[p] = idx;
          sel_key[p] = key;
        }
      }
    });
  }
  __syncthreads();
  const int n = min(sel_n, kMaxTopk);
  if (tid == 0 && n != kt) atomicOr(status, DEV_ERR_OVERFLOW);
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + tid; i < P; i += kSelThreads) {
    sel_idx[i] = 0x7FFFFFFF;
    sel_key[i] = 0;
  }
  __syncthreads();
  // bitonic sort by key index, ascending
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += kSelThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool asc = (i & k) == 0;
          const int32_t a = sel_idx[i], b = sel_idx[ixj];
          if ((a > b) == asc) {
            sel_idx[i] = b;
            sel_idx[ixj] = a;
            const uint32_t ka = sel_key[i];
            sel_key[i] = sel_key[ixj];
            sel_key[ixj] = ka;
          }
        }
      }
      __syncthreads();
    }
  }
  int32_t* out = idx_out + static_cast<size_t>(t) * topk;
  for (int i = tid; i < topk; i += kSelThreads) out[i] = i < n ? sel_idx[i] - r.x : -1;
  if (score_out) {
    float* so = score_out + static_cast<size_t>(t) * topk;
    for (int i = tid; i < topk; i += kSelThreads) so[i] = i < n ? key_float(sel_key[i]) : -__int_as_float(0x7f800000);
  }
}

}  // namespace

cudaError_t launch_select(int n_q, int n_chunks, int cap, int topk, const int2* row_range, const uint32_t* cand_key,
                          const int32_t* cand_idx, const uint32_t* cand_cnt, int32_t* idx_out, float* score_out,
                          uint32_t* status, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  if (topk > kMaxTopk) return cudaErrorInvalidValue;
  select_kernel<<<n_q, kSelThreads, 0, st>>>(n_chunks, cap, topk, row_range, cand_key, cand_idx, cand_cnt, idx_out,
                                            score_out, status);
  return cudaGetLastError();
}

}  // namespace dsa
