// Final exact top-k of every query row from the indexer's candidate buffers.
//
// Row t keeps k_t = min(topk, ke_t - ks_t) keys: the largest scores, ties to the lower key
// index.  They are written as offsets j - ks_t in ascending order, then -1 up to width topk
// ("GLM-5/5.1/5.2 DSA + LoRA enablement", commit capping top-k at the sequence length and
// padding back with -1).  Candidates are (order-preserving score key, absolute key index)
// pairs in kSub sub-buffers per (row, key chunk); together they hold a superset of the row's
// top-k.  Each chunk also carries an edge key with at least k of its entries at or above it,
// so nothing below the largest edge of the row can be selected.
//
// One block per row: the entries at or above the edge are gathered into shared memory (in any
// order), the exact threshold (v, cut) is found there -- one pass of 2048 bins linear in score,
// then the boundary bin's entries ranked directly, or radix passes when that bin is crowded --
// and the selected entries are sorted by key index (bitonic sort of <= 2048 pairs) for the
// ascending output.  Rows with more gathered entries than shared memory holds take the same
// steps over the buffers in global memory.
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kStage = 6144;        // candidates gathered into shared memory
constexpr int kBins = 2048;         // linear bins over the gathered [min, max] key range
constexpr int kBoundaryMax = 256;   // boundary-bin entries ranked directly; more -> radix passes
constexpr int kSortMax = 2048;      // topk <= 2048
constexpr int kMaxSeg = 64 * kSub;  // (chunk, sub-buffer) segments of a row

struct SelSmem {
  uint32_t key[kStage];
  int32_t idx[kStage];
  unsigned long long sel[kSortMax];   // (key index << 32) | score key of the selected entries
  uint32_t hist[kBins];
  uint32_t bkey[kBoundaryMax];
  int32_t bidx[kBoundaryMax];
  int seg_start[kMaxSeg + 1];
  int n_stage, n_sel, n_bound;
  uint32_t kmin, kmax, edge;
  int misc[4];
  int bc[4];
  int wsum[kSelThreads / 32];
};

// A slot of *counter for every active lane, one shared atomic per warp.
__device__ __forceinline__ int reserve_slot(int* counter) {
  const uint32_t m = __activemask();
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(m, base, leader);
  return base + __popc(m & ((1u << lane) - 1u));
}

// The (chunk, sub-buffer) segments of one row, in order.
struct Segs {
  const uint32_t* key;
  const int32_t* idx;
  int n_seg, cap4;
  size_t row_base;
  __device__ __forceinline__ size_t base(int s) const { return row_base + static_cast<size_t>(s) * cap4; }
};

// Calls f(key, idx) for every entry of every segment at or above `edge` (all threads, any order).
template <class F>
__device__ __forceinline__ void for_each_global(const Segs& S, const SelSmem& sm, uint32_t edge, F&& f) {
  for (int s = 0; s < S.n_seg; ++s) {
    const int n = sm.seg_start[s + 1] - sm.seg_start[s];
    const uint32_t* kp = S.key + S.base(s);
    const int32_t* ip = S.idx + S.base(s);
    for (int e0 = threadIdx.x; e0 < n; e0 += 4 * kSelThreads) {
      uint32_t kk[4];
      int32_t ii[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kSelThreads;
        kk[u] = e < n ? __ldg(kp + e) : 0u;
        ii[u] = e < n ? __ldg(ip + e) : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u * kSelThreads < n && kk[u] >= edge) f(kk[u], ii[u]);
    }
  }
}

// Exact threshold (v, cut) over the entries fe visits: exactly K satisfy topk_keep.  One
// histogram pass of 2048 bins linear in score over [kmin, kmax]; the boundary bin's entries
// (normally a handful) are ranked directly; a crowded boundary bin takes the radix passes.
template <class ForEach>
__device__ void block_threshold(const ForEach& fe, int K, uint32_t kmin, uint32_t kmax, SelSmem& sm, uint32_t& v,
                                uint32_t& cut) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < kBins; i += kSelThreads) sm.hist[i] = 0u;
  if (tid == 0) sm.n_bound = 0;
  __syncthreads();
  const float fmin = key_float(kmin), fmax = key_float(kmax);
  const float span = fmax - fmin;
  const float scale = span > 0.f && span < 3.0e38f ? static_cast<float>(kBins) / span : 0.f;
  auto bin_of = [&](uint32_t key) {
    const float y = (key_float(key) - fmin) * scale;
    return y >= static_cast<float>(kBins - 1) ? kBins - 1 : (y > 0.f ? static_cast<int>(y) : 0);
  };
  fe([&](uint32_t key, int32_t) { atomicAdd(&sm.hist[bin_of(key)], 1u); });
  __syncthreads();
  // thread tid owns the 8 bins [kBins - 8 tid - 8, kBins - 8 tid), visited from the top
  constexpr int kPerT = kBins / kSelThreads;
  int h[kPerT], sum = 0;
#pragma unroll
  for (int j = 0; j < kPerT; ++j) {
    h[j] = static_cast<int>(sm.hist[kBins - 1 - (tid * kPerT + j)]);
    sum += h[j];
  }
  int x = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sm.wsum[w] = x;
  __syncthreads();
  int c = x - sum;
  for (int i = 0; i < w; ++i) c += sm.wsum[i];
  if (c < K && K <= c + sum) {
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
      if (c < K && K <= c + h[j]) {
        sm.misc[0] = kBins - 1 - (tid * kPerT + j);
        sm.misc[1] = c;
        sm.misc[2] = h[j];
      }
      c += h[j];
    }
  }
  __syncthreads();
  const int b = sm.misc[0], above = sm.misc[1], hb = sm.misc[2];
  if (hb <= kBoundaryMax) {
    fe([&](uint32_t key, int32_t idx) {
      if (bin_of(key) == b) {
        const int slot = atomicAdd(&sm.n_bound, 1);
        sm.bkey[slot] = key;
        sm.bidx[slot] = idx;
      }
    });
    __syncthreads();
    const int need = K - above;   // 1 <= need <= hb
    for (int i = tid; i < hb; i += kSelThreads) {
      const uint32_t ki = sm.bkey[i];
      const int32_t ii = sm.bidx[i];
      int rank = 0;
      for (int j = 0; j < hb; ++j) rank += (sm.bkey[j] > ki || (sm.bkey[j] == ki && sm.bidx[j] < ii)) ? 1 : 0;
      if (rank == need - 1) {
        sm.misc[2] = static_cast<int>(ki);
        sm.misc[3] = ii;
      }
    }
    __syncthreads();
    v = static_cast<uint32_t>(sm.misc[2]);
    cut = static_cast<uint32_t>(sm.misc[3]);
    __syncthreads();
    return;
  }
  __syncthreads();
  radix_threshold<kSelThreads>([] { __syncthreads(); }, fe, tid, K, sm.hist, sm.bc, v, cut);
}

// Ascending bitonic sort of sm.sel[0, n) (n <= kSortMax), padded to a power of two.
__device__ void block_sort_sel(SelSmem& sm, int n) {
  int p = 1;
  while (p < n) p <<= 1;
  for (int i = n + threadIdx.x; i < p; i += kSelThreads) sm.sel[i] = ~0ull;
  __syncthreads();
  for (int size = 2; size <= p; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < p / 2; i += kSelThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const unsigned long long a = sm.sel[lo], c = sm.sel[hi];
        if ((a > c) == asc) {
          sm.sel[lo] = c;
          sm.sel[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(int n_chunks, int cap4, int topk, int trivial_len,
                                                             const int2* __restrict__ row_range,
                                                             const uint32_t* __restrict__ cand_edge,
                                                             const uint32_t* __restrict__ cand_key,
                                                             const int32_t* __restrict__ cand_idx,
                                                             const uint32_t* __restrict__ cand_cnt,
                                                             int32_t* __restrict__ idx_out, float* score_out,
                                                             uint32_t* status) {
  extern __shared__ __align__(16) uint8_t sel_smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(sel_smem_raw);
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int2 r = row_range[t];
  int32_t* out = idx_out + static_cast<size_t>(t) * topk;
  float* so = score_out ? score_out + static_cast<size_t>(t) * topk : nullptr;
  const int L = r.y - r.x;
  if (L <= trivial_len) {
    // the whole range is selected: offsets 0 .. L-1 in order, no candidates read.  The host
    // passes trivial_len = 0 whenever scores are requested, so only empty rows get here then.
    for (int i = tid; i < topk; i += kSelThreads) {
      out[i] = i < L ? i : -1;
      if (so) so[i] = -__int_as_float(0x7f800000);
    }
    return;
  }
  const int n_seg = n_chunks * kSub;
  if (tid == 0) {
    int s = 0;
    uint32_t e = 0u;
    for (int c = 0; c < n_chunks; ++c) {
      e = max(e, __ldg(cand_edge + static_cast<size_t>(t) * n_chunks + c));
      for (int q = 0; q < kSub; ++q) {
        sm.seg_start[c * kSub + q] = s;
        s += min(static_cast<int>(__ldg(cand_cnt + (static_cast<size_t>(t) * n_chunks + c) * kSub + q)), cap4);
      }
    }
    sm.seg_start[n_seg] = s;
    sm.edge = e;
    sm.n_stage = 0;
    sm.n_sel = 0;
    sm.kmin = 0xFFFFFFFFu;
    sm.kmax = 0u;
  }
  __syncthreads();
  const uint32_t edge = sm.edge;
  const Segs S{cand_key, cand_idx, n_seg, cap4, static_cast<size_t>(t) * n_seg * cap4};
  const int kt = min(topk, L);

  // gather the entries at or above the edge into shared memory, with their key range
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for_each_global(S, sm, edge, [&](uint32_t key, int32_t idx) {
    const int slot = reserve_slot(&sm.n_stage);
    if (slot < kStage) {
      sm.key[slot] = key;
      sm.idx[slot] = idx;
    }
    mn = min(mn, key);
    mx = max(mx, key);
  });
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((tid & 31) == 0) {
    atomicMin(&sm.kmin, mn);
    atomicMax(&sm.kmax, mx);
  }
  __syncthreads();
  const int n = sm.n_stage;
  const bool staged = n <= kStage;
  auto fe_stage = [&](auto&& f) {
    for (int e = tid; e < n; e += kSelThreads) f(sm.key[e], sm.idx[e]);
  };
  auto fe_global = [&](auto&& f) { for_each_global(S, sm, edge, f); };

  uint32_t v = 0, cut = 0x7FFFFFFFu;
  const bool all = n <= kt;
  if (!all) {
    if (staged) block_threshold(fe_stage, kt, sm.kmin, sm.kmax, sm, v, cut);
    else block_threshold(fe_global, kt, sm.kmin, sm.kmax, sm, v, cut);
  }
  // the selected entries, in any order, as (key index, score key) pairs
  auto take = [&](uint32_t key, int32_t idx) {
    if (all || topk_keep(key, idx, v, cut)) {
      const int slot = reserve_slot(&sm.n_sel);
      if (slot < kSortMax)
        sm.sel[slot] = (static_cast<unsigned long long>(static_cast<uint32_t>(idx)) << 32) | key;
    }
  };
  if (staged) fe_stage(take);
  else fe_global(take);
  __syncthreads();
  const int n_sel = min(sm.n_sel, kSortMax);
  if (tid == 0 && sm.n_sel != kt) atomicOr(status, DEV_ERR_OVERFLOW);
  block_sort_sel(sm, n_sel);
  for (int i = tid; i < topk; i += kSelThreads) {
    if (i < n_sel) {
      const unsigned long long e = sm.sel[i];
      out[i] = static_cast<int32_t>(e >> 32) - r.x;
      if (so) so[i] = key_float(static_cast<uint32_t>(e));
    } else {
      out[i] = -1;
      if (so) so[i] = -__int_as_float(0x7f800000);
    }
  }
}

}  // namespace

cudaError_t launch_select(int n_q, int n_chunks, int cap, int topk, int trivial_len, const int2* row_range,
                          const uint32_t* cand_edge, const uint32_t* cand_key, const int32_t* cand_idx,
                          const uint32_t* cand_cnt, int32_t* idx_out, float* score_out, uint32_t* status,
                          cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  if (n_chunks > kMaxSeg / kSub || topk > kSortMax || cap % kSub) return cudaErrorInvalidValue;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(SelSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  select_kernel<<<n_q, kSelThreads, sizeof(SelSmem), st>>>(n_chunks, cap / kSub, topk, trivial_len, row_range,
                                                          cand_edge, cand_key, cand_idx, cand_cnt, idx_out, score_out,
                                                          status);
  return cudaGetLastError();
}

}  // namespace dsa
