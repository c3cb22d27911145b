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
// One block per row.  When every row has at most 8192 keys, each gathered entry is stored at
// its offset in the row, the exact threshold (v, cut) is found over them and the kept offsets
// are written in order by a ballot compaction.  Otherwise the entries at or above the edge are
// gathered into shared memory (in any order), the threshold is found there -- one pass of 2048
// bins linear in score, then the boundary bin's entries ranked directly, or radix passes when
// that bin is crowded -- and the selected entries are put in key-index order by a counting
// pass over index buckets (at most 2048 buckets over the row; an entry's place is its bucket's
// start plus the number of smaller indices in its bucket).  Rows with more gathered entries
// than shared memory holds take the same steps over the buffers in global memory.  Block
// shapes: 256 threads and 4096 or 8192 score keys for short rows; 5120 staged entries and 256
// threads for single-chunk rows and where a row's buffers cannot hold more; else 10240 entries
// and 512 threads, or 24576 entries and 1024 threads when there are no more rows than SMs.
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int kBins = 2048;         // linear bins over the gathered [min, max] key range
constexpr int kBoundaryMax = 256;   // boundary-bin entries ranked directly; more -> radix passes
constexpr int kSortMax = 2048;      // topk <= 2048
constexpr int kMaxSeg = 64 * kSub;  // (chunk, sub-buffer) segments of a row
constexpr int kSmallStage = 5120, kSmallThreads = 256;
constexpr int kBigStage = 24576, kBigThreads = 512;
constexpr int kMidStage = 10240;   // 107 KB: two rows per SM
constexpr int kDenseKeys = 4096, kDenseThreads = 256;

template <int STAGE>
struct SelSmem {
  // staged entries; once the threshold is known, the region holds the bucketed selection
  // (kSortMax pairs) and the bucket fill counters
  uint32_t key[STAGE];
  int32_t idx[STAGE];
  unsigned long long sel[kSortMax];   // (key index << 32) | score key of the selected entries
  uint32_t hist[kBins];               // threshold bins, then index-bucket counts / starts
  uint32_t bkey[kBoundaryMax];
  int32_t bidx[kBoundaryMax];
  int seg_start[kMaxSeg + 1];
  int n_stage, n_sel, n_bound;
  uint32_t kmin, kmax, edge;
  int misc[4];
  int bc[4];
  int wsum[32];
};
static_assert(kSmallStage * 8 >= kSortMax * 8 + kBins * 4, "bucketed selection fits the stage region");

// Rows of at most KEYS keys: one score key per offset of the row, no staging or sort region.
template <int KEYS>
struct DenseSmem {
  uint32_t key[KEYS];
  uint32_t hist[kBins];
  uint32_t bkey[kBoundaryMax];
  int32_t bidx[kBoundaryMax];
  int seg_start[kMaxSeg + 1];
  int n_stage, n_sel, n_bound;
  uint32_t kmin, kmax, edge;
  int misc[4];
  int bc[4];
  int wsum[32];
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

// Exclusive prefix sum of x over the NT threads of the block (returns it; *total gets the sum).
// Every thread of the block calls it.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int x, int* wsum, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int y = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int z = __shfl_up_sync(0xffffffffu, y, off);
    if (lane >= off) y += z;
  }
  __syncthreads();   // wsum free for reuse
  if (lane == 31) wsum[w] = y;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    const int s = wsum[i];
    before += i < w ? s : 0;
    all += s;
  }
  *total = all;
  return before + y - x;
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
template <int NT, class Sm, class F>
__device__ __forceinline__ void for_each_global(const Segs& S, const Sm& sm, uint32_t edge, F&& f) {
  for (int s = 0; s < S.n_seg; ++s) {
    const int n = sm.seg_start[s + 1] - sm.seg_start[s];
    const uint32_t* kp = S.key + S.base(s);
    const int32_t* ip = S.idx + S.base(s);
    for (int e0 = threadIdx.x; e0 < n; e0 += 4 * NT) {
      uint32_t kk[4];
      int32_t ii[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * NT;
        kk[u] = e < n ? __ldg(kp + e) : 0u;
        ii[u] = e < n ? __ldg(ip + e) : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u * NT < n && kk[u] >= edge) f(kk[u], ii[u]);
    }
  }
}

// Exact threshold (v, cut) over the entries fe visits: exactly K satisfy topk_keep.  One
// histogram pass of 2048 bins linear in score over [kmin, kmax]; the boundary bin's entries
// (normally a handful) are ranked directly; a crowded boundary bin takes the radix passes.
template <int NT, class Sm, class ForEach>
__device__ void block_threshold(const ForEach& fe, int K, uint32_t kmin, uint32_t kmax, Sm& sm, uint32_t& v,
                                uint32_t& cut) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < kBins; i += NT) sm.hist[i] = 0u;
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
  // thread tid owns the kPerT bins [kBins - kPerT (tid + 1), kBins - kPerT tid), from the top
  constexpr int kPerT = kBins / NT;
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
    for (int i = tid; i < hb; i += NT) {
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
  radix_threshold<NT>([] { __syncthreads(); }, fe, tid, K, sm.hist, sm.bc, v, cut);
}

// Writes the n selected entries of sm.sel in ascending key index (offsets from rx; scores to
// so when given) into out[0, n), then -1 up to topk.  Key indices lie in [rx, rx + L); one
// outside (buffers the indexer never filled, after it stopped on an error) is flagged and put
// in the nearest bucket, so the writes stay in bounds.
template <int NT, int STAGE>
__device__ void block_write_ordered(SelSmem<STAGE>& sm, int n, int L, int rx, int topk, int32_t* out, float* so,
                                    uint32_t* status) {
  const int tid = threadIdx.x;
  unsigned long long* tmp = reinterpret_cast<unsigned long long*>(sm.key);   // kSortMax bucketed pairs
  uint32_t* fill = reinterpret_cast<uint32_t*>(tmp + kSortMax);              // kBins fill counters
  int sh = 0;
  while (((L - 1) >> sh) >= kBins) ++sh;   // bucket of offset o: o >> sh < kBins
  auto bucket = [&](int j) {
    const int o = j - rx;
    if (o < 0 || o >= L) {
      atomicOr(status, DEV_ERR_BAD_INDEX);
      return o < 0 ? 0 : (L - 1) >> sh;
    }
    return o >> sh;
  };
  for (int i = tid; i < kBins; i += NT) {
    sm.hist[i] = 0u;
    fill[i] = 0u;
  }
  __syncthreads();
  for (int e = tid; e < n; e += NT) atomicAdd(&sm.hist[bucket(static_cast<int>(sm.sel[e] >> 32))], 1u);
  __syncthreads();
  // exclusive scan of the bucket counts in place: thread tid owns kPerT consecutive buckets
  constexpr int kPerT = kBins / NT;
  int h[kPerT], sum = 0;
#pragma unroll
  for (int j = 0; j < kPerT; ++j) {
    h[j] = static_cast<int>(sm.hist[tid * kPerT + j]);
    sum += h[j];
  }
  int total = 0;
  int c = block_exclusive_scan<NT>(sum, sm.wsum, &total);
#pragma unroll
  for (int j = 0; j < kPerT; ++j) {
    sm.hist[tid * kPerT + j] = static_cast<uint32_t>(c);
    c += h[j];
  }
  __syncthreads();
  for (int e = tid; e < n; e += NT) {
    const unsigned long long x = sm.sel[e];
    const int b = bucket(static_cast<int>(x >> 32));
    tmp[sm.hist[b] + atomicAdd(&fill[b], 1u)] = x;
  }
  __syncthreads();
  for (int p = tid; p < n; p += NT) {
    const unsigned long long x = tmp[p];
    const int j = static_cast<int>(x >> 32);
    const int b = bucket(j);
    const int lo = static_cast<int>(sm.hist[b]), m = static_cast<int>(fill[b]);
    int rank = lo;
    for (int q = lo; q < lo + m; ++q) rank += static_cast<int>(tmp[q] >> 32) < j ? 1 : 0;
    out[rank] = j - rx;
    if (so) so[rank] = key_float(static_cast<uint32_t>(x));
  }
  for (int i = n + tid; i < topk; i += NT) {
    out[i] = -1;
    if (so) so[i] = -__int_as_float(0x7f800000);
  }
}

// A row of at most KEYS keys.  Every gathered entry goes to its own offset in the row (0 marks
// an offset without an entry; a real key of 0 -- the all-ones NaN pattern -- is stored as 1),
// the exact threshold is found over the present offsets, and the selection is written in
// offset order by a ballot compaction: warp w walks its own contiguous span of offsets twice,
// once to count its kept entries, once to write them after the earlier warps'.
template <int NT, int KEYS>
__device__ void dense_row(const Segs& S, DenseSmem<KEYS>& sm, uint32_t edge, int L, int rx, int kt, int topk,
                          int32_t* out, float* so, uint32_t* status) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  uint32_t* dk = sm.key;
  for (int o = tid; o < L; o += NT) dk[o] = 0u;
  __syncthreads();
  int cnt = 0;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for_each_global<NT>(S, sm, edge, [&](uint32_t key, int32_t idx) {
    const int o = idx - rx;
    if (o < 0 || o >= L) {
      atomicOr(status, DEV_ERR_BAD_INDEX);
      return;
    }
    const uint32_t k1 = key ? key : 1u;
    dk[o] = k1;
    ++cnt;
    mn = min(mn, k1);
    mx = max(mx, k1);
  });
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    atomicAdd(&sm.n_stage, cnt);
    atomicMin(&sm.kmin, mn);
    atomicMax(&sm.kmax, mx);
  }
  __syncthreads();
  const bool all = sm.n_stage <= kt;
  uint32_t v = 0, cut = 0x7FFFFFFFu;
  if (!all) {
    auto fe = [&](auto&& f) {
      for (int o = tid; o < L; o += NT) {
        const uint32_t k = dk[o];
        if (k) f(k, rx + o);
      }
    };
    block_threshold<NT>(fe, kt, sm.kmin, sm.kmax, sm, v, cut);
  }
  const int span = ((L + NW - 1) / NW + 31) & ~31;
  const int o0 = w * span, o1 = min(L, o0 + span);
  auto keep = [&](int o) {
    const uint32_t k = o < o1 ? dk[o] : 0u;
    return k != 0u && (all || topk_keep(k, rx + o, v, cut));
  };
  int c = 0;
  for (int b = o0; b < o1; b += 32) c += __popc(__ballot_sync(0xffffffffu, keep(b + lane)));
  __syncthreads();
  if (lane == 0) sm.wsum[w] = c;
  __syncthreads();
  int pre = 0, total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int s = sm.wsum[i];
    pre += i < w ? s : 0;
    total += s;
  }
  for (int b = o0; b < o1; b += 32) {
    const int o = b + lane;
    const bool kp = keep(o);
    const uint32_t m = __ballot_sync(0xffffffffu, kp);
    const int pos = pre + __popc(m & ((1u << lane) - 1u));
    if (kp && pos < topk) {
      out[pos] = o;
      if (so) so[pos] = key_float(dk[o]);
    }
    pre += __popc(m);
  }
  for (int i = total + tid; i < topk; i += NT) {
    out[i] = -1;
    if (so) so[i] = -__int_as_float(0x7f800000);
  }
  if (tid == 0 && total != kt) atomicOr(status, DEV_ERR_OVERFLOW);
}

// A row gathered as (key, index) entries: staged in shared memory when they fit, else read
// from the buffers in global memory on every pass; threshold, then index-bucket ordering.
template <int NT, int STAGE>
__device__ void select_sparse(const Segs& S, SelSmem<STAGE>& sm, uint32_t edge, int L, int rx, int kt, int topk,
                              int32_t* out, float* so, uint32_t* status) {
  const int tid = threadIdx.x;
  // gather the entries at or above the edge into shared memory, with their key range
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for_each_global<NT>(S, sm, edge, [&](uint32_t key, int32_t idx) {
    const int slot = reserve_slot(&sm.n_stage);
    if (slot < STAGE) {
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
  const bool staged = n <= STAGE;
  auto fe_stage = [&](auto&& f) {
    for (int e = tid; e < n; e += NT) f(sm.key[e], sm.idx[e]);
  };
  auto fe_global = [&](auto&& f) { for_each_global<NT>(S, sm, edge, f); };

  uint32_t v = 0, cut = 0x7FFFFFFFu;
  const bool all = n <= kt;
  if (!all) {
    if (staged) block_threshold<NT>(fe_stage, kt, sm.kmin, sm.kmax, sm, v, cut);
    else block_threshold<NT>(fe_global, kt, sm.kmin, sm.kmax, sm, v, cut);
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
  block_write_ordered<NT>(sm, n_sel, L, rx, topk, out, so, status);
}

// One row per block.  SM: SelSmem<STAGE> (any row) or DenseSmem<KEYS> (DENSE: rows of at most
// KEYS keys, which the host guarantees by choosing this shape only when max_len <= KEYS).
template <class SM, int NT, bool DENSE>
__device__ __forceinline__ void select_row(int n_chunks, int cap4, int topk, int trivial_len,
                                           const int2* __restrict__ row_range, const uint32_t* __restrict__ cand_edge,
                                           const uint32_t* __restrict__ cand_key, const int32_t* __restrict__ cand_idx,
                                           const uint32_t* __restrict__ cand_cnt, int32_t* __restrict__ idx_out,
                                           float* score_out, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t sel_smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(sel_smem_raw);
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int2 r = row_range[t];
  int32_t* out = idx_out + static_cast<size_t>(t) * topk;
  float* so = score_out ? score_out + static_cast<size_t>(t) * topk : nullptr;
  const int L = r.y - r.x;
  if (L <= trivial_len) {
    // the whole range is selected: offsets 0 .. L-1 in order, no candidates read.  The host
    // passes trivial_len = 0 whenever scores are requested, so only empty rows get here then.
    for (int i = tid; i < topk; i += NT) {
      out[i] = i < L ? i : -1;
      if (so) so[i] = -__int_as_float(0x7f800000);
    }
    return;
  }
  const int n_seg = n_chunks * kSub;
  if (tid == 0) {
    sm.edge = 0u;
    sm.n_stage = 0;
    sm.n_sel = 0;
    sm.kmin = 0xFFFFFFFFu;
    sm.kmax = 0u;
  }
  __syncthreads();
  // segment starts (one thread per segment) and the row's edge (largest chunk edge)
  const int cnt_s =
      tid < n_seg ? static_cast<int>(min(__ldg(cand_cnt + static_cast<size_t>(t) * n_seg + tid), static_cast<uint32_t>(cap4)))
                  : 0;
  if (tid < n_chunks) atomicMax(&sm.edge, __ldg(cand_edge + static_cast<size_t>(t) * n_chunks + tid));
  int n_all = 0;
  const int start_s = block_exclusive_scan<NT>(cnt_s, sm.wsum, &n_all);
  if (tid < n_seg) sm.seg_start[tid] = start_s;
  if (tid == 0) sm.seg_start[n_seg] = n_all;
  __syncthreads();
  const uint32_t edge = sm.edge;
  const Segs S{cand_key, cand_idx, n_seg, cap4, static_cast<size_t>(t) * n_seg * cap4};
  const int kt = min(topk, L);
  if constexpr (DENSE) {
    if (L <= static_cast<int>(sizeof(sm.key) / sizeof(sm.key[0]))) {
      dense_row<NT>(S, sm, edge, L, r.x, kt, topk, out, so, status);
    } else {
      if (tid == 0) atomicOr(status, DEV_ERR_RANGE);
      for (int i = tid; i < topk; i += NT) {
        out[i] = -1;
        if (so) so[i] = -__int_as_float(0x7f800000);
      }
    }
  } else {
    select_sparse<NT>(S, sm, edge, L, r.x, kt, topk, out, so, status);
  }
}

#define DSA_SEL_PARAMS                                                                                        \
  int n_chunks, int cap4, int topk, int trivial_len, const int2 *__restrict__ row_range,                     \
      const uint32_t *__restrict__ cand_edge, const uint32_t *__restrict__ cand_key,                         \
      const int32_t *__restrict__ cand_idx, const uint32_t *__restrict__ cand_cnt, int32_t *__restrict__ idx_out, \
      float *score_out, uint32_t *status
#define DSA_SEL_FWD \
  n_chunks, cap4, topk, trivial_len, row_range, cand_edge, cand_key, cand_idx, cand_cnt, idx_out, score_out, status

template <class SM, int NT>
__global__ void __launch_bounds__(NT) select_kernel(DSA_SEL_PARAMS) {
  select_row<SM, NT, false>(DSA_SEL_FWD);
}
// six short rows an SM (40 registers a thread)
template <class SM, int NT>
__global__ void __launch_bounds__(NT, 6) select_dense_kernel(DSA_SEL_PARAMS) {
  select_row<SM, NT, true>(DSA_SEL_FWD);
}
#undef DSA_SEL_PARAMS
#undef DSA_SEL_FWD

template <class SM, int NT, bool DENSE>
cudaError_t launch_shape(int n_q, int n_chunks, int cap, int topk, int trivial_len, const int2* row_range,
                         const uint32_t* cand_edge, const uint32_t* cand_key, const int32_t* cand_idx,
                         const uint32_t* cand_cnt, int32_t* idx_out, float* score_out, uint32_t* status,
                         cudaStream_t st) {
  auto kern = [] {
    if constexpr (DENSE) return select_dense_kernel<SM, NT>;
    else return select_kernel<SM, NT>;
  }();
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(SM));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  kern<<<n_q, NT, sizeof(SM), st>>>(n_chunks, cap / kSub, topk, trivial_len, row_range, cand_edge, cand_key, cand_idx,
                                    cand_cnt, idx_out, score_out, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(int n_q, int n_chunks, int cap, int topk, int trivial_len, int max_len, const int2* row_range,
                          const uint32_t* cand_edge, const uint32_t* cand_key, const int32_t* cand_idx,
                          const uint32_t* cand_cnt, int32_t* idx_out, float* score_out, uint32_t* status,
                          cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  if (n_chunks > kMaxSeg / kSub || topk > kSortMax || cap % kSub) return cudaErrorInvalidValue;
#define DSA_SEL_ARGS                                                                                          \
  n_q, n_chunks, cap, topk, trivial_len, row_range, cand_edge, cand_key, cand_idx, cand_cnt, idx_out, score_out, \
      status, st
  // short rows (prefill of a few thousand keys): one score key per offset, 27 or 43 KB a row,
  // so six to eight rows share an SM
  if (max_len <= kDenseKeys) return launch_shape<DenseSmem<kDenseKeys>, kDenseThreads, true>(DSA_SEL_ARGS);
  if (max_len <= 2 * kDenseKeys) return launch_shape<DenseSmem<2 * kDenseKeys>, kDenseThreads, true>(DSA_SEL_ARGS);
  // the small shape (68 KB: three CTAs per SM) when a row's buffers cannot hold more than its stage, or
  // when a row has one chunk: the indexer leaves a filtered row's chunk compacted to its
  // entries at or above the final threshold (about k + a bin of them); a row that still
  // gathers more takes the global path
  if (static_cast<long long>(n_chunks) * cap <= kSmallStage || n_chunks == 1)
    return launch_shape<SelSmem<kSmallStage>, kSmallThreads, false>(DSA_SEL_ARGS);
  // few rows (decode): one CTA per row leaves most SMs idle, so each row gets 1024 threads
  if (n_q <= device_sm_count()) return launch_shape<SelSmem<kBigStage>, 2 * kBigThreads, false>(DSA_SEL_ARGS);
  // many multi-chunk rows (chunk_1m): the entries at or above the row's edge (the largest of its
  // chunks' edges) number a few k, so two rows share an SM
  return launch_shape<SelSmem<kMidStage>, kBigThreads, false>(DSA_SEL_ARGS);
#undef DSA_SEL_ARGS
}

}  // namespace dsa
