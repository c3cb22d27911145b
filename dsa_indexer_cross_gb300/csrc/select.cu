// Final exact top-k of every query row from the indexer's per-chunk candidate buffers.
//
// Row t keeps k_t = min(topk, ke_t - ks_t) keys: the largest scores, ties to the lower key
// index.  They are written as offsets j - ks_t in ascending order, then -1 up to width topk
// ("GLM-5/5.1/5.2 DSA + LoRA enablement", commit capping top-k at the sequence length and
// padding back with -1).  Candidates are (order-preserving score key, absolute key index)
// pairs; every chunk buffer holds a superset of that chunk's top-k and is already sorted by
// key index (the indexer appends in key order and cuts back stably), and chunks cover
// increasing key ranges, so the concatenated list is sorted and a stable compaction of the
// selected entries is the sorted output.
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kBins = 2048;         // linear bins over the row's [min, max] key range
constexpr int kBoundaryMax = 256;   // boundary-bin entries ranked directly; more -> radix passes
constexpr int kSelPer = 17;    // entries per thread kept in registers (rows up to 4352 candidates)
constexpr int kMaxChunks = 64;

// Exact top-K threshold in one histogram pass for rows whose scores are spread out: 2048
// bins linear in score over [min, max] locate the bin holding the K-th entry, and the entries
// of that bin (normally a handful) are ranked directly by (key desc, index asc).  Returns
// false, before touching (v, cut), when that bin holds more than kBoundaryMax entries (many
// equal or nearly equal scores); the caller then runs the radix passes.  Same contract as
// radix_threshold: exactly K entries satisfy key > v || (key == v && idx <= cut).
struct LinearSmem {
  uint32_t hist[kBins];
  uint32_t bkey[kBoundaryMax];
  int32_t bidx[kBoundaryMax];
  uint32_t wmin[kSelThreads / 32], wmax[kSelThreads / 32];
  int wsum[kSelThreads / 32];
  int misc[8];
};

template <class ForEach>
__device__ bool linear_threshold(const ForEach& fe, int tid, int K, LinearSmem& L, uint32_t& v, uint32_t& cut) {
  const int lane = tid & 31, w = tid >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  fe([&](uint32_t key, int32_t) {
    mn = min(mn, key);
    mx = max(mx, key);
  });
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    L.wmin[w] = mn;
    L.wmax[w] = mx;
  }
  for (int i = tid; i < kBins; i += kSelThreads) L.hist[i] = 0u;
  if (tid == 0) L.misc[3] = 0;
  __syncthreads();
  uint32_t kmin = L.wmin[0], kmax = L.wmax[0];
#pragma unroll
  for (int i = 1; i < kSelThreads / 32; ++i) {
    kmin = min(kmin, L.wmin[i]);
    kmax = max(kmax, L.wmax[i]);
  }
  // bins are linear in score value (keys are log-spaced); (f - fmin) * scale is monotone
  // non-decreasing in f under round-to-nearest, so a higher bin never holds a smaller score
  const float fmin = key_float(kmin), fmax = key_float(kmax);
  const float span = fmax - fmin;
  const float scale = span > 0.f && span < 3.0e38f ? static_cast<float>(kBins) / span : 0.f;
  auto bin_of = [&](uint32_t key) {
    const float y = (key_float(key) - fmin) * scale;
    return y >= static_cast<float>(kBins - 1) ? kBins - 1 : (y > 0.f ? static_cast<int>(y) : 0);
  };
  fe([&](uint32_t key, int32_t) { atomicAdd(&L.hist[bin_of(key)], 1u); });
  __syncthreads();
  // thread tid owns the 8 bins [kBins - 8 tid - 8, kBins - 8 tid), visited from the top
  constexpr int kPerT = kBins / kSelThreads;
  int h[kPerT], sum = 0;
#pragma unroll
  for (int j = 0; j < kPerT; ++j) {
    h[j] = static_cast<int>(L.hist[kBins - 1 - (tid * kPerT + j)]);
    sum += h[j];
  }
  int x = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) L.wsum[w] = x;
  __syncthreads();
  int c = x - sum;
  for (int i = 0; i < w; ++i) c += L.wsum[i];
  if (c < K && K <= c + sum) {
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
      if (c < K && K <= c + h[j]) {
        L.misc[0] = kBins - 1 - (tid * kPerT + j);
        L.misc[1] = c;
        L.misc[2] = h[j];
      }
      c += h[j];
    }
  }
  __syncthreads();
  const int b = L.misc[0], above = L.misc[1], hb = L.misc[2];
  if (hb > kBoundaryMax) return false;
  fe([&](uint32_t key, int32_t idx) {
    if (bin_of(key) == b) {
      const int slot = atomicAdd(&L.misc[3], 1);
      L.bkey[slot] = key;
      L.bidx[slot] = idx;
    }
  });
  __syncthreads();
  const int need = K - above;   // 1 <= need <= hb
  for (int i = tid; i < hb; i += kSelThreads) {
    const uint32_t ki = L.bkey[i];
    const int32_t ii = L.bidx[i];
    int rank = 0;
    for (int j = 0; j < hb; ++j) rank += (L.bkey[j] > ki || (L.bkey[j] == ki && L.bidx[j] < ii)) ? 1 : 0;
    if (rank == need - 1) {
      L.misc[4] = static_cast<int>(ki);
      L.misc[5] = ii;
    }
  }
  __syncthreads();
  v = static_cast<uint32_t>(L.misc[4]);
  cut = static_cast<uint32_t>(L.misc[5]);
  return true;
}

template <bool kRegs>
__global__ void __launch_bounds__(kSelThreads) select_kernel(int n_chunks, int cap, int topk, int trivial_len,
                                                             const int2* __restrict__ row_range,
                                                             const uint32_t* __restrict__ cand_edge,
                                                             const uint32_t* __restrict__ cand_key,
                                                             const int32_t* __restrict__ cand_idx,
                                                             const uint32_t* __restrict__ cand_cnt,
                                                             int32_t* __restrict__ idx_out, float* score_out,
                                                             uint32_t* status) {
  __shared__ uint32_t hist[256];
  __shared__ int bc[4];
  __shared__ int start[kMaxChunks + 1];
  __shared__ int warp_tot[2][kSelThreads / 32];
  __shared__ LinearSmem lin;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int2 r = row_range[t];
  if (r.y - r.x <= trivial_len) {
    // the whole range is selected: offsets 0 .. L-1 in order, no candidates read.  The host
    // passes trivial_len = 0 whenever scores are requested, so only empty rows get here then.
    int32_t* out = idx_out + static_cast<size_t>(t) * topk;
    float* so = score_out ? score_out + static_cast<size_t>(t) * topk : nullptr;
    const int L = r.y - r.x;
    for (int i = tid; i < topk; i += kSelThreads) {
      out[i] = i < L ? i : -1;
      if (so) so[i] = -__int_as_float(0x7f800000);
    }
    return;
  }
  const size_t base = static_cast<size_t>(t) * n_chunks * cap;
  const uint32_t* cnt_row = cand_cnt + static_cast<size_t>(t) * n_chunks;
  __shared__ uint32_t s_edge;
  if (tid == 0) {
    int s = 0;
    uint32_t e = 0u;
    for (int c = 0; c < n_chunks; ++c) {
      start[c] = s;
      s += min(static_cast<int>(cnt_row[c]), cap);
      e = max(e, __ldg(cand_edge + static_cast<size_t>(t) * n_chunks + c));
    }
    start[n_chunks] = s;
    s_edge = e;
  }
  __syncthreads();
  // a chunk's edge has at least k of that chunk's entries at or above it, so nothing below the
  // largest edge can be in the row's top-k: the threshold passes skip those entries
  const uint32_t edge = s_edge;
  const int total = start[n_chunks];
  int kt = min(topk, r.y - r.x);
  if (total < kt) {
    if (tid == 0) atomicOr(status, DEV_ERR_OVERFLOW);
    kt = total;
  }
  int32_t* out = idx_out + static_cast<size_t>(t) * topk;
  float* so = score_out ? score_out + static_cast<size_t>(t) * topk : nullptr;
  auto finish = [&](int n_sel) {
    if (tid == 0 && n_sel != kt) atomicOr(status, DEV_ERR_OVERFLOW);
    for (int i = n_sel + tid; i < topk; i += kSelThreads) {
      out[i] = -1;
      if (so) so[i] = -__int_as_float(0x7f800000);
    }
  };
  const bool take_all = total <= kt;
  uint32_t v = 0, cut = 0x7FFFFFFFu;
  if constexpr (kRegs) {
    // Up to kSelPer entries per thread, held in registers: thread tid owns the contiguous list
    // positions [p0, p1), so a block scan of per-thread counts gives the stable order.
    const int per = (total + kSelThreads - 1) / kSelThreads;
    const int p0 = min(total, tid * per), p1 = min(total, p0 + per);
    uint32_t rk[kSelPer];
    int32_t ri[kSelPer];
#pragma unroll
    for (int i = 0; i < kSelPer; ++i) {
      if (p0 + i < p1) {
        int c = 0;
        while (p0 + i >= start[c + 1]) ++c;
        const size_t o = base + static_cast<size_t>(c) * cap + (p0 + i - start[c]);
        rk[i] = __ldg(cand_key + o);
        ri[i] = __ldg(cand_idx + o);
      }
    }
    auto fe = [&](auto&& f) {
#pragma unroll
      for (int i = 0; i < kSelPer; ++i)
        if (p0 + i < p1 && rk[i] >= edge) f(rk[i], ri[i]);
    };
    if (kt > 0 && !take_all && !linear_threshold(fe, tid, kt, lin, v, cut)) {
      __syncthreads();
      radix_threshold<kSelThreads>([] { __syncthreads(); }, fe, tid, kt, hist, bc, v, cut);
    }
    int keep = 0;
    fe([&](uint32_t key, int32_t idx) { keep += (take_all || topk_keep(key, idx, v, cut)) ? 1 : 0; });
    int x = keep;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[0][wid] = x;
    __syncthreads();
    int pos = x - keep;
    for (int w = 0; w < wid; ++w) pos += warp_tot[0][w];
    fe([&](uint32_t key, int32_t idx) {
      if (take_all || topk_keep(key, idx, v, cut)) {
        if (pos < topk) {
          out[pos] = idx - r.x;
          if (so) so[pos] = key_float(key);
        }
        ++pos;
      }
    });
    int n_sel = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) n_sel += warp_tot[0][w];
    finish(n_sel);
  } else {
    // Larger rows stay in the buffers (L2).  The threshold passes only need every entry
    // once, in any order: thread tid reads positions tid, tid + 256, ... chunk by chunk, with
    // four loads in flight.
    auto fe = [&](auto&& f) {
      for (int c = 0; c < n_chunks; ++c) {
        const int n = start[c + 1] - start[c];
        const uint32_t* kp = cand_key + base + static_cast<size_t>(c) * cap;
        const int32_t* ip = cand_idx + base + static_cast<size_t>(c) * cap;
        for (int e0 = tid; e0 < n; e0 += 4 * kSelThreads) {
          uint32_t kk[4];
          int32_t ii[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kSelThreads;
            if (e < n) {
              kk[u] = __ldg(kp + e);
              ii[u] = __ldg(ip + e);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (e0 + u * kSelThreads < n && kk[u] >= edge) f(kk[u], ii[u]);
        }
      }
    };
    if (kt > 0 && !take_all && !linear_threshold(fe, tid, kt, lin, v, cut)) {
      __syncthreads();
      radix_threshold<kSelThreads>([] { __syncthreads(); }, fe, tid, kt, hist, bc, v, cut);
    }
    // Stable compaction in list order, in rounds of 1024 entries of one chunk: thread tid
    // takes the four consecutive entries 4 tid .. 4 tid + 3 of the round (one 16-byte load
    // each of keys and indices when all four exist), and a block scan of the per-thread
    // counts places them.  The warp totals alternate between two arrays, so one barrier
    // per round suffices.
    int written = 0, round = 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int n = start[c + 1] - start[c];
      const uint32_t* kp = cand_key + base + static_cast<size_t>(c) * cap;
      const int32_t* ip = cand_idx + base + static_cast<size_t>(c) * cap;
      for (int r0 = 0; r0 < n; r0 += 4 * kSelThreads, ++round) {
        const int e = r0 + 4 * tid;
        uint32_t kk[4] = {0u, 0u, 0u, 0u};
        int32_t ii[4] = {0, 0, 0, 0};
        if (e + 3 < n) {
          const uint4 k4 = __ldg(reinterpret_cast<const uint4*>(kp + e));
          const int4 i4 = __ldg(reinterpret_cast<const int4*>(ip + e));
          kk[0] = k4.x; kk[1] = k4.y; kk[2] = k4.z; kk[3] = k4.w;
          ii[0] = i4.x; ii[1] = i4.y; ii[2] = i4.z; ii[3] = i4.w;
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (e + u < n) {
              kk[u] = __ldg(kp + e + u);
              ii[u] = __ldg(ip + e + u);
            }
        }
        bool kf[4];
        int keep = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          kf[u] = e + u < n && (take_all || topk_keep(kk[u], ii[u], v, cut));
          keep += kf[u] ? 1 : 0;
        }
        int x = keep;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, off);
          if (lane >= off) x += y;
        }
        const int par = round & 1;
        if (lane == 31) warp_tot[par][wid] = x;
        __syncthreads();
        int pos = written + x - keep, tot = 0;
#pragma unroll
        for (int w = 0; w < kSelThreads / 32; ++w) {
          const int t = warp_tot[par][w];
          pos += w < wid ? t : 0;
          tot += t;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (kf[u]) {
            if (pos < topk) {
              out[pos] = ii[u] - r.x;
              if (so) so[pos] = key_float(kk[u]);
            }
            ++pos;
          }
        }
        written += tot;
      }
    }
    finish(written);
  }
}

}  // namespace

cudaError_t launch_select(int n_q, int n_chunks, int cap, int topk, int trivial_len, const int2* row_range,
                          const uint32_t* cand_edge,
                          const uint32_t* cand_key,
                          const int32_t* cand_idx, const uint32_t* cand_cnt, int32_t* idx_out, float* score_out,
                          uint32_t* status, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  if (n_chunks > kMaxChunks) return cudaErrorInvalidValue;
  if (static_cast<long long>(n_chunks) * cap <= static_cast<long long>(kSelThreads) * kSelPer)
    select_kernel<true><<<n_q, kSelThreads, 0, st>>>(n_chunks, cap, topk, trivial_len, row_range, cand_edge, cand_key, cand_idx, cand_cnt,
                                                    idx_out, score_out, status);
  else
    select_kernel<false><<<n_q, kSelThreads, 0, st>>>(n_chunks, cap, topk, trivial_len, row_range, cand_edge, cand_key, cand_idx, cand_cnt,
                                                     idx_out, score_out, status);
  return cudaGetLastError();
}

}  // namespace dsa
