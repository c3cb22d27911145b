// Block-cooperative exact top-k threshold search (radix select on order-preserving keys).
//
// Given a set of (key, idx) entries spread over the threads of a group, radix_threshold
// finds (v, cut) such that exactly K entries satisfy
//     key > v   ||   (key == v  &&  idx <= cut)
// which is the top-K by key descending with ties going to the lower idx -- the tie rule
// of the top-k.  Four 8-bit passes fix v, and only when the entries equal to v do not all
// fit, four more passes over idx (ascending) fix `cut`.  Requires K >= 1 and at least K
// entries.  idx values are non-negative.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace dsa {

// Warp 0 helper: bins 8*lane .. 8*lane+7 belong to `lane`.  Finds bin b with
// c(b) < need <= c(b) + hist[b], where c(b) counts entries in bins above b (descending)
// or below b (ascending).  Writes bc[0] = b, bc[1] = c(b), bc[2] = hist[b].
template <bool kDescending>
__device__ __forceinline__ void find_bin(const uint32_t* hist, int need, int* bc) {
  const int lane = threadIdx.x & 31;
  uint32_t h[8];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = hist[lane * 8 + i];
    s += h[i];
  }
  uint32_t x = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = kDescending ? __shfl_down_sync(0xffffffffu, x, off) : __shfl_up_sync(0xffffffffu, x, off);
    if (kDescending ? (lane + off < 32) : (lane >= off)) x += y;
  }
  int c = static_cast<int>(x - s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int bi = kDescending ? 7 - i : i;
    const int hv = static_cast<int>(h[bi]);
    if (c < need && need <= c + hv) {
      bc[0] = lane * 8 + bi;
      bc[1] = c;
      bc[2] = hv;
    }
    c += hv;
  }
}

// Histogram increment aggregated over the lanes of a warp that hit the same bin (scores
// cluster in few high-order bins, so plain shared atomics would serialise).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin) {
  const uint32_t act = __activemask();
  const uint32_t peers = __match_any_sync(act, bin);
  if ((threadIdx.x & 31u) == static_cast<uint32_t>(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
}

// `sync()` synchronises the NT cooperating threads; `tid` is this thread's rank in
// [0, NT) with rank 0..31 forming one warp.  `fe(f)` calls f(key, idx) for every entry
// this thread owns.  hist: 256 words of shared memory; bc: 4 ints of shared memory.
template <int NT, class Sync, class ForEach>
__device__ void radix_threshold(const Sync& sync, const ForEach& fe, int tid, int K, uint32_t* hist, int* bc,
                                uint32_t& v_out, uint32_t& cut_out) {
  uint32_t prefix = 0, mask = 0;
  int need = K, eq = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    sync();
    fe([&](uint32_t key, int32_t) {
      if ((key & mask) == prefix) hist_add(hist, (key >> shift) & 255u);
    });
    sync();
    if (tid < 32) find_bin<true>(hist, need, bc);
    sync();
    const int b = bc[0];
    need -= bc[1];
    eq = bc[2];
    prefix |= static_cast<uint32_t>(b) << shift;
    mask |= 0xFFu << shift;
    sync();
  }
  v_out = prefix;
  if (eq == need) {
    cut_out = 0x7FFFFFFFu;
    return;
  }
  uint32_t p2 = 0, m2 = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    sync();
    fe([&](uint32_t key, int32_t idx) {
      const uint32_t u = static_cast<uint32_t>(idx);
      if (key == prefix && (u & m2) == p2) hist_add(hist, (u >> shift) & 255u);
    });
    sync();
    if (tid < 32) find_bin<false>(hist, need, bc);
    sync();
    const int b = bc[0];
    need -= bc[1];
    p2 |= static_cast<uint32_t>(b) << shift;
    m2 |= 0xFFu << shift;
    sync();
  }
  cut_out = p2;
}

__device__ __forceinline__ bool topk_keep(uint32_t key, int32_t idx, uint32_t v, uint32_t cut) {
  return key > v || (key == v && static_cast<uint32_t>(idx) <= cut);
}

}  // namespace dsa
