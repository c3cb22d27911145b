// Backward of the MLA-absorbed sparse attention: gradients of q and of the latent rows.
//
// The forward (sparse_attn.cu) computes, for token t, head h and the selected rows j,
//   s_j = tau q . kv_j,   p_j = exp(s_j - lse),   o = sum_j p_j kv_j[:512].
// Given the upstream d_o, with D = d_o . o (from the forward's own output):
//   dp_j = d_o . kv_j[:512],   ds_j = p_j (dp_j - D),
//   dq   = tau sum_j ds_j kv_j,
//   dkv_j += tau ds_j q + p_j d_o (first 512 dims), summed over every (token, head) selecting j.
// "GLM-5/5.1/5.2 DSA + LoRA enablement" (Megatron-Bridge pull request #15), in the commit that
// vendors the fused sparse-MLA and lightning-indexer kernels for training, names a backward for
// each but defines neither; this is the exact gradient of the forward.
//
// One CTA per (token, block of HB = 16 or 32 heads; 16 when the layer has at most 16), eight
// warps, bf16 tensor-core MMAs (m16n8k16, fp32 accumulate) fed from shared memory by ldmatrix.
// The token's selected rows are walked in chunks of 64, double-buffered: cp.async fetches chunk
// c + 1's latent rows while chunk c is computed.  Per chunk:
//   A  S = Q KV^T and dP = dO V^T (HB heads x 64 rows; K = 576 and 512), then P and
//      dS' = tau dS in registers, stored to shared memory in bf16;
//   B  dQ += dS' KV (HB x 576, K = 64 rows), held in registers across chunks;
//   C  dKV = dS'^T Q + P^T dO (64 rows x 576, K = HB heads), added to HBM with 16-byte atomics
//      (a row is selected by many tokens).
// Shared-memory rows are padded by 16 bytes so the eight row addresses of every ldmatrix fall
// in distinct bank groups.  No wait in this kernel spins: its only synchronisation is
// cp.async group waits and CTA barriers.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kR = 64;                   // selected rows per chunk
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDq = 576, kDv = 512;
constexpr int kQS = kDq + 8;             // padded bf16 row strides (1168 B, 1040 B, 144 B)
constexpr int kOS = kDv + 8;
constexpr int kPS = kR + 8;
constexpr int kQPieces = kDq / 8;        // 16-byte pieces per latent / q row

template <int HB>
struct BwdSmem {
  __nv_bfloat16 q[HB * kQS];
  __nv_bfloat16 dout[HB * kOS];
  __nv_bfloat16 kv[2][kR * kQS];
  __nv_bfloat16 p[HB * kPS];
  __nv_bfloat16 ds[HB * kPS];
  float lse[HB];
  float dsum[HB];
  long long row[2][kR];
};
static_assert(sizeof(BwdSmem<32>) <= 232448, "backward shared memory");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// d += a (16x16, row) . b (16x8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Issue the cp.async copies of chunk c's latent rows into buffer b (rows past the token's
// selection, -1 slots and out-of-range rows are zero-filled and marked -1 in S.row).
template <class Smem>
__device__ __forceinline__ void issue_chunk(Smem& S, int c, int b, const int32_t* irow, int topk, long long kst,
                                            int n_kv, const uint16_t* kv, bool count_bad, uint32_t* status,
                                            uint32_t* bad_count) {
  const int tid = threadIdx.x;
  const uint32_t base = smem_u32(S.kv[b]);
  for (int e = tid; e < kR * kQPieces; e += kThreads) {
    const int r = e / kQPieces, piece = e - r * kQPieces;
    const int slot = c * kR + r;
    const int j = slot < topk ? __ldg(irow + slot) : -1;
    long long row = j >= 0 ? kst + j : -1;
    const bool ok = row >= 0 && row < n_kv;
    if (!ok) row = -1;
    cp_async_16_zfill(base + static_cast<uint32_t>((r * kQS + piece * 8) * 2),
                      ok ? static_cast<const void*>(kv + static_cast<size_t>(row) * kDq + piece * 8) : kv, ok);
    if (piece == 0) {
      S.row[b][r] = row;
      if (j >= 0 && !ok && count_bad) {
        atomicOr(status, DEV_ERR_BAD_INDEX);
        atomicAdd(bad_count, 1u);
      }
    }
  }
}

template <int HB>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_bwd_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ ks, const uint16_t* __restrict__ out, const float* __restrict__ lse,
    const uint16_t* __restrict__ dout, float* __restrict__ dq, float* __restrict__ dkv, int n_kv, int H, int topk,
    float scale, uint32_t* status, uint32_t* bad_count) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr int MT = HB / 16;              // 16-head m-tiles
  constexpr int NTA = MT;                   // S / dP n-tiles (8 rows) per warp
  constexpr int NTB = 9 * MT;               // dQ n-tiles (8 dims) per warp
  constexpr int TPH = kThreads / HB;        // threads per head computing D
  BwdSmem<HB>& S = *reinterpret_cast<BwdSmem<HB>*>(smem_raw);
  const int t = blockIdx.x;
  const int h0 = blockIdx.y * HB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3;
  const long long kst = __ldg(ks + t);
  const int32_t* irow = idx + static_cast<size_t>(t) * topk;
  const bool count_bad = blockIdx.y == 0;
  const int n_chunks = (topk + kR - 1) / kR;

  issue_chunk(S, 0, 0, irow, topk, kst, n_kv, kv, count_bad, status, bad_count);
  cp_async_commit();

  // ---- stage q and d_o of the block's heads (zeros past the last head), lse and D = d_o . o
  for (int e = tid; e < HB * kQPieces; e += kThreads) {
    const int h = e / kQPieces, piece = e - h * kQPieces;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h0 + h < H) v = __ldg(reinterpret_cast<const uint4*>(q + (static_cast<size_t>(t) * H + h0 + h) * kDq) + piece);
    *reinterpret_cast<uint4*>(S.q + h * kQS + piece * 8) = v;
  }
  for (int e = tid; e < HB * (kDv / 8); e += kThreads) {
    const int h = e / (kDv / 8), piece = e - h * (kDv / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h0 + h < H)
      v = __ldg(reinterpret_cast<const uint4*>(dout + (static_cast<size_t>(t) * H + h0 + h) * kDv) + piece);
    *reinterpret_cast<uint4*>(S.dout + h * kOS + piece * 8) = v;
  }
  {
    // D: TPH threads per head, each over 64 / TPH 16-byte pieces, then a shuffle reduction
    const int h = tid / TPH, part = tid % TPH;
    float acc = 0.f;
    if (h0 + h < H) {
      const uint4* o4 = reinterpret_cast<const uint4*>(out + (static_cast<size_t>(t) * H + h0 + h) * kDv);
      const uint4* d4 = reinterpret_cast<const uint4*>(dout + (static_cast<size_t>(t) * H + h0 + h) * kDv);
      for (int piece = part; piece < kDv / 8; piece += TPH) {
        const uint4 a = __ldg(o4 + piece), b = __ldg(d4 + piece);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(b2[i]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
      }
    }
#pragma unroll
    for (int off = TPH / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (part == 0) {
      S.dsum[h] = acc;
      S.lse[h] = h0 + h < H ? __ldg(lse + static_cast<size_t>(t) * H + h0 + h) : 0.f;
    }
  }

  __syncthreads();   // staged q / d_o / lse / D and chunk 0's row markers are visible to all

  // dQ accumulators: warp (mq = warp % MT, nq = warp / MT) owns heads 16 mq.. and the NTB
  // 8-wide n-tiles of dims 8 NTB nq..
  const int mq = warp % MT, nq = warp / MT;
  float acc_dq[NTB][4];
#pragma unroll
  for (int i = 0; i < NTB; ++i) acc_dq[i][0] = acc_dq[i][1] = acc_dq[i][2] = acc_dq[i][3] = 0.f;

  const uint32_t sq = smem_u32(S.q), sdo = smem_u32(S.dout), sp = smem_u32(S.p), sds = smem_u32(S.ds);
  for (int c = 0; c < n_chunks; ++c) {
    const int b = c & 1;
    if (c + 1 < n_chunks) issue_chunk(S, c + 1, b ^ 1, irow, topk, kst, n_kv, kv, count_bad, status, bad_count);
    cp_async_commit();
    cp_async_wait<1>();
    if (!__syncthreads_or(tid < kR && S.row[b][tid] >= 0)) continue;   // nothing selected in this chunk
    const uint32_t skv = smem_u32(S.kv[b]);

    // ---- A: S and dP for heads 16 ma.. x chunk rows 8 NTA na.. (NTA n-tiles)
    {
      const int ma = warp % MT, na = warp / MT;
      float s[NTA][4] = {}, dp[NTA][4] = {};
      const uint32_t a_row = static_cast<uint32_t>(ma * 16 + (lane & 15));
      const uint32_t a_col = static_cast<uint32_t>((lane >> 4) * 8);
      const uint32_t b_row = static_cast<uint32_t>(na * NTA * 8 + (lane & 7) + (NTA == 2 ? ((lane >> 4) << 3) : 0));
      const uint32_t b_col = static_cast<uint32_t>(((lane >> 3) & 1) * 8);
#pragma unroll 4
      for (int k = 0; k < kDq / 16; ++k) {
        uint32_t a[4], bb[4];
        ldsm_x4(sq + (a_row * kQS + a_col + k * 16) * 2, a);
        if constexpr (NTA == 2) {
          ldsm_x4(skv + (b_row * kQS + b_col + k * 16) * 2, bb);
        } else {
          ldsm_x2(skv + (b_row * kQS + b_col + k * 16) * 2, bb[0], bb[1]);
        }
        mma16816(s[0], a, bb[0], bb[1]);
        if constexpr (NTA == 2) mma16816(s[1], a, bb[2], bb[3]);
        if (k < kDv / 16) {
          uint32_t ad[4];
          ldsm_x4(sdo + (a_row * kOS + a_col + k * 16) * 2, ad);
          mma16816(dp[0], ad, bb[0], bb[1]);
          if constexpr (NTA == 2) mma16816(dp[1], ad, bb[2], bb[3]);
        }
      }
      const int ha = ma * 16 + g, hb = ha + 8;
      const bool va = h0 + ha < H, vb = h0 + hb < H;
      const float la = S.lse[ha], lb = S.lse[hb], da = S.dsum[ha], db = S.dsum[hb];
#pragma unroll
      for (int j = 0; j < NTA; ++j) {
        const int r0 = na * NTA * 8 + j * 8 + 2 * tig;
        const bool v0 = S.row[b][r0] >= 0, v1 = S.row[b][r0 + 1] >= 0;
        const float p00 = va && v0 ? expf(scale * s[j][0] - la) : 0.f;
        const float p01 = va && v1 ? expf(scale * s[j][1] - la) : 0.f;
        const float p10 = vb && v0 ? expf(scale * s[j][2] - lb) : 0.f;
        const float p11 = vb && v1 ? expf(scale * s[j][3] - lb) : 0.f;
        *reinterpret_cast<uint32_t*>(S.p + ha * kPS + r0) = pack_bf16(p00, p01);
        *reinterpret_cast<uint32_t*>(S.p + hb * kPS + r0) = pack_bf16(p10, p11);
        *reinterpret_cast<uint32_t*>(S.ds + ha * kPS + r0) =
            pack_bf16(scale * p00 * (dp[j][0] - da), scale * p01 * (dp[j][1] - da));
        *reinterpret_cast<uint32_t*>(S.ds + hb * kPS + r0) =
            pack_bf16(scale * p10 * (dp[j][2] - db), scale * p11 * (dp[j][3] - db));
      }
    }
    __syncthreads();

    // ---- B: dQ += dS' KV over the chunk's 64 rows
    {
      const uint32_t a_row = static_cast<uint32_t>(mq * 16 + (lane & 15));
      const uint32_t a_col = static_cast<uint32_t>((lane >> 4) * 8);
      const uint32_t b_row = static_cast<uint32_t>((lane & 7) + ((lane >> 3) & 1) * 8);
      const uint32_t n0 = static_cast<uint32_t>(nq * NTB * 8);
      const uint32_t b_col = n0 + static_cast<uint32_t>((lane >> 4) * 8);
#pragma unroll
      for (int k = 0; k < kR / 16; ++k) {
        uint32_t a[4];
        ldsm_x4(sds + (a_row * kPS + a_col + k * 16) * 2, a);
#pragma unroll
        for (int pr = 0; pr < NTB / 2; ++pr) {
          uint32_t bb[4];
          ldsm_x4_t(skv + ((b_row + k * 16) * kQS + b_col + pr * 16) * 2, bb);
          mma16816(acc_dq[2 * pr], a, bb[0], bb[1]);
          mma16816(acc_dq[2 * pr + 1], a, bb[2], bb[3]);
        }
        if constexpr (NTB % 2 == 1) {
          uint32_t b0, b1;
          ldsm_x2_t(skv + ((b_row + k * 16) * kQS + n0 + (NTB - 1) * 8) * 2, b0, b1);
          mma16816(acc_dq[NTB - 1], a, b0, b1);
        }
      }
    }

    // ---- C: dKV for chunk rows 16 mc.. x dims 288 nc.., scattered with 16-byte atomics
    {
      const int mc = warp & 3, nc = warp >> 2;
      const int i4 = lane >> 3;
      uint32_t ads[MT][4], ap[MT][4];
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        const uint32_t hrow = static_cast<uint32_t>(kk * 16 + (lane & 7) + (i4 >> 1) * 8);
        const uint32_t rcol = static_cast<uint32_t>(mc * 16 + (i4 & 1) * 8);
        ldsm_x4_t(sds + (hrow * kPS + rcol) * 2, ads[kk]);
        ldsm_x4_t(sp + (hrow * kPS + rcol) * 2, ap[kk]);
      }
      const int ra = mc * 16 + g;
      const long long row_a = S.row[b][ra], row_b = S.row[b][ra + 8];
      const uint32_t b_row = static_cast<uint32_t>((lane & 7) + ((lane >> 3) & 1) * 8);
      for (int pr = 0; pr < 18; ++pr) {
        const int d0 = nc * 288 + pr * 16;
        float o[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
          uint32_t bb[4];
          ldsm_x4_t(sq + ((b_row + kk * 16) * kQS + d0 + (lane >> 4) * 8) * 2, bb);
          mma16816(o[0], ads[kk], bb[0], bb[1]);
          mma16816(o[1], ads[kk], bb[2], bb[3]);
        }
        if (d0 < kDv) {
#pragma unroll
          for (int kk = 0; kk < MT; ++kk) {
            uint32_t bb[4];
            ldsm_x4_t(sdo + ((b_row + kk * 16) * kOS + d0 + (lane >> 4) * 8) * 2, bb);
            mma16816(o[0], ap[kk], bb[0], bb[1]);
            mma16816(o[1], ap[kk], bb[2], bb[3]);
          }
        }
        // lanes tig and tig ^ 1 swap halves so that each holds four consecutive dims of one
        // row (even tig: row ra, dims 2 tig..+3; odd: row ra + 8, dims 2 tig - 2..+3), then one
        // 16-byte atomic add each
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const bool odd = tig & 1;
          const float y0 = __shfl_xor_sync(0xffffffffu, odd ? o[j][0] : o[j][2], 1);
          const float y1 = __shfl_xor_sync(0xffffffffu, odd ? o[j][1] : o[j][3], 1);
          const int d = d0 + j * 8 + 2 * (tig & 2);
          const long long row = odd ? row_b : row_a;
          const float4 v = odd ? make_float4(y0, y1, o[j][2], o[j][3]) : make_float4(o[j][0], o[j][1], y0, y1);
          if (row >= 0) atomicAdd(reinterpret_cast<float4*>(dkv + row * kDq + d), v);
        }
      }
    }
    __syncthreads();   // the chunk's buffers are free for chunk c + 2 and the next P / dS'
  }
  cp_async_wait<0>();

  // ---- dQ out: heads 16 mq + g (+8), dims 8 NTB nq + 8 i + 2 tig
  const int ha = h0 + mq * 16 + g, hb = ha + 8;
#pragma unroll
  for (int i = 0; i < NTB; ++i) {
    const int d = nq * NTB * 8 + i * 8 + 2 * tig;
    if (ha < H)
      *reinterpret_cast<float2*>(dq + (static_cast<size_t>(t) * H + ha) * kDq + d) = make_float2(acc_dq[i][0], acc_dq[i][1]);
    if (hb < H)
      *reinterpret_cast<float2*>(dq + (static_cast<size_t>(t) * H + hb) * kDq + d) = make_float2(acc_dq[i][2], acc_dq[i][3]);
  }
}

}  // namespace

cudaError_t launch_sparse_attn_bwd(int n_q, int n_kv, int n_heads, int topk, float scale, const void* q,
                                   const void* kv, const int32_t* idx, const int32_t* ks, const void* out,
                                   const float* lse, const void* dout, float* dq, float* dkv, uint32_t* status,
                                   cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  auto run = [&](auto kernel, int hb, int smem, cudaError_t attr) {
    if (attr != cudaSuccess) return attr;
    dim3 grid(n_q, (n_heads + hb - 1) / hb);
    kernel<<<grid, kThreads, smem, st>>>(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(kv), idx, ks,
                                         static_cast<const uint16_t*>(out), lse, static_cast<const uint16_t*>(dout), dq,
                                         dkv, n_kv, n_heads, topk, scale, status, status + 1);
    return cudaGetLastError();
  };
  if (n_heads <= 16) {
    constexpr int smem = static_cast<int>(sizeof(BwdSmem<16>));
    return run(sparse_attn_bwd_kernel<16>, 16, smem, smem_attr_once<sparse_attn_bwd_kernel<16>>(smem));
  }
  constexpr int smem = static_cast<int>(sizeof(BwdSmem<32>));
  return run(sparse_attn_bwd_kernel<32>, 32, smem, smem_attr_once<sparse_attn_bwd_kernel<32>>(smem));
}

}  // namespace dsa
