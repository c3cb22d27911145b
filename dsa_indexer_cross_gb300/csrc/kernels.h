// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dsa {

// Sets Kern's maximum dynamic shared memory once per device (the attribute persists for the
// device's context, so later launches skip the driver call).
template <auto Kern>
inline cudaError_t smem_attr_once(int bytes) {
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// Layout of the 256-byte header at the start of every workspace.
struct WsHeader {
  uint32_t status;       // DEV_ERR_* bits
  uint32_t bad_count;    // number of out-of-range indices met
  uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Paged latent / index-key caches: pages of kPageRows rows; row t's logical key j lives at
// cache row block_table[t * max_pages + j / kPageRows] * kPageRows + j % kPageRows and is
// valid for j < seq_len[t].  block_table == nullptr means a contiguous cache (rows ks[t] + j).
constexpr int kPageShift = 7;
constexpr int kPageRows = 1 << kPageShift;
struct PagedRows {
  const int32_t* block_table = nullptr;
  const int32_t* seq_len = nullptr;
  int max_pages = 0;
  int n_pages = 0;
};

// ---------------------------------------------------------------------------- RoPE pre-pass
// out[row] = in[row] with its last `rope` dims rotated at position pos[row / rows_per_pos];
// only dims from the first 64-dim block holding rotary dims on are written
// (rope_split_blocks gives how many leading blocks are left to the unrotated input).
cudaError_t launch_rope_rows(const void* in, void* out, const int32_t* pos, int64_t n_rows, int rows_per_pos, int d,
                             int rope, const float* cs, int n_pos, uint32_t* status, cudaStream_t st);

// ---------------------------------------------------------------------------- indexer
// Candidate buffers: per (row, key chunk) kSub sub-buffers of cap / kSub entries, one per
// lane quarter of the indexer's 128-key tiles (keys j with (j - chunk start) % 128 in
// [32 q, 32 q + 32) go to sub-buffer q, in key order).
constexpr int kSub = 4;
// Rows with at most kDirectMax keys in a chunk keep every key (no streaming threshold).
constexpr int kDirectMax = 4096;
struct IndexerPlan {
  int n_heads, head_dim, group;      // group = query rows sharing one key stream (G)
  int n_groups, n_chunks, chunk;     // key chunking of every group's range
  int cap;                           // candidate capacity per (row, chunk), multiple of 128
  int grid;                          // persistent CTAs
  int topk;
  bool unit_list;                    // the kernel reads the dense unit list (independent rows)
};

// Fills row_range[t] = (ks, ke) when valid (ks == nullptr: every range starts at 0), else
// (0, 0) and flags; group_range[g] = union of the ranges of the group's rows longer than
// trivial_len (shorter rows keep every key and are not scored), at most span_limit keys long
// (a longer union is cut there and flagged: the plan's key chunks cover span_limit keys).
// In-place transpose of the index RoPE on fp32 rows (the backward of launch_rope_rows): the
// rotated pair (a, b) of dims (d - r + i, d - r/2 + i) becomes (a c + b s, b c - a s).
cudaError_t launch_rope_rows_transpose_f32(float* x, const int32_t* pos, int64_t n_rows, int rows_per_pos, int d,
                                           int rope, const float* cs, int n_pos, uint32_t* status, cudaStream_t st);

cudaError_t launch_ranges(const int32_t* ks, const int32_t* ke, int n_q, int group, int n_kv, int max_len,
                          int trivial_len, long long span_limit, int2* row_range, int2* group_range,
                          uint32_t* status, cudaStream_t st);

// The indexer's work units, listed densely: every (group, chunk) pair whose chunk holds keys
// of the group's range, chunk-major, later groups first within a chunk, as int2 (group,
// chunk), followed by (-1, -1) up to n_groups * n_chunks entries.  The candidate counts and
// edges of every (row, chunk) pair left out are zeroed, so the final select reads them as
// empty.  One block.
cudaError_t launch_units(const int2* group_range, int n_groups, int n_chunks, int chunk_len, int group, int n_q,
                         int2* units, uint32_t* cand_cnt, uint32_t* cand_edge, cudaStream_t st);

// Bound of every pipeline wait and a test hook that stops a kernel's producer after a number
// of tiles (so the waits behind it run out); see dsa_debug_pipeline.
struct PipelineDebug {
  unsigned long long wait_ns = 2000000000ull;
  int stop_after_tiles = -1;
};
PipelineDebug pipeline_debug();

// Lightning-indexer backward (head_dim 128, n_heads a multiple of 4 up to 64): dq~ written,
// dk~ and dw accumulated (both zeroed by the caller), all fp32.  q_split / k_split: 64-dim
// blocks read from the unrotated inputs, as in launch_indexer.
cudaError_t launch_indexer_bwd(int n_q, int n_kv, int n_heads, int head_dim, int topk, const void* q_rot,
                               const void* q_in, const void* k_rot, const void* k_in, int q_split, int k_split,
                               const float* w, const int32_t* ks, const int32_t* ke, const int32_t* idx,
                               const float* d_score, float* dq, float* dk, float* dw, int grid, uint32_t* status,
                               const PipelineDebug& dbg, cudaStream_t st);

// Scores + streaming top-k candidates.  tmap_q covers rotated q as [(n_q*H_I) x d_I] bf16,
// tmap_k covers rotated k as [n_kv x d_I] bf16, both 128-byte swizzled, boxes {64, N} and
// {64, 128}.  Per (row, chunk) it leaves up to p.cap candidates in key order, their count and
// an edge key (no entry below it can be in the row's top-k; 0 when unknown) for
// launch_select.  Rows of at most trivial_len keys are not scored (count 0).
inline int rope_split_blocks(int d, int rope) { return rope > 0 ? (d - rope) / 64 : 0; }
// tmap_q / tmap_k: rotated copies; tmap_q_in / tmap_k_in: the unrotated inputs, read for the
// 64-dim blocks below q_split / k_split.
cudaError_t launch_indexer(const IndexerPlan& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                           const CUtensorMap& tmap_q_in, const CUtensorMap& tmap_k_in, int q_split, int k_split,
                           const PagedRows& pg, const float* w, int n_q, const int2* row_range,
                           const int2* group_range, int trivial_len, uint32_t* cand_key, int32_t* cand_idx,
                           uint32_t* cand_cnt, uint32_t* cand_edge, const int2* units, uint32_t* status, const PipelineDebug& dbg, cudaStream_t st);

// Exact top-k of every row from its candidates; writes offsets (ascending) and -1 padding.
// Rows of at most trivial_len keys are written as 0..L-1 without reading candidates; entries
// below the largest of a row's chunk edges are skipped.
// max_len bounds every row's length (the ranges kernel empties longer rows).
cudaError_t launch_select(int n_q, int n_chunks, int cap, int topk, int trivial_len, int max_len, const int2* row_range,
                          const uint32_t* cand_edge,
                          const uint32_t* cand_key,
                          const int32_t* cand_idx, const uint32_t* cand_cnt, int32_t* idx_out, float* score_out,
                          uint32_t* status, cudaStream_t st);

// ---------------------------------------------------------------------------- sparse attention
// Block-dense walk: an item is kDenseCols (token, head) columns, kDenseCols / H consecutive
// tokens with all H heads, and its tokens' selections over the item's key range are one
// bitmask of kDenseMaskBytes (kDenseMaskBytes * 8 / tokens bits a token).
constexpr int kDenseCols = 64;
constexpr int kDenseMaskBytes = 4096;
// Heads of the block-dense walk for this shape, or 0 for the per-token gather walk.
int sparse_attn_dense_heads(int n_heads, int n_kv, int topk);
// The block-dense pre-pass over idx, one CTA per item (hd = heads of the walk): block_range[b]
// = [min, max + 1) of the in-range latent rows the item's tokens select ((0, 0) for none),
// block_mask[b] = per token, bit o set when row min + o is selected.  Bad offsets are counted in
// status[0..1].  dense_scratch splits a scratch of sparse_attn_ws_bytes into the two arrays.
struct DenseScratch {
  int2* block_range;
  uint32_t* block_mask;
};
DenseScratch dense_scratch(void* scratch, int n_q, int hd);
cudaError_t launch_block_mask(int hd, const int32_t* idx, const int32_t* ks, int n_q, int n_kv, int topk,
                              const DenseScratch& ds, uint32_t* status, cudaStream_t st);
// Scratch bytes launch_sparse_attn needs (per-row tile counts, or per-block key ranges and
// selection bitmasks).
size_t sparse_attn_ws_bytes(int n_q, int n_heads, int n_kv, int topk);
// Rows of q (consecutive (token, head) rows) that one work item of the chosen walk reads:
// the box height of tmap_q (a paged cache always takes the gather walk).
int sparse_attn_q_box_rows(int n_heads, int n_kv, int topk, bool paged);
// tmap_kv: block-dense walk -- kv [n_kv x 576] bf16 viewed as (64 dims, n_kv rows, 9 dim
// blocks) with 128-byte swizzled boxes of {64, 64, 9} = one 64-row tile; gather walk -- kv as
// a 2-D [n_kv][576] tensor with 128-byte swizzled boxes of {64, 1} (four-row gathers).
// tmap_q: q as a 2-D [n_q * n_heads][576] tensor, 128-byte swizzled boxes of
// {64, sparse_attn_q_box_rows(...)}.
// reuse_prepass: the scratch already holds the pre-pass results (tile counts, or key ranges and
// bitmasks) for these idx and ks rows, from the previous call on the same scratch and shape.
cudaError_t launch_sparse_attn(const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q, int n_q, int n_kv, int n_heads,
                               int topk, float scale, const void* kv, const int32_t* idx, const int32_t* ks,
                               const PagedRows& pg, void* out, float* lse, uint32_t* status, void* scratch,
                               cudaStream_t st, bool reuse_prepass = false);

// ---------------------------------------------------------------------------- indexer projections
// One GEMM job of the projection kernel, Y = A[T][k] . W^T in N tiles of n_tile weight rows.
//   kProjEpiBf16:        W = one matrix [n_total][k], output bf16 [T][n_total], n_tile <= 256;
//   kProjEpiLayerNormF32: W = two matrices stacked in one tile -- n_total rows (LayerNorm'd,
//                        output bf16 [T][n_total]) then n2 rows (output fp32 out2 [T][n2]) --
//                        so both share one pass over the activations; n_tile = n_total + the
//                        second matrix's box height.
enum { kProjEpiBf16 = 0, kProjEpiLayerNormF32 = 1 };
struct ProjJob {
  int n_total, k, n_tile, epi;
  void* out;
  const float* gamma;    // LayerNorm weight / bias [n_total]
  const float* beta;
  float eps;
  float* out2;           // fp32 tail outputs [T][n2]
  int n2;
};
struct ProjJobs {
  ProjJob job[2];
  int n_jobs;
  int first_unit[3];     // first unit of each job; first_unit[n_jobs] = total units
};
// ta[j]: the activations of job j ([T][k] bf16, boxes {64, 128}); tb[j]: its weights ([rows][k],
// boxes {64, rows of the tile}); tb2: the second weight matrix of the LayerNorm job.
cudaError_t launch_projections(const CUtensorMap* ta, const CUtensorMap* tb, const CUtensorMap& tb2,
                               const ProjJobs& J, int n_tokens, uint32_t* status, cudaStream_t st);

// ---------------------------------------------------------------------------- attention backward
// dq [n_q][H][576] fp32 (written), dkv [n_kv][576] fp32 (accumulated: zero it first), given the
// forward's out (bf16) and lse (fp32) and the upstream gradient dout [n_q][H][512] bf16.
cudaError_t launch_sparse_attn_bwd(int n_q, int n_kv, int n_heads, int topk, float scale, const void* q,
                                   const void* kv, const int32_t* idx, const int32_t* ks, const void* out,
                                   const float* lse, const void* dout, float* dq, float* dkv, uint32_t* status,
                                   cudaStream_t st);

// The same gradients on the block-dense walk (hd = sparse_attn_dense_heads(...) != 0), on
// tcgen05: delta [n_q * hd] fp32 scratch for D = d_out . out, scratch of sparse_attn_ws_bytes
// for the walk's pre-pass.  tmap_kv as for launch_sparse_attn's block-dense walk; tmap_q and
// tmap_do: q [n_q * hd][576] and dout [n_q * hd][512] bf16 with 128-byte swizzled boxes of
// {64, kDenseCols}.
size_t sparse_attn_bwd_dense_delta_bytes(int n_q, int n_heads);
// The same gradients on the gather walk (every other shape), on tcgen05: item = (token, 64-head
// block), each 64-slot tile of the token's selections gathered with cp.async.  delta as above;
// row_nt: n_q int32 scratch (64-slot tiles per token).
cudaError_t launch_sparse_attn_bwd_gather(const CUtensorMap& tmap_q, const CUtensorMap& tmap_do, int n_q, int n_kv,
                                          int n_heads, int topk, float scale, const void* kv, const int32_t* idx,
                                          const int32_t* ks, const void* out, const float* lse, const void* dout,
                                          float* dq, float* dkv, uint32_t* status, float* delta, int32_t* row_nt,
                                          cudaStream_t st);
// row_nt[t] = number of 64-slot tiles of idx row t up to its last index >= 0.
cudaError_t launch_row_tiles(const int32_t* idx, int n_q, int topk, int32_t* row_nt, cudaStream_t st);
cudaError_t launch_sparse_attn_bwd_dense(int hd, const CUtensorMap& tmap_kv, const CUtensorMap& tmap_q,
                                         const CUtensorMap& tmap_do, int n_q, int n_kv, int topk, float scale,
                                         const int32_t* idx, const int32_t* ks, const void* out, const float* lse,
                                         const void* dout, float* dq, float* dkv, uint32_t* status, float* delta,
                                         void* scratch, cudaStream_t st);

int device_sm_count();

// ---------------------------------------------------------------------------- launch log
// While profiling is switched on (dsa_profile_enable), every kernel launch of the library is
// bracketed by a pair of CUDA events on its stream, tagged with the kernel's kind, so that a
// caller can read each launch's device time afterwards (dsa_profile_read).  Off, both calls
// do nothing.  prof_begin returns the record's slot (-1 when nothing is recorded).
enum ProfKind : int {
  kProfRope = 0, kProfRanges = 1, kProfIndexer = 2, kProfSelect = 3, kProfAttnPrep = 4, kProfAttn = 5,
  kProfAttnBwd = 6, kProfProj = 7, kProfIndexerBwd = 8
};
int prof_begin(int kind, cudaStream_t st);
void prof_end(int slot, cudaStream_t st);

}  // namespace dsa
