/*
 * dsa.h -- C ABI of libdsa: the DeepSeek Sparse Attention lightning indexer with a fused
 * causal top-k, GLM-5.2 cross-layer IndexShare, and MLA-absorbed sparse attention, for
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * What the operations compute is defined on three public pages:
 *   [MT] "add glm5.2 indexshare" (MaxText pull request #4832), Description and Code Review;
 *   [MB] "GLM-5/5.1/5.2 DSA + LoRA enablement" (Megatron-Bridge pull request #15), the
 *        commits on the indexer RoPE half swap, on capping top-k at the sequence length,
 *        on cross-layer top-k sharing and on the per-query key ranges (cu_seqlens
 *        starts/ends) of the indexer;
 *   [EX] "GLM-5.2 IndexShare" (explainer), sections 1-2, "Layer execution pattern",
 *        "Public config evidence", "What is actually shared?".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Device pointers point to GPU global memory owned by the caller.  The library never
 *    allocates device memory: every call that needs scratch space takes a workspace
 *    (`ws`, `ws_bytes`) whose size the matching *_workspace_size query returns.  A
 *    workspace must be 256-byte aligned and must not be used by two calls that can run
 *    at the same time.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only enqueue
 *    work and return; results are ready when the stream reaches them.
 *  - Arrays are dense and row-major ("[a][b]" = b fastest).  bf16 tensors must be
 *    16-byte aligned (they are read by the Tensor Memory Accelerator or by 16-byte
 *    vector loads).
 *  - Every function returns a dsa_status and never throws or aborts.  Argument and shape
 *    errors are detected on the host before anything is enqueued; the reason is then
 *    available from dsa_last_error() on the calling thread.
 *  - Faults found on the device (an index outside its range, a pipeline wait that ran
 *    past its 2 s bound) are recorded in the first word of the workspace and read back
 *    with dsa_workspace_status().  No kernel traps.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_ARG = 1,         /* a NULL or misaligned pointer, or a value out of range        */
  DSA_ERR_SHAPE = 2,       /* sizes that are inconsistent with each other                  */
  DSA_ERR_NO_DONOR = 3,    /* a shared layer precedes every full layer                     */
  DSA_ERR_UNSUPPORTED = 4, /* a valid size this library has no kernel for, or no sm_10x GPU */
  DSA_ERR_CUDA = 5,        /* a CUDA runtime call failed (message in dsa_last_error)       */
  DSA_ERR_WORKSPACE = 6,   /* ws_bytes smaller than the *_workspace_size query             */
  DSA_ERR_TIMEOUT = 7,     /* a device pipeline wait ran past its bound                    */
  DSA_ERR_DEVICE = 8       /* the device counted out-of-range indices or a buffer overflow */
} dsa_status;

/* Human-readable name of a status code (static storage). */
const char* dsa_status_string(dsa_status s);

/* Message describing the last error returned on the calling thread ("" if none). */
const char* dsa_last_error(void);

/* ------------------------------------------------------------------ layer schedule -- */

/* Values of an indexer_types array.  [EX] "Public config evidence": the released config
 * lists one of "full" / "shared" per layer; [MT] Description: full layers run the
 * lightning indexer, shared layers reuse the donor full layer's top-k indices. */
#define DSA_LAYER_SHARED 0u
#define DSA_LAYER_FULL 1u

/* Donor of every layer: donors[l] = l for a full layer, else the nearest preceding full
 * layer ([EX] "Layer execution pattern"; [MT] Code Review: shared layers 5, 6, 7 reuse
 * layer 4).  indexer_types and donors are host arrays of n_layers entries.
 * Errors: DSA_ERR_ARG (NULL, n_layers < 1, a value other than 0/1), DSA_ERR_NO_DONOR
 * (a shared layer before the first full layer -- [MB] build-time stage assert). */
dsa_status dsa_donor_table(int32_t n_layers, const uint8_t* indexer_types, int32_t* donors);

/* ------------------------------------------------------------------ index RoPE ------- */

/* Fill the host table rope_cs[p][i] = {cos(p * f_i), sin(p * f_i)} (float32, evaluated in
 * float64) with f_i = theta^(-2i/rope_dim), for p in [0, n_pos), i in [0, rope_dim/2).
 * The indexer rotates the LAST rope_dim dims of each index head with this table, pairing
 * dim (d - r + i) with dim (d - r/2 + i) ([MB] RoPE half-swap commit: rotary dims sit in
 * the last qk_pos_emb_head_dim of each index head).  host_out holds n_pos * rope_dim
 * floats, caller-owned.  Errors: DSA_ERR_ARG (NULL, odd or negative rope_dim, n_pos < 1,
 * theta <= 0). */
dsa_status dsa_rope_table(double theta, int32_t rope_dim, int32_t n_pos, float* host_out);

/* ------------------------------------------------------------------ indexer + top-k -- */

/* Flags of dsa_indexer_desc. */
#define DSA_IDX_ROPE_Q (1u << 0)           /* rotate q_idx before scoring                  */
#define DSA_IDX_ROPE_K (1u << 1)           /* rotate k_idx before scoring (clear when the  */
                                           /*  caller keeps an already-rotated key cache)  */
#define DSA_IDX_INDEPENDENT_ROWS (1u << 2) /* rows do not share key ranges (batched decode:*/
                                           /*  each row is its own sequence)               */

typedef struct dsa_indexer_desc {
  int32_t n_q;       /* query rows                                                       */
  int32_t n_kv;      /* key rows in k_idx                                                */
  int32_t n_heads;   /* index heads H_I: 4, 8, 16, 32 or 64                              */
  int32_t head_dim;  /* index head dim d_I: 64 or 128                                    */
  int32_t rope_dim;  /* RoPE dims r at the end of each head: even, 0 <= r <= d_I         */
  int32_t topk;      /* index_topk k: 1 .. 2048                                          */
  int32_t max_len;   /* an upper bound on every ke_t - ks_t (0 < max_len <= n_kv)        */
  uint32_t flags;    /* DSA_IDX_*                                                        */
} dsa_indexer_desc;

/* Workspace bytes dsa_indexer_topk needs for this descriptor on the current device. */
dsa_status dsa_indexer_workspace_size(const dsa_indexer_desc* desc, size_t* bytes);

/* Lightning indexer with a fused streaming causal top-k ([EX] section 1: score the prefix
 * tokens of every query and keep the top-k positions; the score of the problem statement):
 *
 *   s[t, j] = sum_h w[t, h] * max(0, rope(q_idx[t, h]) . rope(k_idx[j]))   j in [ks_t, ke_t)
 *
 * and idx_out[t] = the offsets j - ks_t of the min(topk, ke_t - ks_t) largest s[t, .]
 * (ties to the lower j), sorted ascending, then -1 up to width topk ([MB] commit capping
 * top-k at the sequence length and padding with -1).  One key head is shared by all index
 * heads ([MB] one wk / k_norm per index head dim; weights_proj is a per-head scalar).
 * The T x L score matrix is never written to memory: candidates above a running
 * per-row threshold are kept in the workspace and cut back to k as they accumulate.
 *
 *   q_idx  bf16  [n_q][n_heads][head_dim]     k_idx bf16 [n_kv][head_dim]
 *   w      f32   [n_q][n_heads]               q_pos int32 [n_q], k_pos int32 [n_kv]
 *   ks, ke int32 [n_q]  key row range of row t: 0 <= ks_t <= ke_t <= n_kv,
 *                       ke_t - ks_t <= max_len
 *   rope_cs f32  [rope_n_pos][rope_dim/2][2]  table from dsa_rope_table (device copy);
 *                may be NULL when neither ROPE flag is set or rope_dim == 0.  Positions
 *                must lie in [0, rope_n_pos).
 *   idx_out   int32 [n_q][topk]   (output)
 *   score_out f32   [n_q][topk]   (optional output, NULL to skip): s of each selected key,
 *                                  -inf on padding.
 * q_pos / k_pos may be NULL when the matching ROPE flag is clear.
 * Errors: DSA_ERR_ARG, DSA_ERR_UNSUPPORTED (n_heads / head_dim / topk outside the lists
 * above), DSA_ERR_WORKSPACE, DSA_ERR_CUDA.  Device-side: a position outside the table,
 * or a key range outside [0, n_kv) or longer than max_len, sets DSA_ERR_DEVICE in the
 * workspace status. */
dsa_status dsa_indexer_topk(const dsa_indexer_desc* desc, const void* q_idx, const void* k_idx, const float* w,
                            const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                            const float* rope_cs, int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws,
                            size_t ws_bytes, void* stream);

/* Indexer + top-k for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot hand the library a
 * workspace -- for example a plugin that a host framework calls with only its input and
 * output buffers (the framework owns the device allocator), or a latency-critical loop in
 * which a cudaMalloc and its implicit synchronisation are not acceptable.
 * Same arguments, results and errors as dsa_indexer_topk, minus ws / ws_bytes.  Scratch
 * comes from one file-scope device array of DSA_STATIC_SCRATCH_BYTES held on every GPU
 * that uses this call until the process exits; no allocation routine is called.  The first
 * call on a device (with that device current) looks up the array's address once; make that
 * call before any stream capture.  Problems that need more scratch than the array holds are
 * rejected with DSA_ERR_WORKSPACE.  All calls on a device share the array: calls whose work
 * overlaps on the GPU race and must be serialised by the caller.  Device-side faults (bad
 * positions or key ranges, a timed-out pipeline wait) are recorded in the array's status
 * word, which dsa_indexer_static_status reads; the next call clears it.  The cached address
 * belongs to the device's primary context: after cudaDeviceReset (or anything else that
 * destroys and re-creates that context) this entry point must not be called again in the
 * same process. */
#define DSA_STATIC_SCRATCH_BYTES (32u << 20)
dsa_status dsa_indexer_topk_static(const dsa_indexer_desc* desc, const void* q_idx, const void* k_idx, const float* w,
                                   const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                                   const float* rope_cs, int32_t rope_n_pos, int32_t* idx_out, float* score_out,
                                   void* stream);

/* Status of the last dsa_indexer_topk_static call on the current device, the counterpart of
 * dsa_workspace_status for that variant: synchronises `stream` (pass the stream of that
 * call), reads the status word of the static array and maps it the same way (DSA_OK,
 * DSA_ERR_TIMEOUT, DSA_ERR_DEVICE); the raw bits go to *device_bits when it is not NULL.
 * Allocates nothing.  Errors: DSA_ERR_UNSUPPORTED (no static call made on this device yet),
 * DSA_ERR_CUDA. */
dsa_status dsa_indexer_static_status(void* stream, uint32_t* device_bits);

/* ------------------------------------------------------------------ sparse attention - */

typedef struct dsa_attn_desc {
  int32_t n_q;          /* query rows                                                    */
  int32_t n_kv;         /* latent rows in kv                                             */
  int32_t n_heads;      /* attention heads H: 1 .. 128                                   */
  int32_t d_qk;         /* 576 = 512 latent + 64 rope ([MB] qk_rope_head_dim commit)     */
  int32_t d_v;          /* 512: V is the first d_v dims of each latent row               */
  int32_t topk;         /* width of each idx row                                         */
  float softmax_scale;  /* tau, e.g. 1/sqrt(576)                                         */
  uint32_t flags;       /* reserved, 0                                                   */
} dsa_attn_desc;

dsa_status dsa_sparse_attn_workspace_size(const dsa_attn_desc* desc, size_t* bytes);

/* MLA-absorbed sparse attention over the selected latent rows ([EX] section 1: the main
 * attention runs only on the selected positions; "What is actually shared?": every layer
 * computes its own attention):
 *
 *   o[t, h]   = sum_{j in I_t} softmax_j(tau * q[t, h] . kv[ks_t + j]) * kv[ks_t + j, :d_v]
 *   lse[t, h] = log sum_{j in I_t} exp(tau * q[t, h] . kv[ks_t + j])
 *
 * with I_t the entries of idx[t] that are >= 0, which must be distinct (as the indexer's
 * rows are); repeated offsets in one row are not supported.  All heads of a token read the
 * same rows.
 *   q   bf16 [n_q][n_heads][d_qk]     kv  bf16 [n_kv][d_qk]
 *   idx int32 [n_q][topk]  offsets relative to ks_t, -1 = unused slot
 *   ks  int32 [n_q]
 *   out bf16 [n_q][n_heads][d_v]      (output)
 *   lse f32  [n_q][n_heads]           (optional output, NULL to skip)
 * A row with no valid index gives o = 0 and lse = -inf.  An index with ks_t + j outside
 * [0, n_kv) is skipped and counted (DSA_ERR_DEVICE in the workspace status).
 * Errors: DSA_ERR_ARG, DSA_ERR_UNSUPPORTED (d_qk != 576 or d_v != 512, n_heads > 128),
 * DSA_ERR_WORKSPACE, DSA_ERR_CUDA. */
dsa_status dsa_sparse_attn(const dsa_attn_desc* desc, const void* q, const void* kv, const int32_t* idx,
                           const int32_t* ks, void* out, float* lse, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ index cache ------ */

/* Host object mapping every layer to the device buffer holding its donor's indices
 * ([EX] "Implementation checklist": cache the top-k of full layers, shared layers read
 * the preceding full layer's; [MB] anchors publish top-k, skip layers reuse it).
 * idx_buffers has n_layers entries; entry l must be a device buffer of n_q * topk int32
 * for every full layer l and is ignored (may be NULL) for shared layers.  The cache
 * stores the pointers, not the memory: the caller keeps the buffers alive.
 * Errors: DSA_ERR_ARG, DSA_ERR_NO_DONOR. */
typedef struct dsa_index_cache dsa_index_cache;

dsa_status dsa_index_cache_create(int32_t n_layers, const uint8_t* indexer_types, int32_t n_q, int32_t topk,
                                  int32_t* const* idx_buffers, dsa_index_cache** cache_out);
/* Donor layer of `layer`.  Errors: DSA_ERR_ARG (NULL, layer out of range). */
dsa_status dsa_index_cache_donor(const dsa_index_cache* cache, int32_t layer, int32_t* donor);
/* Device buffer holding the indices `layer` attends with (its donor's), NULL on error. */
int32_t* dsa_index_cache_indices(const dsa_index_cache* cache, int32_t layer);
void dsa_index_cache_destroy(dsa_index_cache* cache);

/* ------------------------------------------------------------------ layer loop ------- */

/* Per-layer tensors.  q_idx, k_idx and w are read on full layers only (NULL allowed on
 * shared layers); q, kv, out (and lse, optional) on every layer. */
typedef struct dsa_layer_io {
  const void* q_idx;
  const void* k_idx;
  const float* w;
  const void* q;
  const void* kv;
  void* out;
  float* lse;
} dsa_layer_io;

dsa_status dsa_layers_workspace_size(const dsa_indexer_desc* idx_desc, const dsa_attn_desc* attn_desc, size_t* bytes);

/* The IndexShare layer loop ([EX] section 2 and "Layer execution pattern"; [MT] Key
 * Changes: full layers compute, shared layers pass the cached state through).  For each
 * layer l in order: if indexer_types[l] is full, run dsa_indexer_topk into the cache
 * buffer of l; then run dsa_sparse_attn of layer l with the buffer of donor(l).  Shared
 * layers launch no indexer work and read their donor's buffer unchanged.  indexer_types
 * must equal the array the cache was created with.  Everything is enqueued on `stream`
 * with no host synchronisation.  Errors: those of the two calls, DSA_ERR_SHAPE when the
 * descriptors disagree (n_q, topk, n_kv) or do not match the cache. */
dsa_status indexshare_layers_forward(const dsa_indexer_desc* idx_desc, const dsa_attn_desc* attn_desc,
                                     int32_t n_layers, const uint8_t* indexer_types, const dsa_layer_io* layer_io,
                                     const int32_t* ks, const int32_t* ke, const int32_t* q_pos,
                                     const int32_t* k_pos, const float* rope_cs, int32_t rope_n_pos,
                                     dsa_index_cache* cache, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ projections ----- */

/* The indexer's input projections of one full layer ("GLM-5/5.1/5.2 DSA + LoRA enablement",
 * indexer RoPE half-swap commit: wq_b, wk, k_norm -- a LayerNorm with weight and bias applied
 * to the key before RoPE -- and weights_proj, one scalar per index head):
 *   q_idx[t] = q_latent[t] . wq_b^T                               [n_heads * head_dim] bf16
 *   k_idx[t] = LayerNorm_eps(x[t] . wk^T) * k_norm_w + k_norm_b   [head_dim]           bf16
 *   w[t]     = x[t] . weights_proj^T                              [n_heads]            fp32
 * (no further scaling: fold any into weights_proj).  The outputs feed dsa_indexer_topk
 * (which applies the RoPE).  All three run in one tensor-core kernel (fp32 accumulation, the
 * LayerNorm in fp32 on the accumulator, outputs rounded once).
 * Layouts, row-major device arrays: x [n_tokens][d_hidden], q_latent [n_tokens][d_q] bf16;
 * wq_b [n_heads * head_dim][d_q], wk [head_dim][d_hidden], weights_proj [n_heads][d_hidden]
 * bf16; k_norm_w, k_norm_b [head_dim] fp32.  d_hidden and d_q multiples of 64; n_heads in
 * {4, 8, 16, 32, 64}, head_dim in {64, 128} (the indexer's lists); ws: at least 256 bytes,
 * 256-byte aligned (its first word is the status read by dsa_workspace_status).
 * Errors: DSA_ERR_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA. */
typedef struct dsa_proj_desc {
  int32_t n_tokens;
  int32_t d_hidden;  /* width of x (K of wk and weights_proj)        */
  int32_t d_q;       /* width of the query latent (K of wq_b)       */
  int32_t n_heads;   /* index heads H_I                              */
  int32_t head_dim;  /* d_I                                          */
  float ln_eps;      /* k_norm epsilon                               */
} dsa_proj_desc;

dsa_status dsa_indexer_projections(const dsa_proj_desc* desc, const void* x, const void* q_latent, const void* wq_b,
                                   const void* wk, const float* k_norm_w, const float* k_norm_b,
                                   const void* weights_proj, void* q_idx, void* k_idx, float* w, void* ws,
                                   size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ training ------- */

/* Gradients of dsa_sparse_attn.  [MB]'s commit that vendors the fused sparse-MLA and
 * lightning-indexer kernels for training names a backward for each but defines neither; this
 * is the exact gradient of the forward above.  With p_j = exp(tau q . kv_j - lse) and
 * D = d_out . out:
 *   dq[t, h]  = tau sum_j p_j (d_out . kv_j[:512] - D) kv_j
 *   dkv[row] += tau p_j (d_out . kv_j[:512] - D) q[t, h] + p_j d_out[t, h] (first 512 dims)
 * summed over every (t, h) selecting the row.  Inputs as in dsa_sparse_attn plus the forward's
 * out [n_q][n_heads][512] bf16 and lse [n_q][n_heads] fp32, and d_out [n_q][n_heads][512]
 * bf16.  Outputs fp32: dq [n_q][n_heads][576] (written) and dkv [n_kv][576] (zeroed here, then
 * accumulated; rows shared by several tokens receive atomic adds, so the order of the
 * additions, and the last bits of dkv, vary from run to run).  All tensors 16-byte aligned.
 * Out-of-range indices are counted in the status word and skipped.  Shapes that take the
 * forward's block-dense walk (at most 16 heads, selections dense in a short key range) run
 * on the tensor cores with P and dS rounded to bf16; the others take a per-token kernel.
 * ws: dsa_sparse_attn_backward_workspace_size bytes (at least 256), 256-byte aligned.
 * Errors: DSA_ERR_ARG, DSA_ERR_UNSUPPORTED (d_qk != 576 or d_v != 512), DSA_ERR_WORKSPACE,
 * DSA_ERR_CUDA. */
dsa_status dsa_sparse_attn_backward_workspace_size(const dsa_attn_desc* desc, size_t* bytes);
dsa_status dsa_sparse_attn_backward(const dsa_attn_desc* desc, const void* q, const void* kv, const int32_t* idx,
                                    const int32_t* ks, const void* out, const float* lse, const void* d_out,
                                    float* dq, float* dkv, void* ws, size_t ws_bytes, void* stream);

/* Gradients of the indexer scores that dsa_indexer_topk selected.  [MB]'s commit vendoring
 * the fused lighting_indexer "with fwd/bwd" names this backward without defining it; it is
 * the exact derivative of the score above.  For row t, slot n < min(topk, ke_t - ks_t) with
 * idx[t][n] = j >= 0 (key row ks_t + j) and upstream g = d_score[t][n]:
 *   x_h = rope(q_idx[t, h]) . rope(k_idx[ks_t + j])
 *   dw[t][h]          += g max(0, x_h)
 *   dq_idx[t][h]      += R(q_pos_t)^T  g w[t][h] [x_h > 0] rope(k_idx[ks_t + j])
 *   dk_idx[ks_t + j]  += R(k_pos_j)^T  g sum_h w[t][h] [x_h > 0] rope(q_idx[t, h])
 * with ReLU'(0) = 0, R^T the rotation by the negated angle (only when the matching ROPE flag
 * is set), and the bf16 rounding of the rotated inputs taken as the identity.  The products
 * run on the tensor core with g w [x > 0] rounded to bf16 and fp32 accumulation.  Slots past
 * min(topk, ke_t - ks_t) are not read; -1 slots are skipped; an offset >= ke_t - ks_t is
 * skipped and flagged (DSA_ERR_DEVICE).  The loss that produces d_score (for example a KL
 * term between the indexer's and the attention's distributions) is the caller's: the pages
 * do not define one.
 *   desc: as for dsa_indexer_topk; head_dim must be 128, n_heads <= 64, and
 *         DSA_IDX_INDEPENDENT_ROWS is not supported.
 *   inputs as for dsa_indexer_topk (w 16-byte aligned), plus
 *   idx     int32 [n_q][topk]  the forward's idx_out        d_score f32 [n_q][topk]
 *   outputs f32: dq_idx [n_q][n_heads][head_dim] (written), dk_idx [n_kv][head_dim] and
 *          dw [n_q][n_heads] (zeroed here, then accumulated; rows of dk_idx selected by
 *          several queries receive atomic adds, so the order of the additions, and the last
 *          bits, vary from run to run).  q_idx, k_idx, dq_idx, dk_idx 16-byte aligned.
 * ws: dsa_indexer_backward_workspace_size bytes, 256-byte aligned.  Errors: DSA_ERR_ARG,
 * DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA; device-side faults go to the
 * workspace status (dsa_workspace_status). */
dsa_status dsa_indexer_backward_workspace_size(const dsa_indexer_desc* desc, size_t* bytes);
dsa_status dsa_indexer_backward(const dsa_indexer_desc* desc, const void* q_idx, const void* k_idx, const float* w,
                                const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                                const float* rope_cs, int32_t rope_n_pos, const int32_t* idx, const float* d_score,
                                float* dq_idx, float* dk_idx, float* dw, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ paged caches ---- */

/* Paged decode caches (a serving layout; the pages describe per-query key ranges only -- the
 * Megatron-Bridge commits' per-query starts/ends -- so the paging is this library's own):
 * the index-key cache [n_pages * page_rows][d_I] bf16 (stored already rotated) and the
 * latent cache [n_pages * page_rows][576] bf16 hold pages of page_rows rows; query row t's
 * logical key j (j < seq_len[t]) sits at cache row
 *   block_table[t * max_pages + j / page_rows] * page_rows + j % page_rows.
 * All arrays are device memory owned by the caller.  page_rows must be DSA_PAGE_ROWS (one
 * 128-key indexer tile per page, so every tile is one TMA box). */
#define DSA_PAGE_ROWS 128
typedef struct dsa_paged_cache {
  const int32_t* block_table; /* [n_q][max_pages] int32 physical page ids                    */
  const int32_t* seq_len;     /* [n_q] int32: keys of row t are logical positions [0, seq_len) */
  int32_t max_pages;          /* columns of block_table                                       */
  int32_t n_pages;            /* pages in the cache arrays: desc->n_kv == n_pages * page_rows */
  int32_t page_rows;          /* DSA_PAGE_ROWS                                                */
} dsa_paged_cache;

/* dsa_indexer_topk over a paged, pre-rotated index-key cache: row t scores its logical keys
 * [0, seq_len[t]) and idx_out holds logical positions (offsets from 0), same selection and
 * order rules as dsa_indexer_topk.  Requires DSA_IDX_INDEPENDENT_ROWS, no DSA_IDX_ROPE_K,
 * n_heads == 64 (one row per key stream) and max_len <= max_pages * page_rows; the workspace
 * is dsa_indexer_workspace_size(desc).  A block-table entry outside [0, n_pages) is counted in
 * the workspace status.  Errors: those of dsa_indexer_topk, DSA_ERR_SHAPE (n_kv !=
 * n_pages * page_rows), DSA_ERR_UNSUPPORTED (page_rows, n_heads). */
dsa_status dsa_indexer_topk_paged(const dsa_indexer_desc* desc, const void* q_idx, const void* k_cache, const float* w,
                                  const int32_t* q_pos, const dsa_paged_cache* pages, const float* rope_cs,
                                  int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws, size_t ws_bytes,
                                  void* stream);

/* dsa_sparse_attn over a paged latent cache: idx[t] holds logical positions of row t (as
 * dsa_indexer_topk_paged writes them); an entry >= seq_len[t] or on a page outside the cache
 * is skipped and counted.  Always the per-token gather walk.  Workspace:
 * dsa_sparse_attn_workspace_size(desc).  Errors: those of dsa_sparse_attn, DSA_ERR_SHAPE,
 * DSA_ERR_UNSUPPORTED (page_rows). */
dsa_status dsa_sparse_attn_paged(const dsa_attn_desc* desc, const void* q, const void* kv_cache, const int32_t* idx,
                                 const dsa_paged_cache* pages, void* out, float* lse, void* ws, size_t ws_bytes,
                                 void* stream);

/* ------------------------------------------------------------------ MTP drafting ---- */

/* One step of multi-step MTP drafting with IndexShare ([EX] "MTP path: IndexShare +
 * KVShare": for multi-step MTP the indexer runs at the first step and the following steps
 * reuse its top-k indices; "Public config evidence": index_share_for_mtp_iteration).
 *   step == 0: dsa_indexer_topk of this step's query rows into mtp_idx, then
 *              dsa_sparse_attn with mtp_idx;
 *   step  > 0: no indexer work; dsa_sparse_attn of this step's q over its kv with the
 *              indices left in mtp_idx by step 0, read unchanged.
 * Row t of every step is the draft token of the same sequence t.  The indices are offsets
 * from ks[t], so every step must pass the same ks; a later step's range [ks_t, ke_t) may be
 * longer than step 0's (the drafts' own latent rows appended), and the step-0 selection,
 * all inside step 0's range, stays causal for it.  io: q_idx, k_idx and w are read at step 0
 * only (NULL allowed after); q, kv, out (and lse, optional) at every step.  mtp_idx:
 * caller-owned device buffer of n_q * topk int32, written at step 0 and only read after.
 * idx_desc is used at step 0 only; attn_desc describes this step (its n_kv may grow with the
 * step).  Workspace: dsa_layers_workspace_size(idx_desc, attn_desc) bytes.  Errors: those
 * of the two calls, DSA_ERR_ARG (step < 0, NULL io / mtp_idx / ws, missing tensors),
 * DSA_ERR_SHAPE (the descriptors disagree on n_q or topk). */
dsa_status dsa_mtp_indexshare_step(const dsa_indexer_desc* idx_desc, const dsa_attn_desc* attn_desc, int32_t step,
                                   const dsa_layer_io* io, const int32_t* ks, const int32_t* ke,
                                   const int32_t* q_pos, const int32_t* k_pos, const float* rope_cs,
                                   int32_t rope_n_pos, int32_t* mtp_idx, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ device status ---- */

/* Synchronise `stream`, read the device status word of workspace `ws`, and map it:
 * DSA_OK, DSA_ERR_TIMEOUT (a pipeline wait hit its bound) or DSA_ERR_DEVICE (bad index,
 * range or overflow).  The raw bits are stored in *device_bits when it is not NULL.
 * The word is cleared at the start of every call that takes the workspace. */
dsa_status dsa_workspace_status(const void* ws, void* stream, uint32_t* device_bits);

/* ------------------------------------------------------------------ profiling ------- */

/* Process-wide switch (off by default).  While on, every indexer call (dsa_indexer_topk,
 * its static-scratch variant and the full layers of indexshare_layers_forward) records CUDA
 * events on its stream between its phases, so that dsa_profile_indexer_last can report
 * device time per phase.  The events add no work to the kernels.  Not meant for calls that
 * run concurrently from several host threads.  The pages have no counterpart: this exists to
 * measure the score kernel on its own.  Errors: none (DSA_OK). */
dsa_status dsa_profile_enable(int32_t on);

/* Device time, in milliseconds, of each phase of the last profiled indexer call made on the
 * current device: ms[0] = RoPE of the index q and k, ms[1] = key-range plan, ms[2] = scores
 * with the streaming top-k (the tensor-core kernel), ms[3] = final top-k select.  Writes the
 * first min(n, 4) values; waits for that call to finish.  Errors: DSA_ERR_ARG (ms NULL or
 * n < 1), DSA_ERR_UNSUPPORTED (no profiled call yet on this device), DSA_ERR_CUDA. */
dsa_status dsa_profile_indexer_last(float* ms, int32_t n);

/* Launch log.  While profiling is on, every kernel launch of the library (in every call,
 * any stream) is also bracketed by two CUDA events on its stream and logged with its kind;
 * dsa_profile_enable(1) empties the log of every device.  dsa_profile_read waits for the
 * logged launches of the current device to finish and copies up to `cap` records, in launch
 * order, into out; *n receives the number logged.  The log holds 8192 records per device;
 * later launches are not logged and dsa_profile_read then returns DSA_ERR_WORKSPACE (the
 * records it copied are valid).  Errors: DSA_ERR_ARG, DSA_ERR_WORKSPACE, DSA_ERR_CUDA. */
enum {
  DSA_PROF_ROPE = 0,          /* index q or k RoPE pre-pass                                 */
  DSA_PROF_RANGES = 1,        /* key-range plan                                             */
  DSA_PROF_INDEXER = 2,       /* tcgen05 scores + streaming top-k                           */
  DSA_PROF_SELECT = 3,        /* final top-k select                                         */
  DSA_PROF_ATTN_PREP = 4,     /* attention pre-pass (tile counts or block masks)            */
  DSA_PROF_ATTN = 5,          /* sparse attention kernel                                    */
  DSA_PROF_ATTN_BWD = 6,      /* sparse attention backward                                  */
  DSA_PROF_PROJ = 7,          /* indexer projections                                        */
  DSA_PROF_INDEXER_BWD = 8    /* indexer backward                                           */
};
typedef struct dsa_profile_record {
  int32_t kind;   /* DSA_PROF_*                        */
  float ms;       /* device time of the launch, in ms  */
} dsa_profile_record;
dsa_status dsa_profile_read(dsa_profile_record* out, int32_t cap, int32_t* n);

/* ------------------------------------------------------------------ testing --------- */

/* Test hook for the bounded pipeline waits (the pages have no counterpart).  Every
 * mbarrier wait inside the library's pipelined kernels gives up after wait_ns nanoseconds of
 * device time (0 restores the default, 2 s): the waiting warp records a timeout in the
 * workspace status word (DSA_ERR_TIMEOUT from dsa_workspace_status), every other warp of its
 * block stops at its next wait, copies already in flight are allowed to land, and the kernel
 * returns -- the context stays usable.  stop_after_tiles >= 0 makes the TMA producer of the
 * indexer and sparse-attention kernels stop after that many tiles, so that the waits behind
 * it run out; -1 (the default) never stops.  Process-wide; applies to calls made after it.
 * Meant for tests only.  Errors: DSA_ERR_ARG (stop_after_tiles < -1). */
dsa_status dsa_debug_pipeline(int32_t stop_after_tiles, uint64_t wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
