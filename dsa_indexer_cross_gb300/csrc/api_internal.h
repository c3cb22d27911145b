// Internal entry points shared between the C-ABI translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

// Workspace bytes of dsa_indexer_topk for `d` on the current device (validates `d`).
dsa_status indexer_workspace_bytes(const dsa_indexer_desc* d, size_t* bytes);

// dsa_indexer_topk on an explicit workspace (clears its status header first).
dsa_status indexer_run(const dsa_indexer_desc* d, const void* q_idx, const void* k_idx, const float* w,
                       const int32_t* q_pos, const int32_t* k_pos, const int32_t* ks, const int32_t* ke,
                       const float* rope_cs, int32_t rope_n_pos, int32_t* idx_out, float* score_out, void* ws,
                       size_t ws_bytes, cudaStream_t st);

// Records `msg` as the calling thread's last error and returns `s`.
dsa_status set_error(dsa_status s, const char* msg);

}  // namespace dsa
