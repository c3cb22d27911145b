// dsa_indexer_topk_static: the indexer + top-k entry point for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a plugin that a host framework calls
// with only its input and output buffers (the framework owns the device allocator and
// exposes none of it), or a latency-critical loop in which a cudaMalloc, with its implicit
// device synchronisation, is not acceptable.  This entry point runs exactly the same kernels
// as dsa_indexer_topk but keeps its scratch (rotated q/k, key ranges, candidate buffers and
// the status word) in one file-scope device array of DSA_STATIC_SCRATCH_BYTES per GPU.  It
// calls no allocation routine.
//
// Set-up: the first call on a device (with that device current) looks up the array's
// device address once with cudaGetSymbolAddress and caches it; make that first call before
// any stream capture.  The cached address belongs to the device's primary context, so the
// entry point must not be used again after that context is reset.  Every call on a device
// shares the array and it keeps the previous call's contents: the status word is cleared at
// the start of each call and every other scratch word is written before it is read.  Calls
// whose work overlaps on the GPU (other streams, other host threads) race on the array and
// must be serialised by the caller.  dsa_indexer_static_status reads the status word of the
// last call (a device-to-host copy of the array's first 256 bytes; nothing is allocated).
#include <mutex>

#include "../../include/dsa.h"

#include "api_internal.h"
#include "kernels.h"

namespace dsa {
namespace {

static __device__ __align__(256) uint8_t g_static_scratch[DSA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
dsa_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return set_error(DSA_ERR_UNSUPPORTED, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) return set_error(DSA_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_indexer_topk_static(const dsa_indexer_desc* desc, const void* q_idx, const void* k_idx,
                                              const float* w, const int32_t* q_pos, const int32_t* k_pos,
                                              const int32_t* ks, const int32_t* ke, const float* rope_cs,
                                              int32_t rope_n_pos, int32_t* idx_out, float* score_out,
                                              void* stream) {
  size_t need = 0;
  dsa_status s = dsa::indexer_workspace_bytes(desc, &need);
  if (s != DSA_OK) return s;
  if (need > DSA_STATIC_SCRATCH_BYTES)
    return dsa::set_error(DSA_ERR_WORKSPACE,
                          "problem needs more scratch than the static array holds (DSA_STATIC_SCRATCH_BYTES); "
                          "use dsa_indexer_topk with a caller workspace");
  void* ws = nullptr;
  if ((s = dsa::scratch_address(&ws)) != DSA_OK) return s;
  return dsa::indexer_run(desc, q_idx, k_idx, w, q_pos, k_pos, ks, ke, rope_cs, rope_n_pos, idx_out, score_out, ws,
                          DSA_STATIC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_indexer_static_status(void* stream, uint32_t* device_bits) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return dsa::set_error(DSA_ERR_CUDA, "cudaGetDevice failed");
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(dsa::g_mu);
    if (dev >= 0 && dev < dsa::kMaxDevices) ws = dsa::g_addr[dev];
  }
  if (!ws) return dsa::set_error(DSA_ERR_UNSUPPORTED, "no dsa_indexer_topk_static call has been made on this device");
  return dsa_workspace_status(ws, stream, device_bits);
}
