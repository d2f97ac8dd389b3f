// topk_noalloc.cu — dsv_topk_blocks for callers that cannot allocate device memory.
//
// The DSV pages have no counterpart of this entry point; it exists for
// deployment.  Some callers of the top-k cannot call cudaMalloc (or any
// allocating routine, torch's caching allocator included): code that runs
// while a CUDA graph is being captured on another thread, plugins embedded in
// a host framework that owns the whole device heap, or real-time loops where
// an allocation may block or fail.  They pass scores and output lists as
// usual; the scratch space the top-k needs (the group x block bitmask and the
// per-block counts) comes from a fixed device array that this file declares.
//
// That array is DSV_TOPK_NOALLOC_SCRATCH_BYTES (64 MiB) and is held on every
// GPU that loads libdsv until the process exits.  Its device address is looked
// up once per device, with that device current, on the first call made on it;
// make that first call before any stream capture.  All calls share the array
// and it keeps the last call's contents: nothing in it has to start at zero
// (every mask word and every count a call reads is written earlier in the
// same call), but two calls whose kernels overlap on the GPU race on it.
#include <mutex>

#include "dsv_launch.h"

namespace {

constexpr size_t kScratchBytes = DSV_TOPK_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// In host code this name is only a stand-in: kernels must be given the device
// address returned by cudaGetSymbolAddress, never the host-side symbol.
static __device__ __align__(256) unsigned char g_topk_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" dsv_status dsv_topk_blocks_noalloc(const float* scores, dsv_shape s, const int32_t* k_per_head,
                                              int32_t* fwd_ptr, int32_t* fwd_col, int32_t* bwd_ptr,
                                              int32_t* bwd_col, dsv_stream_t stream) {
  const size_t need = dsv_topk_workspace_bytes(s);
  if (need > kScratchBytes) return DSV_ERR_UNSUPPORTED;  // problem too large for the fixed scratch
  void* ws = nullptr;
  if (need > 0 && scratch_address(&ws) != cudaSuccess) return DSV_ERR_CUDA;
  return dsv_topk_blocks(scores, s, k_per_head, fwd_ptr, fwd_col, bwd_ptr, bwd_col, ws, kScratchBytes, stream);
}
