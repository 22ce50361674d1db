// moe_noalloc.cu -- a W4A4 forward for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: plugins that run inside a host
// framework which owns every device allocation (and counts or pools them),
// code that runs while a CUDA graph is being captured on a stream whose
// allocator is locked, and embedded runtimes that work inside a fixed memory
// budget set at start-up.  Such a caller can still pass its own inputs and
// outputs, but has no way to hand the layer a scratch workspace.  For them this
// file keeps the forward's scratch in one file-scope device array of fixed size
// that is reserved when the library is loaded on a device and held until the
// process exits.  Nothing here allocates, frees or calls an allocating routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_nvfp4.h"

namespace {

// Maximum scratch of the allocation-free forward: 64 MiB on every device that
// loads the library.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// The scratch itself.  Host code must never pass this name to a kernel: on the
// host it is only a stand-in symbol, not a device address.  The device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Per-device set-up, run on the first call on each device with that device
// current: look up the device address of the scratch array.  The address is
// kept for the life of the process; a cudaDeviceReset on that device makes it
// stale (the array is re-created at a new address), so callers must not reset a
// device on which they use this entry point.
moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_nvfp4_forward_noalloc(const moe_dims* d, const moe_nvfp4_weights* w,
                                                int32_t T, int32_t K, const uint8_t* codes,
                                                const uint8_t* sf, const float* scale,
                                                const int32_t* topk_ids, const float* topk_w,
                                                void* out_bf16, moe_stream_t stream) {
  // the shape checks of moe_nvfp4_forward first, so a bad shape gets the same
  // status code here as there; then the size of the fixed scratch
  moe_ws_layout L;
  const moe_status shape = moe_nvfp4_workspace_layout(d, T, K, 0, &L);
  if (shape != MOE_OK) return shape;
  if (L.total > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  moe_status st = scratch_for_current_device(&scratch);
  if (st != MOE_OK) return st;
  // The forward rewrites the scratch's status words itself (in its routing
  // step); every other scratch region is written before it is read, so
  // whatever an earlier call left in the array does not matter.
  return moe_nvfp4_forward(d, w, T, K, codes, sf, scale, topk_ids, topk_w, out_bf16, scratch,
                           kNoAllocScratchBytes, stream);
}
