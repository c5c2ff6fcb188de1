// The layer with its scratch memory in a fixed device array of this library,
// for callers that cannot allocate device memory. Such callers include code
// that runs while a CUDA graph is being captured or replayed, real-time or
// embedded loops that forbid cudaMalloc after start-up (it can synchronise
// the device and fail when memory is fragmented), and plug-in hosts that own
// the device allocator and give their plug-ins only input and output
// buffers.
//
// The scratch array below is part of the library image: every GPU that loads
// the library holds it until the process exits, whether or not this entry
// point is used. It is shared by all calls on a device and keeps the contents
// of the last call. The calls clear what has to start at zero themselves (the
// status word and the fp32 combine accumulator), so nothing carries over into
// the result. Two calls whose work overlaps on the GPU (different streams, or
// different host threads, without ordering between them) race on the array
// and may both produce wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"

namespace {

constexpr size_t kStaticScratchBytes = MOE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device. Host code may
// not take the array's address directly (the host-side symbol is only a
// stand-in), so it is looked up once per device with that device current.
void* static_scratch_on_current_device() {
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" moe_status moe_layer_forward_static(const moe_weights* w, const uint16_t* x, int T, uint16_t* y,
                                               void* stream) {
  const size_t need = moe_workspace_size(w, T);
  if (need == 0) return moe_layer_forward(w, x, T, y, nullptr, 0, stream);  // names the argument or shape error
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = static_scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  return moe_layer_forward(w, x, T, y, scratch, kStaticScratchBytes, stream);
}
