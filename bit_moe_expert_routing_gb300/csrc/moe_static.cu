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

// Largest token count, at most T, whose workspace fits the array (0 if even
// one token does not). The size grows with the token count up to the chunk
// size and is flat beyond it, so a bisection finds it.
int tokens_fitting(const moe_weights* w, int T) {
  if (moe_workspace_size(w, T) <= kStaticScratchBytes) return T;
  int lo = 0, hi = T;  // size(lo) fits (or lo = 0), size(hi) does not
  while (hi - lo > 1) {
    const int mid = lo + (hi - lo) / 2;
    if (moe_workspace_size(w, mid) <= kStaticScratchBytes)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

}  // namespace

extern "C" moe_status moe_layer_forward_static(const moe_weights* w, const uint16_t* x, int T, uint16_t* y,
                                               void* stream) {
  const size_t need = moe_workspace_size(w, T);
  if (need == 0 || T == 0) return moe_layer_forward(w, x, T, y, nullptr, 0, stream);  // names the error, or T = 0
  const int step = tokens_fitting(w, T);
  if (step == 0) return MOE_ERR_WORKSPACE;
  void* scratch = static_scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  if (!x || !y) return MOE_ERR_ARG;
  for (int t0 = 0; t0 < T; t0 += step) {
    const int n = T - t0 < step ? T - t0 : step;
    const size_t at = size_t(t0) * w->D;
    if (moe_status s = moe_layer_forward(w, x + at, n, y + at, scratch, kStaticScratchBytes, stream)) return s;
  }
  return MOE_OK;
}
