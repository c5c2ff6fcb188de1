// The layer with its scratch memory in a fixed device array of this library,
// for callers that cannot allocate device memory. Such callers include
// real-time or embedded loops that forbid cudaMalloc after start-up (it can
// synchronise the device and fail when memory is fragmented), and plug-in
// hosts that own the device allocator and give their plug-ins only input
// and output buffers.
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
#include "internal.h"

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

// Largest token count, at most the call's pass size, whose workspace fits the
// array (0 if even one token does not). The size grows with the token count,
// so a bisection finds it.
int tokens_fitting(const moe_weights* w, int T, const moe::Options& opt) {
  const int cap = moe::pass_tokens(T, opt);
  if (moe::pass_workspace_bytes(w, cap) <= kStaticScratchBytes) return cap;
  int lo = 0, hi = cap;  // size(lo) fits (or lo = 0), size(hi) does not
  while (hi - lo > 1) {
    const int mid = lo + (hi - lo) / 2;
    if (moe::pass_workspace_bytes(w, mid) <= kStaticScratchBytes)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" moe_status moe_layer_forward_static(const moe_weights* w, const uint16_t* x, int T, uint16_t* y,
                                               void* stream) {
  const moe::Options opt = moe::options_snapshot();
  if (moe_status s = moe::check_weights(w)) return s;
  if (T < 0 || T > moe::kMaxTokens) return MOE_ERR_ARG;
  if (T == 0) {  // a no-op, as for the workspace entry point
    moe::reset_launch_count();
    return MOE_OK;
  }
  if (!x || !y || !aligned16(x) || !aligned16(y) || x == y) return MOE_ERR_ARG;
  const int step = tokens_fitting(w, T, opt);
  if (step == 0) return MOE_ERR_WORKSPACE;
  void* scratch = static_scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  return moe::forward_passes(w, x, T, y, scratch, kStaticScratchBytes, stream, step, opt);
}

extern "C" moe_status moe_get_device_status_static(void* stream) {
  void* scratch = static_scratch_on_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  return moe_get_device_status(scratch, stream);  // the status word heads the array
}
