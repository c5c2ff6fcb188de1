// Inline-PTX wrappers shared by the kernels: shared-memory addresses,
// mbarriers with bounded waits, proxy fences and bulk (TMA) copies.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// About 2 s of SM cycles: far beyond any legal wait in these kernels.
constexpr long long kWaitLimit = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous proxy.
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// One try of a phase wait. The thread may be suspended in hardware (not
// issuing) until the phase completes or, at most, kTrySuspendNs pass, so a
// waiting warp does not take issue slots from the warps doing work.
constexpr uint32_t kTrySuspendNs = 20000;
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kTrySuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete. Gives up when the CTA's
// abort flag is set (unless draining) or after `limit` cycles (then sets the
// flag and records MOE_ERR_DEVICE_TIMEOUT with `site` as its detail). The flag
// and the clock are checked every 16 tries: the loop's own instructions take
// issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, WsHeader* hdr,
                                          long long limit = kWaitLimit, bool draining = false, int site = 100) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (!draining && *abort_flag) return false;
      if (clock64() - t0 > limit) {
        *abort_flag = 1;
        report(hdr, MOE_ERR_DEVICE_TIMEOUT, site);
        return false;
      }
    }
  }
}

// Programmatic dependent launch. A kernel launched with launch_pdl may start
// while the previous kernel of its stream is finishing: griddep_wait() returns
// once that kernel has completed and its memory writes are visible (at once
// for a kernel launched the ordinary way); griddep_launch() lets the next
// such kernel start. A kernel triggers only after its own wait, so a kernel
// that starts early can rely on everything before its predecessor.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Contiguous global -> shared copy by the TMA engine; completes `bytes` of
// the barrier's transaction count. Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

}  // namespace moe
