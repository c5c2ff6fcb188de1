// Device helpers shared by the kernels of the 4-bit MoE layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kGroup = 64;  // weights per quantisation group

// Workspace header, at offset 0 of every workspace.
struct WsHeader {
  int status;        // first device-side error (moe_status), 0 = none
  int detail;        // kernel-specific detail of that error
  unsigned counter;  // scratch counter (last-block patterns), reset by its user
  int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte slot");

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Records the first device-side error of a call in the workspace header.
__device__ __forceinline__ void report(WsHeader* hdr, int status, int detail) {
  if (atomicCAS(&hdr->status, 0, status) == 0) hdr->detail = detail;
}

// SiLU(g) * u with the hardware exponential and approximate division: a few
// ulp of fp32, far below the bf16 rounding of the result. For g below about
// -88 the denominator is +inf and the quotient the limit 0.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Low-half and high-half bf16 of a packed pair, as fp32.
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace moe

namespace moe {

// Raises a kernel's dynamic shared-memory limit once per device (host side).
bool ensure_smem_limit(const void* func, int bytes);

// Eight 4-bit codes of one word -> eight bf16 weights s*q + b, each rounded
// once to nearest even (the tensor-core operand format). out[i] holds
// elements 2i (low half) and 2i+1 (high half).
// 0x4300 | q is the bf16 value 128 + q (q in the low mantissa bits), so one
// AND-OR builds two of them; subtracting 128 is exact, and the fused
// multiply-add rounds s*q + b once.
__device__ __forceinline__ void dq8_bf16(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 b2, uint32_t out[4]) {
  const __nv_bfloat162 k128 = __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300));
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;  // (128+q_i, 128+q_{i+4})
    __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p), k128);
    __nv_bfloat162 r = __hfma2(q, s2, b2);
    v[i] = *reinterpret_cast<uint32_t*>(&r);
  }
  out[0] = __byte_perm(v[0], v[1], 0x5410);  // (w0, w1)
  out[1] = __byte_perm(v[2], v[3], 0x5410);  // (w2, w3)
  out[2] = __byte_perm(v[0], v[1], 0x7632);  // (w4, w5)
  out[3] = __byte_perm(v[2], v[3], 0x7632);  // (w6, w7)
}

// The same eight weights in the paired order (below): out[i] holds
// elements i (low half) and i + 4 (high half), with no reordering step. A
// matrix product over K is unchanged when both operands take this order
// inside every group of eight (the activations are permuted once to match).
__device__ __forceinline__ void dq8_bf16_paired(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 b2, uint32_t out[4]) {
  const __nv_bfloat162 k128 = __halves2bfloat162(__ushort_as_bfloat16(0x4300), __ushort_as_bfloat16(0x4300));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;  // (128+q_i, 128+q_{i+4})
    __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p), k128);
    __nv_bfloat162 r = __hfma2(q, s2, b2);
    out[i] = *reinterpret_cast<uint32_t*>(&r);
  }
}

// Paired order of eight consecutive K elements (positions 0..7 hold elements
// 0, 4, 1, 5, 2, 6, 3, 7): the order dq8_bf16_paired emits weights in.
// pair_order8_first/second(lo, hi) take elements 0..3 (lo) and 4..7 (hi), two bf16 per
// word, and returns positions 0..3 (first) or 4..7 (second) of the permuted
// chunk.
__device__ __forceinline__ uint2 pair_order8_first(uint2 lo, uint2 hi) {
  return make_uint2(__byte_perm(lo.x, hi.x, 0x5410), __byte_perm(lo.x, hi.x, 0x7632));  // (0,4), (1,5)
}
__device__ __forceinline__ uint2 pair_order8_second(uint2 lo, uint2 hi) {
  return make_uint2(__byte_perm(lo.y, hi.y, 0x5410), __byte_perm(lo.y, hi.y, 0x7632));  // (2,6), (3,7)
}

}  // namespace moe
