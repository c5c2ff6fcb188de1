// Dequantising dot products of the row-parallel (GEMV) kernels, on the CUDA
// cores ("Optimizing on-device inference for Apple Silicon", section
// "Optimise the single-row weight path").
//
// Per group of 64 weights w = s*q + b, so a dot product over a 32-code chunk
// of one group is s * sum(x*q) + b * sum(x). The codes enter the sum as fp32
// values 128 + q built by bit operations (the code placed into the mantissa
// of 128.0f), and 128 * sum(x) is removed per chunk. The per-chunk sums of x are
// computed once per staged row and shared by every weight row.
//
// Activations live in shared memory chunk-major: for a row of K values with
// nch = K/32 chunks, float4 number (jq * nch + c) holds values
// 32c+4jq..32c+4jq+3. Lane l working on chunk c = l + 32m reads consecutive
// float4s, as do the lanes reading consecutive 16-byte code chunks.
#pragma once

#include "common.cuh"

namespace moe {

// acc += sum_j x[j] * (128 + q_j) over the 8 codes of word w; xa holds
// activations 0..3 of the word, xb 4..7. Even and odd terms go to .x and .y.
// lo = w & 0x0F0F0F0F holds codes 0, 2, 4, 6 in its four bytes and hi the
// odd ones; one byte permute with 0x43000000 puts a code into bits 16..19 of
// the fp32 value 128.0, which is then exactly 128 + q (one instruction per
// code).
__device__ __forceinline__ float2 dot8_128(uint32_t w, float4 xa, float4 xb, float2 acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu, k128 = 0x43000000u;
  auto q = [&](uint32_t src, uint32_t byte_sel) { return __uint_as_float(__byte_perm(src, k128, byte_sel)); };
  acc = __ffma2_rn(make_float2(xa.x, xa.y), make_float2(q(lo, 0x7054), q(hi, 0x7054)), acc);
  acc = __ffma2_rn(make_float2(xa.z, xa.w), make_float2(q(lo, 0x7154), q(hi, 0x7154)), acc);
  acc = __ffma2_rn(make_float2(xb.x, xb.y), make_float2(q(lo, 0x7254), q(hi, 0x7254)), acc);
  acc = __ffma2_rn(make_float2(xb.z, xb.w), make_float2(q(lo, 0x7354), q(hi, 0x7354)), acc);
  return acc;
}

// s * sum(x*q) + b * sum(x) over one 32-code chunk of a row: w4 holds its
// codes, xv its 32 activations (chunk-major float4s), xsum their sum, s and b
// the bf16 scale and bias of its group.
__device__ __forceinline__ float chunk_dot_r(const uint4 w4, const float4 (&xv)[8], float xsum, uint16_t s,
                                             uint16_t b) {
  float2 d0 = make_float2(0.f, 0.f), d1 = d0;
  d0 = dot8_128(w4.x, xv[0], xv[1], d0);
  d1 = dot8_128(w4.y, xv[2], xv[3], d1);
  d0 = dot8_128(w4.z, xv[4], xv[5], d0);
  d1 = dot8_128(w4.w, xv[6], xv[7], d1);
  return bf16_to_f32(s) * ((d0.x + d0.y) + (d1.x + d1.y) - 128.f * xsum) + bf16_to_f32(b) * xsum;
}

// Stages 8 bf16 values (number q8 of a row) into a chunk-major fp32 row.
__device__ __forceinline__ void stage_bf16x8(float4* rowdst, int nch, int q8, uint4 v) {
  const int c = q8 >> 2, jq = (q8 & 3) * 2;
  rowdst[jq * nch + c] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
  rowdst[(jq + 1) * nch + c] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
}

// Per-chunk sums of `rows` staged rows (thread per (row, chunk)).
__device__ __forceinline__ void chunk_sums(const float4* xs4, float* xsum, int rows, int nch) {
  for (int q = threadIdx.x; q < rows * nch; q += blockDim.x) {
    const int r = q / nch, c = q % nch;
    const float4* xr = xs4 + size_t(r) * 8 * nch;
    float s = 0.f;
#pragma unroll
    for (int jq = 0; jq < 8; ++jq) {
      const float4 v = xr[jq * nch + c];
      s += (v.x + v.y) + (v.z + v.w);
    }
    xsum[q] = s;
  }
}

}  // namespace moe
