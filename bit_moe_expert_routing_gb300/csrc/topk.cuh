// Top-k selection of one token's router logits by one warp, shared by the
// routing kernels and the fused decode kernel.
#pragma once

#include <climits>

#include "common.cuh"

namespace moe {

// Top-k of one token's logits (larger logit first, lower expert index on
// ties) by one warp; lane l holds logits l, l+32, ... On return lane j < k
// holds slot j: its expert and its weight, the softmax renormalised over the
// k kept, exp(l_j - l_max) / sum.
// MPL >= ceil(E / 32) logits per lane (E <= 1024).
template <int MPL>
__device__ __forceinline__ void select_topk(const float* __restrict__ lg, int E, int k, int& myi, float& myw) {
  const int lane = threadIdx.x & 31;
  const int M = (E + 31) / 32;
  float v[MPL];
  unsigned taken = 0;
#pragma unroll
  for (int m = 0; m < MPL; ++m) {
    const int e = lane + 32 * m;
    v[m] = (m < M && e < E) ? lg[e] : 0.f;
    if (!(m < M && e < E)) taken |= 1u << m;
  }
  float first = 0.f, myv = 0.f;
  myi = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int m = 0; m < MPL; ++m) {
      const int e = lane + 32 * m;
      if (!((taken >> m) & 1u) && (v[m] > bv || (v[m] == bv && e < bi))) {
        bv = v[m];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) first = bv;
    if (lane == j) {
      myv = bv;
      myi = bi;
    }
  }
  const float ex = lane < k ? expf(myv - first) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  myw = ex / sum;
}

}  // namespace moe
