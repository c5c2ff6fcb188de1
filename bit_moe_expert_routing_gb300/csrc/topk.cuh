// Top-k selection of one token's router logits by one warp, shared by the
// routing kernels and the fused decode kernel.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving map of a logit onto an unsigned key: a larger float gives
// a larger key. NaN is taken as -inf and -0 as +0, so floats that compare
// equal give equal keys; every real logit's key is above 0, the key of an
// empty or taken place.
__device__ __forceinline__ unsigned logit_key(float v) {
  if (v != v) v = -INFINITY;
  if (v == 0.f) v = 0.f;
  const unsigned b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The logits of one token as keys, lane l holding logits l, l+32, ...:
// MPL >= ceil(E / 32) keys per lane (E <= 1024), 0 past E. L2 = true reads
// the logits through L2 only (they were written by other CTAs of the grid).
template <int MPL, bool L2 = false>
__device__ __forceinline__ void load_logit_keys(const float* __restrict__ lg, int E, unsigned (&key)[MPL]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < MPL; ++m) {
    const int e = lane + 32 * m;
    key[m] = e < E ? logit_key(L2 ? __ldcg(lg + e) : lg[e]) : 0u;
  }
}

// Top-k of one token's keys (larger logit first, lower expert index on ties)
// by one warp. On return lane j < k holds slot j: its expert and its weight,
// the softmax renormalised over the k kept, exp(l_j - l_max) / sum. The keys
// of the chosen places are cleared.
// Each of the k rounds takes the warp's largest key with one max reduction
// and, among the places holding it, the lowest expert index with one min
// reduction (redux.sync), then clears that place.
template <int MPL>
__device__ __forceinline__ void select_topk_keys(unsigned (&key)[MPL], int k, int& myi, float& myw) {
  const int lane = threadIdx.x & 31;
  float first = 0.f, myv = 0.f;
  myi = 0;
  for (int j = 0; j < k; ++j) {
    unsigned lb = key[0];
    int lm = 0;
#pragma unroll
    for (int m = 1; m < MPL; ++m)
      if (key[m] > lb) {  // strict: the lowest place of equal keys stays
        lb = key[m];
        lm = m;
      }
    const unsigned top = __reduce_max_sync(0xffffffffu, lb);
    const unsigned bi = __reduce_min_sync(0xffffffffu, lb == top ? unsigned(lane + 32 * lm) : 0xffffffffu);
#pragma unroll
    for (int m = 0; m < MPL; ++m)
      if (unsigned(lane + 32 * m) == bi) key[m] = 0u;
    const float bv = key_logit(top);
    if (j == 0) first = bv;
    if (lane == j) {
      myv = bv;
      myi = int(bi);
    }
  }
  const float ex = lane < k ? expf(myv - first) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  myw = ex / sum;
}

// Top-k of one token's logits: load_logit_keys, then select_topk_keys.
template <int MPL, bool L2 = false>
__device__ __forceinline__ void select_topk(const float* __restrict__ lg, int E, int k, int& myi, float& myw) {
  unsigned key[MPL];
  load_logit_keys<MPL, L2>(lg, E, key);
  select_topk_keys<MPL>(key, k, myi, myw);
}

}  // namespace moe
