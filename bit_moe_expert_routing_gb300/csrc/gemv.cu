// Decode path for one to a few token rows: row-parallel dequantising GEMVs on
// the CUDA cores ("Optimizing on-device inference for Apple Silicon", sections
// "Optimise the single-row weight path" and "Reduce intermediate and state
// traffic"; the switch to matrix kernels above a row count follows
// "Why continuous batching halved LLM throughput on an M2 Mac mini").
//
//   gemv_gateup: one warp per (expert block, intermediate row i). Lanes stream
//     the gate and up rows of i with 128-bit loads (32 codes per load), dot
//     them with every token row of the block, reduce with shuffles and write
//     h = bf16(silu(g) * u) in the permuted order.
//   gemv_down: one warp per output column d. For each token it reads row d of
//     the down matrix of each of its k experts and of the shared expert, dots
//     it with h, scales by the routing weight and sums, then writes
//     y = bf16(sum). No atomics: the result is deterministic.
//
// The kernels are bound by weight reads, so each warp issues its weight loads
// before anything else (the activations are staged while those loads fly),
// and register use is capped so that four CTAs share an SM.
//
// Per group of 64 weights w = s*q + b, so a dot product over a 32-code chunk
// of one group is s * sum(x*q) + b * sum(x). The codes enter the sum as fp32
// values 128 + q built by bit operations (OR the code into the mantissa of
// 128.0f), and 128 * sum(x) is removed per chunk. The per-chunk sums of x are
// computed once per token and shared by every row.
//
// Activations live in shared memory chunk-major: for a row of K values with
// nch = K/32 chunks, float4 number (jq * nch + c) holds values 32c+4jq..32c+4jq+3.
// Lane l works on chunk c = l + 32m, so the lanes of a warp read consecutive
// float4s (no bank conflicts).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxGemvRows = 8;
constexpr int kGemvWarps = 8;

// fp32 value 128 + q of the nibble in bits 16..19 of w_shifted.
__device__ __forceinline__ float q128(uint32_t w_shifted) {
  return __uint_as_float((w_shifted & 0x000F0000u) | 0x43000000u);
}

// acc += sum_j x[j] * (128 + q_j) over the 8 codes of word w; xa holds
// activations 0..3 of the word, xb 4..7. Even and odd terms go to .x and .y.
__device__ __forceinline__ float2 dot8_128(uint32_t w, float4 xa, float4 xb, float2 acc) {
  const uint32_t sw = __byte_perm(w, 0, 0x1032);  // codes 0..3 into bits 16..31
  acc = __ffma2_rn(make_float2(xa.x, xa.y), make_float2(q128(sw), q128(sw >> 4)), acc);
  acc = __ffma2_rn(make_float2(xa.z, xa.w), make_float2(q128(sw >> 8), q128(sw >> 12)), acc);
  acc = __ffma2_rn(make_float2(xb.x, xb.y), make_float2(q128(w), q128(w >> 4)), acc);
  acc = __ffma2_rn(make_float2(xb.z, xb.w), make_float2(q128(w >> 8), q128(w >> 12)), acc);
  return acc;
}

// s * sum(x*q) + b * sum(x) over one 32-code chunk; sb = (scale, bias) bf16 pair.
__device__ __forceinline__ float chunk_dot(const uint4 w4, const float4* xr, int nch, int c, float xsum,
                                           uint32_t sb) {
  float2 d = make_float2(0.f, 0.f);
  d = dot8_128(w4.x, xr[0 * nch + c], xr[1 * nch + c], d);
  d = dot8_128(w4.y, xr[2 * nch + c], xr[3 * nch + c], d);
  d = dot8_128(w4.z, xr[4 * nch + c], xr[5 * nch + c], d);
  d = dot8_128(w4.w, xr[6 * nch + c], xr[7 * nch + c], d);
  return bf16lo(sb) * (d.x + d.y - 128.f * xsum) + bf16hi(sb) * xsum;
}

struct GemvArgs {
  const uint16_t* x;
  moe_qmatrix gate, up, down, s_gate, s_up, s_down;
  const int32_t* blocks;
  const int32_t* n_blocks;
  const int32_t* perm;
  const int32_t* inv;
  const int32_t* topk_idx;
  const float* topk_w;
  uint16_t* h;
  uint16_t* y;
  WsHeader* hdr;
  int T, D, E, k, I;
};

// Stages bf16 row `r` (K values, 16-byte aligned) into chunk-major fp32;
// called by all threads of the CTA for q8 = thread, thread + blockDim, ...
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

// Shared memory: xs4 [R][8*nch] float4 (chunk-major x rows), xsum [R][nch],
// then the gate and up results of the CTA's rows. Warp w streams row
// blockIdx.y * 4 + w/2 of the gate (even w) or up (odd w) matrix; the pair
// meets in shared memory for h = silu(g) * u. CPL = 32-code chunks per lane
// (ceil(D/1024)).
constexpr int kGateupRowsPerCta = kGemvWarps / 2;

template <int CPL>
__global__ void __launch_bounds__(kGemvWarps * 32, CPL == 1 ? 4 : 3) gemv_gateup_kernel(GemvArgs a) {
  extern __shared__ float4 gv_smem[];
  float4* xs4 = gv_smem;
  __shared__ float s_gu[kGemvWarps][kMaxGemvRows];
  if (blockIdx.x >= *a.n_blocks) return;
  const int g = a.blocks[3 * blockIdx.x], p0 = a.blocks[3 * blockIdx.x + 1], R = a.blocks[3 * blockIdx.x + 2];
  const int A = a.T * a.k;
  if (g < 0 || g > a.E || R < 1 || R > kMaxGemvRows || R > a.T || p0 < 0 || p0 + R > A + a.T) {
    if (threadIdx.x == 0) report(a.hdr, MOE_ERR_DEVICE_CHECK, 3);
    return;
  }
  const int D = a.D, I = a.I, nch = D / 32;
  float* xsum = reinterpret_cast<float*>(xs4 + size_t(R) * 8 * nch);
  const bool shared = (g == a.E);
  const int ex = shared ? 0 : g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const moe_qmatrix m = (warp & 1) ? (shared ? a.s_up : a.up) : (shared ? a.s_gate : a.gate);
  const int i = blockIdx.y * kGateupRowsPerCta + (warp >> 1);
  const bool row_ok = i < I;
  const size_t row = size_t(ex) * I + (row_ok ? i : 0);

  // this warp's weights first: they do not depend on x
  uint4 w4[CPL];
  uint32_t sb[CPL];
#pragma unroll
  for (int mm = 0; mm < CPL; ++mm) {
    const int c = lane + 32 * mm;
    w4[mm] = make_uint4(0u, 0u, 0u, 0u);
    sb[mm] = 0u;
    if (c < nch && row_ok) {
      w4[mm] = __ldcs(reinterpret_cast<const uint4*>(m.codes + row * (D / 8)) + c);
      sb[mm] = uint32_t(m.scales[row * (D / 64) + c / 2]) | (uint32_t(m.biases[row * (D / 64) + c / 2]) << 16);
    }
  }

  for (int q = threadIdx.x; q < R * (D / 8); q += blockDim.x) {
    const int r = q / (D / 8), q8 = q % (D / 8);
    const int p = p0 + r;
    const int t = shared ? p - A : a.perm[p] / a.k;
    stage_bf16x8(xs4 + size_t(r) * 8 * nch, nch, q8, *reinterpret_cast<const uint4*>(a.x + size_t(t) * D + q8 * 8));
  }
  __syncthreads();
  chunk_sums(xs4, xsum, R, nch);
  __syncthreads();

#pragma unroll 1
  for (int r = 0; r < R; ++r) {
    const float4* xr = xs4 + size_t(r) * 8 * nch;
    float v = 0.f;
#pragma unroll
    for (int mm = 0; mm < CPL; ++mm) {
      const int c = lane + 32 * mm;  // 32-code chunk c lies in group c/2
      if (c < nch) v += chunk_dot(w4[mm], xr, nch, c, xsum[r * nch + c], sb[mm]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) s_gu[warp][r] = v;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < kGateupRowsPerCta * R; q += blockDim.x) {
    const int rr = q / R, r = q % R, ii = blockIdx.y * kGateupRowsPerCta + rr;
    if (ii < I) a.h[size_t(p0 + r) * I + ii] = f32_to_bf16(silu_mul(s_gu[2 * rr][r], s_gu[2 * rr + 1][r]));
  }
}

// Shared memory: hs4 [T*(k+1)][8*nch] float4 (chunk-major h rows in
// (token, slot) order, slot k = shared expert), hsum [T*(k+1)][nch], and the
// routing weight of each row. One warp per output column d; the (slot, chunk)
// items of a token are spread over the lanes, kDownBatch per lane per pass.
constexpr int kDownBatch = 6;

__global__ void __launch_bounds__(kGemvWarps * 32, 4) gemv_down_kernel(GemvArgs a) {
  extern __shared__ float4 gv_smem[];
  const int T = a.T, k = a.k, I = a.I, D = a.D, nch = I / 32;
  const int nrows = T * (k + 1), A = T * k, nitems = (k + 1) * nch;
  float4* hs4 = gv_smem;
  float* hsum = reinterpret_cast<float*>(hs4 + size_t(nrows) * 8 * nch);
  float* s_w = hsum + nrows * nch;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d = blockIdx.x * kGemvWarps + warp;
  const bool d_ok = d < D;

  uint4 w4[kDownBatch];
  uint32_t sb[kDownBatch];
  auto load = [&](int t, int base) {
#pragma unroll
    for (int u = 0; u < kDownBatch; ++u) {
      const int it = base + 32 * u + lane;
      w4[u] = make_uint4(0u, 0u, 0u, 0u);
      sb[u] = 0u;
      if (d_ok && it < nitems) {
        const int j = it / nch, c = it % nch;
        const bool sh = (j == k);
        const int ex = sh ? 0 : a.topk_idx[t * k + j];
        const moe_qmatrix& m = sh ? a.s_down : a.down;
        const size_t row = size_t(ex) * D + d;
        w4[u] = __ldcs(reinterpret_cast<const uint4*>(m.codes + row * (I / 8)) + c);
        sb[u] = uint32_t(m.scales[row * (I / 64) + c / 2]) | (uint32_t(m.biases[row * (I / 64) + c / 2]) << 16);
      }
    }
  };
  load(0, 0);  // the first token's weights fly while h is staged

  for (int q = threadIdx.x; q < nrows * (I / 8); q += blockDim.x) {
    const int rr = q / (I / 8), q8 = q % (I / 8);
    const int t = rr / (k + 1), j = rr % (k + 1);
    const int p = j < k ? a.inv[t * k + j] : A + t;
    stage_bf16x8(hs4 + size_t(rr) * 8 * nch, nch, q8, *reinterpret_cast<const uint4*>(a.h + size_t(p) * I + q8 * 8));
  }
  for (int rr = threadIdx.x; rr < nrows; rr += blockDim.x) {
    const int t = rr / (k + 1), j = rr % (k + 1);
    s_w[rr] = j < k ? a.topk_w[t * k + j] : 1.f;
  }
  __syncthreads();
  chunk_sums(hs4, hsum, nrows, nch);
  __syncthreads();
  if (!d_ok) return;

  for (int t = 0; t < T; ++t) {
    float part = 0.f;
    for (int base = 0; base < nitems; base += 32 * kDownBatch) {
      if (t > 0 || base > 0) load(t, base);
#pragma unroll
      for (int u = 0; u < kDownBatch; ++u) {
        const int it = base + 32 * u + lane;
        if (it < nitems) {
          const int j = it / nch, c = it % nch;
          const int rr = t * (k + 1) + j;
          part += s_w[rr] * chunk_dot(w4[u], hs4 + size_t(rr) * 8 * nch, nch, c, hsum[rr * nch + c], sb[u]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) a.y[size_t(t) * D + d] = f32_to_bf16(part);
  }
}

size_t gateup_smem(const Ctx& c) {
  return size_t(std::min(c.T, kMaxGemvRows)) * (size_t(c.D) * 4 + size_t(c.D / 32) * 4);
}
size_t down_smem(const Ctx& c) {
  return size_t(c.T) * (c.k + 1) * (size_t(c.I) * 4 + size_t(c.I / 32) * 4 + 4);
}

}  // namespace

bool gemv_supported(const Ctx& c) {
  return c.T >= 1 && c.T <= kMaxGemvRows && c.D <= 4096 && gateup_smem(c) <= 200 * 1024 &&
         down_smem(c) <= 200 * 1024;
}

cudaError_t gemv(const Ctx& c) {
  const moe_weights* w = c.w;
  GemvArgs a{c.x, w->gate, w->up, w->down, w->s_gate, w->s_up, w->s_down, c.blocks, c.n_blocks,
             c.perm, c.inv, c.topk_idx, c.topk_w, c.h, c.y, c.hdr, c.T, c.D, c.E, c.k, c.I};
  const size_t s1 = gateup_smem(c), s2 = down_smem(c);
  const int cpl = (c.D / 32 + 31) / 32;
  void (*gk)(GemvArgs) = cpl <= 1 ? gemv_gateup_kernel<1> : cpl <= 2 ? gemv_gateup_kernel<2> : gemv_gateup_kernel<4>;
  if (!ensure_smem_limit(reinterpret_cast<const void*>(gk), int(s1)) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(gemv_down_kernel), int(s2)))
    return cudaErrorInvalidValue;
  cudaError_t err;
  gk<<<dim3(c.max_blocks, (c.I + kGateupRowsPerCta - 1) / kGateupRowsPerCta), kGemvWarps * 32, s1, c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("gemv_gateup", c.stream);
  gemv_down_kernel<<<(c.D + kGemvWarps - 1) / kGemvWarps, kGemvWarps * 32, s2, c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("gemv_down", c.stream);
  return cudaSuccess;
}

}  // namespace moe
