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
//     it with h, scales by the routing weight and sums in slot order, then
//     writes y = bf16(sum). No atomics: the result is deterministic.
//
// Per group of 64 weights w = s*q + b, so a dot product over a 32-code chunk
// of one group is s * sum(x*q) + b * sum(x). The codes enter the sum as
// fp32 values 128 + q built by bit operations (OR the code into the mantissa
// of 128.0f), and 128 * sum(x) is removed per chunk. The per-chunk sums of x
// are computed once per token and shared by every row.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxGemvRows = 8;
constexpr int kGemvWarps = 8;

// fp32 value 128 + q for the code at bits [sh, sh+3] of w, for sh in {16..28}
// after the caller has shifted the nibble into bits 16..19.
__device__ __forceinline__ float q128(uint32_t w_shifted) {
  return __uint_as_float((w_shifted & 0x000F0000u) | 0x43000000u);
}

// sum_j x[j] * (128 + q_j) over the 8 codes of one word, packed in pairs.
// x8 holds the 8 activations in element order.
__device__ __forceinline__ float2 dot8_128(uint32_t w, const float* x8, float2 acc) {
  // codes 4..7 sit at bits 16..31; codes 0..3 at bits 0..15 (swap halves)
  const uint32_t sw = __byte_perm(w, 0, 0x1032);
  const float q0 = q128(sw), q1 = q128(sw >> 4), q2 = q128(sw >> 8), q3 = q128(sw >> 12);
  const float q4 = q128(w), q5 = q128(w >> 4), q6 = q128(w >> 8), q7 = q128(w >> 12);
  acc = __ffma2_rn(make_float2(x8[0], x8[1]), make_float2(q0, q1), acc);
  acc = __ffma2_rn(make_float2(x8[2], x8[3]), make_float2(q2, q3), acc);
  acc = __ffma2_rn(make_float2(x8[4], x8[5]), make_float2(q4, q5), acc);
  acc = __ffma2_rn(make_float2(x8[6], x8[7]), make_float2(q6, q7), acc);
  return acc;
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

// Shared memory: xs [R][D] fp32, xsum [R][D/32] fp32 (sum of each 32-chunk).
// One warp per intermediate row i; CPL = 32-code chunks per lane
// (ceil(D/1024)). The warp issues its weight loads before the CTA stages x.
template <int CPL>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_gateup_kernel(GemvArgs a) {
  extern __shared__ float4 gv_smem[];
  float* xs = reinterpret_cast<float*>(gv_smem);
  if (blockIdx.x >= *a.n_blocks) return;
  const int g = a.blocks[3 * blockIdx.x], p0 = a.blocks[3 * blockIdx.x + 1], R = a.blocks[3 * blockIdx.x + 2];
  const int A = a.T * a.k;
  if (g < 0 || g > a.E || R < 1 || R > kMaxGemvRows || R > a.T || p0 < 0 || p0 + R > A + a.T) {
    if (threadIdx.x == 0) report(a.hdr, MOE_ERR_DEVICE_CHECK, 3);
    return;
  }
  const int D = a.D, I = a.I, nch = D / 32;
  float* xsum = xs + R * D;
  const bool shared = (g == a.E);
  const int ex = shared ? 0 : g;
  const moe_qmatrix mg = shared ? a.s_gate : a.gate;
  const moe_qmatrix mu = shared ? a.s_up : a.up;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.y * kGemvWarps + warp;
  const bool row_ok = i < I;
  const size_t row = size_t(ex) * I + (row_ok ? i : 0);

  uint4 gw[CPL], uw[CPL];
  uint32_t gsb[CPL], usb[CPL];  // (scale, bias) bf16 pairs
#pragma unroll
  for (int m = 0; m < CPL; ++m) {
    const int c = lane + 32 * m;
    gw[m] = uw[m] = make_uint4(0u, 0u, 0u, 0u);
    gsb[m] = usb[m] = 0u;
    if (c < nch && row_ok) {
      gw[m] = __ldcs(reinterpret_cast<const uint4*>(mg.codes + row * (D / 8)) + c);
      uw[m] = __ldcs(reinterpret_cast<const uint4*>(mu.codes + row * (D / 8)) + c);
      gsb[m] = uint32_t(mg.scales[row * (D / 64) + c / 2]) | (uint32_t(mg.biases[row * (D / 64) + c / 2]) << 16);
      usb[m] = uint32_t(mu.scales[row * (D / 64) + c / 2]) | (uint32_t(mu.biases[row * (D / 64) + c / 2]) << 16);
    }
  }

  // token rows of this block, and the per-chunk sums
  for (int q = threadIdx.x; q < R * D / 8; q += blockDim.x) {
    const int r = q / (D / 8), c8 = q % (D / 8);
    const int p = p0 + r;
    const int t = shared ? p - A : a.perm[p] / a.k;
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + size_t(t) * D + c8 * 8);
    float* dst = xs + r * D + c8 * 8;
    dst[0] = bf16lo(v.x); dst[1] = bf16hi(v.x); dst[2] = bf16lo(v.y); dst[3] = bf16hi(v.y);
    dst[4] = bf16lo(v.z); dst[5] = bf16hi(v.z); dst[6] = bf16lo(v.w); dst[7] = bf16hi(v.w);
  }
  __syncthreads();
  for (int q = threadIdx.x; q < R * nch; q += blockDim.x) {
    const float* src = xs + (q / nch) * D + (q % nch) * 32;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) s += src[j];
    xsum[q] = s;
  }
  __syncthreads();
  if (!row_ok) return;

#pragma unroll 1
  for (int r = 0; r < R; ++r) {
    const float* xr = xs + r * D;
    float gv = 0.f, uv = 0.f;
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
      const int c = lane + 32 * m;  // 32-code chunk c lies in group c/2
      if (c < nch) {
        const float* x32 = xr + c * 32;
        float2 dg = make_float2(0.f, 0.f), du = make_float2(0.f, 0.f);
        dg = dot8_128(gw[m].x, x32 + 0, dg);  du = dot8_128(uw[m].x, x32 + 0, du);
        dg = dot8_128(gw[m].y, x32 + 8, dg);  du = dot8_128(uw[m].y, x32 + 8, du);
        dg = dot8_128(gw[m].z, x32 + 16, dg); du = dot8_128(uw[m].z, x32 + 16, du);
        dg = dot8_128(gw[m].w, x32 + 24, dg); du = dot8_128(uw[m].w, x32 + 24, du);
        const float sx = xsum[r * nch + c];
        gv += bf16lo(gsb[m]) * (dg.x + dg.y - 128.f * sx) + bf16hi(gsb[m]) * sx;
        uv += bf16lo(usb[m]) * (du.x + du.y - 128.f * sx) + bf16hi(usb[m]) * sx;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      gv += __shfl_xor_sync(0xffffffffu, gv, off);
      uv += __shfl_xor_sync(0xffffffffu, uv, off);
    }
    if (lane == 0) a.h[size_t(p0 + r) * I + i] = f32_to_bf16(silu_mul(gv, uv));
  }
}

// Shared memory: hs [T*(k+1)][I] fp32 (rows in (token, slot) order, slot k =
// shared expert) and hsum [T*(k+1)][I/32]. One warp per output column d and
// token: the (slot, chunk) items of all k+1 rows are spread over the lanes and
// loaded in batches of kDownBatch per lane before any arithmetic.
constexpr int kDownBatch = 4;

__global__ void __launch_bounds__(kGemvWarps * 32) gemv_down_kernel(GemvArgs a) {
  extern __shared__ float4 gv_smem[];
  float* hs = reinterpret_cast<float*>(gv_smem);
  const int T = a.T, k = a.k, I = a.I, D = a.D, nch = I / 32;
  const int nrows = T * (k + 1);
  float* hsum = hs + size_t(nrows) * I;
  const int A = T * k;
  for (int i = threadIdx.x; i < nrows * I / 8; i += blockDim.x) {
    const int rr = i / (I / 8), c8 = i % (I / 8);
    const int t = rr / (k + 1), j = rr % (k + 1);
    const int p = j < k ? a.inv[t * k + j] : A + t;
    const uint4 v = *reinterpret_cast<const uint4*>(a.h + size_t(p) * I + c8 * 8);
    float* dst = hs + size_t(rr) * I + c8 * 8;
    dst[0] = bf16lo(v.x); dst[1] = bf16hi(v.x); dst[2] = bf16lo(v.y); dst[3] = bf16hi(v.y);
    dst[4] = bf16lo(v.z); dst[5] = bf16hi(v.z); dst[6] = bf16lo(v.w); dst[7] = bf16hi(v.w);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nrows * nch; i += blockDim.x) {
    const float* src = hs + size_t(i / nch) * I + (i % nch) * 32;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) s += src[j];
    hsum[i] = s;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d = blockIdx.x * kGemvWarps + warp;
  if (d >= D) return;
  const int nitems = (k + 1) * nch;
  for (int t = 0; t < T; ++t) {
    float part = 0.f;
    for (int base = 0; base < nitems; base += 32 * kDownBatch) {
      uint4 w4[kDownBatch];
      uint16_t sb[kDownBatch][2];
      float wgt[kDownBatch];
      int hrow[kDownBatch], cc[kDownBatch];
#pragma unroll
      for (int u = 0; u < kDownBatch; ++u) {
        const int it = base + 32 * u + lane;
        w4[u] = make_uint4(0u, 0u, 0u, 0u);
        sb[u][0] = sb[u][1] = 0;
        wgt[u] = 0.f;
        hrow[u] = 0;
        cc[u] = 0;
        if (it < nitems) {
          const int j = it / nch, c = it % nch;
          const bool sh = (j == k);
          const int ex = sh ? 0 : a.topk_idx[t * k + j];
          const moe_qmatrix& m = sh ? a.s_down : a.down;
          const size_t row = size_t(ex) * D + d;
          w4[u] = __ldcs(reinterpret_cast<const uint4*>(m.codes + row * (I / 8)) + c);
          sb[u][0] = m.scales[row * (I / 64) + c / 2];
          sb[u][1] = m.biases[row * (I / 64) + c / 2];
          wgt[u] = sh ? 1.f : a.topk_w[t * k + j];
          hrow[u] = t * (k + 1) + j;
          cc[u] = c;
        }
      }
#pragma unroll
      for (int u = 0; u < kDownBatch; ++u) {
        const float* hr = hs + size_t(hrow[u]) * I + cc[u] * 32;
        const float sx = hsum[hrow[u] * nch + cc[u]];
        float2 dd = make_float2(0.f, 0.f);
        dd = dot8_128(w4[u].x, hr + 0, dd);
        dd = dot8_128(w4[u].y, hr + 8, dd);
        dd = dot8_128(w4[u].z, hr + 16, dd);
        dd = dot8_128(w4[u].w, hr + 24, dd);
        const float s = bf16_to_f32(sb[u][0]), b = bf16_to_f32(sb[u][1]);
        part += wgt[u] * (s * (dd.x + dd.y - 128.f * sx) + b * sx);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) a.y[size_t(t) * D + d] = f32_to_bf16(part);
  }
}

size_t gateup_smem(const Ctx& c) { return sizeof(float) * size_t(std::min(c.T, kMaxGemvRows)) * (c.D + c.D / 32); }
size_t down_smem(const Ctx& c) { return sizeof(float) * size_t(c.T) * (c.k + 1) * (c.I + c.I / 32); }

}  // namespace

bool gemv_supported(const Ctx& c) {
  return c.T >= 1 && c.T <= kMaxGemvRows && c.D <= 4096 && gateup_smem(c) <= 200 * 1024 && down_smem(c) <= 200 * 1024;
}

cudaError_t gemv(const Ctx& c) {
  const moe_weights* w = c.w;
  GemvArgs a{c.x, w->gate, w->up, w->down, w->s_gate, w->s_up, w->s_down, c.blocks, c.n_blocks,
             c.perm, c.inv, c.topk_idx, c.topk_w, c.h, c.y, c.hdr, c.T, c.D, c.E, c.k, c.I};
  const size_t s1 = gateup_smem(c), s2 = down_smem(c);
  cudaError_t err;
  const int cpl = (c.D / 32 + 31) / 32;
  void (*gk)(GemvArgs) = cpl <= 1 ? gemv_gateup_kernel<1> : cpl <= 2 ? gemv_gateup_kernel<2> : gemv_gateup_kernel<4>;
  if (!ensure_smem_limit(reinterpret_cast<const void*>(gk), int(s1)) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(gemv_down_kernel), int(s2)))
    return cudaErrorInvalidValue;
  const int rows_per_cta = kGemvWarps;
  gk<<<dim3(c.max_blocks, (c.I + rows_per_cta - 1) / rows_per_cta), kGemvWarps * 32, s1,
                       c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("gemv_gateup", c.stream);
  gemv_down_kernel<<<(c.D + kGemvWarps - 1) / kGemvWarps, kGemvWarps * 32, s2, c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("gemv_down", c.stream);
  return cudaSuccess;
}

}  // namespace moe
