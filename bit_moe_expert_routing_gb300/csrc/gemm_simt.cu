// Grouped GEMMs on the CUDA cores (fp32 FMA). This is the comparison
// baseline for the tensor-core kernels and the simplest complete form of the
// prefill expert path ("Optimizing on-device inference for Apple Silicon",
// sections "Dequantise weights during matrix multiplication" and "Reduce
// intermediate and state traffic"):
//   gate/up: for each block-map entry (expert, up to 128 permuted rows) and 64
//     intermediate columns: g = x_rows . dq(W_gate)^T, u = x_rows . dq(W_up)^T,
//     h = bf16(silu(g) * u) in the permuted order;
//   down: for each entry and 64 output columns: y_acc[t] += w[t,j] * (h . dq(W_down)^T),
//     shared expert rows with weight 1;
//   then y = bf16(y_acc).
// Weights are dequantised one 64-wide group at a time into shared memory and
// never exist expanded in global memory.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int SBM = 128, SBN = 64, SBK = 64;

struct SimtArgs {
  const uint16_t* x;  // gate/up A source
  const uint16_t* h;  // down A source
  moe_qmatrix m0, m1;       // routed: gate, up (or down in m0)
  moe_qmatrix s0, s1;       // shared
  const int32_t* blocks;
  const int32_t* n_blocks;
  const int32_t* perm;
  const float* topk_w;
  uint16_t* h_out;
  float* y_acc;
  WsHeader* hdr;
  int T, D, E, k, I;
};

// Dequantises 8 codes of one word into fp32: s*q + b (one fp32 rounding).
__device__ __forceinline__ void dq8(uint32_t word, float s, float b, float* out) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float q = __uint_as_float(0x4B000000u | ((word >> (4 * j)) & 0xFu)) - 8388608.0f;
    out[j] = fmaf(s, q, b);
  }
}

template <bool GATEUP>
__global__ void __launch_bounds__(256) gemm_simt_kernel(SimtArgs a) {
  constexpr int NB = GATEUP ? 2 : 1;
  extern __shared__ float4 simt_smem[];
  float (*As)[SBM] = reinterpret_cast<float (*)[SBM]>(simt_smem);
  float (*Bs)[SBK][SBN] = reinterpret_cast<float (*)[SBK][SBN]>(&As[SBK][0]);
  __shared__ int s_row_src[SBM];  // token (gate/up) or permuted row (down) of each tile row
  __shared__ float s_row_w[SBM];

  if (blockIdx.x >= *a.n_blocks) return;
  const int g = a.blocks[3 * blockIdx.x], p0 = a.blocks[3 * blockIdx.x + 1], R = a.blocks[3 * blockIdx.x + 2];
  const int A = a.T * a.k;
  if (g < 0 || g > a.E || R < 1 || R > SBM || p0 < 0 || p0 + R > A + a.T) {
    if (threadIdx.x == 0) report(a.hdr, MOE_ERR_DEVICE_CHECK, 2);
    return;
  }
  const bool shared = (g == a.E);
  const int ex = shared ? 0 : g;
  const int K = GATEUP ? a.D : a.I;      // reduction length
  const int N = GATEUP ? a.I : a.D;      // output columns of the matrix
  const int n0 = blockIdx.y * SBN;
  const moe_qmatrix m0 = shared ? a.s0 : a.m0;
  const moe_qmatrix m1 = shared ? a.s1 : a.m1;

  for (int r = threadIdx.x; r < SBM; r += blockDim.x) {
    int src = -1;
    float wgt = 0.f;
    if (r < R) {
      const int p = p0 + r;
      if (shared) {
        src = GATEUP ? (p - A) : p;
        wgt = 1.f;
      } else {
        const int asg = a.perm[p];
        src = GATEUP ? asg / a.k : p;
        wgt = a.topk_w[asg];
      }
      if (!GATEUP) s_row_w[r] = wgt;
    }
    s_row_src[r] = src;
    if (GATEUP) s_row_w[r] = 0.f;
  }
  __syncthreads();

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[NB][8][4];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[b][i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += SBK) {
    // A tile: row r = tid/2, 32 consecutive elements of half tid%2
    {
      const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
      const int src = s_row_src[r];
      uint4 v[4] = {};
      if (src >= 0) {
        const uint16_t* base = GATEUP ? a.x + size_t(src) * a.D : a.h + size_t(src) * a.I;
        const uint4* p = reinterpret_cast<const uint4*>(base + k0 + half * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = p[q];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t wds[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
          const int kk = half * 32 + q * 8 + h2 * 2;
          As[kk][r] = bf16lo(wds[h2]);
          As[kk + 1][r] = bf16hi(wds[h2]);
        }
      }
    }
    // B tiles: NB matrices x 64 rows x 8 words
    for (int wi = threadIdx.x; wi < NB * SBN * 8; wi += blockDim.x) {
      const int b = wi / (SBN * 8), n = (wi / 8) % SBN, wrd = wi % 8;
      const moe_qmatrix& m = b == 0 ? m0 : m1;
      const size_t row = size_t(ex) * N + n0 + n;
      const uint32_t word = m.codes[row * (K / 8) + k0 / 8 + wrd];
      const float s = bf16_to_f32(m.scales[row * (K / 64) + k0 / 64]);
      const float bb = bf16_to_f32(m.biases[row * (K / 64) + k0 / 64]);
      float wv[8];
      dq8(word, s, bb, wv);
#pragma unroll
      for (int j = 0; j < 8; ++j) Bs[b][wrd * 8 + j][n] = wv[j];
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < SBK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][ty * 8 + 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float4 bv4 = *reinterpret_cast<const float4*>(&Bs[b][kk][tx * 4]);
        const float bv[4] = {bv4.x, bv4.y, bv4.z, bv4.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[b][i][j] = fmaf(av[i], bv[j], acc[b][i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = ty * 8 + i;
    if (r >= R) continue;
    if (GATEUP) {
      uint16_t hv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) hv[j] = f32_to_bf16(silu_mul(acc[0][i][j], acc[NB - 1][i][j]));
      uint2 pk = make_uint2(uint32_t(hv[0]) | (uint32_t(hv[1]) << 16), uint32_t(hv[2]) | (uint32_t(hv[3]) << 16));
      *reinterpret_cast<uint2*>(a.h_out + size_t(p0 + r) * a.I + n0 + tx * 4) = pk;
    } else {
      const int p = s_row_src[r];
      const int t = shared ? p - A : a.perm[p] / a.k;
      const float wgt = s_row_w[r];
      float* dst = a.y_acc + size_t(t) * a.D + n0 + tx * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) atomicAdd(dst + j, wgt * acc[0][i][j]);
    }
  }
}

}  // namespace

__global__ void zero_f32_kernel(float4* p, size_t n4) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void cast_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, size_t n4) {
  griddep_wait();  // the down projection's accumulator
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_uint2(uint32_t(f32_to_bf16(v.x)) | (uint32_t(f32_to_bf16(v.y)) << 16),
                        uint32_t(f32_to_bf16(v.z)) | (uint32_t(f32_to_bf16(v.w)) << 16));
  }
}

cudaError_t zero_yacc(const Ctx& c) {
  const size_t n4 = size_t(c.T) * c.D / 4;
  zero_f32_kernel<<<4 * 152, 256, 0, c.stream>>>(reinterpret_cast<float4*>(c.y_acc), n4);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) launch_done(c, "zero_yacc");
  return err;
}

cudaError_t cast_y(const Ctx& c) {
  const size_t n4 = size_t(c.T) * c.D / 4;
  cudaError_t err = launch_pdl(c, cast_bf16_kernel, dim3(4 * 152), dim3(256), 0,
                               reinterpret_cast<const float4*>(c.y_acc), reinterpret_cast<uint2*>(c.y), n4);
  if (err == cudaSuccess) launch_done(c, "cast_y");
  return err;
}

constexpr size_t simt_smem_bytes(int nb) { return sizeof(float) * SBK * (SBM + nb * SBN); }

cudaError_t gemm_simt(const Ctx& c) {
  const moe_weights* w = c.w;
  if (!ensure_smem_limit(reinterpret_cast<const void*>(gemm_simt_kernel<true>), int(simt_smem_bytes(2))) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(gemm_simt_kernel<false>), int(simt_smem_bytes(1))))
    return cudaErrorInvalidValue;
  SimtArgs a{c.x, c.h, w->gate, w->up, w->s_gate, w->s_up, c.blocks, c.n_blocks, c.perm, c.topk_w,
             c.h, c.y_acc, c.hdr, c.T, c.D, c.E, c.k, c.I};
  cudaError_t err = c.yacc_zeroed ? cudaSuccess : zero_yacc(c);
  if (err != cudaSuccess) return err;
  gemm_simt_kernel<true><<<dim3(c.max_blocks, c.I / SBN), 256, simt_smem_bytes(2), c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done(c, "gateup_simt");
  a.m0 = w->down;
  a.s0 = w->s_down;
  gemm_simt_kernel<false><<<dim3(c.max_blocks, c.D / SBN), 256, simt_smem_bytes(1), c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done(c, "down_simt");
  return cast_y(c);
}

}  // namespace moe
