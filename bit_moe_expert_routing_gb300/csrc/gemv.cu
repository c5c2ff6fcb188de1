// Decode path for one to a few token rows: row-parallel dequantising GEMVs on
// the CUDA cores ("Optimizing on-device inference for Apple Silicon", sections
// "Optimise the single-row weight path" and "Reduce intermediate and state
// traffic"; the switch to matrix kernels above a row count follows
// "Why continuous batching halved LLM throughput on an M2 Mac mini").
//
//   gemv_gateup: a CTA owns 16 consecutive intermediate rows of one expert
//     block. Their gate and up codes, scales and biases are contiguous in
//     memory, so one thread fetches all of them into shared memory with six
//     bulk (TMA) copies on one mbarrier while the CTA stages every token row
//     (they do not depend on the routing). A warp takes two rows: per
//     32-code chunk it loads the activations once and runs four independent
//     dot products (gate and up of each row); then h = bf16(silu(g) * u) in
//     the permuted order.
//   gemv_down: a CTA owns 8 output columns of one token. It bulk-copies the
//     8 rows of the down matrix of each of the token's k experts and of the
//     shared expert and stages the token's k+1 h rows. A thread takes one
//     (expert slot, 32-code chunk) item and adds w_j * (h_j . row) for all 8
//     columns; lanes and warps are then summed in a fixed order, y = bf16(sum).
//     No atomics: deterministic.
//
// The kernels are bound by weight reads: every byte a CTA needs is in flight
// at once (bulk copies do not hold registers), and the grids fill the GPU in
// about one wave.
//
// The dequantising dot products are in dot.cuh.
#include <algorithm>
#include <cstddef>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "dot.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kMaxGemvRows = 8;
constexpr int kGemvWarps = 8;
constexpr int kGateupRows = 16;  // intermediate rows per gate/up CTA
constexpr int kDownCols = 8;     // output columns per down CTA

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

// Shared-memory layout of a gate/up CTA (D input columns, R token rows).
struct GateupSmem {
  size_t codes_g, codes_u, sg, bg, su, bu, xs4, xsum, total;
  __host__ __device__ GateupSmem(int D, int R) {
    const size_t cb = size_t(kGateupRows) * D / 2, sbb = size_t(kGateupRows) * (D / 64) * 2;
    codes_g = 16;  // bytes 0..15: mbarrier and abort flag
    codes_u = codes_g + cb;
    sg = codes_u + cb;
    bg = sg + sbb;
    su = bg + sbb;
    bu = su + sbb;
    xs4 = (bu + sbb + 15) & ~size_t(15);
    xsum = xs4 + size_t(R) * D * 4;
    total = xsum + size_t(R) * (D / 32) * 4;
  }
};

__global__ void __launch_bounds__(kGemvWarps * 32) gemv_gateup_kernel(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t gsm[];
  __shared__ int s_tok[kMaxGemvRows];
  if (blockIdx.x >= *a.n_blocks) return;
  const int D = a.D, I = a.I, nch = D / 32, G = D / 64;
  const int nt = min(a.T, kMaxGemvRows);
  const GateupSmem L(D, nt);
  const uint32_t bar = smem_u32(gsm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gsm + 8);
  const int g = a.blocks[3 * blockIdx.x], p0 = a.blocks[3 * blockIdx.x + 1], R = a.blocks[3 * blockIdx.x + 2];
  const int A = a.T * a.k;
  if (g < 0 || g > a.E || R < 1 || R > kMaxGemvRows || R > a.T || p0 < 0 || p0 + R > A + a.T) {
    if (threadIdx.x == 0) report(a.hdr, MOE_ERR_DEVICE_CHECK, 3);
    return;
  }
  const bool shared = (g == a.E);
  const int ex = shared ? 0 : g;
  const moe_qmatrix mg = shared ? a.s_gate : a.gate;
  const moe_qmatrix mu = shared ? a.s_up : a.up;
  const int i0 = blockIdx.y * kGateupRows;
  const int nr = min(kGateupRows, I - i0);

  if (threadIdx.x == 0) {  // all of this CTA's weights, in six bulk copies
    *abort_flag = 0;
    mbar_init(bar, 1);
    mbar_init_fence();
    const uint32_t cb = uint32_t(nr) * D / 2, sbb = uint32_t(nr) * G * 2;
    const size_t row0 = size_t(ex) * I + i0;
    mbar_arrive_tx(bar, 2 * cb + 4 * sbb);
    bulk_g2s(bar + uint32_t(L.codes_g), mg.codes + row0 * (D / 8), cb, bar);
    bulk_g2s(bar + uint32_t(L.codes_u), mu.codes + row0 * (D / 8), cb, bar);
    bulk_g2s(bar + uint32_t(L.sg), mg.scales + row0 * G, sbb, bar);
    bulk_g2s(bar + uint32_t(L.bg), mg.biases + row0 * G, sbb, bar);
    bulk_g2s(bar + uint32_t(L.su), mu.scales + row0 * G, sbb, bar);
    bulk_g2s(bar + uint32_t(L.bu), mu.biases + row0 * G, sbb, bar);
  }
  // every token row (T <= 8), staged while the weights are in flight
  float4* xs4 = reinterpret_cast<float4*>(gsm + L.xs4);
  float* xsum = reinterpret_cast<float*>(gsm + L.xsum);
  for (int q = threadIdx.x; q < nt * (D / 8); q += blockDim.x) {
    const int t = q / (D / 8), q8 = q % (D / 8);
    stage_bf16x8(xs4 + size_t(t) * 8 * nch, nch, q8, *reinterpret_cast<const uint4*>(a.x + size_t(t) * D + q8 * 8));
  }
  if (threadIdx.x < R) {
    const int p = p0 + threadIdx.x;
    int t = shared ? p - A : a.perm[p] / a.k;
    if (t < 0 || t >= nt) {
      report(a.hdr, MOE_ERR_DEVICE_CHECK, 4);
      t = 0;
    }
    s_tok[threadIdx.x] = t;
  }
  __syncthreads();
  chunk_sums(xs4, xsum, nt, nch);
  __syncthreads();
  if (!mbar_wait(bar, 0, abort_flag, a.hdr, kWaitLimit, true)) return;

  // warp w takes rows w, w+8, w+16, w+24: for each 32-code chunk of the token
  // row the activations are loaded once and feed eight independent dot products
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kRowsPerWarp = kGateupRows / kGemvWarps;
  const uint8_t* cg = gsm + L.codes_g;
  const uint8_t* cu = gsm + L.codes_u;
  const uint16_t* sg = reinterpret_cast<const uint16_t*>(gsm + L.sg);
  const uint16_t* bg = reinterpret_cast<const uint16_t*>(gsm + L.bg);
  const uint16_t* su = reinterpret_cast<const uint16_t*>(gsm + L.su);
  const uint16_t* bu = reinterpret_cast<const uint16_t*>(gsm + L.bu);
#pragma unroll 1
  for (int r = 0; r < R; ++r) {
    const int t = s_tok[r];
    const float4* xr = xs4 + size_t(t) * 8 * nch;
    float gacc[kRowsPerWarp], uacc[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) gacc[i] = uacc[i] = 0.f;
    for (int c = lane; c < nch; c += 32) {  // 32-code chunk c lies in group c/2
      float4 xv[8];
#pragma unroll
      for (int jq = 0; jq < 8; ++jq) xv[jq] = xr[jq * nch + c];
      const float sx = xsum[t * nch + c];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int rr = warp + kGemvWarps * i;
        if (rr < nr) {
          const uint4 wg = reinterpret_cast<const uint4*>(cg + size_t(rr) * D / 2)[c];
          const uint4 wu = reinterpret_cast<const uint4*>(cu + size_t(rr) * D / 2)[c];
          const int gi = rr * G + c / 2;
          gacc[i] += chunk_dot_r(wg, xv, sx, sg[gi], bg[gi]);
          uacc[i] += chunk_dot_r(wu, xv, sx, su[gi], bu[gi]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        gacc[i] += __shfl_xor_sync(0xffffffffu, gacc[i], off);
        uacc[i] += __shfl_xor_sync(0xffffffffu, uacc[i], off);
      }
      const int rr = warp + kGemvWarps * i;
      if (lane == 0 && rr < nr) a.h[size_t(p0 + r) * I + i0 + rr] = f32_to_bf16(silu_mul(gacc[i], uacc[i]));
    }
  }
}

// Shared-memory layout of a down CTA (k+1 slots, I input columns).
struct DownSmem {
  size_t codes, sc, bi, hs4, hsum, w, red, total;
  __host__ __device__ DownSmem(int k, int I) {
    const size_t S = size_t(k) + 1;
    codes = 16;  // bytes 0..15: mbarrier and abort flag
    sc = codes + S * kDownCols * (I / 2);
    bi = sc + S * kDownCols * (I / 64) * 2;
    hs4 = (bi + S * kDownCols * (I / 64) * 2 + 15) & ~size_t(15);
    hsum = hs4 + S * size_t(I) * 4;
    w = hsum + S * size_t(I / 32) * 4;
    red = (w + S * 4 + 15) & ~size_t(15);
    total = red + size_t(kGemvWarps) * kDownCols * 4;
  }
};

// grid (D / kDownCols, T): blockIdx.y is the token.
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_down_kernel(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int k = a.k, I = a.I, D = a.D, nch = I / 32, G = I / 64, S = k + 1;
  const int t = blockIdx.y, d0 = blockIdx.x * kDownCols, A = a.T * k;
  const DownSmem L(k, I);
  const uint32_t bar = smem_u32(dsm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(dsm + 8);
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar, S);  // one arrival (with its byte count) per slot
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x < S) {  // slot j: rows d0..d0+15 of its expert's down matrix
    const int j = threadIdx.x;
    const bool sh = (j == k);
    int ex = sh ? 0 : a.topk_idx[t * k + j];
    if (ex < 0 || ex >= a.E) {
      report(a.hdr, MOE_ERR_DEVICE_CHECK, 8);
      ex = 0;
    }
    const moe_qmatrix& m = sh ? a.s_down : a.down;
    const size_t row0 = size_t(ex) * D + d0;
    const uint32_t cb = kDownCols * (I / 2), sbb = kDownCols * G * 2;
    mbar_arrive_tx(bar, cb + 2 * sbb);
    bulk_g2s(bar + uint32_t(L.codes + size_t(j) * cb), m.codes + row0 * (I / 8), cb, bar);
    bulk_g2s(bar + uint32_t(L.sc + size_t(j) * sbb), m.scales + row0 * G, sbb, bar);
    bulk_g2s(bar + uint32_t(L.bi + size_t(j) * sbb), m.biases + row0 * G, sbb, bar);
  }
  float4* hs4 = reinterpret_cast<float4*>(dsm + L.hs4);
  float* hsum = reinterpret_cast<float*>(dsm + L.hsum);
  float* s_w = reinterpret_cast<float*>(dsm + L.w);
  for (int q = threadIdx.x; q < S * (I / 8); q += blockDim.x) {
    const int j = q / (I / 8), q8 = q % (I / 8);
    const int p = j < k ? a.inv[t * k + j] : A + t;
    stage_bf16x8(hs4 + size_t(j) * 8 * nch, nch, q8, *reinterpret_cast<const uint4*>(a.h + size_t(p) * I + q8 * 8));
  }
  for (int j = threadIdx.x; j < S; j += blockDim.x) s_w[j] = j < k ? a.topk_w[t * k + j] : 1.f;
  __syncthreads();
  chunk_sums(hs4, hsum, S, nch);
  __syncthreads();
  if (!mbar_wait(bar, 0, abort_flag, a.hdr, kWaitLimit, true)) return;

  // thread item it = (slot j, 32-code chunk c): its activations are loaded
  // once and feed the dot products of all 16 output columns; the partial sums
  // are then reduced over the lanes and over the warps in a fixed order
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint8_t* codes = dsm + L.codes;
  const uint16_t* sc = reinterpret_cast<const uint16_t*>(dsm + L.sc);
  const uint16_t* bi = reinterpret_cast<const uint16_t*>(dsm + L.bi);
  float part[kDownCols];
#pragma unroll
  for (int cl = 0; cl < kDownCols; ++cl) part[cl] = 0.f;
  for (int it = threadIdx.x; it < S * nch; it += blockDim.x) {
    const int j = it / nch, c = it % nch;
    float4 xv[8];
    const float4* xr = hs4 + size_t(j) * 8 * nch;
#pragma unroll
    for (int jq = 0; jq < 8; ++jq) xv[jq] = xr[jq * nch + c];
    const float sx = hsum[j * nch + c], wj = s_w[j];
#pragma unroll
    for (int cl = 0; cl < kDownCols; ++cl) {
      const int rowi = j * kDownCols + cl;  // row of slot j's copy
      const uint4 w4 = reinterpret_cast<const uint4*>(codes + size_t(rowi) * (I / 2))[c];
      const int gi = rowi * G + c / 2;
      part[cl] += wj * chunk_dot_r(w4, xv, sx, sc[gi], bi[gi]);
    }
  }
  float* red = reinterpret_cast<float*>(dsm + L.red);  // [kGemvWarps][kDownCols]
#pragma unroll
  for (int cl = 0; cl < kDownCols; ++cl) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part[cl] += __shfl_xor_sync(0xffffffffu, part[cl], off);
  }
  if (lane == 0) {
#pragma unroll
    for (int cl = 0; cl < kDownCols; ++cl) red[warp * kDownCols + cl] = part[cl];
  }
  __syncthreads();
  if (threadIdx.x < kDownCols) {
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) y += red[w * kDownCols + threadIdx.x];
    a.y[size_t(t) * D + d0 + threadIdx.x] = f32_to_bf16(y);
  }
}

// ---------------------------------------------------------------------------
// Fused decode for one token: router logits, top-k, gate/up + SwiGLU and the
// down projection in one cooperative kernel with a single grid barrier.
//
// A CTA owns one item: 32 consecutive intermediate rows of one expert slot
// (slot j < k is the token's j-th expert, slot k the shared expert). It
// computes those 32 values of h and multiplies them with the matching 32
// columns of the expert's down matrix, which is its share of every output
// value, and adds that share, times the routing weight, into the fp32
// accumulator. So no CTA waits for another CTA's h.
//   1. At entry: bulk copies of the CTA's router rows (experts blockIdx.x +
//      m * gridDim.x). x is staged and the accumulator cleared.
//   2. Logits of its experts in the canonical order; grid barrier.
//   3. Every CTA takes the top-k of all logits itself (the same deterministic
//      selection), then starts its item's copies: gate/up codes, scales and
//      biases by bulk copy in four sub-items of 8 rows (one mbarrier each);
//      the down matrix's 32-code column block (16 bytes of each of its D
//      rows) by 2-D tensor copies of 64 rows; the scale and bias words of
//      the block's group for this thread's output columns into registers.
//   4. Gate/up dot products as the sub-items land: warps 4s .. 4s + 3 (one
//      per scheduler) take sub-item s, warp 4s + q its rows 2q and 2q + 1,
//      gate and up (four dot products sharing each load of x); h =
//      bf16(silu(g) * u); the down partials of output columns d =
//      threadIdx.x + 512 c; red.add into the accumulator.
//   5. The last CTA to finish (counted on the barrier's counter) converts the
//      accumulator to bf16 y.
// The accumulator's fp32 additions land in arrival order, as in the grouped
// GEMM's combine: results agree up to the summation order.
constexpr int kFdRows = 32;     // intermediate rows per item: one 32-code chunk of a down row
constexpr int kFdSubRows = 8;   // rows per sub-item (one mbarrier)
constexpr int kFdSubs = kFdRows / kFdSubRows;
constexpr int kFdWarps = 16;
constexpr int kFdCopies = 6;        // bulk copies per sub-item: gate codes, up codes, four scale/bias rows
constexpr int kFdRouterRows = 2;    // router rows (experts) per CTA
constexpr int kFdColsPerThread = 4;  // output columns per thread in the down step, 512 apart
constexpr int kFdDownBox = 64;       // down rows per tensor copy (one lane each)
static_assert(kFdWarps == 4 * kFdSubs && kFdSubRows == 8, "four warps per sub-item, two rows per warp");
static_assert(kFdRows == 32, "h of an item is one warp's lanes and one 32-code chunk of a down row");
static_assert(kFdCopies * kFdSubs <= 32, "one lane per bulk copy");
static_assert(kFdColsPerThread * kFdWarps * 32 == 32 * kFdDownBox, "one lane per tensor copy of the down columns");

struct FusedSmem {
  size_t xs4, xsum, xraw, wr, item, dcodes, gu, hv, total;
  size_t sub_codes, sub_sb, sub_bytes;  // per sub-item: one matrix's codes, one scale or bias row set, all
  __host__ __device__ explicit FusedSmem(int D) {
    sub_codes = size_t(kFdSubRows) * D / 2;
    sub_sb = size_t(kFdSubRows) * (D / 64) * 2;
    sub_bytes = 2 * sub_codes + 4 * sub_sb;
    xs4 = 64;  // bytes 0..63: six mbarriers, abort flag, grid-barrier result, last-CTA flag
    xsum = xs4 + size_t(D) * 4;
    xraw = (xsum + size_t(D / 32) * 4 + 15) & ~size_t(15);  // the token row as bf16
    wr = (xraw + size_t(D) * 2 + 127) & ~size_t(127);       // router rows, fp32
    item = (wr + size_t(kFdRouterRows) * D * 4 + 127) & ~size_t(127);
    dcodes = (item + kFdSubs * sub_bytes + 127) & ~size_t(127);  // the down column block: [D][16 bytes]
    gu = dcodes + size_t(D) * 16;         // the item's gate and up dot products, [2][kFdRows] fp32
    hv = gu + 2 * kFdRows * 4;        // the item's h as fp32 [kFdRows], then their sum
    total = hv + (kFdRows + 4) * 4;
  }
};

struct FusedArgs {
  const uint16_t* x;
  moe_qmatrix gate, up, down, s_gate, s_up, s_down;
  const float* router_w;
  const float* router_bias;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* count;
  int32_t* off;
  int32_t* perm;
  int32_t* inv;
  int32_t* blocks;
  int32_t* n_blocks;
  uint16_t* h;  // [k+1][I]: slot-major for the one token
  float* y_acc;
  uint16_t* y;
  WsHeader* hdr;
  int D, E, k, I;
  int n_items;
};

// Grid-wide barrier of a cooperative launch: every CTA arrives once on the
// header's counter (zeroed on the stream before the launch) and waits, for at
// most kWaitLimit cycles, until `target` arrivals in all. Returns false on
// expiry (MOE_ERR_DEVICE_TIMEOUT recorded).
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned target, volatile int* result) {
  __syncthreads();
  if (threadIdx.x == 0) {
    // release: the CTA's writes (ordered before this thread by the CTA
    // barrier) are visible to every CTA that sees the arrival
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&hdr->counter) : "memory");
    const long long t0 = clock64();
    int ok = 1;
    while (true) {  // relaxed polls with a short sleep, then one acquire fence
      unsigned v;
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&hdr->counter) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > kWaitLimit) {
        report(hdr, MOE_ERR_DEVICE_TIMEOUT, 110);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    *result = ok;
  }
  __syncthreads();
  return *result != 0;
}

// Tensor maps of the down codes as [rows][I/8] 32-bit words, boxes of 4
// words x kFdDownBox rows: every expert's matrix (rows E*D) and the shared
// expert's (rows D).
struct DownMaps {
  CUtensorMap routed, shared;
};

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void red_add_f32(float* dst, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(v) : "memory");
}

template <int MPL>
__global__ void __launch_bounds__(kFdWarps * 32, 1)
    decode_fused_kernel(FusedArgs a, const __grid_constant__ DownMaps dm) {
  extern __shared__ __align__(128) uint8_t fsm[];
  __shared__ int s_exp[kMaxGemvRows * 8 + 1];
  __shared__ float s_w[kMaxGemvRows * 8 + 1];
  const int D = a.D, I = a.I, k = a.k, E = a.E, nch = D / 32, G = D / 64, Gi = I / 64;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const FusedSmem L(D);
  const uint32_t bar0 = smem_u32(fsm);  // mbarriers: sub-items 0..3, the router rows, the down codes
  const uint32_t rbar = bar0 + 8u * kFdSubs, dbar = rbar + 8u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(fsm + 48);
  volatile int* gb_result = reinterpret_cast<volatile int*>(fsm + 52);
  volatile int* last_flag = reinterpret_cast<volatile int*>(fsm + 56);
  const int RB = I / kFdRows;  // items per slot
  const bool has_item = int(blockIdx.x) < a.n_items;
  const int slot = blockIdx.x / RB, i0 = (blockIdx.x % RB) * kFdRows;
  int n_rt = 0;  // router rows (experts) of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  for (int m = 0; m < kFdRouterRows; ++m) n_rt += (blockIdx.x + m * int(gridDim.x) < E);

  // Copy q (lane q of warp 0) of the item of expert e: sub-item q / 6, part
  // q % 6 = gate codes, up codes, gate scales, gate biases, up scales, up
  // biases of the sub-item's 8 rows, each a contiguous block.
  auto item_copy = [&](int q, int e) {
    const int sub = q / kFdCopies, part = q % kFdCopies;
    const bool sh = (e == E);
    const moe_qmatrix& mq = part == 0 || part == 2 || part == 3 ? (sh ? a.s_gate : a.gate) : (sh ? a.s_up : a.up);
    const size_t row0 = size_t(sh ? 0 : e) * I + i0 + sub * kFdSubRows;
    const uint32_t dst = bar0 + uint32_t(L.item + sub * L.sub_bytes), bar = bar0 + 8u * sub;
    if (part < 2)
      bulk_g2s(dst + part * uint32_t(L.sub_codes), mq.codes + row0 * (D / 8), uint32_t(L.sub_codes), bar);
    else
      bulk_g2s(dst + uint32_t(2 * L.sub_codes + (part - 2) * L.sub_sb), ((part & 1) ? mq.biases : mq.scales) + row0 * G,
               uint32_t(L.sub_sb), bar);
  };
  // The item's copies for expert e: warp 0 the gate/up sub-items, warp 1 the
  // down column block (lane l: rows 64 l .. 64 l + 63); every thread loads
  // the aligned 32-bit word holding the scale (and the bias) of the block's
  // group for its down columns d = threadIdx.x + c * blockDim.x. Element
  // (row, g) is number row * Gi + g of its array; the word is number (that
  // >> 1) from the 16-byte-aligned base, so it never crosses the end of the
  // array (D is even, so every array holds an even number of elements).
  uint32_t dsc[kFdColsPerThread], dbi[kFdColsPerThread];
  auto item_start = [&](int e) {
    const bool sh = (e == E);
    if (warp == 0 && lane < kFdCopies * kFdSubs) item_copy(lane, e);
    if (warp == 1 && lane * kFdDownBox < D)
      tma_2d(bar0 + uint32_t(L.dcodes) + lane * kFdDownBox * 16, sh ? &dm.shared : &dm.routed, i0 / 8,
             (sh ? 0 : e) * D + lane * kFdDownBox, dbar);
    const moe_qmatrix& md = sh ? a.s_down : a.down;
    const size_t r0 = size_t(sh ? 0 : e) * D;
#pragma unroll
    for (int c = 0; c < kFdColsPerThread; ++c) {
      const int d = threadIdx.x + c * blockDim.x;
      if (d < D) {
        const size_t el = (r0 + d) * Gi + i0 / 64;
        dsc[c] = __ldg(reinterpret_cast<const uint32_t*>(md.scales) + (el >> 1));
        dbi[c] = __ldg(reinterpret_cast<const uint32_t*>(md.biases) + (el >> 1));
      }
    }
  };

  // --- entry: barriers and byte counts; copies that need no routing
  if (warp == 0) {
    if (lane == 0) {
      *abort_flag = 0;
      for (int i = 0; i < kFdSubs + 2; ++i) mbar_init(bar0 + 8u * i, 1);
      mbar_init_fence();
      if (has_item) {
        for (int sub = 0; sub < kFdSubs; ++sub) mbar_arrive_tx(bar0 + 8u * sub, uint32_t(L.sub_bytes));
        mbar_arrive_tx(dbar, uint32_t(D) * 16);
      }
      if (n_rt) mbar_arrive_tx(rbar, uint32_t(n_rt) * D * 4);
    }
    __syncwarp();
    if (lane < n_rt)
      bulk_g2s(bar0 + uint32_t(L.wr) + lane * D * 4, a.router_w + size_t(blockIdx.x + lane * gridDim.x) * D, D * 4,
               rbar);
  }
  // the token row: bf16 as is (router) and chunk-major fp32 (expert dot products)
  float4* xs4 = reinterpret_cast<float4*>(fsm + L.xs4);
  float* xsum = reinterpret_cast<float*>(fsm + L.xsum);
  uint4* xraw4 = reinterpret_cast<uint4*>(fsm + L.xraw);
  for (int q = threadIdx.x; q < D / 8; q += blockDim.x) {
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + size_t(q) * 8);
    xraw4[q] = v;
    stage_bf16x8(xs4, nch, q, v);
  }
  // the accumulator starts at zero; the grid barrier orders this before any red.add
  for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < D / 4; q += gridDim.x * blockDim.x)
    reinterpret_cast<float4*>(a.y_acc)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (threadIdx.x == 0) {
    s_exp[k] = E;  // slot k: the shared expert
    s_w[k] = 1.f;
  }
  __syncthreads();
  chunk_sums(xs4, xsum, 1, nch);

  // --- router logits of this CTA's experts, in the canonical order (lane l: elements 32c + l, then the tree)
  if (warp < n_rt && mbar_wait(rbar, 0, abort_flag, a.hdr, kWaitLimit, true)) {
    const int e = blockIdx.x + warp * gridDim.x;
    const float* wrow = reinterpret_cast<const float*>(fsm + L.wr) + size_t(warp) * D;
    const uint16_t* xr = reinterpret_cast<const uint16_t*>(fsm + L.xraw);
    float acc = 0.f;
    for (int c = 0; c < nch; ++c) acc = fmaf(bf16_to_f32(xr[32 * c + lane]), wrow[32 * c + lane], acc);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_down_sync(0xffffffffu, acc, off));
    if (lane == 0) a.logits[e] = a.router_bias ? __fadd_rn(acc, a.router_bias[e]) : acc;
  }
  if (n_rt && warp == kFdWarps - 1) mbar_wait(rbar, 0, abort_flag, a.hdr, kWaitLimit, true);  // landed before any exit
  const bool gb1 = grid_barrier(a.hdr, gridDim.x, gb_result);

  // --- top-k (every CTA, the same selection), then the routed item's copies
  if (warp == 0) {
    int myi = 0;
    float myw = 0.f;
    if (gb1) select_topk<MPL, true>(a.logits, E, k, myi, myw);
    if (lane < k && (myi < 0 || myi >= E)) {
      report(a.hdr, MOE_ERR_DEVICE_CHECK, 111);
      myi = 0;
    }
    if (lane < k) {
      s_exp[lane] = myi;
      s_w[lane] = myw;
      if (blockIdx.x == 0) {
        a.topk_idx[lane] = myi;
        a.topk_w[lane] = myw;
      }
    }
  }
  __syncthreads();
  if (has_item) item_start(s_exp[slot]);

  // --- gate/up: warps 4s .. 4s + 3 take sub-item s; warp 4s + q its rows
  // 2q and 2q + 1, gate and up: dot products j = 2 * row + matrix
  float* gu = reinterpret_cast<float*>(fsm + L.gu);
  float* hv = reinterpret_cast<float*>(fsm + L.hv);
  bool item_ok = has_item && gb1;
  if (has_item) {
    const int sub = warp >> 2, r0 = 2 * (warp & 3);
    // every copy is waited for (draining), so none is in flight at exit;
    // warp 15 also waits for the down block
    if (!mbar_wait(bar0 + 8u * sub, 0, abort_flag, a.hdr, kWaitLimit, true)) {
      item_ok = false;
    } else {
      const uint8_t* base = fsm + L.item + sub * L.sub_bytes;
      const uint16_t* sb = reinterpret_cast<const uint16_t*>(base + 2 * L.sub_codes);  // [4][kFdSubRows][G]
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = lane; c < nch; c += 32) {
        float4 xv[8];
#pragma unroll
        for (int jq = 0; jq < 8; ++jq) xv[jq] = xs4[jq * nch + c];
        const float sx = xsum[c];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = r0 + (j >> 1), mat = j & 1;
          const uint4 w4 = reinterpret_cast<const uint4*>(base + mat * L.sub_codes + size_t(r) * (D / 2))[c];
          const uint16_t* srow = sb + (2 * mat) * (kFdSubRows * G) + r * G;  // scales; the biases follow
          acc[j] += chunk_dot_r(w4, xv, sx, srow[c / 2], srow[kFdSubRows * G + c / 2]);
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
      }
      if (lane < 4) {
        float v = acc[0];
#pragma unroll
        for (int j = 1; j < 4; ++j)
          if (lane == j) v = acc[j];
        gu[(lane & 1) * kFdRows + sub * kFdSubRows + r0 + (lane >> 1)] = v;
      }
    }
  }
  if (has_item && warp == kFdWarps - 1 && !mbar_wait(dbar, 0, abort_flag, a.hdr, kWaitLimit, true)) item_ok = false;
  if (!item_ok && has_item) *abort_flag = 1;
  __syncthreads();
  item_ok = has_item && gb1 && !*abort_flag;
  // h of the item's 32 rows (lane i: row i0 + i), rounded to bf16, and their sum
  if (item_ok && warp == 0) {
    const uint16_t hb = f32_to_bf16(silu_mul(gu[lane], gu[kFdRows + lane]));
    const float h = bf16_to_f32(hb);
    hv[lane] = h;
    float hs = h;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) hs += __shfl_xor_sync(0xffffffffu, hs, off);
    if (lane == 0) hv[kFdRows] = hs;
    a.h[size_t(slot) * I + i0 + lane] = hb;
  }
  __syncthreads();
  // --- down: this thread's output columns from the item's 32 rows
  if (item_ok) {
    float4 hx[8];
#pragma unroll
    for (int jq = 0; jq < 8; ++jq) hx[jq] = reinterpret_cast<const float4*>(hv)[jq];
    const float hs = hv[kFdRows], wj = s_w[slot];
    const uint4* dc = reinterpret_cast<const uint4*>(fsm + L.dcodes);
#pragma unroll
    for (int c = 0; c < kFdColsPerThread; ++c) {
      const int d = threadIdx.x + c * blockDim.x;
      if (d < D) {
        // the element's half of the loaded word (the expert's first row is
        // even: D is even)
        const int sh16 = 16 * ((d * Gi + i0 / 64) & 1);
        const uint16_t sc = uint16_t(dsc[c] >> sh16), bi = uint16_t(dbi[c] >> sh16);
        red_add_f32(a.y_acc + d, wj * chunk_dot_r(dc[d], hx, hs, sc, bi));
      }
    }
  }

  // CTA 0: the routing tables for inspection (one token: each selected
  // expert holds one row; the permutation orders the slots by expert)
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int cnt = 0, below = 0;
      for (int j = 0; j < k; ++j) {
        cnt += (s_exp[j] == e);
        below += (s_exp[j] < e);
      }
      a.count[e] = cnt;
      a.off[e] = below;
    }
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      int rank = 0;
      for (int j2 = 0; j2 < k; ++j2) rank += (s_exp[j2] < s_exp[j]);
      a.perm[rank] = j;
      a.inv[j] = rank;
      a.blocks[3 * rank + 0] = s_exp[j];
      a.blocks[3 * rank + 1] = rank;
      a.blocks[3 * rank + 2] = 1;
    }
    if (threadIdx.x == 0) {
      a.off[E] = k;
      a.blocks[3 * k + 0] = E;  // the shared expert's row
      a.blocks[3 * k + 1] = k;
      a.blocks[3 * k + 2] = 1;
      *a.n_blocks = k + 1;
    }
  }

  // --- the last CTA to arrive (2 * gridDim.x arrivals on the counter, the
  // barrier's included) converts the accumulator. The CTA barrier orders the
  // CTA's red.adds before thread 0's arrival, whose release makes them
  // visible to the CTA that acquires the final count; that CTA's threads read
  // after its own CTA barrier.
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned before;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(&a.hdr->counter) : "memory");
    *last_flag = before == 2u * gridDim.x - 1u;
  }
  __syncthreads();
  if (*last_flag) {
    for (int q = threadIdx.x; q < D / 4; q += blockDim.x) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.y_acc) + q);
      uint2 o;
      o.x = uint32_t(f32_to_bf16(v.x)) | (uint32_t(f32_to_bf16(v.y)) << 16);
      o.y = uint32_t(f32_to_bf16(v.z)) | (uint32_t(f32_to_bf16(v.w)) << 16);
      reinterpret_cast<uint2*>(a.y)[q] = o;
    }
  }
}

}  // namespace

bool gemv_supported(const Ctx& c) {
  if (c.T < 1 || c.T > kMaxGemvRows || c.k + 1 > kGemvWarps * 32) return false;
  const size_t lim = 200 * 1024;
  return GateupSmem(c.D, std::min(c.T, kMaxGemvRows)).total <= lim && DownSmem(c.k, c.I).total <= lim;
}

cudaError_t gemv(const Ctx& c) {
  const moe_weights* w = c.w;
  GemvArgs a{c.x, w->gate, w->up, w->down, w->s_gate, w->s_up, w->s_down, c.blocks, c.n_blocks,
             c.perm, c.inv, c.topk_idx, c.topk_w, c.h, c.y, c.hdr, c.T, c.D, c.E, c.k, c.I};
  const size_t s1 = GateupSmem(c.D, std::min(c.T, kMaxGemvRows)).total, s2 = DownSmem(c.k, c.I).total;
  if (!ensure_smem_limit(reinterpret_cast<const void*>(gemv_gateup_kernel), int(s1)) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(gemv_down_kernel), int(s2)))
    return cudaErrorInvalidValue;
  cudaError_t err;
  gemv_gateup_kernel<<<dim3(c.max_blocks, (c.I + kGateupRows - 1) / kGateupRows), kGemvWarps * 32, s1, c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done(c, "gemv_gateup");
  gemv_down_kernel<<<dim3(c.D / kDownCols, c.T), kGemvWarps * 32, s2, c.stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done(c, "gemv_down");
  return cudaSuccess;
}

namespace {

struct FusedPlan {
  int grid = 0, n_items = 0, mpl = 0;
  size_t smem = 0;
};

// Launch shape of the fused decode for this layer, or grid 0 when it does not
// apply (more than one token, shared memory, too many logits per lane, or not
// all CTAs co-resident).
FusedPlan fused_plan_uncached(const Ctx& c) {
  FusedPlan p;
  if (c.T != 1 || c.I % 64 != 0 || c.D % kFdDownBox != 0 || c.D > kFdColsPerThread * kFdWarps * 32 ||
      c.E > 512 || c.k + 1 > kMaxGemvRows * 8 + 1 || !tmap_encoder_available())
    return p;
  p.mpl = (c.E + 31) / 32 <= 8 ? 8 : 16;
  p.smem = FusedSmem(c.D).total;
  if (p.smem > 227 * 1024) return p;
  p.n_items = (c.k + 1) * (c.I / kFdRows);
  const int grid = std::max(p.n_items, (c.E + kFdRouterRows - 1) / kFdRouterRows);
  int dev = 0, coop = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return p;
  const void* f = p.mpl == 8 ? reinterpret_cast<const void*>(decode_fused_kernel<8>)
                             : reinterpret_cast<const void*>(decode_fused_kernel<16>);
  if (!ensure_smem_limit(f, int(p.smem)) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kFdWarps * 32, p.smem) != cudaSuccess)
    return p;
  if (grid > per_sm * sms) return p;
  p.grid = grid;
  return p;
}

// The plan depends on the device and the layer shape only: computed once.
FusedPlan fused_plan(const Ctx& c) {
  struct Entry {
    int dev, T, D, I, k, E;
    FusedPlan p;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FusedPlan{};
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.T == c.T && e.D == c.D && e.I == c.I && e.k == c.k && e.E == c.E) return e.p;
  const FusedPlan p = fused_plan_uncached(c);
  cache.push_back({dev, c.T, c.D, c.I, c.k, c.E, p});
  return p;
}

// The down codes' tensor maps for this layer's weights, encoded once per
// weight pointers and shape.
bool down_maps(const Ctx& c, DownMaps* out) {
  struct Entry {
    const void* routed;
    const void* shared;
    int E, D, I;
    DownMaps m;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  const moe_weights* w = c.w;
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.routed == w->down.codes && e.shared == w->s_down.codes && e.E == c.E && e.D == c.D && e.I == c.I) {
      *out = e.m;
      return true;
    }
  Entry e{w->down.codes, w->s_down.codes, c.E, c.D, c.I, DownMaps{}};
  const auto U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  const auto NOL2 = CU_TENSOR_MAP_L2_PROMOTION_NONE;
  if (!make_tmap_2d(&e.m.routed, U32, 4, w->down.codes, uint64_t(c.E) * c.D, c.I / 8, 4, kFdDownBox, NOSW, NOL2) ||
      !make_tmap_2d(&e.m.shared, U32, 4, w->s_down.codes, c.D, c.I / 8, 4, kFdDownBox, NOSW, NOL2))
    return false;
  if (cache.size() >= 16) cache.erase(cache.begin());
  cache.push_back(e);
  *out = e.m;
  return true;
}

}  // namespace

bool decode_fused_supported(const Ctx& c) { return fused_plan(c).grid > 0; }

cudaError_t decode_fused(const Ctx& c) {
  const FusedPlan p = fused_plan(c);
  if (p.grid == 0) return cudaErrorInvalidValue;
  const moe_weights* w = c.w;
  FusedArgs a{c.x,        w->gate,        w->up,    w->down,    w->s_gate,   w->s_up, w->s_down,
              w->router_w, w->router_bias, c.logits, c.topk_idx, c.topk_w,    c.count, c.off,
              c.perm,      c.inv,          c.blocks, c.n_blocks, c.h,         c.y_acc, c.y,
              c.hdr,       c.D,            c.E,      c.k,        c.I,         p.n_items};
  // the grid-barrier counter starts at zero; on the call's first pass the
  // status does too (later passes keep what earlier ones recorded)
  static_assert(offsetof(WsHeader, counter) == 8, "status, detail, counter");
  cudaError_t err = c.first_pass ? cudaMemsetAsync(c.hdr, 0, 12, c.stream)
                                 : cudaMemsetAsync(&c.hdr->counter, 0, 4, c.stream);
  if (err != cudaSuccess) return err;
  DownMaps dm;
  if (!down_maps(c, &dm)) return cudaErrorInvalidValue;
  void* args[] = {&a, &dm};
  const void* f = p.mpl == 8 ? reinterpret_cast<const void*>(decode_fused_kernel<8>)
                             : reinterpret_cast<const void*>(decode_fused_kernel<16>);
  err = cudaLaunchCooperativeKernel(f, dim3(p.grid), dim3(kFdWarps * 32), args, p.smem, c.stream);
  if (err != cudaSuccess) return err;
  launch_done(c, "decode_fused");
  return cudaSuccess;
}

}  // namespace moe
