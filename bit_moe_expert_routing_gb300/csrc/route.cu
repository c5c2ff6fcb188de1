// GPU-resident expert routing: router logits, top-k with renormalised
// weights, per-expert histogram, exclusive scan, scatter into expert groups
// and the block map of fixed-size row blocks. All on the caller's stream,
// with no host synchronisation ("Optimizing on-device inference for Apple
// Silicon", section "Keep expert routing on the GPU").
//
// Router logits use one fixed fp32 evaluation order so that the top-k
// decision (an integer result) is reproducible by any implementation: the
// plain dot product as one fused multiply-add chain in index order,
//   acc = 0;  for d = 0 .. D-1:  acc = fma(float(x[t, d]), W_r[e, d], acc)
//   logit = acc (+ bias[e])
// Each logit is one thread's accumulator; the parallelism is across logits.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Router logits as a register-tiled SIMT GEMM: a CTA computes BT tokens x BE
// experts, a thread TT tokens x TE experts, each logit one sequential FMA chain.
// D is walked in chunks of kRgK: the chunk of x (bf16 -> fp32) and of W_r is
// stored transposed in shared memory ([k][token], [k][expert]) so that a
// thread reads its tokens and its experts of one k with 16-byte loads (each
// shared by the lanes with the same tokens or experts). The next chunk
// is loaded into registers, consecutive lanes along a row, while the current
// one is used. The transposed rows are XOR-swizzled in groups of four (tokens
// by (k/8)%4, experts by (k/4)%8) so that the transposing stores hit 32
// different banks and a 4-group stays one aligned 16-byte word.
constexpr int kRgK = 32;

template <int BT, int BE, int TT, int TE>
__global__ void __launch_bounds__(BT * BE / (TT * TE), BT >= 128 ? 3 : 1)
    router_gemm_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
                       int T, int D, int E, float* __restrict__ logits, WsHeader* hdr) {
  constexpr int N = BT * BE / (TT * TE);  // threads
  constexpr int XP = BT * 4 / N;          // 16-byte x pieces per thread per chunk
  constexpr int WP = BE * 8 / N;          // 16-byte W pieces per thread per chunk
  constexpr int XG = TT / 4, WG = TE / 4;  // 16-byte reads of x and of W per k
  static_assert(BT >= 32 && BE >= 32 && XP >= 1 && WP >= 1 && TT % 4 == 0 && TE % 4 == 0, "tile shape");
  // First kernel of every call: start the call's device status afresh. No
  // other CTA of this kernel reports, so nothing races with the clear.
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    hdr->status = 0;
    hdr->detail = 0;
  }
  __shared__ __align__(16) float xs[2][kRgK][BT];
  __shared__ __align__(16) float ws[2][kRgK][BE];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * BT, e0 = blockIdx.y * BE;
  const int ti = tid / (BE / TE), ei = tid % (BE / TE);  // tokens TT ti .., experts TE ei ..
  // piece c of x: token row c/4 of the tile, columns 8(c%4) .. +7 of the chunk;
  // piece c of W: expert row c/8, columns 4(c%8) .. +3. Consecutive lanes
  // take consecutive pieces, so a warp reads whole row segments.
  const uint16_t* xsrc[XP];
  const float* wsrc[WP];
#pragma unroll
  for (int m = 0; m < XP; ++m) {
    const int c = tid + m * N, t = t0 + (c >> 2);
    xsrc[m] = t < T ? x + size_t(t) * D + 8 * (c & 3) : nullptr;
  }
#pragma unroll
  for (int m = 0; m < WP; ++m) {
    const int c = tid + m * N;
    wsrc[m] = wr + size_t(min(e0 + (c >> 3), E - 1)) * D + 4 * (c & 7);
  }
  uint4 xr[XP];
  float4 wv_in[WP];
  auto load = [&](int d0) {
#pragma unroll
    for (int m = 0; m < XP; ++m)
      xr[m] = xsrc[m] ? *reinterpret_cast<const uint4*>(xsrc[m] + d0) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int m = 0; m < WP; ++m) wv_in[m] = *reinterpret_cast<const float4*>(wsrc[m] + d0);
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int m = 0; m < XP; ++m) {
      const int c = tid + m * N, r = c >> 2, ch = c & 3;
      const int col = r ^ (ch << 3);  // k = 8 ch + i: (k / 8) % 4 = ch
      const uint32_t xw[4] = {xr[m].x, xr[m].y, xr[m].z, xr[m].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xs[buf][8 * ch + 2 * i][col] = __uint_as_float(xw[i] << 16);
        xs[buf][8 * ch + 2 * i + 1][col] = __uint_as_float(xw[i] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int m = 0; m < WP; ++m) {
      const int c = tid + m * N, r = c >> 3, ch = c & 7;
      const int col = r ^ (ch << 2);  // k = 4 ch + i: (k / 4) % 8 = ch
      const float wa[4] = {wv_in[m].x, wv_in[m].y, wv_in[m].z, wv_in[m].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) ws[buf][4 * ch + i][col] = wa[i];
    }
  };

  float2 acc[TT / 2][TE];  // [token pair][expert]: .x token TT ti + 2p, .y token TT ti + 2p + 1
#pragma unroll
  for (int p = 0; p < TT / 2; ++p)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[p][j] = make_float2(0.f, 0.f);

  const int nk = D / kRgK;
  load(0);
  store(0);
  __syncthreads();
  for (int kc = 0; kc < nk; ++kc) {
    const int buf = kc & 1;
    if (kc + 1 < nk) load((kc + 1) * kRgK);
    auto rd = [&](int k, float4 (&xv)[XG], float4 (&wv)[WG]) {
#pragma unroll
      for (int g = 0; g < XG; ++g)
        xv[g] = *reinterpret_cast<const float4*>(&xs[buf][k][(TT * ti + 4 * g) ^ (((k >> 3) & 3) << 3)]);
#pragma unroll
      for (int g = 0; g < WG; ++g)
        wv[g] = *reinterpret_cast<const float4*>(&ws[buf][k][(TE * ei + 4 * g) ^ (((k >> 2) & 7) << 2)]);
    };
    // shared-memory reads run one k ahead of the FMAs that use them
    float4 xv[XG], wv[WG];
    rd(0, xv, wv);
#pragma unroll
    for (int k = 0; k < kRgK; ++k) {
      float4 xn[XG], wn[WG];
      if (k + 1 < kRgK) rd(k + 1, xn, wn);
#pragma unroll
      for (int g = 0; g < WG; ++g) {
        const float wj[4] = {wv[g].x, wv[g].y, wv[g].z, wv[g].w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int q = 0; q < XG; ++q) {
            acc[2 * q][4 * g + jj] =
                __ffma2_rn(make_float2(xv[q].x, xv[q].y), make_float2(wj[jj], wj[jj]), acc[2 * q][4 * g + jj]);
            acc[2 * q + 1][4 * g + jj] =
                __ffma2_rn(make_float2(xv[q].z, xv[q].w), make_float2(wj[jj], wj[jj]), acc[2 * q + 1][4 * g + jj]);
          }
      }
      if (k + 1 < kRgK) {
#pragma unroll
        for (int g = 0; g < XG; ++g) xv[g] = xn[g];
#pragma unroll
        for (int g = 0; g < WG; ++g) wv[g] = wn[g];
      }
    }
    if (kc + 1 < nk) store(buf ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int p = 0; p < TT / 2; ++p)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + TT * ti + 2 * p + h;
      if (t >= T) continue;
#pragma unroll
      for (int j = 0; j < TE; ++j) {
        const int e = e0 + TE * ei + j;
        if (e >= E) continue;
        const float a = h ? acc[p][j].y : acc[p][j].x;
        logits[size_t(t) * E + e] = bias ? __fadd_rn(a, bias[e]) : a;
      }
    }
}
// 8 tokens x 4 experts per thread measured fastest at T = 4096, E = 256
// (113 us with 128-token tiles, 117 us with 64; 8 x 8 and 4 x 4 per thread
// were slower): the reads of x, shared by a thread's four neighbours with the
// same tokens, dominate the shared-memory traffic.
constexpr int kRgE = 64, kRgTT = 8, kRgTE = 4;

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

// Top-k and weights of each token of a chunk, and the chunk's per-expert
// assignment counts. One warp per token.
constexpr int kTopkThreads = 512;
template <int MPL>
__global__ void __launch_bounds__(kTopkThreads)
    topk_hist_kernel(const float* __restrict__ logits, int T, int E, int k,
                     int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                     int32_t* __restrict__ chunk_count) {
  extern __shared__ int hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int tt = warp; tt < kChunkTokens; tt += blockDim.x / 32) {
    const int t = blockIdx.x * kChunkTokens + tt;
    if (t >= T) break;
    int myi;
    float myw;
    select_topk<MPL>(logits + size_t(t) * E, E, k, myi, myw);
    if (lane < k) {
      topk_idx[size_t(t) * k + lane] = myi;
      topk_w[size_t(t) * k + lane] = myw;
      atomicAdd(&hist[myi], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_count[size_t(blockIdx.x) * E + e] = hist[e];
}

// Exclusive scan over the threads of one CTA (blockDim.x <= 1024, a multiple of 32).
__device__ int block_exclusive_scan(int v, int* s_warp, int* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < nw) s_warp[lane] = wi - w;
    if (lane == nw - 1) *s_total = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + inc - v;
  __syncthreads();
  return r;
}

// Totals, offsets, per-chunk bases and the block map. One CTA of 1024 threads;
// thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024)
    scan_blocks_kernel(int T, int E, int k, int BM, int n_chunks, int max_blocks,
                       int32_t* __restrict__ chunk, int32_t* __restrict__ count,
                       int32_t* __restrict__ off, int32_t* __restrict__ blocks,
                       int32_t* __restrict__ n_blocks, WsHeader* hdr) {
  __shared__ int s_warp[32];
  __shared__ int s_tot_rows, s_tot_blocks;
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      const int v = chunk[size_t(c) * E + e];
      chunk[size_t(c) * E + e] = total;
      total += v;
    }
  }
  const int nb = (total + BM - 1) / BM;
  const int ex_off = block_exclusive_scan(total, s_warp, &s_tot_rows);
  const int ex_nb = block_exclusive_scan(nb, s_warp, &s_tot_blocks);
  if (e < E) {
    count[e] = total;
    off[e] = ex_off;
    for (int c = 0; c < n_chunks; ++c) chunk[size_t(c) * E + e] += ex_off;
    for (int b = 0; b < nb; ++b) {
      const int idx = ex_nb + b;
      if (idx < max_blocks) {
        blocks[3 * idx + 0] = e;
        blocks[3 * idx + 1] = ex_off + b * BM;
        blocks[3 * idx + 2] = min(BM, total - b * BM);
      }
    }
  }
  if (e == 0) off[E] = s_tot_rows;
  const int routed_blocks = s_tot_blocks;
  const int shared_blocks = (T + BM - 1) / BM;
  for (int s = threadIdx.x; s < shared_blocks; s += blockDim.x) {
    const int idx = routed_blocks + s;
    if (idx < max_blocks) {
      blocks[3 * idx + 0] = E;
      blocks[3 * idx + 1] = T * k + s * BM;
      blocks[3 * idx + 2] = min(BM, T - s * BM);
    }
  }
  if (threadIdx.x == 0) {
    const int total_blocks = routed_blocks + shared_blocks;
    *n_blocks = min(total_blocks, max_blocks);
    if (total_blocks > max_blocks || s_tot_rows != T * k) report(hdr, MOE_ERR_DEVICE_CHECK, 1);
  }
}

// Scatter: position of assignment a = its expert's base for this chunk plus
// the number of earlier assignments of the chunk to the same expert, so the
// permutation is unique (ascending a inside every expert segment).
__global__ void __launch_bounds__(256)
    scatter_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                   const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm,
                   int32_t* __restrict__ inv, WsHeader* hdr) {
  extern __shared__ int sm[];
  int* base = sm;      // [E]
  int* wh = sm + E;    // [8][E] per-warp counts of the current round
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = chunk_base[size_t(blockIdx.x) * E + e];
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kChunkTokens * k;
  const int a1 = min(T, (blockIdx.x + 1) * kChunkTokens) * k;
  const unsigned lt = (1u << lane) - 1u;
  for (int r0 = a0; r0 < a1; r0 += blockDim.x) {
    const int a = r0 + threadIdx.x;
    const bool valid = a < a1;
    int e = valid ? topk_idx[a] : -1;
    if (valid && (e < 0 || e >= E)) {
      report(hdr, MOE_ERR_DEVICE_CHECK, 5);
      e = 0;
    }
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    unsigned peers = 0;
    int rank = 0;
    if (valid) {
      peers = __match_any_sync(act, e);
      rank = __popc(peers & lt);
      if (rank == 0) wh[warp * E + e] = __popc(peers);
    }
    __syncthreads();
    if (valid) {
      int pos = base[e] + rank;
      for (int w2 = 0; w2 < warp; ++w2) pos += wh[w2 * E + e];
      if (pos >= 0 && pos < T * k) {
        perm[pos] = a;
        inv[a] = pos;
      } else {
        report(hdr, MOE_ERR_DEVICE_CHECK, 4);
      }
    }
    __syncthreads();
    if (valid && rank == 0) {
      atomicAdd(&base[e], __popc(peers));
      wh[warp * E + e] = 0;
    }
    __syncthreads();
  }
}

// ---- small token counts (decode): two kernels for the whole routing ----------------------

// Router logits for T <= TT tokens: one warp per expert, every token of the
// call in the same warp. The CTA's kRouterSmallExperts rows of W_r are
// contiguous, so one bulk (TMA) copy brings them into shared memory while the
// token rows are staged; each lane then runs its fixed-order FMA chain.
constexpr int kRouterSmallExperts = 2;

// Token rows are staged D/8 + 1 16-byte words apart so that the tokens' reads
// of one column fall in different banks.
__host__ __device__ constexpr size_t router_small_smem(int TT, int D) {
  return 16 + size_t(kRouterSmallExperts) * D * 4 + size_t(TT) * (D / 8 + 1) * 16;
}

template <int TT>
__global__ void __launch_bounds__(kRouterSmallExperts * 32)
    router_small_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                        const float* __restrict__ bias, int T, int D, int E, float* __restrict__ logits,
                        WsHeader* hdr) {
  extern __shared__ __align__(128) uint8_t rsm[];
  const uint32_t bar = smem_u32(rsm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(rsm + 8);
  const float* ws = reinterpret_cast<const float*>(rsm + 16);
  uint4* xsm4 = reinterpret_cast<uint4*>(rsm + 16 + size_t(kRouterSmallExperts) * D * 4);
  const int e0 = blockIdx.x * kRouterSmallExperts;
  const int ne = min(kRouterSmallExperts, E - e0);
  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) {  // first kernel of the call: start its status afresh
      hdr->status = 0;
      hdr->detail = 0;
    }
    *abort_flag = 0;
    mbar_init(bar, 1);
    mbar_init_fence();
    mbar_arrive_tx(bar, uint32_t(ne) * D * 4);
    bulk_g2s(bar + 16, wr + size_t(e0) * D, uint32_t(ne) * D * 4, bar);
  }
  for (int i = threadIdx.x; i < TT * (D / 8); i += blockDim.x) {
    const int t = i / (D / 8), c8 = i % (D / 8);
    xsm4[t * (D / 8 + 1) + c8] =
        t < T ? *reinterpret_cast<const uint4*>(x + size_t(t) * D + c8 * 8) : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  if (!mbar_wait(bar, 0, abort_flag, hdr, kWaitLimit, true)) return;
  // thread (token t, expert el): one FMA chain over d, 8 columns per step
  const int t = threadIdx.x % TT, el = threadIdx.x / TT;
  if (el >= ne || t >= T) return;
  const int e = e0 + el;
  const float4* w4 = reinterpret_cast<const float4*>(ws + size_t(el) * D);
  const uint4* x4 = xsm4 + size_t(t) * (D / 8 + 1);
  float acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    const uint4 xv = x4[c];
    const float4 wa = w4[2 * c], wb = w4[2 * c + 1];
    acc = fmaf(__uint_as_float(xv.x << 16), wa.x, acc);
    acc = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wa.y, acc);
    acc = fmaf(__uint_as_float(xv.y << 16), wa.z, acc);
    acc = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wa.w, acc);
    acc = fmaf(__uint_as_float(xv.z << 16), wb.x, acc);
    acc = fmaf(__uint_as_float(xv.z & 0xFFFF0000u), wb.y, acc);
    acc = fmaf(__uint_as_float(xv.w << 16), wb.z, acc);
    acc = fmaf(__uint_as_float(xv.w & 0xFFFF0000u), wb.w, acc);
  }
  logits[size_t(t) * E + e] = bias ? __fadd_rn(acc, bias[e]) : acc;
}

// Top-k, weights, histogram, scan, scatter and block map of up to
// kSmallRouteTokens tokens in one CTA of 1024 threads (thread e owns expert e
// for the scan; warp t selects token t's experts).
constexpr int kSmallRouteTokens = 16;

template <int MPL>
__global__ void __launch_bounds__(1024)
    route_small_kernel(const float* __restrict__ logits, int T, int E, int k, int BM, int max_blocks,
                       int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ count,
                       int32_t* __restrict__ off, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                       int32_t* __restrict__ blocks, int32_t* __restrict__ n_blocks, WsHeader* hdr) {
  __shared__ int s_idx[kSmallRouteTokens * 32];
  __shared__ int s_cnt[1024];
  __shared__ int s_warp[32];
  __shared__ int s_tot_rows, s_tot_blocks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int A = T * k;
  s_cnt[threadIdx.x] = 0;
  __syncthreads();
  if (warp < T) {
    int myi;
    float myw;
    select_topk<MPL>(logits + size_t(warp) * E, E, k, myi, myw);
    if (lane < k) {
      topk_idx[warp * k + lane] = myi;
      topk_w[warp * k + lane] = myw;
      s_idx[warp * k + lane] = myi;
      atomicAdd(&s_cnt[myi], 1);
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int total = e < E ? s_cnt[e] : 0;
  const int nb = (total + BM - 1) / BM;
  const int ex_off = block_exclusive_scan(total, s_warp, &s_tot_rows);
  const int ex_nb = block_exclusive_scan(nb, s_warp, &s_tot_blocks);
  if (e < E) {
    count[e] = total;
    off[e] = ex_off;
    for (int b = 0; b < nb; ++b) {
      const int idx = ex_nb + b;
      if (idx < max_blocks) {
        blocks[3 * idx + 0] = e;
        blocks[3 * idx + 1] = ex_off + b * BM;
        blocks[3 * idx + 2] = min(BM, total - b * BM);
      }
    }
    s_cnt[e] = ex_off;  // now the segment start of expert e
  }
  if (e == 0) off[E] = s_tot_rows;
  const int shared_blocks = (T + BM - 1) / BM;
  for (int sb = threadIdx.x; sb < shared_blocks; sb += blockDim.x) {
    const int idx = s_tot_blocks + sb;
    if (idx < max_blocks) {
      blocks[3 * idx + 0] = E;
      blocks[3 * idx + 1] = A + sb * BM;
      blocks[3 * idx + 2] = min(BM, T - sb * BM);
    }
  }
  if (threadIdx.x == 0) {
    const int total_blocks = s_tot_blocks + shared_blocks;
    *n_blocks = min(total_blocks, max_blocks);
    if (total_blocks > max_blocks || s_tot_rows != A) report(hdr, MOE_ERR_DEVICE_CHECK, 6);
  }
  __syncthreads();
  // scatter: rank of assignment a among earlier assignments to the same expert
  const int a = threadIdx.x;
  if (a < A) {
    const int ea = s_idx[a];
    int pos = s_cnt[ea];
    for (int b = 0; b < a; ++b) pos += (s_idx[b] == ea);
    if (pos >= 0 && pos < A) {
      perm[pos] = a;
      inv[a] = pos;
    } else {
      report(hdr, MOE_ERR_DEVICE_CHECK, 7);
    }
  }
}

}  // namespace

cudaError_t route(const Ctx& c) {
  const moe_weights* w = c.w;
  cudaError_t err;
  if (c.T <= kSmallRouteTokens && c.D <= 4096) {
    const int tt = c.T <= 2 ? 2 : c.T <= 8 ? 8 : 16;
    void (*rk)(const uint16_t*, const float*, const float*, int, int, int, float*, WsHeader*) =
        tt == 2 ? router_small_kernel<2> : tt == 8 ? router_small_kernel<8> : router_small_kernel<16>;
    const size_t smem = router_small_smem(tt, c.D);
    if (!ensure_smem_limit(reinterpret_cast<const void*>(rk), int(smem))) return cudaErrorInvalidValue;
    rk<<<(c.E + kRouterSmallExperts - 1) / kRouterSmallExperts, kRouterSmallExperts * 32, smem, c.stream>>>(
        c.x, w->router_w, w->router_bias, c.T, c.D, c.E, c.logits, c.hdr);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    launch_done("router_small", c.stream);
    const int mpl = (c.E + 31) / 32;
    void (*rs)(const float*, int, int, int, int, int, int32_t*, float*, int32_t*, int32_t*, int32_t*, int32_t*,
               int32_t*, int32_t*, WsHeader*) =
        mpl <= 4 ? route_small_kernel<4> : mpl <= 8 ? route_small_kernel<8> : mpl <= 16 ? route_small_kernel<16>
                                                                                    : route_small_kernel<32>;
    rs<<<1, 1024, 0, c.stream>>>(c.logits, c.T, c.E, c.k, c.BM, c.max_blocks, c.topk_idx,
                                                 c.topk_w, c.count, c.off, c.perm, c.inv, c.blocks, c.n_blocks,
                                                 c.hdr);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    launch_done("route_small", c.stream);
    return cudaSuccess;
  }
  if (c.T >= 4096) {  // 128-token tiles still fill the GPU
    dim3 grid((c.T + 127) / 128, (c.E + kRgE - 1) / kRgE);
    router_gemm_kernel<128, kRgE, kRgTT, kRgTE>
        <<<grid, 128 * kRgE / (kRgTT * kRgTE), 0, c.stream>>>(c.x, w->router_w, w->router_bias, c.T, c.D, c.E,
                                                              c.logits, c.hdr);
  } else {
    dim3 grid((c.T + 63) / 64, (c.E + kRgE - 1) / kRgE);
    router_gemm_kernel<64, kRgE, kRgTT, kRgTE>
        <<<grid, 64 * kRgE / (kRgTT * kRgTE), 0, c.stream>>>(c.x, w->router_w, w->router_bias, c.T, c.D, c.E,
                                                             c.logits, c.hdr);
  }
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("router_logits", c.stream);

  {
    const int mpl = (c.E + 31) / 32;
    void (*tk)(const float*, int, int, int, int32_t*, float*, int32_t*) =
        mpl <= 4 ? topk_hist_kernel<4> : mpl <= 8 ? topk_hist_kernel<8> : mpl <= 16 ? topk_hist_kernel<16>
                                                                                  : topk_hist_kernel<32>;
    tk<<<c.n_chunks, kTopkThreads, c.E * sizeof(int), c.stream>>>(c.logits, c.T, c.E, c.k, c.topk_idx, c.topk_w,
                                                                  c.chunk);
  }
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("topk_hist", c.stream);

  scan_blocks_kernel<<<1, 1024, 0, c.stream>>>(c.T, c.E, c.k, c.BM, c.n_chunks, c.max_blocks, c.chunk,
                                               c.count, c.off, c.blocks, c.n_blocks, c.hdr);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("scan_blocks", c.stream);

  scatter_kernel<<<c.n_chunks, 256, 9 * c.E * sizeof(int), c.stream>>>(c.topk_idx, c.T, c.E, c.k, c.chunk,
                                                                       c.perm, c.inv, c.hdr);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done("scatter", c.stream);
  return cudaSuccess;
}

}  // namespace moe
