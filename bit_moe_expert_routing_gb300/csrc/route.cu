// GPU-resident expert routing: router logits, top-k with renormalised
// weights, per-expert histogram, exclusive scan, scatter into expert groups
// and the block map of fixed-size row blocks. All on the caller's stream,
// with no host synchronisation ("Optimizing on-device inference for Apple
// Silicon", section "Keep expert routing on the GPU").
//
// Router logits use one fixed fp32 evaluation order so that the top-k
// decision (an integer result) is reproducible by any implementation:
//   acc[l] = 0, l = 0..31
//   for c = 0 .. D/32-1:  acc[l] = fma(float(x[t, 32c+l]), W_r[e, 32c+l], acc[l])
//   for off = 16, 8, 4, 2, 1:  acc[l] = acc[l] + acc[l+off]   (l < off)
//   logit = acc[0] (+ bias[e])
// Lane l of a warp owns partial sum l; the tree's additions are done with
// warp shuffles.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

// Router logits in the order above for larger T. A warp computes 16 tokens x
// 8 experts: lane l holds partial sum l of each of those 128 logits (as 64
// pairs of tokens for the packed FMA), and the tree reduces them at the end.
// A CTA of kRtWarps warps covers kRtTok tokens x kRtExp experts. D is walked
// in chunks of kRtDC, staged in shared memory one chunk ahead: W (router-
// weight rows) fp32 as in memory, by cp.async; x as words holding one column
// of two tokens in bf16.
constexpr int kRtTok = 32, kRtExp = 32, kRtWarps = 8, kRtDC = 256;
constexpr int kRtWT = 16, kRtWE = 8;  // tokens and experts of a warp
constexpr size_t kRtWBytes = size_t(2) * kRtExp * kRtDC * 4;
constexpr size_t kRtSmem = kRtWBytes + size_t(2) * (kRtTok / 2) * kRtDC * 4;
static_assert((kRtTok / kRtWT) * (kRtExp / kRtWE) == kRtWarps, "one 16 x 8 logit tile per warp");
constexpr int kRtXItems = (kRtTok / 2) * (kRtDC / 4) / (kRtWarps * 32);  // token-pair items per thread and chunk
constexpr int kRtWItems = kRtExp * (kRtDC / 4) / (kRtWarps * 32);        // router-weight pieces per thread and chunk
static_assert(kRtXItems * kRtWarps * 32 == (kRtTok / 2) * (kRtDC / 4), "whole token-pair items");
static_assert(kRtWItems * kRtWarps * 32 == kRtExp * (kRtDC / 4), "whole router-weight pieces");

__device__ __forceinline__ void cp_async16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_all() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// One level of the recursive halving: values 0..2H-1 of each lane, partner
// lane ^ o; the lane keeps the lower H (o bit clear) or the upper H, moved
// down, each plus the partner's value of the same index.
template <int H>
__device__ __forceinline__ void halve_level(float (&v)[128], int lane, int o) {
  const bool upper = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float send = upper ? v[i] : v[i + H];
    const float keep = upper ? v[i + H] : v[i];
    v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
  }
}

__global__ void __launch_bounds__(kRtWarps * 32, 1)
    router_tree_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
                       int T, int D, int E, float* __restrict__ logits, WsHeader* hdr,
                       float4* __restrict__ yacc, size_t yacc_n4) {
  // First kernel of a call: start the call's device status afresh (hdr is
  // null for the later launches of a sliced router and for the later passes
  // of a call, which keep what earlier passes recorded). No other CTA of
  // this kernel reports, so nothing races with the clear.
  if (hdr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    hdr->status = 0;
    hdr->detail = 0;
    hdr->counter = 0;
  }
  // When the grouped GEMM follows, its combine accumulator is cleared here,
  // a slice per CTA (the stores overlap this kernel's arithmetic)
  if (yacc) {
    const size_t cta = size_t(blockIdx.y) * gridDim.x + blockIdx.x, n_cta = size_t(gridDim.x) * gridDim.y;
    for (size_t i = cta * blockDim.x + threadIdx.x; i < yacc_n4; i += n_cta * blockDim.x)
      yacc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  extern __shared__ __align__(16) uint8_t rt_smem_raw[];
  float* wsb = reinterpret_cast<float*>(rt_smem_raw);                    // [2][kRtExp][kRtDC]
  uint32_t* xpb = reinterpret_cast<uint32_t*>(rt_smem_raw + kRtWBytes);  // [2][kRtTok/2][kRtDC]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kRtTok, eb = blockIdx.y * kRtExp;
  const int tg = warp / (kRtExp / kRtWE), eg = warp % (kRtExp / kRtWE);  // token pairs 8tg.., experts 8eg..

  // W pieces m: 16 bytes (4 columns) of router-weight row r (clamped to E-1)
  auto issue_w = [&](int buf, int d0, int dc) {
#pragma unroll
    for (int m = 0; m < kRtWItems; ++m) {
      const int i = threadIdx.x + m * blockDim.x, r = i / (kRtDC / 4), c4 = i % (kRtDC / 4);
      if (4 * c4 < dc)
        cp_async16_cg(smem_u32(wsb + (size_t(buf) * kRtExp + r) * kRtDC + c4 * 4),
                      wr + size_t(min(eb + r, E - 1)) * D + d0 + c4 * 4);
    }
    cp_async_commit_all();
  };
  // x items m: token pair ip, columns 4 dq .. +3 of the chunk
  uint2 xa[kRtXItems], xb[kRtXItems];
  auto load_x = [&](int d0, int dc) {
#pragma unroll
    for (int m = 0; m < kRtXItems; ++m) {
      const int i = threadIdx.x + m * blockDim.x, ip = i / (kRtDC / 4), dq = i % (kRtDC / 4);
      const int ta = t0 + 2 * ip, tb = ta + 1;
      const bool in = 4 * dq < dc;
      xa[m] = (in && ta < T) ? *reinterpret_cast<const uint2*>(x + size_t(ta) * D + d0 + 4 * dq) : make_uint2(0u, 0u);
      xb[m] = (in && tb < T) ? *reinterpret_cast<const uint2*>(x + size_t(tb) * D + d0 + 4 * dq) : make_uint2(0u, 0u);
    }
  };
  auto store_x = [&](int buf) {  // word = (token ta, token tb) of one column, bf16
#pragma unroll
    for (int m = 0; m < kRtXItems; ++m) {
      const int i = threadIdx.x + m * blockDim.x, ip = i / (kRtDC / 4), dq = i % (kRtDC / 4);
      *reinterpret_cast<uint4*>(xpb + (size_t(buf) * (kRtTok / 2) + ip) * kRtDC + 4 * dq) =
          make_uint4(__byte_perm(xa[m].x, xb[m].x, 0x5410), __byte_perm(xa[m].x, xb[m].x, 0x7632),
                     __byte_perm(xa[m].y, xb[m].y, 0x5410), __byte_perm(xa[m].y, xb[m].y, 0x7632));
    }
  };

  float2 acc[8][8];  // [token pair][expert]: .x token 16tg+2p, .y token 16tg+2p+1
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[p][j] = make_float2(0.f, 0.f);

  const int nchunks = (D + kRtDC - 1) / kRtDC;
  issue_w(0, 0, min(kRtDC, D));
  load_x(0, min(kRtDC, D));
  store_x(0);
  cp_async_wait_all();
  __syncthreads();
  for (int kc = 0; kc < nchunks; ++kc) {
    const int buf = kc & 1, d0 = kc * kRtDC, dc = min(kRtDC, D - d0);
    const bool nxt = kc + 1 < nchunks;
    if (nxt) {
      const int dn = min(kRtDC, D - d0 - kRtDC);
      issue_w(buf ^ 1, d0 + kRtDC, dn);
      load_x(d0 + kRtDC, dn);
    }
    const float* wrow = wsb + (size_t(buf) * kRtExp + kRtWE * eg) * kRtDC + lane;
    const uint32_t* xrow = xpb + (size_t(buf) * (kRtTok / 2) + (kRtWT / 2) * tg) * kRtDC + lane;
#pragma unroll 1
    for (int c = 0; c < dc / 32; ++c) {
      float2 wv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = wrow[j * kRtDC + 32 * c];
        wv[j] = make_float2(w, w);
      }
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint32_t w2 = xrow[p * kRtDC + 32 * c];
        const float2 xv = make_float2(__uint_as_float(w2 << 16), __uint_as_float(w2 & 0xFFFF0000u));
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[p][j] = __ffma2_rn(xv, wv[j], acc[p][j]);
      }
    }
    if (nxt) {
      store_x(buf ^ 1);
      cp_async_wait_all();
    }
    __syncthreads();
  }

  // The 32 partial sums of each of the 128 logits are reduced by the tree of
  // the canonical order (lane offsets 16, 8, 4, 2, 1) as a recursive halving:
  // at each level a lane keeps half of its values, sends the other half to
  // its partner and adds what it receives. Every addition joins the same two
  // sub-tree sums as the shuffle-down tree (fp32 addition is commutative), so
  // the logits are bit-identical, with 124 shuffles instead of 640. Value n =
  // 2(8p + j) + b is token 16tg+2p+b, expert 8eg+j; lane l ends with values
  // n = 4l .. 4l+3 in v[0..3].
  float v[128];
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[2 * (8 * p + j)] = acc[p][j].x;
      v[2 * (8 * p + j) + 1] = acc[p][j].y;
    }
  halve_level<64>(v, lane, 16);
  halve_level<32>(v, lane, 8);
  halve_level<16>(v, lane, 4);
  halve_level<8>(v, lane, 2);
  halve_level<4>(v, lane, 1);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int q = 2 * lane + m, p = q >> 3, j = q & 7;
    const int e = eb + kRtWE * eg + j, t = t0 + kRtWT * tg + 2 * p;
    if (e < E) {
      const float be = bias ? bias[e] : 0.f;
      if (t < T) logits[size_t(t) * E + e] = bias ? __fadd_rn(v[2 * m], be) : v[2 * m];
      if (t + 1 < T) logits[size_t(t + 1) * E + e] = bias ? __fadd_rn(v[2 * m + 1], be) : v[2 * m + 1];
    }
  }
}

// Top-k and weights of each token of a chunk, and the chunk's per-expert
// assignment counts. A warp takes kChunkTokens / (kTopkThreads / 32) of the
// chunk's tokens.
constexpr int kTopkThreads = 1024;
template <int MPL>
__global__ void __launch_bounds__(kTopkThreads)
    topk_hist_kernel(const float* __restrict__ logits, int T, int E, int k,
                     int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                     int32_t* __restrict__ chunk_count, int n_chunks, const uint16_t* __restrict__ x, int D,
                     uint16_t* __restrict__ xperm) {
  griddep_wait();  // the logits
  griddep_launch();
  if (int(blockIdx.x) >= n_chunks) {
    // CTAs past the chunks write the paired-order copy of x for the
    // tensor-memory gate/up GEMM (see dq8_bf16_paired), on SMs the top-k
    // leaves idle
    const size_t n8 = size_t(T) * D / 8, step = size_t(gridDim.x - n_chunks) * blockDim.x;
    for (size_t i = size_t(blockIdx.x - n_chunks) * blockDim.x + threadIdx.x; i < n8; i += step) {
      const uint4 v = reinterpret_cast<const uint4*>(x)[i];
      const uint2 lo = make_uint2(v.x, v.y), hi = make_uint2(v.z, v.w);
      const uint2 a = pair_order8_first(lo, hi), b = pair_order8_second(lo, hi);
      reinterpret_cast<uint4*>(xperm)[i] = make_uint4(a.x, a.y, b.x, b.y);
    }
    return;
  }
  extern __shared__ int hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // a warp's tokens: their logits are all loaded first (the loads overlap),
  // then selected one after another
  constexpr int kPerWarp = kChunkTokens / (kTopkThreads / 32);
  constexpr int kAhead = MPL <= 8 ? kPerWarp : 1;  // keys held at once
  static_assert(kPerWarp * (kTopkThreads / 32) == kChunkTokens && kPerWarp % kAhead == 0, "tokens per warp");
  for (int g0 = 0; g0 < kPerWarp; g0 += kAhead) {
    unsigned key[kAhead][MPL];
#pragma unroll
    for (int i = 0; i < kAhead; ++i) {
      const int t = blockIdx.x * kChunkTokens + warp + (g0 + i) * (kTopkThreads / 32);
      if (t < T) load_logit_keys<MPL>(logits + size_t(t) * E, E, key[i]);
    }
#pragma unroll
    for (int i = 0; i < kAhead; ++i) {
      const int t = blockIdx.x * kChunkTokens + warp + (g0 + i) * (kTopkThreads / 32);
      if (t >= T) break;
      int myi;
      float myw;
      select_topk_keys<MPL>(key[i], k, myi, myw);
      if (lane < k) {
        topk_idx[size_t(t) * k + lane] = myi;
        topk_w[size_t(t) * k + lane] = myw;
        atomicAdd(&hist[myi], 1);
      }
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
// a group of adjacent threads owns each expert (E <= 1024).
__global__ void __launch_bounds__(1024)
    scan_blocks_kernel(int T, int E, int k, int BM, int n_chunks, int max_blocks,
                       int32_t* __restrict__ chunk, int32_t* __restrict__ count,
                       int32_t* __restrict__ off, int32_t* __restrict__ blocks,
                       int32_t* __restrict__ n_blocks, WsHeader* hdr) {
  griddep_wait();  // the per-chunk counts
  griddep_launch();
  __shared__ int s_warp_rows[32], s_warp_blocks[32];
  __shared__ int s_tot_rows, s_tot_blocks;
  // tpe threads per expert (adjacent lanes, tpe a power of two dividing 32):
  // thread q of expert e owns the chunks [c0, c1). Its counts are loaded in
  // one batch and kept in registers for the second pass when they fit
  // (kKeep), so the whole scan costs one round of dependent loads.
  constexpr int kKeep = 32;
  int tpe = 1;
  while (tpe < 8 && 2 * tpe * E <= int(blockDim.x)) tpe *= 2;
  const int e = threadIdx.x / tpe, q = threadIdx.x % tpe;
  const bool mine = e < E;
  const int per = (n_chunks + tpe - 1) / tpe;
  const int c0 = min(n_chunks, q * per), c1 = min(n_chunks, c0 + per);
  const bool keep = (c1 - c0) <= kKeep;
  int v[kKeep];
  int part = 0;
  if (mine) {
    if (keep) {
#pragma unroll
      for (int j = 0; j < kKeep; ++j) v[j] = c0 + j < c1 ? chunk[size_t(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kKeep; ++j) part += v[j];
    } else {
      for (int c = c0; c < c1; c += 8) {
        int w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = c + j < c1 ? chunk[size_t(c + j) * E + e] : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) part += w[j];
      }
    }
  }
  // the expert's total and this thread's offset inside it, over its group
  int total = part, q_pre = part;
  for (int o = 1; o < tpe; o <<= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  for (int o = 1; o < tpe; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, q_pre, o);
    if (q >= o) q_pre += u;
  }
  q_pre -= part;  // exclusive
  const bool lead = mine && q == 0;
  const int nb = lead ? (total + BM - 1) / BM : 0;
  const int ex_off_l = block_exclusive_scan(lead ? total : 0, s_warp_rows, &s_tot_rows);
  const int ex_nb_l = block_exclusive_scan(nb, s_warp_blocks, &s_tot_blocks);
  // the group leader's scan results, to every thread of the group
  const int src = (threadIdx.x & 31) & ~(tpe - 1);
  const int ex_off = __shfl_sync(0xffffffffu, ex_off_l, src);
  const int ex_nb = __shfl_sync(0xffffffffu, ex_nb_l, src);
  const int nb_e = __shfl_sync(0xffffffffu, nb, src);
  if (mine) {
    if (q == 0) {
      count[e] = total;
      off[e] = ex_off;
    }
    // each chunk's count becomes its base: the expert's offset plus the
    // counts of the expert's earlier chunks
    int run = ex_off + q_pre;
    if (keep) {
#pragma unroll
      for (int j = 0; j < kKeep; ++j)
        if (c0 + j < c1) {
          chunk[size_t(c0 + j) * E + e] = run;
          run += v[j];
        }
    } else {
      for (int c = c0; c < c1; c += 8) {
        int w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = c + j < c1 ? chunk[size_t(c + j) * E + e] : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c + j < c1) {
            chunk[size_t(c + j) * E + e] = run;
            run += w[j];
          }
      }
    }
    for (int b = q; b < nb_e; b += tpe) {
      const int idx = ex_nb + b;
      if (idx < max_blocks) {
        blocks[3 * idx + 0] = e;
        blocks[3 * idx + 1] = ex_off + b * BM;
        blocks[3 * idx + 2] = min(BM, total - b * BM);
      }
    }
  }
  if (threadIdx.x == 0) off[E] = s_tot_rows;
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
  griddep_wait();  // the chunk bases
  griddep_launch();
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

__host__ __device__ constexpr size_t router_small_smem(int TT, int D) {
  return 16 + size_t(kRouterSmallExperts) * D * 4 + size_t(TT) * D * 2;
}

template <int TT>
__global__ void __launch_bounds__(kRouterSmallExperts * 32)
    router_small_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                        const float* __restrict__ bias, int T, int D, int E, float* __restrict__ logits,
                        WsHeader* hdr, int clear_status, uint16_t* __restrict__ xperm, float4* __restrict__ yacc) {
  griddep_wait();  // launched as a programmatic dependent: everything before is done
  griddep_launch();
  extern __shared__ __align__(128) uint8_t rsm[];
  const uint32_t bar = smem_u32(rsm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(rsm + 8);
  const float* ws = reinterpret_cast<const float*>(rsm + 16);
  uint4* xsm4 = reinterpret_cast<uint4*>(rsm + 16 + size_t(kRouterSmallExperts) * D * 4);
  const uint16_t* xsm = reinterpret_cast<const uint16_t*>(xsm4);
  const int e0 = blockIdx.x * kRouterSmallExperts;
  const int ne = min(kRouterSmallExperts, E - e0);
  if (threadIdx.x == 0) {
    if (blockIdx.x == 0 && clear_status) {  // first kernel of the call: start its status afresh
      hdr->status = 0;
      hdr->detail = 0;
    }
    *abort_flag = 0;
    mbar_init(bar, 1);
    mbar_init_fence();
    mbar_arrive_tx(bar, uint32_t(ne) * D * 4);
    bulk_g2s(bar + 16, wr + size_t(e0) * D, uint32_t(ne) * D * 4, bar);
  }
  // the token rows by cp.async, every copy of a thread in flight at once
  // (rows past T, which the unrolled loop below also reads, are zeroed)
  for (int i = threadIdx.x; i < TT * (D / 8); i += blockDim.x) {
    const int t = i / (D / 8), c8 = i % (D / 8);
    if (t < T)
      cp_async16_cg(smem_u32(xsm4 + i), x + size_t(t) * D + c8 * 8);
    else
      xsm4[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit_all();
  cp_async_wait_all();
  __syncthreads();
  // For the tensor-memory GEMM that follows: the CTAs share out the
  // paired-order copy of x (see dq8_bf16_paired), from the staged rows, and
  // the clearing of the combine accumulator y_acc [T, D].
  const size_t n8 = size_t(T) * (D / 8);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += size_t(gridDim.x) * blockDim.x) {
    if (xperm) {
      const uint4 v = xsm4[i];
      const uint2 lo = make_uint2(v.x, v.y), hi = make_uint2(v.z, v.w);
      const uint2 pa = pair_order8_first(lo, hi), pb = pair_order8_second(lo, hi);
      reinterpret_cast<uint4*>(xperm)[i] = make_uint4(pa.x, pa.y, pb.x, pb.y);
    }
    if (yacc) {  // y_acc holds 2 float4 per chunk of 8 columns
      yacc[2 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
      yacc[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (!mbar_wait(bar, 0, abort_flag, hdr, kWaitLimit, true)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp >= ne) return;
  const int e = e0 + warp;
  const float* w = ws + size_t(warp) * D;
  float acc[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t] = 0.f;
  for (int c = 0; c < D / 32; ++c) {
    const float wv = w[c * 32 + lane];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = fmaf(bf16_to_f32(xsm[t * D + c * 32 + lane]), wv, acc[t]);
  }
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    float a = acc[t];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = __fadd_rn(a, __shfl_down_sync(0xffffffffu, a, off));
    if (lane == 0 && t < T) logits[size_t(t) * E + e] = bias ? __fadd_rn(a, bias[e]) : a;
  }
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
  griddep_wait();  // the logits
  griddep_launch();
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

cudaError_t route_logits_small(const Ctx& c, uint16_t* xperm, float* yacc) {
  const moe_weights* w = c.w;
  if (c.T > kSmallRouteTokens || c.D > 4096) return cudaErrorInvalidValue;
  const int tt = c.T <= 2 ? 2 : c.T <= 8 ? 8 : 16;
  void (*rk)(const uint16_t*, const float*, const float*, int, int, int, float*, WsHeader*, int, uint16_t*, float4*) =
      tt == 2 ? router_small_kernel<2> : tt == 8 ? router_small_kernel<8> : router_small_kernel<16>;
  const size_t smem = router_small_smem(tt, c.D);
  if (!ensure_smem_limit(reinterpret_cast<const void*>(rk), int(smem))) return cudaErrorInvalidValue;
  cudaError_t err = launch_pdl(c, rk, dim3((c.E + kRouterSmallExperts - 1) / kRouterSmallExperts),
                               dim3(kRouterSmallExperts * 32), smem, c.x, w->router_w, w->router_bias, c.T, c.D,
                               c.E, c.logits, c.hdr, c.first_pass ? 1 : 0, xperm, reinterpret_cast<float4*>(yacc));
  if (err != cudaSuccess) return err;
  launch_done(c, "router_small");
  return cudaSuccess;
}

int router_wave_tokens(int E) {
  const int expert_tiles = (E + kRtExp - 1) / kRtExp;  // one CTA per SM (254 registers per thread)
  return kRtTok * std::max(1, num_sms() / expert_tiles);
}

cudaError_t wait_x(const Ctx& c) {
  for (int i = 0; i < c.n_x_slices; ++i) {
    const cudaError_t err = cudaStreamWaitEvent(c.stream, c.x_ready[i], 0);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t route(const Ctx& c, bool* yacc_zeroed) {
  const moe_weights* w = c.w;
  cudaError_t err;
  // one CTA of 1024 threads does the small-T top-k: up to 16 logits per lane
  if (c.T <= kSmallRouteTokens && c.D <= 4096 && c.E <= 512) {
    if ((err = wait_x(c)) != cudaSuccess) return err;
    // the router also writes the paired-order x and, when the grouped GEMM
    // follows, clears y_acc
    if ((err = route_logits_small(c, c.xperm, yacc_zeroed ? c.y_acc : nullptr)) != cudaSuccess) return err;
    if (yacc_zeroed) *yacc_zeroed = true;
    const int mpl = (c.E + 31) / 32;
    void (*rs)(const float*, int, int, int, int, int, int32_t*, float*, int32_t*, int32_t*, int32_t*, int32_t*,
               int32_t*, int32_t*, WsHeader*) =
        mpl <= 4 ? route_small_kernel<4> : mpl <= 8 ? route_small_kernel<8> : route_small_kernel<16>;
    if ((err = launch_pdl(c, rs, dim3(1), dim3(1024), 0, c.logits, c.T, c.E, c.k, c.BM, c.max_blocks, c.topk_idx,
                          c.topk_w, c.count, c.off, c.perm, c.inv, c.blocks, c.n_blocks, c.hdr)) != cudaSuccess)
      return err;
    launch_done(c, "route_small");
    return cudaSuccess;
  }
  {
    auto* rk = router_tree_kernel;
    const size_t smem = kRtSmem;
    if (!ensure_smem_limit(reinterpret_cast<const void*>(rk), int(smem))) return cudaErrorInvalidValue;
    const bool zero = yacc_zeroed != nullptr;
    // one launch per slice of x still arriving from the host (one launch for
    // all of x otherwise); each clears the y_acc rows of its own tokens
    const int n_sl = c.n_x_slices > 0 ? c.n_x_slices : 1;
    for (int i = 0, t0 = 0; i < n_sl; ++i) {
      const int t1 = c.n_x_slices > 0 ? c.x_slice_end[i] : c.T;
      if (c.n_x_slices > 0 && (err = cudaStreamWaitEvent(c.stream, c.x_ready[i], 0)) != cudaSuccess) return err;
      if (t1 > t0) {
        const int n = t1 - t0;
        rk<<<dim3((n + kRtTok - 1) / kRtTok, (c.E + kRtExp - 1) / kRtExp), kRtWarps * 32, smem, c.stream>>>(
            c.x + size_t(t0) * c.D, w->router_w, w->router_bias, n, c.D, c.E, c.logits + size_t(t0) * c.E,
            (t0 == 0 && c.first_pass) ? c.hdr : nullptr, zero ? reinterpret_cast<float4*>(c.y_acc + size_t(t0) * c.D) : nullptr,
            zero ? size_t(n) * c.D / 4 : 0);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        launch_done(c, "router_logits");
      }
      t0 = t1;
    }
    if (zero) *yacc_zeroed = true;
  }

  {
    const int mpl = (c.E + 31) / 32;
    void (*tk)(const float*, int, int, int, int32_t*, float*, int32_t*, int, const uint16_t*, int, uint16_t*) =
        mpl <= 4 ? topk_hist_kernel<4> : mpl <= 8 ? topk_hist_kernel<8> : mpl <= 16 ? topk_hist_kernel<16>
                                                                                  : topk_hist_kernel<32>;
    // with the paired-order copy of x to write, the SMs the chunks leave idle
    // (at least 16 CTAs) take it
    const int n_copy = c.xperm ? std::max(16, num_sms() - c.n_chunks) : 0;
    err = launch_pdl(c, tk, dim3(c.n_chunks + n_copy), dim3(kTopkThreads), c.E * sizeof(int), c.logits, c.T, c.E,
                     c.k, c.topk_idx, c.topk_w, c.chunk, c.n_chunks, c.x, c.D, c.xperm);
  }
  if (err != cudaSuccess) return err;
  launch_done(c, "topk_hist");

  err = launch_pdl(c, scan_blocks_kernel, dim3(1), dim3(1024), 0, c.T, c.E, c.k, c.BM, c.n_chunks, c.max_blocks,
                   c.chunk, c.count, c.off, c.blocks, c.n_blocks, c.hdr);
  if (err != cudaSuccess) return err;
  launch_done(c, "scan_blocks");

  err = launch_pdl(c, scatter_kernel, dim3(c.n_chunks), dim3(256), 9 * c.E * sizeof(int), c.topk_idx, c.T, c.E,
                   c.k, c.chunk, c.perm, c.inv, c.hdr);
  if (err != cudaSuccess) return err;
  launch_done(c, "scatter");
  return cudaSuccess;
}

}  // namespace moe
