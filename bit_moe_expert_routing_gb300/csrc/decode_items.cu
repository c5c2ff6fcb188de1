// The whole layer for 2..8 token rows in one cooperative launch, as items
// ("Optimizing on-device inference for Apple Silicon": "Optimise the
// single-row weight path", "Keep expert routing on the GPU", "Reduce
// intermediate and state traffic").
//
// An item is 32 consecutive intermediate rows of one expert of the union of
// the rows' selected experts (the shared expert last). For every row routed to
// that expert, the CTA that owns the item computes those 32 values of h and
// multiplies them with the matching 32-code column block of the expert's down
// matrix: its share of that row's output, which it adds, times the routing
// weight, into the fp32 accumulator. Each expert's weights are read once,
// whatever the number of rows that selected it, and no CTA waits for another
// CTA's h: the CTAs wait on each other once, for the router logits.
//   1. Entry: bulk copies of the CTA's router rows; every row of x staged
//      chunk-major in fp32; the accumulator cleared.
//   2. Logits of the CTA's experts for every row, in the canonical order;
//      grid barrier.
//   3. Every CTA takes the same top-k of every row (warp t: row t), the union
//      of the selected experts in ascending index and the (row, expert) pairs
//      in the permuted order (expert-major, rows ascending), then the shared
//      expert's pairs. CTA 0 writes the routing tables.
//   4. Work units n = blockIdx.x, + gridDim.x, ...: a unit is an item and a
//      group of at most two of its expert's pairs, so that an expert that many
//      rows selected is spread over several CTAs (which read its weights from
//      L2 side by side); the shared expert's units come first. Per unit:
//      gate/up codes, scales and biases in four 8-row sub-items (bulk copies,
//      one mbarrier each), the down column block (2-D tensor copies of 64
//      rows), the scale and bias words of each thread's output columns (loads
//      into registers). Warps 4s..4s+3 take sub-item s: rows 2q, 2q+1 of warp
//      4s+q, gate and up, for each pair of the unit. Once every sub-item has
//      been read, the next unit's gate/up copies start; once the down block
//      has been read, its down copies.
//   5. The last CTA to arrive on the counter converts the accumulator to
//      bf16 y.
// The accumulator's fp32 additions land in arrival order, as in the grouped
// GEMM's combine: results agree up to the summation order.
//
// Every wait is bounded: an expired wait records MOE_ERR_DEVICE_TIMEOUT in the
// workspace status word and the CTA skips its remaining units, but still
// arrives on the counter; no copy of a later unit is started after it, and
// copies already started are waited for (bounded) before the CTA exits.
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

constexpr int kDiWarps = 16;
constexpr int kDiThreads = kDiWarps * 32;
constexpr int kDiMaxT = 8;           // token rows
constexpr int kDiMaxPairs = 128;     // (row, expert) pairs T * (k + 1); also bounds the union
constexpr int kDiRows = 32;          // intermediate rows per item: one 32-code chunk of a down row
constexpr int kDiSubRows = 8;        // rows per sub-item (one mbarrier)
constexpr int kDiSubs = kDiRows / kDiSubRows;
constexpr int kDiCopies = 6;         // bulk copies per sub-item: gate codes, up codes, four scale/bias rows
constexpr int kDiRouterRows = 2;     // router rows (experts) per CTA, at most
constexpr int kDiColsPerThread = 4;  // output columns per thread in the down step, blockDim.x apart
constexpr int kDiDownBox = 64;       // down rows per tensor copy (one lane each)
constexpr int kDiPairsPerUnit = 2;   // pairs of one expert a work unit computes, at most
static_assert(kDiWarps == 4 * kDiSubs && kDiSubRows == 8, "four warps per sub-item, two rows per warp");
static_assert(kDiCopies * kDiSubs <= 32, "one lane per bulk copy");
static_assert(kDiColsPerThread * kDiThreads == 32 * kDiDownBox, "one lane per tensor copy of the down block");

// Shared-memory plan (bytes from the dynamic base) for D and T rows.
struct ItemsSmem {
  size_t xs4, xsum, wr, item, dcodes, gu, hv, total;
  size_t sub_codes, sub_sb, sub_bytes;  // per sub-item: one matrix's codes, one scale or bias row set, all
  int xst;                              // float4 stride of a quarter-row of x (D/32 + 1: conflict-free)
  __host__ __device__ ItemsSmem(int D, int T) {
    xst = D / 32 + 1;
    sub_codes = size_t(kDiSubRows) * D / 2;
    sub_sb = size_t(kDiSubRows) * (D / 64) * 2;
    sub_bytes = 2 * sub_codes + 4 * sub_sb;
    xs4 = 128;  // bytes 0..127: six mbarriers and the flags
    xsum = xs4 + size_t(T) * 8 * xst * 16;
    wr = (xsum + size_t(T) * (D / 32) * 4 + 127) & ~size_t(127);
    item = (wr + size_t(kDiRouterRows) * D * 4 + 127) & ~size_t(127);
    dcodes = (item + kDiSubs * sub_bytes + 127) & ~size_t(127);
    gu = dcodes + size_t(D) * 16;         // [kDiMaxT][2][kDiRows] gate and up dot products
    hv = gu + size_t(kDiMaxT) * 2 * kDiRows * 4;  // [kDiMaxT][kDiRows + 4]: h as fp32, then its sum
    total = hv + size_t(kDiMaxT) * (kDiRows + 4) * 4;
  }
};

// Tensor maps of the down codes as [rows][I/8] 32-bit words, boxes of 4
// words x kDiDownBox rows: every expert's matrix (rows E*D) and the shared
// expert's (rows D).
struct ItemMaps {
  CUtensorMap routed, shared;
};

struct ItemsArgs {
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
  uint16_t* h;  // [T*k + T][I]: the routed pairs in permuted order, then the shared expert's rows T*k + t
  float* y_acc;  // [T][D]
  uint16_t* y;
  WsHeader* hdr;
  int T, D, E, k, I, max_blocks;
};

__device__ __forceinline__ void tma_2d_load(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void red_add(float* dst, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(v) : "memory");
}

// Grid-wide barrier of a cooperative launch on the header's counter (zeroed
// before the launch): every CTA arrives once (release) and thread 0 polls,
// for at most kWaitLimit cycles, until `target` arrivals, then one acquire
// fence. Returns false on expiry (MOE_ERR_DEVICE_TIMEOUT recorded).
__device__ __forceinline__ bool items_barrier(WsHeader* hdr, unsigned target, volatile int* result) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&hdr->counter) : "memory");
    const long long t0 = clock64();
    int ok = 1;
    while (true) {
      unsigned v;
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&hdr->counter) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > kWaitLimit) {
        report(hdr, MOE_ERR_DEVICE_TIMEOUT, 140);
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

template <int MPL>
__global__ void __launch_bounds__(kDiThreads, 1)
    decode_items_kernel(ItemsArgs a, const __grid_constant__ ItemMaps dm) {
  extern __shared__ __align__(128) uint8_t ism[];
  __shared__ int s_sel[kDiMaxPairs];                // [T][k] expert of slot j
  __shared__ float s_selw[kDiMaxPairs];             // its routing weight
  __shared__ unsigned s_tmask[(kDiMaxT + 1) * 32];  // per row (then the union): its experts as bits (E <= 1024)
  __shared__ int s_tpre[(kDiMaxT + 1) * 33];        // set bits of each mask below each word, and in all
  __shared__ int s_ulist[kDiMaxPairs];              // union: selected experts ascending, then E (shared)
  __shared__ int s_ucnt[kDiMaxPairs];               // pairs of each union entry
  __shared__ int s_ubase[kDiMaxPairs + 1];          // its first pair
  __shared__ int s_ptok[kDiMaxPairs];               // pair -> row
  __shared__ int s_pa[kDiMaxPairs];                 // pair -> assignment t*k + j (T*k + t: shared)
  __shared__ float s_pw[kDiMaxPairs];               // pair -> routing weight (1 for the shared expert)
  __shared__ int s_uoff[kDiMaxPairs + 1];           // first work unit of each union entry, shared expert first

  const int T = a.T, D = a.D, E = a.E, k = a.k, I = a.I;
  const int nch = D / 32, G = D / 64, Gi = I / 64;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const ItemsSmem L(D, T);
  const int xst = L.xst;
  const uint32_t bar0 = smem_u32(ism);  // mbarriers: sub-items 0..3, the down block, the router rows
  const uint32_t dbar = bar0 + 8u * kDiSubs, rbar = dbar + 8u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ism + 64);
  volatile int* gb_ok = reinterpret_cast<volatile int*>(ism + 68);
  volatile int* last_flag = reinterpret_cast<volatile int*>(ism + 72);
  float4* xs4 = reinterpret_cast<float4*>(ism + L.xs4);
  float* xsum = reinterpret_cast<float*>(ism + L.xsum);
  float* gu = reinterpret_cast<float*>(ism + L.gu);
  float* hv = reinterpret_cast<float*>(ism + L.hv);
  const int RB = I / kDiRows;  // items per expert
  int n_rt = 0;                // router rows (experts) of this CTA: cta, cta + ncta
  for (int m = 0; m < kDiRouterRows; ++m) n_rt += (cta + m * ncta < E);

  // --- entry: barriers, the router rows' copies, x, the accumulator
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kDiSubs + 2; ++i) mbar_init(bar0 + 8u * i, 1);
    mbar_init_fence();
    if (n_rt) mbar_arrive_tx(rbar, uint32_t(n_rt) * D * 4);
  }
  __syncthreads();
  if (warp == 0 && lane < n_rt)
    bulk_g2s(bar0 + uint32_t(L.wr) + lane * D * 4, a.router_w + size_t(cta + lane * ncta) * D, D * 4, rbar);
  for (int q0 = tid; q0 < T * (D / 8); q0 += 4 * blockDim.x) {  // four 16-byte loads in flight a thread
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = q0 + j * blockDim.x;
      if (q < T * (D / 8)) v[j] = __ldg(reinterpret_cast<const uint4*>(a.x) + q);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = q0 + j * blockDim.x;
      if (q < T * (D / 8)) stage_bf16x8(xs4 + size_t(q / (D / 8)) * 8 * xst, xst, q % (D / 8), v[j]);
    }
  }
  // the accumulator starts at zero; the grid barrier orders this before any red.add
  for (int q = cta * blockDim.x + tid; q < T * D / 4; q += ncta * blockDim.x)
    reinterpret_cast<float4*>(a.y_acc)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  for (int q = tid; q < T * nch; q += blockDim.x) {  // per-chunk sums of x
    const int t = q / nch, c = q % nch;
    const float4* xr = xs4 + size_t(t) * 8 * xst;
    float sum = 0.f;
#pragma unroll
    for (int jq = 0; jq < 8; ++jq) {
      const float4 v = xr[jq * xst + c];
      sum += (v.x + v.y) + (v.z + v.w);
    }
    xsum[q] = sum;
  }

  // --- router logits of this CTA's experts (warp m: expert cta + m * ncta) for
  // every row, in the canonical order: lane l sums elements 32c + l with
  // fused multiply-adds, then the pairwise tree, then the bias
  if (warp < n_rt) {
    const bool landed = __all_sync(0xffffffffu, mbar_wait(rbar, 0, abort_flag, a.hdr, kWaitLimit, true, 141));
    if (landed) {
      const int e = cta + warp * ncta;
      const float* w = reinterpret_cast<const float*>(ism + L.wr) + size_t(warp) * D;
      // element 32c + lane of row t: float (lane / 4) * xst * 4 + 4c + lane % 4 of the row
      const float* xf = reinterpret_cast<const float*>(xs4) + (lane >> 2) * xst * 4 + (lane & 3);
      float acc[kDiMaxT];
#pragma unroll
      for (int t = 0; t < kDiMaxT; ++t) acc[t] = 0.f;
#pragma unroll 4
      for (int c = 0; c < nch; ++c) {
        const float wv = w[32 * c + lane];
#pragma unroll
        for (int t = 0; t < kDiMaxT; ++t)
          if (t < T) acc[t] = fmaf(xf[t * 8 * xst * 4 + c * 4], wv, acc[t]);
      }
#pragma unroll
      for (int t = 0; t < kDiMaxT; ++t) {
        if (t >= T) break;
        float v = acc[t];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
        if (lane == 0) a.logits[size_t(t) * E + e] = a.router_bias ? __fadd_rn(v, a.router_bias[e]) : v;
      }
    }
  }
  if (n_rt && warp == kDiWarps - 1) mbar_wait(rbar, 0, abort_flag, a.hdr, kWaitLimit, true, 141);  // landed before any exit
  const bool ok1 = items_barrier(a.hdr, unsigned(ncta), gb_ok);

  // --- top-k of every row (warp t), the union and the pairs. Each row's
  // experts also go into a bit mask of its own, so that every assignment
  // finds its union entry, its place among the entry's rows and the entry's
  // first pair from counts of set bits, with no search.
  for (int i = tid; i < (T + 1) * 32; i += blockDim.x) s_tmask[i] = 0u;  // mask T: the union
  __syncthreads();
  if (warp < T) {
    int myi = 0;
    float myw = 0.f;
    if (ok1) select_topk<MPL, true>(a.logits + size_t(warp) * E, E, k, myi, myw);
    if (lane < k) {
      if (myi < 0 || myi >= E) {
        report(a.hdr, MOE_ERR_DEVICE_CHECK, 142);
        myi = 0;
      }
      s_sel[warp * k + lane] = myi;
      s_selw[warp * k + lane] = myw;
      atomicOr(&s_tmask[warp * 32 + (myi >> 5)], 1u << (myi & 31));
      atomicOr(&s_tmask[T * 32 + (myi >> 5)], 1u << (myi & 31));
      if (cta == 0) {
        a.topk_idx[warp * k + lane] = myi;
        a.topk_w[warp * k + lane] = myw;
      }
    }
  }
  __syncthreads();
  if (warp <= T) {  // per mask (a row's, or the union's): set bits below each word, a warp scan
    const int c = __popc(s_tmask[warp * 32 + lane]);
    int v = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    s_tpre[warp * 33 + lane] = v - c;
    if (lane == 31) s_tpre[warp * 33 + 32] = v;
  }
  __syncthreads();
  const int n_routed = s_tpre[T * 33 + 32];
  const int n_union = n_routed + 1;
  // bits below expert e in mask m (m = T: the union; its rank there is its entry)
  auto below = [&](int m, int e) {
    return s_tpre[m * 33 + (e >> 5)] + __popc(s_tmask[m * 32 + (e >> 5)] & ((1u << (e & 31)) - 1u));
  };
  for (int q = tid; q < T * k; q += blockDim.x) {  // assignment q = t*k + j
    const int t = q / k, e = s_sel[q];
    const unsigned bit = 1u << (e & 31);
    int pos = 0, cnt = 0, base = 0;  // among the expert's rows; its rows; pairs of lower experts
    for (int t2 = 0; t2 < T; ++t2) {
      const int has = (s_tmask[t2 * 32 + (e >> 5)] & bit) ? 1 : 0;
      cnt += has;
      pos += (t2 < t) ? has : 0;
      base += below(t2, e);
    }
    const int u = below(T, e), p = base + pos;
    if (pos == 0) {
      s_ulist[u] = e;
      s_ucnt[u] = cnt;
      s_ubase[u] = base;
    }
    s_ptok[p] = t;
    s_pa[p] = q;
    s_pw[p] = s_selw[q];
  }
  for (int t = tid; t < T; t += blockDim.x) {  // the shared expert: pairs T*k + t
    const int p = T * k + t;
    s_ptok[p] = t;
    s_pa[p] = p;
    s_pw[p] = 1.f;
  }
  if (tid == 0) {
    s_ulist[n_routed] = E;
    s_ucnt[n_routed] = T;
    s_ubase[n_routed] = T * k;
    s_ubase[n_union] = T * k + T;
  }
  __syncthreads();
  // work units: processing order v = 0 (the shared expert), 1.. (entry v - 1);
  // entry of order v has RB * ceil(pairs / kDiPairsPerUnit) units (warp 0 scan)
  if (warp == 0) {
    int run = 0;
    for (int v0 = 0; v0 < n_union; v0 += 32) {
      const int v = v0 + lane;
      const int u = v == 0 ? n_routed : v - 1;
      const int nu = v < n_union ? RB * ((s_ucnt[u] + kDiPairsPerUnit - 1) / kDiPairsPerUnit) : 0;
      int inc = nu;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
      }
      if (v < n_union) s_uoff[v] = run + inc - nu;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) s_uoff[n_union] = run;
  }
  __syncthreads();

  // CTA 0: the routing tables for inspection (count, offsets, permutation,
  // block map: one block per selected expert, then the shared expert's)
  if (cta == 0) {
    for (int e = tid; e < E; e += blockDim.x) {
      int cnt = 0, base = 0;
      for (int t = 0; t < T; ++t) {
        cnt += (s_tmask[t * 32 + (e >> 5)] >> (e & 31)) & 1u;
        base += below(t, e);
      }
      a.count[e] = cnt;
      a.off[e] = base;
    }
    if (tid == 0) a.off[E] = T * k;
    for (int p = tid; p < T * k; p += blockDim.x) {
      a.perm[p] = s_pa[p];
      a.inv[s_pa[p]] = p;
    }
    for (int u = tid; u < n_union && u < a.max_blocks; u += blockDim.x) {
      a.blocks[3 * u + 0] = s_ulist[u];
      a.blocks[3 * u + 1] = s_ubase[u];
      a.blocks[3 * u + 2] = s_ucnt[u];
    }
    if (tid == 0) *a.n_blocks = min(n_union, a.max_blocks);
  }

  // --- work units n = cta, cta + ncta, ... Unit n: the order v with
  // s_uoff[v] <= n < s_uoff[v + 1]; within it, row block j / ng and pair
  // group j % ng (ng groups), so the groups of one row block sit on
  // neighbouring CTAs
  const int n_items = ok1 ? s_uoff[n_union] : 0;
  struct Unit {
    int u, ii, p0, np;  // union entry, first intermediate row, first pair, pairs
  };
  auto unit = [&](int n) {
    int lo = 0, hi = n_union;  // s_uoff[lo] <= n < s_uoff[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_uoff[mid] <= n)
        lo = mid;
      else
        hi = mid;
    }
    Unit r;
    r.u = lo == 0 ? n_routed : lo - 1;
    const int cnt = s_ucnt[r.u], ng = (cnt + kDiPairsPerUnit - 1) / kDiPairsPerUnit, j = n - s_uoff[lo];
    r.ii = (j / ng) * kDiRows;
    const int g = j % ng;
    r.p0 = s_ubase[r.u] + g * kDiPairsPerUnit;
    r.np = min(kDiPairsPerUnit, cnt - g * kDiPairsPerUnit);
    return r;
  };
  // The gate/up copies of item n (warp 0): lane 0 sets the byte counts, then
  // lane q < 24 issues part q % 6 (gate codes, up codes, gate scales, gate
  // biases, up scales, up biases) of sub-item q / 6: contiguous blocks.
  auto issue_gateup = [&](int n) {
    const Unit un = unit(n);
    const int ii = un.ii, e = s_ulist[un.u];
    const bool sh = (e == E);
    if (lane == 0)
      for (int sub = 0; sub < kDiSubs; ++sub) mbar_arrive_tx(bar0 + 8u * sub, uint32_t(L.sub_bytes));
    __syncwarp();
    if (lane < kDiCopies * kDiSubs) {
      const int sub = lane / kDiCopies, part = lane % kDiCopies;
      const moe_qmatrix& mq =
          part == 0 || part == 2 || part == 3 ? (sh ? a.s_gate : a.gate) : (sh ? a.s_up : a.up);
      const size_t row0 = size_t(sh ? 0 : e) * I + ii + sub * kDiSubRows;
      const uint32_t dst = bar0 + uint32_t(L.item + sub * L.sub_bytes), bar = bar0 + 8u * sub;
      if (part < 2)
        bulk_g2s(dst + part * uint32_t(L.sub_codes), mq.codes + row0 * (D / 8), uint32_t(L.sub_codes), bar);
      else
        bulk_g2s(dst + uint32_t(2 * L.sub_codes + (part - 2) * L.sub_sb),
                 ((part & 1) ? mq.biases : mq.scales) + row0 * G, uint32_t(L.sub_sb), bar);
    }
  };
  // The down column block of item n (warp 1): lane l copies rows 64 l .. 64 l + 63.
  auto issue_down = [&](int n) {
    const Unit un = unit(n);
    const int ii = un.ii, e = s_ulist[un.u];
    const bool sh = (e == E);
    if (lane == 0) mbar_arrive_tx(dbar, uint32_t(D) * 16);
    __syncwarp();
    if (lane * kDiDownBox < D)
      tma_2d_load(bar0 + uint32_t(L.dcodes) + lane * kDiDownBox * 16, sh ? &dm.shared : &dm.routed, ii / 8,
                  (sh ? 0 : e) * D + lane * kDiDownBox, dbar);
  };
  // The aligned 32-bit words holding the scale (and the bias) of item n's
  // group for this thread's output columns d = tid + c * blockDim.x. Element
  // (row, g) is number row * Gi + g of its array; the word is number (that
  // >> 1) from the 16-byte-aligned base, so it never crosses the end of the
  // array (D is even, so every array holds an even number of elements).
  uint32_t dsc[kDiColsPerThread], dbi[kDiColsPerThread];
  auto load_sb = [&](int n) {
    const Unit un = unit(n);
    const int ii = un.ii, e = s_ulist[un.u];
    const bool sh = (e == E);
    const moe_qmatrix& md = sh ? a.s_down : a.down;
    const size_t r0 = size_t(sh ? 0 : e) * D;
#pragma unroll
    for (int c = 0; c < kDiColsPerThread; ++c) {
      const int d = tid + c * blockDim.x;
      if (d < D) {
        const size_t el = (r0 + d) * Gi + ii / 64;
        dsc[c] = __ldg(reinterpret_cast<const uint32_t*>(md.scales) + (el >> 1));
        dbi[c] = __ldg(reinterpret_cast<const uint32_t*>(md.biases) + (el >> 1));
      }
    }
  };

  if (cta < n_items) {
    if (warp == 0) issue_gateup(cta);
    if (warp == 1) issue_down(cta);
    load_sb(cta);
  }
  bool go = cta < n_items;
  int it = 0;
  bool g_next = false;  // the next item's gate/up copies are in flight
  for (int n = cta; go; ++it, n += ncta) {
    const uint32_t ph = uint32_t(it) & 1u;  // each barrier completes once per item
    const Unit un = unit(n);
    const int ii = un.ii, pb = un.p0, np = un.np;
    const bool has_next = n + ncta < n_items;

    // gate/up: warps 4s .. 4s + 3 take sub-item s, warp 4s + q its rows 2q
    // and 2q + 1 (dot products j = 2 * row + matrix), for every pair of the
    // item's expert; every wait drains, so no copy is in flight at exit
    {
      const int sub = warp >> 2, r0 = 2 * (warp & 3);
      if (!mbar_wait(bar0 + 8u * sub, ph, abort_flag, a.hdr, kWaitLimit, true, 143)) {
        *abort_flag = 1;
      } else {
        const uint8_t* base = ism + L.item + sub * L.sub_bytes;
        const uint16_t* sb = reinterpret_cast<const uint16_t*>(base + 2 * L.sub_codes);  // [4][kDiSubRows][G]
        for (int pp = 0; pp < np; ++pp) {
          const int t = s_ptok[pb + pp];
          const float4* xr = xs4 + size_t(t) * 8 * xst;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int c = lane; c < nch; c += 32) {
            float4 xv[8];
#pragma unroll
            for (int jq = 0; jq < 8; ++jq) xv[jq] = xr[jq * xst + c];
            const float sx = xsum[t * nch + c];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int r = r0 + (j >> 1), mat = j & 1;
              const uint4 w4 = reinterpret_cast<const uint4*>(base + mat * L.sub_codes + size_t(r) * (D / 2))[c];
              const uint16_t* srow = sb + (2 * mat) * (kDiSubRows * G) + r * G;  // scales; the biases follow
              acc[j] += chunk_dot_r(w4, xv, sx, srow[c / 2], srow[kDiSubRows * G + c / 2]);
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
            gu[(pp * 2 + (lane & 1)) * kDiRows + sub * kDiSubRows + r0 + (lane >> 1)] = v;
          }
        }
      }
    }
    __syncthreads();  // every sub-item has been read
    bool live = !*abort_flag;
    g_next = live && has_next;
    if (g_next && warp == 0) issue_gateup(n + ncta);
    // h of the item's 32 rows for pair pp (warp pp, lane i: row ii + i),
    // rounded to bf16, at the pair's row of h; and the sum of the 32
    if (live && warp < np) {
      const uint16_t hb = f32_to_bf16(silu_mul(gu[(warp * 2) * kDiRows + lane], gu[(warp * 2 + 1) * kDiRows + lane]));
      const float hf = bf16_to_f32(hb);
      hv[warp * (kDiRows + 4) + lane] = hf;
      float hs = hf;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) hs += __shfl_xor_sync(0xffffffffu, hs, off);
      if (lane == 0) hv[warp * (kDiRows + 4) + kDiRows] = hs;
      a.h[size_t(pb + warp) * I + ii + lane] = hb;
    }
    // the down block of this item (every thread waits: it drains the copy)
    if (!mbar_wait(dbar, ph, abort_flag, a.hdr, kWaitLimit, true, 144)) *abort_flag = 1;
    __syncthreads();  // h and the down block are in place
    live = !*abort_flag;
    if (live) {
      const uint4* dc = reinterpret_cast<const uint4*>(ism + L.dcodes);
      for (int pp = 0; pp < np; ++pp) {
        const int t = s_ptok[pb + pp];
        const float wt = s_pw[pb + pp];
        const float* hp = hv + pp * (kDiRows + 4);
        float4 hx[8];
#pragma unroll
        for (int jq = 0; jq < 8; ++jq) hx[jq] = reinterpret_cast<const float4*>(hp)[jq];
        const float hs = hp[kDiRows];
#pragma unroll
        for (int c = 0; c < kDiColsPerThread; ++c) {
          const int d = tid + c * blockDim.x;
          if (d < D) {
            // the group's bf16 inside the loaded word (the expert's first row is even: D is even)
            const int sh16 = 16 * ((d * Gi + ii / 64) & 1);
            const uint16_t sc = uint16_t(dsc[c] >> sh16), bi = uint16_t(dbi[c] >> sh16);
            red_add(a.y_acc + size_t(t) * D + d, wt * chunk_dot_r(dc[d], hx, hs, sc, bi));
          }
        }
      }
    }
    __syncthreads();  // the down block, h and the scale/bias words have been read
    go = !*abort_flag && has_next;
    if (go) {
      if (warp == 1) issue_down(n + ncta);
      load_sb(n + ncta);
    }
  }
  // after an expired wait, the next item's gate/up copies may still be
  // landing: wait for them (bounded) before the CTA exits
  if (g_next && warp < kDiSubs && lane == 0)
    mbar_wait(bar0 + 8u * warp, uint32_t(it) & 1u, abort_flag, a.hdr, kWaitLimit, true, 145);

  // --- the last CTA to arrive (2 * gridDim.x arrivals on the counter, the
  // barrier's included) converts the accumulator. The CTA barrier orders the
  // CTA's red.adds before thread 0's arrival, whose release makes them
  // visible to the CTA that acquires the final count; that CTA's threads read
  // after its own CTA barrier.
  __syncthreads();
  if (tid == 0) {
    unsigned before;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(&a.hdr->counter) : "memory");
    *last_flag = before == 2u * ncta - 1u;
  }
  __syncthreads();
  if (*last_flag) {
    for (int q = tid; q < T * D / 4; q += blockDim.x) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.y_acc) + q);
      uint2 o;
      o.x = uint32_t(f32_to_bf16(v.x)) | (uint32_t(f32_to_bf16(v.y)) << 16);
      o.y = uint32_t(f32_to_bf16(v.z)) | (uint32_t(f32_to_bf16(v.w)) << 16);
      reinterpret_cast<uint2*>(a.y)[q] = o;
    }
  }
}

struct ItemsPlan {
  int grid = 0, mpl = 0;
  size_t smem = 0;
};

const void* items_kernel(int mpl) {
  return mpl == 8 ? reinterpret_cast<const void*>(decode_items_kernel<8>)
                  : mpl == 16 ? reinterpret_cast<const void*>(decode_items_kernel<16>)
                              : reinterpret_cast<const void*>(decode_items_kernel<32>);
}

// Launch shape for this layer and row count, or grid 0 when the kernel does
// not apply (row count, pairs, shapes, shared memory, or not all CTAs
// resident). One CTA per SM.
ItemsPlan items_plan_uncached(const Ctx& c) {
  ItemsPlan p;
  if (c.T < 2 || c.T > kDiMaxT || c.T * (c.k + 1) > kDiMaxPairs || c.E > 1024 || c.I % 64 != 0 ||
      c.D % kDiDownBox != 0 || c.D > kDiColsPerThread * kDiThreads || !tmap_encoder_available())
    return p;
  int dev = 0, coop = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return p;
  if ((c.E + sms - 1) / sms > kDiRouterRows) return p;
  p.mpl = (c.E + 31) / 32 <= 8 ? 8 : (c.E + 31) / 32 <= 16 ? 16 : 32;
  const void* f = items_kernel(p.mpl);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) return p;
  p.smem = ItemsSmem(c.D, c.T).total;
  if (p.smem + fa.sharedSizeBytes > size_t(optin)) return p;
  int per_sm = 0;
  if (!ensure_smem_limit(f, int(p.smem)) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kDiThreads, p.smem) != cudaSuccess || per_sm < 1)
    return p;
  p.grid = sms;
  return p;
}

ItemsPlan items_plan(const Ctx& c) {
  struct Entry {
    int dev, T, D, I, k, E;
    ItemsPlan p;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ItemsPlan{};
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.T == c.T && e.D == c.D && e.I == c.I && e.k == c.k && e.E == c.E) return e.p;
  const ItemsPlan p = items_plan_uncached(c);
  cache.push_back({dev, c.T, c.D, c.I, c.k, c.E, p});
  return p;
}

// The down codes' tensor maps for this layer's weights, encoded once per
// weight pointers and shape.
bool item_maps(const Ctx& c, ItemMaps* out) {
  struct Entry {
    const void* routed;
    const void* shared;
    int E, D, I;
    ItemMaps m;
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
  Entry e{w->down.codes, w->s_down.codes, c.E, c.D, c.I, ItemMaps{}};
  const auto U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  const auto NOL2 = CU_TENSOR_MAP_L2_PROMOTION_NONE;
  if (!make_tmap_2d(&e.m.routed, U32, 4, w->down.codes, uint64_t(c.E) * c.D, c.I / 8, 4, kDiDownBox, NOSW, NOL2) ||
      !make_tmap_2d(&e.m.shared, U32, 4, w->s_down.codes, c.D, c.I / 8, 4, kDiDownBox, NOSW, NOL2))
    return false;
  if (cache.size() >= 16) cache.erase(cache.begin());
  cache.push_back(e);
  *out = e.m;
  return true;
}

}  // namespace

bool decode_items_supported(const Ctx& c) { return items_plan(c).grid > 0; }

cudaError_t decode_items(const Ctx& c) {
  const ItemsPlan p = items_plan(c);
  if (p.grid == 0) return cudaErrorInvalidValue;
  ItemMaps dm;
  if (!item_maps(c, &dm)) return cudaErrorInvalidValue;
  const moe_weights* w = c.w;
  ItemsArgs a{c.x,       w->gate,         w->up,    w->down,     w->s_gate,  w->s_up, w->s_down,
              w->router_w, w->router_bias, c.logits, c.topk_idx,  c.topk_w,   c.count, c.off,
              c.perm,     c.inv,           c.blocks, c.n_blocks,  c.h,        c.y_acc, c.y,
              c.hdr,      c.T,             c.D,      c.E,         c.k,        c.I,     c.max_blocks};
  // the counter starts at zero; on the call's first pass the status does too
  // (later passes keep what earlier ones recorded)
  static_assert(offsetof(WsHeader, counter) == 8, "status, detail, counter");
  cudaError_t err = c.first_pass ? cudaMemsetAsync(c.hdr, 0, 12, c.stream)
                                 : cudaMemsetAsync(&c.hdr->counter, 0, 4, c.stream);
  if (err != cudaSuccess) return err;
  void* args[] = {&a, &dm};
  err = cudaLaunchCooperativeKernel(items_kernel(p.mpl), dim3(p.grid), dim3(kDiThreads), args, p.smem, c.stream);
  if (err != cudaSuccess) return err;
  launch_done(c, "decode_items");
  return cudaSuccess;
}

}  // namespace moe
