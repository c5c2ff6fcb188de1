// The whole layer for a few token rows (1 to 8) in one cooperative launch:
// router logits, top-k, gate/up + SwiGLU and down + combine, on the CUDA
// cores ("Optimizing on-device inference for Apple Silicon": "Optimise the
// single-row weight path", "Keep expert routing on the GPU", "Reduce
// intermediate and state traffic"; the row count where the grouped GEMM takes
// over is measured, after "Why continuous batching halved LLM throughput on an
// M2 Mac mini").
//
// One CTA per SM, all co-resident (cooperative launch), 16 compute warps and
// one copy warp. The weight bytes are what binds this layer, so the design
// keeps as many of them in flight as early as possible:
//   * At entry, before any routing, each CTA's copy warp starts bulk (TMA)
//     copies of its router rows and of its share of the shared expert: a few
//     of its gate/up rows and its output rows of its down matrix. The compute
//     warps stage x in shared memory and compute the router logits of the
//     CTA's experts in the canonical order; then grid barrier 1, overlapped
//     with the shared expert's gate/up rows.
//   * Every CTA takes the same top-k of every token (warp t: token t) and the
//     same union of the selected experts in ascending index, the shared
//     expert last. Each expert in the union is read once, whatever the number
//     of rows that selected it.
//   * Gate/up: the union's intermediate rows (expert-major) are cut evenly
//     over the CTAs; a CTA's range streams through a ring of 8-row slots
//     (gate and up codes, scales and biases; one mbarrier per slot). A warp
//     takes one row of a slot: for each token routed to that expert both dot
//     products, then h = bf16(silu(g) * u) into the workspace at the pair's
//     row in the permuted order. Grid barrier 2.
//   * Down: a CTA owns D/G consecutive output rows. For each expert of the
//     union its rows of that expert's down matrix stream through a second
//     ring (copies of the first ones start right after the top-k, the shared
//     expert's at entry). Half a warp takes one row: for each token of the
//     expert the dot product with its h row, times the routing weight, into a
//     per-(token, expert) partial; finally y[t] sums the token's k+1 partials
//     in slot order (the shared expert last). No atomics: the result is
//     bitwise repeatable.
// CTA 0 also writes the routing tables (top-k, counts, offsets, permutation,
// block map) for inspection.
//
// Every wait is bounded: an expired wait records MOE_ERR_DEVICE_TIMEOUT in the
// workspace status word, the kernel skips the remaining work but still
// arrives at both grid barriers, and each CTA waits (bounded) for its copies
// in flight before it exits.
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

constexpr int kDrWarps = 16;                       // compute warps
constexpr int kDrThreads = (kDrWarps + 1) * 32;    // + the copy warp
constexpr int kDrMaxT = 8;                         // token rows
constexpr int kDrMaxPairs = 128;                   // (token, expert) pairs T * (k + 1); also the union size bound
constexpr int kDrMaxGUnits = 96;                   // gate/up units of one CTA
constexpr int kDrGRows = 8;                        // rows per gate/up unit (one slot)
constexpr int kDrMaxNSG = 8, kDrMaxNSD = 16;       // ring slots
constexpr int kDrBarBytes = 512;                   // mbarriers and flags at the start of shared memory

// Shared-memory plan of one launch shape (computed on the host, passed in).
struct RowsLayout {
  int G;        // CTAs
  int n_rt;     // router rows per CTA, at most
  int nsg, nsd; // gate/up and down ring slots
  int rows_d;   // output rows per CTA, at most
  uint32_t gslot, g_up, g_sb, g_piece;  // gate/up slot: bytes, up codes at, s/b pieces at, bytes per piece
  uint32_t dslot, d_sb, d_piece;        // down slot: bytes, s/b pieces at, bytes per piece
  uint32_t dring, a_xs, a_xsum, a_wr, a_gring;  // offsets (region A: until grid barrier 2)
  uint32_t b_hs, b_hsum, b_part;                // offsets (region B: the down phase; aliases region A)
  uint32_t total;
};

__host__ __device__ inline uint32_t al16(uint32_t v) { return (v + 15u) & ~15u; }
__host__ __device__ inline uint32_t al128(uint32_t v) { return (v + 127u) & ~127u; }

// Bytes of a 16-byte-aligned window covering `bytes` bytes from `addr`.
__host__ __device__ inline uint32_t window_bytes(uintptr_t addr, uint32_t bytes) {
  const uintptr_t lo = addr & ~uintptr_t(15), hi = (addr + bytes + 15) & ~uintptr_t(15);
  return uint32_t(hi - lo);
}

RowsLayout rows_layout(int T, int D, int I, int k, int E, int G, size_t budget) {
  RowsLayout L{};
  L.G = G;
  L.n_rt = (E + G - 1) / G;
  L.rows_d = (D + G - 1) / G;
  const uint32_t gcodes = uint32_t(kDrGRows) * D / 2;
  L.g_up = gcodes;
  L.g_sb = 2 * gcodes;
  L.g_piece = al16(uint32_t(kDrGRows) * (D / 64) * 2 + 32);  // room for a 16-byte-aligned window
  L.gslot = al128(L.g_sb + 4 * L.g_piece);
  L.d_sb = uint32_t(L.rows_d) * I / 2;
  L.d_piece = al16(uint32_t(L.rows_d) * (I / 64) * 2 + 32);
  L.dslot = al128(L.d_sb + 2 * L.d_piece);
  const uint32_t P = uint32_t(T) * (k + 1);
  // every expert's down rows in flight at once for one token; more rows use
  // the room for gate/up slots
  L.nsd = std::min<int>(kDrMaxNSD, std::max(2, std::min(10, k * T + 1)));
  L.dring = kDrBarBytes;
  const uint32_t a0 = al128(L.dring + L.nsd * L.dslot);
  L.a_xs = a0;  // x chunk-major fp32, 8 quarter-rows of D/32 + 1 float4 per token
  L.a_xsum = L.a_xs + uint32_t(T) * 8 * (D / 32 + 1) * 16;
  L.a_wr = al128(L.a_xsum + uint32_t(T) * (D / 32) * 4);
  L.a_gring = al128(L.a_wr + uint32_t(L.n_rt) * D * 4);
  L.b_hs = a0;
  L.b_hsum = L.b_hs + P * I * 4;
  L.b_part = al16(L.b_hsum + P * (I / 32) * 4);
  const uint32_t b_end = L.b_part + P * L.rows_d * 4;
  const size_t room = budget > L.a_gring ? budget - L.a_gring : 0;
  L.nsg = int(std::min<size_t>(kDrMaxNSG, room / L.gslot)) & ~1;  // even: see the gate/up items
  L.total = std::max<uint32_t>(L.a_gring + uint32_t(L.nsg) * L.gslot, b_end);
  if (L.total > budget) L.nsg = 0;  // does not fit
  return L;
}

struct RowsArgs {
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
  uint16_t* h;  // [T*k + T][I]: the routed pairs in permuted order (expert-major, tokens ascending), then the shared expert's rows T*k + t
  uint16_t* y;
  WsHeader* hdr;
  int T, D, E, k, I, BM, max_blocks;
  RowsLayout L;
};

// Grid barrier halves: every CTA adds one to the header counter (zeroed on
// the stream before the launch) once all its threads are past the point, and
// later waits, for at most kWaitLimit cycles, until `target` arrivals. The
// wait polls with relaxed loads and a short sleep (an acquiring load would
// invalidate the SM's L1 on every poll and keep its warp issuing), then one
// acquire fence orders the CTA's later reads after the other CTAs' writes.
__device__ __forceinline__ void grid_arrive(WsHeader* hdr) {
  __threadfence();
  atomicAdd(&hdr->counter, 1u);
}
__device__ __forceinline__ bool grid_wait(WsHeader* hdr, unsigned target, int site) {
  const long long t0 = clock64();
  while (true) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&hdr->counter) : "memory");
    if (v >= target) break;
    if (clock64() - t0 > kWaitLimit) {
      report(hdr, MOE_ERR_DEVICE_TIMEOUT, site);
      return false;
    }
    __nanosleep(32);
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return true;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bulk copy of a 16-byte-aligned window around [src, src + bytes) into dst;
// returns the window's size (what the barrier's transaction count expects).
__device__ __forceinline__ uint32_t bulk_window(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src);
  const uint32_t n = window_bytes(a, bytes);
  bulk_g2s(dst, reinterpret_cast<const void*>(a & ~uintptr_t(15)), n, bar);
  return n;
}
__device__ __forceinline__ uint32_t window_delta(const void* src) {
  return uint32_t(reinterpret_cast<uintptr_t>(src) & 15);
}

// silu(g) * u of one intermediate row for one token: the warp's lanes take
// the 32-code chunks c = lane, lane + 32, ...; the result is on every lane.
__device__ __forceinline__ float gateup_row(const float4* xr, int xst, const float* xsum_t, int nch, const uint8_t* cg,
                                         const uint8_t* cu, const uint16_t* sg, const uint16_t* bg, const uint16_t* su,
                                         const uint16_t* bu) {
  const int lane = threadIdx.x & 31;
  float g = 0.f, uu = 0.f;
  for (int c = lane; c < nch; c += 32) {
    float4 xv[8];
#pragma unroll
    for (int jq = 0; jq < 8; ++jq) xv[jq] = xr[jq * xst + c];
    const float sx = xsum_t[c];
    const uint4 wg = reinterpret_cast<const uint4*>(cg)[c];
    const uint4 wu = reinterpret_cast<const uint4*>(cu)[c];
    g += chunk_dot_r(wg, xv, sx, sg[c >> 1], bg[c >> 1]);
    uu += chunk_dot_r(wu, xv, sx, su[c >> 1], bu[c >> 1]);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    g += __shfl_xor_sync(0xffffffffu, g, off);
    uu += __shfl_xor_sync(0xffffffffu, uu, off);
  }
  return silu_mul(g, uu);
}

// Four down rows rg, rg + 2, rg + 4, rg + 6 (rg = 8 * group + lane / 16) of
// one unit for one pair: lanes take the chunks c = lane % 16, + 16, ...; the
// sums over the chunks are on every lane of the half-warp (rows >= nd: 0).
__device__ __forceinline__ float4 down_rows(const uint8_t* codes, int row_bytes, const uint16_t* sc, const uint16_t* bi,
                                         int Gi, const float4* hr, const float* hsum_p, int nchi, int rg, int nd) {
  const int l16 = threadIdx.x & 15;
  float acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0.f;
  for (int c = l16; c < nchi; c += 16) {
    float4 hv[8];
#pragma unroll
    for (int jq = 0; jq < 8; ++jq) hv[jq] = hr[jq * nchi + c];
    const float hsx = hsum_p[c];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rg + 2 * i;
      if (r < nd)
        acc[i] += chunk_dot_r(reinterpret_cast<const uint4*>(codes + size_t(r) * row_bytes)[c], hv, hsx,
                              sc[r * Gi + (c >> 1)], bi[r * Gi + (c >> 1)]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
  }
  return make_float4(acc[0], acc[1], acc[2], acc[3]);
}

// Top-k of one token's logits (select_topk): lane j < k gets slot j.
struct TopkSlot {
  int idx;
  float w;
};
template <int MPL>
__device__ __forceinline__ TopkSlot topk_row(const float* lg, int E, int k) {
  TopkSlot r;
  select_topk<MPL, true>(lg, E, k, r.idx, r.w);
  return r;
}

template <int MPL>
__global__ void __launch_bounds__(kDrThreads, 1) decode_rows_kernel(RowsArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ int s_sel[kDrMaxPairs];      // [T][k] expert of slot j
  __shared__ float s_selw[kDrMaxPairs];   // its routing weight
  __shared__ unsigned s_tmask[(kDrMaxT + 1) * 32];  // per token (then the union): its experts as bits (E <= 1024)
  __shared__ int s_tpre[(kDrMaxT + 1) * 33];        // set bits of each mask below each word, and in all
  __shared__ int s_ulist[kDrMaxPairs];    // union: selected experts ascending, then E (shared)
  __shared__ int s_ucnt[kDrMaxPairs];     // pairs of each union entry
  __shared__ int s_ubase[kDrMaxPairs + 1];
  __shared__ int s_ptok[kDrMaxPairs];     // pair -> token
  __shared__ int s_pa[kDrMaxPairs];       // pair -> assignment t*k + j (T*k + t: shared)
  __shared__ float s_pw[kDrMaxPairs];     // pair -> routing weight (1 for the shared expert)
  __shared__ int s_pof[kDrMaxPairs];      // [T][k+1]: pair of (token, slot); slot k is the shared expert
  __shared__ int s_gu[kDrMaxGUnits];      // gate/up unit: union index (-1: shared), first row, rows
  __shared__ int s_gi[kDrMaxGUnits];
  __shared__ int s_gn[kDrMaxGUnits];
  __shared__ int s_n_union, s_ng, s_ngs, s_issued_g, s_issued_d;

  const RowsLayout& L = a.L;
  const int T = a.T, D = a.D, E = a.E, k = a.k, I = a.I, G = L.G;
  const int nch = D / 32, nchi = I / 32, Gd = D / 64, Gi = I / 64;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x;
  const bool copier = (warp == kDrWarps);
  const uint32_t bar0 = smem_u32(sm);
  auto full_g = [&](int s) { return bar0 + 8u * s; };
  auto empty_g = [&](int s) { return bar0 + 64u + 8u * s; };
  auto full_d = [&](int s) { return bar0 + 128u + 8u * s; };
  auto empty_d = [&](int s) { return bar0 + 256u + 8u * s; };
  const uint32_t rbar = bar0 + 384u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + 392);
  volatile int* gb_ok = reinterpret_cast<volatile int*>(sm + 396);
  float4* xs4 = reinterpret_cast<float4*>(sm + L.a_xs);
  float* xsum = reinterpret_cast<float*>(sm + L.a_xsum);
  const float* wr = reinterpret_cast<const float*>(sm + L.a_wr);
  // x of token t: float4 (jq * xst + c) of xs4 + t * 8 * xst holds elements
  // 32c + 4jq .. 32c + 4jq + 3. The stride is padded by one float4 so that
  // the router's lanes (element 32c + l) fall in 32 different banks, as do
  // the expert dot products' lanes (chunk c = lane).
  const int xst = nch + 1;

  // this CTA's output rows, shared-expert intermediate rows and router rows
  const int d0 = int(unsigned(cta) * D / G), d1 = int(unsigned(cta + 1) * D / G), nd = d1 - d0;
  const int n_rg = (nd + 7) / 8;  // 8-row groups of a down unit (one warp each)
  const int sh0 = int(unsigned(cta) * I / G), sh1 = int(unsigned(cta + 1) * I / G);
  int n_rt = 0;
  while (n_rt < L.n_rt && cta + n_rt * G < E) ++n_rt;

  // --- P0: barriers, the shared expert's units, copies that need no routing
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < L.nsg; ++s) {
      mbar_init(full_g(s), 1);
      mbar_init(empty_g(s), kDrGRows);  // the warps of the slot's rows
    }
    for (int s = 0; s < L.nsd; ++s) {
      mbar_init(full_d(s), 1);
      mbar_init(empty_d(s), max(n_rg, 1));  // one arrival per row group
    }
    mbar_init(rbar, 1);
    mbar_init_fence();
    int n = 0;
    for (int i = sh0; i < sh1; i += kDrGRows, ++n) {
      s_gu[n] = -1;
      s_gi[n] = i;
      s_gn[n] = min(kDrGRows, sh1 - i);
    }
    s_ngs = n;
    s_ng = n;
    s_issued_g = 0;
    s_issued_d = 0;
  }
  __syncthreads();

  // Copies of gate/up unit n (slot n % nsg) and of down unit n (slot n % nsd;
  // unit 0 is the shared expert, unit n >= 1 the union's entry n - 1).
  auto issue_g = [&](int n) {
    const int s = n % L.nsg;
    const int u = s_gu[n], i0 = s_gi[n], nr = s_gn[n];
    const bool sh = (u < 0);
    const int e = sh ? 0 : s_ulist[u];
    const moe_qmatrix& mg = sh ? a.s_gate : a.gate;
    const moe_qmatrix& mu = sh ? a.s_up : a.up;
    const size_t row0 = size_t(e) * I + i0;
    const uint32_t dst = smem_u32(sm + L.a_gring) + uint32_t(s) * L.gslot;
    const uint32_t cb = uint32_t(nr) * D / 2, sb = uint32_t(nr) * Gd * 2;
    const void* sbs[4] = {mg.scales + row0 * Gd, mg.biases + row0 * Gd, mu.scales + row0 * Gd, mu.biases + row0 * Gd};
    uint32_t tx = 2 * cb;
    for (int p = 0; p < 4; ++p) tx += window_bytes(reinterpret_cast<uintptr_t>(sbs[p]), sb);
    mbar_arrive_tx(full_g(s), tx);
    bulk_g2s(dst, mg.codes + row0 * (D / 8), cb, full_g(s));
    bulk_g2s(dst + L.g_up, mu.codes + row0 * (D / 8), cb, full_g(s));
    for (int p = 0; p < 4; ++p) bulk_window(dst + L.g_sb + p * L.g_piece, sbs[p], sb, full_g(s));
  };
  auto issue_d = [&](int n) {
    const int s = n % L.nsd;
    const bool sh = (n == 0);
    const int e = sh ? 0 : s_ulist[n - 1];
    const moe_qmatrix& md = sh ? a.s_down : a.down;
    const size_t row0 = size_t(e) * D + d0;
    const uint32_t dst = smem_u32(sm + L.dring) + uint32_t(s) * L.dslot;
    const uint32_t cb = uint32_t(nd) * I / 2, sb = uint32_t(nd) * Gi * 2;
    const void* sbs[2] = {md.scales + row0 * Gi, md.biases + row0 * Gi};
    const uint32_t tx = cb + window_bytes(reinterpret_cast<uintptr_t>(sbs[0]), sb) +
                        window_bytes(reinterpret_cast<uintptr_t>(sbs[1]), sb);
    mbar_arrive_tx(full_d(s), tx);
    bulk_g2s(dst, md.codes + row0 * (I / 8), cb, full_d(s));
    for (int p = 0; p < 2; ++p) bulk_window(dst + L.d_sb + p * L.d_piece, sbs[p], sb, full_d(s));
  };

  if (copier) {  // lanes issue in parallel: lane 0 the router rows, lane 1 the shared down rows, lanes 2.. the shared gate/up units
    if (lane == 0 && n_rt) {
      mbar_arrive_tx(rbar, uint32_t(n_rt) * D * 4);
      for (int m = 0; m < n_rt; ++m)
        bulk_g2s(smem_u32(sm + L.a_wr) + uint32_t(m) * D * 4, a.router_w + size_t(cta + m * G) * D, D * 4, rbar);
    }
    if (lane == 1 && nd > 0) issue_d(0);
    for (int n = lane - 2; n >= 0 && n < s_ngs; n += 30) issue_g(n);  // the host checked that they fit the ring
    if (lane == 0) {
      s_issued_g = s_ngs;
      s_issued_d = nd > 0 ? 1 : 0;
    }
  }
  // x, chunk-major fp32 (the expert dot products), and its per-chunk sums
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
  __syncthreads();

  // Gate/up unit items: item q = n * kDrGRows + r (unit n, row r) goes to
  // compute warp (q + 8) % kDrWarps = 8 (1 - n % 2) + r. The warp waits for the unit's
  // slot, computes the row for every token of the unit's expert and releases
  // the slot. The slot count is even, so every unit of slot s goes to the
  // same eight warps (8 (1 - s % 2) + r): a warp consumes the units of a slot in
  // order, and the full barrier it waits on is never more than one phase
  // ahead, which is all a parity wait can tell apart.
  int q_next = (warp + kDrGRows) % kDrWarps;  // this warp's next gate/up item (unit 0, the shared expert's, avoids the router warps)
  auto gateup_items = [&](int n_end) {
    for (; q_next < n_end * kDrGRows; q_next += kDrWarps) {
      const int n = q_next / kDrGRows, r = q_next % kDrGRows, s = n % L.nsg;
      if (!*abort_flag && mbar_wait(full_g(s), (n / L.nsg) & 1, abort_flag, a.hdr, kWaitLimit, false, 131) &&
          r < s_gn[n]) {
        const int u = s_gu[n], i0 = s_gi[n];
        const bool sh = (u < 0);
        const int npairs = sh ? T : s_ucnt[u], pbase = sh ? 0 : s_ubase[u];
        const uint8_t* base = sm + L.a_gring + size_t(s) * L.gslot;
        const uint8_t* cg = base + size_t(r) * D / 2;
        const uint8_t* cu = base + L.g_up + size_t(r) * D / 2;
        const int e = sh ? 0 : s_ulist[u];
        const size_t row0 = size_t(e) * I + i0;
        const moe_qmatrix& mg = sh ? a.s_gate : a.gate;
        const moe_qmatrix& mu = sh ? a.s_up : a.up;
        const uint16_t* sg = reinterpret_cast<const uint16_t*>(base + L.g_sb + 0 * L.g_piece + window_delta(mg.scales + row0 * Gd)) + r * Gd;
        const uint16_t* bg = reinterpret_cast<const uint16_t*>(base + L.g_sb + 1 * L.g_piece + window_delta(mg.biases + row0 * Gd)) + r * Gd;
        const uint16_t* su = reinterpret_cast<const uint16_t*>(base + L.g_sb + 2 * L.g_piece + window_delta(mu.scales + row0 * Gd)) + r * Gd;
        const uint16_t* bu = reinterpret_cast<const uint16_t*>(base + L.g_sb + 3 * L.g_piece + window_delta(mu.biases + row0 * Gd)) + r * Gd;
        for (int pp = 0; pp < npairs; ++pp) {
          const int t = sh ? pp : s_ptok[pbase + pp];
          const int arow = sh ? T * k + pp : pbase + pp;  // the pair's row of h: its permuted position
          const float hv = gateup_row(xs4 + size_t(t) * 8 * xst, xst, xsum + t * nch, nch, cg, cu, sg, bg, su, bu);
          if (lane == 0) a.h[size_t(arow) * I + i0 + r] = f32_to_bf16(hv);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_g(s));
    }
  };

  // --- P1: router logits of this CTA's experts (warp m: expert cta + m*G),
  // all tokens, in the canonical order: lane l sums elements 32c + l with
  // fused multiply-adds, then the pairwise tree, then the bias.
  if (warp < n_rt) {
    if (mbar_wait(rbar, 0, abort_flag, a.hdr, kWaitLimit, false, 132)) {
      const int e = cta + warp * G;
      const float* w = wr + size_t(warp) * D;
      float acc[kDrMaxT];
#pragma unroll
      for (int t = 0; t < kDrMaxT; ++t) acc[t] = 0.f;
      const float* xf = reinterpret_cast<const float*>(xs4) + (lane >> 2) * xst * 4 + (lane & 3);
#pragma unroll 4
      for (int c = 0; c < nch; ++c) {
        const float wv = w[32 * c + lane];
#pragma unroll
        for (int t = 0; t < kDrMaxT; ++t)
          if (t < T) acc[t] = fmaf(xf[t * 8 * xst * 4 + c * 4], wv, acc[t]);
      }
#pragma unroll
      for (int t = 0; t < kDrMaxT; ++t) {
        if (t >= T) break;
        float v = acc[t];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
        if (lane == 0) a.logits[size_t(t) * E + e] = a.router_bias ? __fadd_rn(v, a.router_bias[e]) : v;
      }
    }
  }
  // the router warps (warp 0 among them, or warp 0 alone) are done: arrive
  if (warp < max(n_rt, 1)) {
    named_sync(1, max(n_rt, 1) * 32);
    if (tid == 0) grid_arrive(a.hdr);
  }
  if (!copier) gateup_items(s_ngs);  // the shared expert's rows, while the barrier completes
  __syncthreads();
  if (tid == 0) *gb_ok = grid_wait(a.hdr, unsigned(G), 121) ? 1 : 0;
  __syncthreads();
  const bool ok1 = *gb_ok != 0;

  // --- P2: top-k of every token (warp t), then the union and the pairs.
  // Each token's experts also go into a bit mask of its own, so that every
  // assignment finds its unit, its position among the unit's tokens and the
  // unit's first pair from counts of set bits, with no search.
  for (int i = tid; i < (T + 1) * 32; i += blockDim.x) s_tmask[i] = 0u;  // row T: the union
  __syncthreads();
  if (warp < T) {
    int myi = 0;
    float myw = 0.f;
    if (ok1) {
      const TopkSlot ts = topk_row<MPL>(a.logits + size_t(warp) * E, E, k);
      myi = ts.idx;
      myw = ts.w;
    }
    if (lane < k) {
      if (myi < 0 || myi >= E) {
        report(a.hdr, MOE_ERR_DEVICE_CHECK, 123);
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
  if (warp <= T) {  // per mask (a token's, or the union's): set bits below each word, a warp scan
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
  // bits below expert e in mask m (m = T: the union; its rank there is its unit)
  auto below = [&](int m, int e) {
    return s_tpre[m * 33 + (e >> 5)] + __popc(s_tmask[m * 32 + (e >> 5)] & ((1u << (e & 31)) - 1u));
  };
  for (int q = tid; q < T * k; q += blockDim.x) {  // assignment q = t*k + j
    const int t = q / k, e = s_sel[q];
    const unsigned bit = 1u << (e & 31);
    int pos = 0, cnt = 0, base = 0;  // among the expert's tokens; its tokens; pairs of lower experts
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
    s_pof[t * (k + 1) + q % k] = p;
  }
  for (int t = tid; t < T; t += blockDim.x) {  // the shared expert: pairs T*k + t
    const int p = T * k + t;
    s_ptok[p] = t;
    s_pa[p] = p;
    s_pw[p] = 1.f;
    s_pof[t * (k + 1) + k] = p;
  }
  if (tid == 0) {
    s_ulist[n_routed] = E;
    s_ucnt[n_routed] = T;
    s_ubase[n_routed] = T * k;
    s_ubase[n_union] = T * k + T;
    s_n_union = n_union;
  }
  if (copier) {  // this CTA's share of the routed gate/up rows, as units of at most kDrGRows rows
    const unsigned N = unsigned(n_routed) * I;  // at most 128 * 4096: products below stay under 2^32
    const int r0 = int(unsigned(cta) * N / G), r1 = int(unsigned(cta + 1) * N / G);
    const int u0 = r0 / I, n_seg = (r1 > r0) ? (r1 - 1) / I - u0 + 1 : 0;  // experts the range touches
    int n_at = s_ngs;
    for (int j0 = 0; j0 < n_seg; j0 += 32) {
      const int j = j0 + lane, u = u0 + j;
      const int lo = max(r0, u * I), hi = min(r1, (u + 1) * I);
      const int nu = (j < n_seg) ? (hi - lo + kDrGRows - 1) / kDrGRows : 0;
      int v = nu;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      const int first = n_at + v - nu;
      for (int i = 0; i < nu; ++i) {
        const int n = first + i;
        if (n < kDrMaxGUnits) {
          s_gu[n] = u;
          s_gi[n] = lo - u * I + i * kDrGRows;
          s_gn[n] = min(kDrGRows, hi - lo - i * kDrGRows);
        }
      }
      n_at += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
      if (n_at > kDrMaxGUnits) report(a.hdr, MOE_ERR_DEVICE_CHECK, 124);
      s_ng = min(n_at, kDrMaxGUnits);
    }
  }
  __syncthreads();

  // --- P3: gate/up of the routed experts. The copy warp keeps both rings
  // full: gate/up units first, then (while down slots are free) down units.
  const int ng = s_ng, n_dunits = (nd > 0) ? n_union : 0;
  // the free slots first, one unit per compute warp, issued side by side:
  // gate/up units, then down units; the copy warp refills the rings after
  const int g0 = s_issued_g, g_free = max(0, min(ng, L.nsg) - g0);
  const int d0u = s_issued_d, d_free = max(0, min(n_dunits, L.nsd) - d0u);
  if (!copier && lane == 0)
    for (int j = warp; j < g_free + d_free; j += kDrWarps) {
      if (j < g_free)
        issue_g(g0 + j);
      else
        issue_d(d0u + j - g_free);
    }
  if (copier) {
    if (lane == 0) {
      int nd_issued = d0u + d_free;
      int n = g0 + g_free;
      for (; n < ng; ++n) {
        const int s = n % L.nsg;
        if (*abort_flag || !mbar_wait(empty_g(s), ((n / L.nsg) - 1) & 1, abort_flag, a.hdr, kWaitLimit, false, 133))
          break;
        issue_g(n);
      }
      s_issued_g = n;
      s_issued_d = nd_issued;
    }
  } else {
    gateup_items(ng);
  }

  // --- grid barrier 2: every h row is written
  __syncthreads();
  if (tid == 0) {
    grid_arrive(a.hdr);
    *gb_ok = grid_wait(a.hdr, 2u * G, 122) ? 1 : 0;
  }
  __syncthreads();
  const bool ok2 = ok1 && *gb_ok != 0 && !*abort_flag;

  // --- P4: down. Stage every pair's h row (chunk-major fp32) and its chunk sums.
  float4* hs4 = reinterpret_cast<float4*>(sm + L.b_hs);
  float* hsum = reinterpret_cast<float*>(sm + L.b_hsum);
  float* part = reinterpret_cast<float*>(sm + L.b_part);
  const int P = T * (k + 1);
  if (ok2) {
    for (int q0 = tid; q0 < P * (I / 8); q0 += 4 * blockDim.x) {  // four 16-byte loads in flight a thread
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = q0 + j * blockDim.x;
        if (q < P * (I / 8)) v[j] = __ldcg(reinterpret_cast<const uint4*>(a.h) + q);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = q0 + j * blockDim.x;
        if (q < P * (I / 8)) stage_bf16x8(hs4 + size_t(q / (I / 8)) * 8 * nchi, nchi, q % (I / 8), v[j]);
      }
    }
  }
  __syncthreads();
  if (ok2) chunk_sums(hs4, hsum, P, nchi);
  __syncthreads();

  if (copier) {
    if (lane == 0) {
      int n = s_issued_d;
      for (; n < n_dunits; ++n) {
        const int s = n % L.nsd;
        if (*abort_flag || !mbar_wait(empty_d(s), ((n / L.nsd) - 1) & 1, abort_flag, a.hdr, kWaitLimit, false, 134))
          break;
        issue_d(n);
      }
      s_issued_d = n;
    }
  } else {
    // Down item (unit n, row group g: rows 8g .. 8g + 7 of the CTA's rows of
    // one expert) belongs to warp (slot * n_rg + g) % kDrWarps, the same warp
    // for every unit of the slot; a warp takes its items in unit order, so it
    // consumes the units of a slot in order and no parity wait is more than
    // one phase ahead. Lane l takes the chunks c = l % 16, l % 16 + 16, ... of
    // rows 8g + l / 16 + 2i, i < 4: the token's h chunk is loaded once for
    // the four rows, whose dot products are independent.
    const int hh = lane >> 4, l16 = lane & 15;
    for (int n0 = 0; n0 < n_dunits; n0 += L.nsd)
      for (int idx = warp; idx < L.nsd * n_rg; idx += kDrWarps) {
        const int s = idx / n_rg, gq = idx - s * n_rg, n = n0 + s;
        if (n >= n_dunits) break;
        if (!*abort_flag && ok2 && mbar_wait(full_d(s), (n / L.nsd) & 1, abort_flag, a.hdr, kWaitLimit, false, 135)) {
          const int u = (n == 0) ? n_routed : n - 1;
          const bool sh = (n == 0);
          const int e = sh ? 0 : s_ulist[u];
          const moe_qmatrix& md = sh ? a.s_down : a.down;
          const size_t row0 = size_t(e) * D + d0;
          const uint8_t* base = sm + L.dring + size_t(s) * L.dslot;
          const uint16_t* sc = reinterpret_cast<const uint16_t*>(base + L.d_sb + window_delta(md.scales + row0 * Gi));
          const uint16_t* bi =
              reinterpret_cast<const uint16_t*>(base + L.d_sb + L.d_piece + window_delta(md.biases + row0 * Gi));
          const int npairs = s_ucnt[u], pbase = s_ubase[u], rg = 8 * gq + hh;
          for (int pp = 0; pp < npairs; ++pp) {
            const int p = pbase + pp;
            const float4 acc4 = down_rows(base, I / 2, sc, bi, Gi, hs4 + size_t(p) * 8 * nchi, hsum + p * nchi, nchi, rg, nd);
            const float acc[4] = {acc4.x, acc4.y, acc4.z, acc4.w};
            const float wp = s_pw[p];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = rg + 2 * i;
              if (l16 == 0 && r < nd) part[p * L.rows_d + r] = acc[i] * wp;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_d(s));
      }
  }
  __syncthreads();

  // y[t] = sum over the token's slots (its k experts in top-k order, then the
  // shared expert) of the weighted partials
  if (ok2) {
    for (int q = tid; q < T * nd; q += blockDim.x) {
      const int t = q / nd, r = q % nd;
      float v = 0.f;
      for (int j = 0; j <= k; ++j) v += part[s_pof[t * (k + 1) + j] * L.rows_d + r];
      a.y[size_t(t) * D + d0 + r] = f32_to_bf16(v);
    }
  }

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

  // no copy may still be landing when the CTA exits (only after an abort is
  // one left unconsumed): wait, bounded, for the last phase of every slot used
  if (tid == 0) {
    const int ig = s_issued_g, id = s_issued_d;
    for (int s = 0; s < L.nsg && s < ig; ++s) {
      const int last = s + ((ig - 1 - s) / L.nsg) * L.nsg;
      mbar_wait(full_g(s), (last / L.nsg) & 1, abort_flag, a.hdr, kWaitLimit, true, 136);
    }
    for (int s = 0; s < L.nsd && s < id; ++s) {
      const int last = s + ((id - 1 - s) / L.nsd) * L.nsd;
      mbar_wait(full_d(s), (last / L.nsd) & 1, abort_flag, a.hdr, kWaitLimit, true, 137);
    }
    if (n_rt) mbar_wait(rbar, 0, abort_flag, a.hdr, kWaitLimit, true, 138);
  }
}

struct RowsPlan {
  int grid = 0, mpl = 0;
  RowsLayout L{};
};

const void* rows_kernel(int mpl) {
  return mpl == 8 ? reinterpret_cast<const void*>(decode_rows_kernel<8>)
                  : mpl == 16 ? reinterpret_cast<const void*>(decode_rows_kernel<16>)
                              : reinterpret_cast<const void*>(decode_rows_kernel<32>);
}

// Launch shape for this layer and row count, or grid 0 when the kernel does
// not apply (too many rows or pairs, shared memory, not all CTAs resident).
RowsPlan rows_plan_uncached(const Ctx& c) {
  RowsPlan p;
  if (c.T < 1 || c.T > kDrMaxT || c.T * (c.k + 1) > kDrMaxPairs || c.E > 1024) return p;
  int dev = 0, coop = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return p;
  p.mpl = (c.E + 31) / 32 <= 8 ? 8 : (c.E + 31) / 32 <= 16 ? 16 : 32;
  const void* f = rows_kernel(p.mpl);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) return p;
  const size_t budget = size_t(optin) - fa.sharedSizeBytes;
  const int G = sms;
  p.L = rows_layout(c.T, c.D, c.I, c.k, c.E, G, budget);
  const RowsLayout& L = p.L;
  if (L.nsg < 2) return p;
  // the shared expert's gate/up units are issued at entry without waiting
  const int sh_rows = (c.I + G - 1) / G, sh_units = (sh_rows + kDrGRows - 1) / kDrGRows;
  if (sh_units > L.nsg - 1) return p;
  // gate/up units per CTA, at most: its routed rows cut at expert boundaries
  const int routed = std::min(c.E, c.T * c.k);
  const long long rows_cta = ((long long)routed * c.I + G - 1) / G;
  if (sh_units + rows_cta / kDrGRows + routed + 1 > kDrMaxGUnits) return p;
  int per_sm = 0;
  if (!ensure_smem_limit(f, int(L.total)) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kDrThreads, L.total) != cudaSuccess || per_sm < 1)
    return p;
  p.grid = G;
  return p;
}

RowsPlan rows_plan(const Ctx& c) {
  struct Entry {
    int dev, T, D, I, k, E;
    RowsPlan p;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return RowsPlan{};
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.T == c.T && e.D == c.D && e.I == c.I && e.k == c.k && e.E == c.E) return e.p;
  const RowsPlan p = rows_plan_uncached(c);
  cache.push_back({dev, c.T, c.D, c.I, c.k, c.E, p});
  return p;
}

}  // namespace

bool decode_rows_supported(const Ctx& c) { return rows_plan(c).grid > 0; }

cudaError_t decode_rows(const Ctx& c) {
  const RowsPlan p = rows_plan(c);
  if (p.grid == 0) return cudaErrorInvalidValue;
  const moe_weights* w = c.w;
  RowsArgs a{c.x,      w->gate,  w->up,         w->down,    w->s_gate, w->s_up,   w->s_down,
             w->router_w, w->router_bias, c.logits, c.topk_idx, c.topk_w, c.count, c.off,
             c.perm,   c.inv,    c.blocks,      c.n_blocks, c.h,       c.y,       c.hdr,
             c.T,      c.D,      c.E,           c.k,        c.I,       c.BM,      c.max_blocks,
             p.L};
  // the grid-barrier counter starts at zero; on the call's first pass the
  // status does too (later passes keep what earlier ones recorded)
  static_assert(offsetof(WsHeader, counter) == 8, "status, detail, counter");
  cudaError_t err = c.first_pass ? cudaMemsetAsync(c.hdr, 0, 12, c.stream)
                                 : cudaMemsetAsync(&c.hdr->counter, 0, 4, c.stream);
  if (err != cudaSuccess) return err;
  void* args[] = {&a};
  err = cudaLaunchCooperativeKernel(rows_kernel(p.mpl), dim3(p.grid), dim3(kDrThreads), args, p.L.total, c.stream);
  if (err != cudaSuccess) return err;
  launch_done(c, "decode_rows");
  return cudaSuccess;
}

}  // namespace moe
