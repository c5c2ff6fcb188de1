// Tensor-core grouped GEMMs of the prefill expert path on sm_103a: tcgen05
// MMAs with fp32 accumulators in tensor memory, operands in shared memory in
// the 128-byte-swizzled K-major layout ("Optimizing on-device inference for
// Apple Silicon", section "Dequantise weights during matrix multiplication":
// weights are expanded to bf16 one small tile at a time on chip, multiplied
// with the routed activation rows, accumulated in fp32 and written as bf16;
// section "Reduce intermediate and state traffic": gate/up fused with the
// gated activation, down fused with the routing weights and the shared
// expert).
//
// One persistent kernel per projection. A tile is one block-map entry (up to
// 128 rows of one expert, MMA M = 128) times 256 weight rows (MMA N = 256):
//   gate/up: 128 gate rows and the 128 up rows of the same intermediate
//            columns, so one accumulator holds both and the epilogue applies
//            h = bf16(silu(g) * u);
//   down:    256 output columns; the epilogue adds w[t,j] * acc into the fp32
//            combine accumulator of token t (shared-expert rows with weight 1).
// The K loop runs one 64-wide quantisation group per step.
//
// A second form of each kernel reads weights that a separate pass has already
// expanded to bf16 in device memory (the design the fused form replaces, kept
// for measuring what fusion saves): the TMA producer then loads the weight
// stage itself and the dequantising warps have no work.
//
// Warp roles (18 warps):
//   0      TMA producer: packed codes of the 256 weight rows (and, for down,
//          the 128 h rows of the tile)
//   1      TMEM allocator and the single MMA-issuing thread
//   2..5   gate/up only: gather the tile's token rows of x with cp.async into
//          the swizzled A stage
//   6..13  dequantisation: one weight row per thread, 8 codes -> 8 bf16 by bit
//          operations and one bf16x2 FMA per pair, stored swizzled
//   14..17 epilogue: TMEM -> registers -> SwiGLU / weighted combine
// Every wait on an mbarrier is bounded: on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT, drains what it has in flight and exits.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;   // A/B operand ring (MMA side)
constexpr int kCStages = 4;  // packed-code ring (TMA side)
constexpr int BM = 128;      // token rows per tile (MMA M)
constexpr int kTileRows = BM;
constexpr int BN = 256;      // weight rows per tile (MMA N)
constexpr int BK = 64;       // one quantisation group per k-step
constexpr uint32_t kABytes = BM * BK * 2;        // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;        // 32 KB
constexpr uint32_t kCBytes = BN * BK / 2;        // 8 KB of codes
constexpr uint32_t kTmemCols = 2 * BN;           // two accumulators: tile i+1 runs while tile i drains
constexpr int kAPipeLag = 3;                     // cp.async groups kept in flight (< kStages)
static_assert(kAPipeLag < kStages, "the gather may not wait on a stage it has not released");

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpA0 = 2, kNumAWarps = 4, kWarpDq0 = 6, kNumDqWarps = 8,
              kWarpEpi0 = 14, kNumEpiWarps = 4;
constexpr int kNumWarps = 18;
constexpr int kNumThreads = kNumWarps * 32;

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffC = kOffB + kStages * kBBytes;
constexpr uint32_t kOffBar = kOffC + kCStages * kCBytes;
// full, empty, afull [kStages]; cfull, cempty [kCStages]; accf, acce [2]; drain; never
constexpr uint32_t kNumBars = 3 * kStages + 2 * kCStages + 6;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024


// ---- PTX wrappers (beyond the shared ones) ---------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// bf16 number gi (0..7) of a 16-byte vector, without indexing registers.
__device__ __forceinline__ uint16_t pick_bf16(uint4 v, int gi) {
  const uint32_t w = (gi & 4) ? ((gi & 2) ? v.w : v.z) : ((gi & 2) ? v.y : v.x);
  return uint16_t((gi & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// Byte offset of 16-byte chunk c of row r inside a 1024-aligned SW128 K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

struct TcArgs {
  const uint16_t* x;
  moe_qmatrix m0, m1;  // routed: gate, up (gate/up kernel) or down in m0
  moe_qmatrix s0, s1;  // shared expert
  const int32_t* blocks;
  const int32_t* n_blocks;
  const int32_t* perm;
  const float* topk_w;
  uint16_t* h;
  float* y_acc;
  WsHeader* hdr;
  int T, D, E, k, I;
  int max_blocks;
  long long epi_wait_limit;  // > 0: test hook, the epilogue first waits this long on a barrier nothing arrives on
};

struct TcMaps {
  CUtensorMap c0, c1;    // routed codes (gate, up) or (down, unused); bf16 weights in the second form
  CUtensorMap cs0, cs1;  // shared-expert codes; bf16 weights in the second form
  CUtensorMap a;         // down only: h rows, bf16, SW128 box 64 x 128
};

// BF16W: the weights arrive as bf16 (128-byte-swizzled TMA tiles of 64 x 128
// rows) on afull, with the h rows for down; full then counts the token
// gather alone (gate/up) or nothing (down).
template <bool GATEUP, bool BF16W>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_tc_kernel(const TcArgs args, const __grid_constant__ TcMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);  // generic pointer of the aligned base
  const uint32_t bar0 = base + kOffBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto afull = [&](int s) { return bar0 + 8u * (2 * kStages + s); };  // TMA loads landed (down: h rows; bf16 weights)
  auto cfull = [&](int s) { return bar0 + 8u * (3 * kStages + s); };
  auto cempty = [&](int s) { return bar0 + 8u * (3 * kStages + kCStages + s); };
  constexpr uint32_t kBarAcc = 3 * kStages + 2 * kCStages;
  auto accf = [&](int b) { return bar0 + 8u * (kBarAcc + b); };
  auto acce = [&](int b) { return bar0 + 8u * (kBarAcc + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (kBarAcc + 4);
  const uint32_t never_bar = bar0 + 8u * (kBarAcc + 5);  // test hook: nothing arrives here
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TcArgs& a = args;
  const int NT = GATEUP ? a.I / 128 : a.D / BN;  // weight-row tiles per block-map entry
  const int KS = GATEUP ? a.D / BK : a.I / BK;   // k-steps per tile
  const int K = GATEUP ? a.D : a.I;
  const int A_rows = a.T * a.k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), GATEUP ? ((BF16W ? 0 : kNumDqWarps) + kNumAWarps) : (BF16W ? 1 : kNumDqWarps));
      mbar_init(empty(s), 1);
      mbar_init(afull(s), 1);
    }
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(cfull(s), 1);
      mbar_init(cempty(s), kNumDqWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf(b), 1);
      mbar_init(acce(b), kNumEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int nb = *a.n_blocks;
  if (nb > a.max_blocks || nb < 0) {
    if (threadIdx.x == 0) report(a.hdr, MOE_ERR_DEVICE_CHECK, 10);
    nb = 0;
  }
  const int n_tiles = nb * NT;

  // decodes a tile into (group, first row, rows, expert, shared, weight-row tile)
  auto tile_info = [&](int tile, int& g, int& p0, int& R, int& j) {
    const int b = tile / NT;
    j = tile % NT;
    g = a.blocks[3 * b];
    p0 = a.blocks[3 * b + 1];
    R = a.blocks[3 * b + 2];
    if (g < 0 || g > a.E || R < 1 || R > kTileRows || p0 < 0 || p0 + R > A_rows + a.T) {
      report(a.hdr, MOE_ERR_DEVICE_CHECK, 11);
      return false;
    }
    return true;
  };

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0, c_issued = 0, a_issued = 0;  // loads issued: iterations [0, *_issued)
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        int g, p0, R, j;
        if (!tile_info(tile, g, p0, R, j)) {
          *abort_flag = 1;
          break;
        }
        const bool sh = (g == a.E);
        const int ex = sh ? 0 : g;
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = it % kStages, cs = it % kCStages;
          const uint32_t ph = (it / kStages) & 1u, cph = (it / kCStages) & 1u;
          if (BF16W) {
            // the weight stage (and the h rows for down) straight from memory
            if (!(ok = mbar_wait(empty(s), ph ^ 1u, abort_flag, a.hdr))) break;
            mbar_arrive_tx(afull(s), kBBytes + (GATEUP ? 0u : kABytes));
            const uint32_t bdst = base + kOffB + s * kBBytes;
            const int row = GATEUP ? ex * a.I + j * 128 : ex * a.D + j * BN;
            tma_load_2d(bdst, sh ? &maps.cs0 : &maps.c0, ks * BK, row, afull(s));
            if (GATEUP)
              tma_load_2d(bdst + kBBytes / 2, sh ? &maps.cs1 : &maps.c1, ks * BK, row, afull(s));
            else
              tma_load_2d(bdst + kBBytes / 2, sh ? &maps.cs0 : &maps.c0, ks * BK, row + 128, afull(s));
            if (!GATEUP) tma_load_2d(base + kOffA + s * kABytes, &maps.a, ks * BK, p0, afull(s));
            a_issued = it + 1;
            continue;
          }
          if (!(ok = mbar_wait(cempty(cs), cph ^ 1u, abort_flag, a.hdr))) break;
          const uint32_t cdst = base + kOffC + cs * kCBytes;
          mbar_arrive_tx(cfull(cs), kCBytes);
          if (GATEUP) {
            const int row = ex * a.I + j * 128;
            tma_load_2d(cdst, sh ? &maps.cs0 : &maps.c0, ks * 8, row, cfull(cs));
            tma_load_2d(cdst + kCBytes / 2, sh ? &maps.cs1 : &maps.c1, ks * 8, row, cfull(cs));
          } else {
            tma_load_2d(cdst, sh ? &maps.cs0 : &maps.c0, ks * 8, ex * a.D + j * BN, cfull(cs));
          }
          c_issued = it + 1;
          if (!GATEUP) {
            if (!(ok = mbar_wait(empty(s), ph ^ 1u, abort_flag, a.hdr))) break;
            mbar_arrive_tx(afull(s), kABytes);
            tma_load_2d(base + kOffA + s * kABytes, &maps.a, ks * BK, p0, afull(s));
            a_issued = it + 1;
          }
        }
      }
      // drain: every load this thread issued lands before the CTA exits
      for (uint32_t s = 0; s < uint32_t(kCStages); ++s) {
        if (s < c_issued) {
          const uint32_t last = c_issued - 1 - ((c_issued - 1 - s) % kCStages);  // last issue to stage s
          mbar_wait(cfull(s), (last / kCStages) & 1u, abort_flag, a.hdr, kWaitLimit, true);
        }
      }
      for (uint32_t s = 0; s < uint32_t(kStages); ++s) {
        if (s < a_issued) {
          const uint32_t last = a_issued - 1 - ((a_issued - 1 - s) % kStages);
          mbar_wait(afull(s), (last / kStages) & 1u, abort_flag, a.hdr, kWaitLimit, true);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
        const int buf = tc & 1;
        if (!(ok = mbar_wait(acce(buf), ((tc >> 1) & 1u) ^ 1u, abort_flag, a.hdr))) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if ((GATEUP || !BF16W) && !(ok = mbar_wait(full(s), ph, abort_flag, a.hdr))) break;
          if ((!GATEUP || BF16W) && !(ok = mbar_wait(afull(s), ph, abort_flag, a.hdr))) break;
          tc_fence_after();
          const uint32_t sa = base + kOffA + s * kABytes, sb = base + kOffB + s * kBBytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma(d, smem_desc(sa + kk * 32), smem_desc(sb + kk * 32), (ks | kk) != 0);
          umma_commit(empty(s));
        }
        if (!ok) break;
        umma_commit(accf(buf));
      }
      // all MMAs issued by this thread complete before TMEM is released
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, abort_flag, a.hdr, kWaitLimit, true);
    }
  } else if (GATEUP && warp >= kWarpA0 && warp < kWarpA0 + kNumAWarps) {
    // ---------------- token-row gather (gate/up A operand) ----------------
    const int r = threadIdx.x - kWarpA0 * 32;  // tile row 0..127
    uint32_t it = 0, pending = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      int g, p0, R, j;
      if (!tile_info(tile, g, p0, R, j)) {
        *abort_flag = 1;
        break;
      }
      int t0 = -1;
      if (r < R) t0 = (g == a.E) ? (p0 + r - A_rows) : (a.perm[p0 + r] / a.k);
      const bool v0 = (t0 >= 0 && t0 < a.T);
      const char* src0 = reinterpret_cast<const char*>(a.x + size_t(v0 ? t0 : 0) * a.D);
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!(ok = mbar_wait(empty(s), ph ^ 1u, abort_flag, a.hdr))) break;
        const uint32_t dst = base + kOffA + s * kABytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) cp_async16(dst + sw128(r, c), src0 + ks * 128 + c * 16, v0 ? 16u : 0u);
        cp_async_commit();
        ++pending;
        if (pending > kAPipeLag) {
          cp_async_wait<kAPipeLag>();
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(full((it - kAPipeLag) % kStages));
          --pending;
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    __syncwarp();
    if (ok && !*abort_flag) {
      for (uint32_t q = it - pending; q < it; ++q)
        if (lane == 0) mbar_arrive(full(q % kStages));
    }
  } else if (!BF16W && warp >= kWarpDq0 && warp < kWarpDq0 + kNumDqWarps) {
    // ---------------- dequantisation: B operand ----------------
    const int r = threadIdx.x - kWarpDq0 * 32;  // weight row 0..255 of the tile
    const bool vec_sb = (K / 64) % 8 == 0;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      int g, p0, R, j;
      if (!tile_info(tile, g, p0, R, j)) {
        *abort_flag = 1;
        break;
      }
      const bool sh = (g == a.E);
      const int ex = sh ? 0 : g;
      const moe_qmatrix& m = GATEUP ? (r < 128 ? (sh ? a.s0 : a.m0) : (sh ? a.s1 : a.m1)) : (sh ? a.s0 : a.m0);
      const size_t row = GATEUP ? size_t(ex) * a.I + j * 128 + (r & 127) : size_t(ex) * a.D + j * BN + r;
      const uint16_t* srow = m.scales + row * (K / 64);
      const uint16_t* brow = m.biases + row * (K / 64);
      // scales and biases: windows of 8 groups (16 bytes) fetched one window
      // ahead when rows hold a multiple of 8 groups; else one group ahead
      uint4 s_cur = make_uint4(0u, 0u, 0u, 0u), b_cur = s_cur, s_nxt = s_cur, b_nxt = s_cur;
      uint16_t s_one = 0, b_one = 0;
      if (vec_sb) {
        s_cur = *reinterpret_cast<const uint4*>(srow);
        b_cur = *reinterpret_cast<const uint4*>(brow);
        if (KS > 8) {
          s_nxt = *reinterpret_cast<const uint4*>(srow + 8);
          b_nxt = *reinterpret_cast<const uint4*>(brow + 8);
        }
      } else {
        s_one = srow[0];
        b_one = brow[0];
      }
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kStages, cs = it % kCStages;
        const uint32_t ph = (it / kStages) & 1u, cph = (it / kCStages) & 1u;
        uint16_t sc, bi;
        if (vec_sb) {
          const int gi = ks & 7;
          sc = pick_bf16(s_cur, gi);
          bi = pick_bf16(b_cur, gi);
          if (gi == 7) {
            s_cur = s_nxt;
            b_cur = b_nxt;
            if (ks + 9 < KS) {
              s_nxt = *reinterpret_cast<const uint4*>(srow + ks + 9);
              b_nxt = *reinterpret_cast<const uint4*>(brow + ks + 9);
            }
          }
        } else {
          sc = s_one;
          bi = b_one;
          if (ks + 1 < KS) {
            s_one = srow[ks + 1];
            b_one = brow[ks + 1];
          }
        }
        if (!(ok = mbar_wait(cfull(cs), cph, abort_flag, a.hdr))) break;
        // the two 16-byte halves of the row's codes, read in an order that
        // spreads a quarter-warp over all banks
        const uint4* cw = reinterpret_cast<const uint4*>(gbase + kOffC + cs * kCBytes + r * 32);
        const int h0 = (r >> 2) & 1;
        const uint4 first = cw[h0], second = cw[h0 ^ 1];
        const uint4 w0 = h0 ? second : first, w1 = h0 ? first : second;
        const __nv_bfloat162 s2 = __halves2bfloat162(__ushort_as_bfloat16(sc), __ushort_as_bfloat16(sc));
        const __nv_bfloat162 b2 = __halves2bfloat162(__ushort_as_bfloat16(bi), __ushort_as_bfloat16(bi));
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t o[8][4];
#pragma unroll
        for (int c = 0; c < 8; ++c) dq8_bf16(words[c], s2, b2, o[c]);
        // The code stage goes back to the TMA (an async-proxy writer) only
        // after every lane's reads of it have returned: the dequantised values
        // above depend on them. The proxy fence orders those generic-proxy
        // reads before the next asynchronous write of the stage.
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(cempty(cs));
        if (!(ok = mbar_wait(empty(s), ph ^ 1u, abort_flag, a.hdr))) break;
        uint8_t* bt = gbase + kOffB + s * kBBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(bt + sw128(r, c)) = make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(full(s));
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kNumEpiWarps) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t tc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
      int g, p0, R, j;
      if (!tile_info(tile, g, p0, R, j)) {
        *abort_flag = 1;
        break;
      }
      // test hook: a wait on a barrier nothing arrives on, bounded by the hook's limit
      if (a.epi_wait_limit > 0 && !(ok = mbar_wait(never_bar, 0, abort_flag, a.hdr, a.epi_wait_limit))) break;
      const int buf = tc & 1;
      if (!(ok = mbar_wait(accf(buf), (tc >> 1) & 1u, abort_flag, a.hdr))) break;
      tc_fence_after();
      {
        const int r = q * 32 + lane;  // tile row of this thread
        const bool valid = r < R;
        const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + buf * BN;
        if (GATEUP) {
          uint16_t* hrow = a.h + size_t(p0 + (valid ? r : 0)) * a.I + j * 128;
#pragma unroll 1
          for (int cc = 0; cc < 128; cc += 16) {
            uint32_t gv[16], uv[16];
            tmem_ld16(tbase + cc, gv);
            tmem_ld16(tbase + 128 + cc, uv);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float h0 = silu_mul(__uint_as_float(gv[2 * i]), __uint_as_float(uv[2 * i]));
              const float h1 = silu_mul(__uint_as_float(gv[2 * i + 1]), __uint_as_float(uv[2 * i + 1]));
              pk[i] = uint32_t(f32_to_bf16(h0)) | (uint32_t(f32_to_bf16(h1)) << 16);
            }
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(hrow + cc);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        } else {
          int t = 0;
          float wgt = 0.f;
          if (valid) {
            const int p = p0 + r;
            if (g == a.E) {
              t = p - A_rows;
              wgt = 1.f;
            } else {
              const int asg = a.perm[p];
              t = asg / a.k;
              wgt = a.topk_w[asg];
            }
          }
          float* yrow = a.y_acc + size_t(t) * a.D + j * BN;
#pragma unroll 1
          for (int cc = 0; cc < BN; cc += 16) {
            uint32_t v[16];
            tmem_ld16(tbase + cc, v);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                red_add_v4(yrow + cc + i, wgt * __uint_as_float(v[i]), wgt * __uint_as_float(v[i + 1]),
                           wgt * __uint_as_float(v[i + 2]), wgt * __uint_as_float(v[i + 3]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---- host side ------------------------------------------------------------------------------



__global__ void debug_dequant_kernel(moe_qmatrix m, int expert, int rows, int K, uint16_t* out) {
  const int words = K / 8;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < rows * words; i += gridDim.x * blockDim.x) {
    const int n = i / words, wi = i % words;
    const size_t row = size_t(expert) * rows + n;
    const uint32_t w = m.codes[row * words + wi];
    const uint16_t s = m.scales[row * (K / 64) + wi / 8], b = m.biases[row * (K / 64) + wi / 8];
    const __nv_bfloat162 s2 = __halves2bfloat162(__ushort_as_bfloat16(s), __ushort_as_bfloat16(s));
    const __nv_bfloat162 b2 = __halves2bfloat162(__ushort_as_bfloat16(b), __ushort_as_bfloat16(b));
    uint32_t o[4];
    dq8_bf16(w, s2, b2, o);
    *reinterpret_cast<uint4*>(out + size_t(n) * K + wi * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The separate expansion pass: the matrices of expert blockIdx.y to bf16,
// each weight rounded once from s * q + b as the fused kernels round it. A
// thread takes four consecutive code words (32 weights of one quantisation
// group: K is a multiple of 64, so four-word runs never straddle a group) in
// one 16-byte load and writes 64 bytes. count: skip experts no row selected
// (null: all).
__global__ void expand_weights_kernel(moe_qmatrix m, int rows, int K, const int32_t* count, uint16_t* out) {
  const int e = blockIdx.y;
  if (count && count[e] == 0) return;
  const int quads = K / 32;  // four-word runs per row
  const size_t n = size_t(rows) * quads;
  const size_t row0 = size_t(e) * rows;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
    const size_t row = row0 + i / quads;
    const int qi = int(i % quads);
    const uint4 w = *reinterpret_cast<const uint4*>(m.codes + row * (K / 8) + size_t(qi) * 4);
    const uint16_t sc = m.scales[row * (K / 64) + qi / 2], bi = m.biases[row * (K / 64) + qi / 2];
    const __nv_bfloat162 s2 = __halves2bfloat162(__ushort_as_bfloat16(sc), __ushort_as_bfloat16(sc));
    const __nv_bfloat162 b2 = __halves2bfloat162(__ushort_as_bfloat16(bi), __ushort_as_bfloat16(bi));
    uint32_t o[4][4];
    dq8_bf16(w.x, s2, b2, o[0]);
    dq8_bf16(w.y, s2, b2, o[1]);
    dq8_bf16(w.z, s2, b2, o[2]);
    dq8_bf16(w.w, s2, b2, o[3]);
    uint4* dst = reinterpret_cast<uint4*>(out + row * K + size_t(qi) * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) dst[c] = make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
  }
}

}  // namespace

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// 2-D tensor map over a row-major [rows, cols] array.
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t elem, const void* ptr, uint64_t rows, uint64_t cols,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * elem};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_encoder_available() { return encoder() != nullptr; }

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t debug_dequant(const moe_qmatrix* m, int expert, int rows, int K, uint16_t* out, cudaStream_t s) {
  debug_dequant_kernel<<<256, 256, 0, s>>>(*m, expert, rows, K, out);
  return cudaGetLastError();
}

bool gemm_tc_supported(const Ctx& c) { return c.I % 128 == 0 && c.D % BN == 0 && encoder() != nullptr; }

ExpandedWeights expanded_weights(const moe_weights* w, void* base) {
  ExpandedWeights x;
  const size_t gu = size_t(w->I) * w->D;  // elements of one expert's gate (or up, or down) matrix
  uint16_t* p = static_cast<uint16_t*>(base);
  x.gate = p;
  x.up = x.gate + size_t(w->E) * gu;
  x.down = x.up + size_t(w->E) * gu;
  x.s_gate = x.down + size_t(w->E) * gu;
  x.s_up = x.s_gate + gu;
  x.s_down = x.s_up + gu;
  x.bytes = (size_t(3) * w->E + 3) * gu * 2;
  return x;
}

cudaError_t expand_weights(const Ctx& c) {
  const moe_weights* w = c.w;
  const ExpandedWeights& x = c.wexp;
  const dim3 blk(256);
  // about four waves of CTAs over the routed experts' matrices
  const int per_e = std::max(1, 4 * num_sms() * 4 / std::max(1, c.E));
  struct Job {
    const moe_qmatrix* m;
    int rows, K, n;
    const int32_t* count;
    uint16_t* out;
  } jobs[6] = {{&w->gate, c.I, c.D, c.E, c.count, x.gate},   {&w->up, c.I, c.D, c.E, c.count, x.up},
               {&w->down, c.D, c.I, c.E, c.count, x.down},   {&w->s_gate, c.I, c.D, 1, nullptr, x.s_gate},
               {&w->s_up, c.I, c.D, 1, nullptr, x.s_up},     {&w->s_down, c.D, c.I, 1, nullptr, x.s_down}};
  for (const Job& j : jobs) {
    const dim3 grid(j.n == 1 ? 4 * num_sms() : per_e, j.n);
    expand_weights_kernel<<<grid, blk, 0, c.stream>>>(*j.m, j.rows, j.K, j.count, j.out);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    launch_done(c, "expand_weights");
  }
  return cudaSuccess;
}

template <bool BF16W>
static cudaError_t gemm_tc_run(const Ctx& c) {
  const moe_weights* w = c.w;
  if (!ensure_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<true, BF16W>), int(kSmemBytes)) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<false, BF16W>), int(kSmemBytes)))
    return cudaErrorInvalidValue;
  const int A = c.T * c.k;
  TcArgs a{c.x,      w->gate,   w->up,      w->s_gate, w->s_up, c.blocks, c.n_blocks, c.perm,
           c.topk_w, c.h,       c.y_acc,    c.hdr,     c.T,     c.D,      c.E,        c.k,
           c.I,      c.max_blocks, (long long)c.opt.test_wait_cycles};
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const auto U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32, BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE, SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const ExpandedWeights& x = c.wexp;
  bool ok = BF16W ? make_tmap_2d(&maps.c0, BF16, 2, x.gate, uint64_t(c.E) * c.I, c.D, BK, 128, SW) &&
                        make_tmap_2d(&maps.c1, BF16, 2, x.up, uint64_t(c.E) * c.I, c.D, BK, 128, SW) &&
                        make_tmap_2d(&maps.cs0, BF16, 2, x.s_gate, c.I, c.D, BK, 128, SW) &&
                        make_tmap_2d(&maps.cs1, BF16, 2, x.s_up, c.I, c.D, BK, 128, SW)
                  : make_tmap_2d(&maps.c0, U32, 4, w->gate.codes, uint64_t(c.E) * c.I, c.D / 8, 8, 128, NOSW) &&
                        make_tmap_2d(&maps.c1, U32, 4, w->up.codes, uint64_t(c.E) * c.I, c.D / 8, 8, 128, NOSW) &&
                        make_tmap_2d(&maps.cs0, U32, 4, w->s_gate.codes, c.I, c.D / 8, 8, 128, NOSW) &&
                        make_tmap_2d(&maps.cs1, U32, 4, w->s_up.codes, c.I, c.D / 8, 8, 128, NOSW);
  if (!ok) return cudaErrorInvalidValue;

  cudaError_t err = c.yacc_zeroed ? cudaSuccess : zero_yacc(c);
  if (err != cudaSuccess) return err;
  const int grid1 = std::max(1, std::min(num_sms(), c.max_blocks * (c.I / 128)));
  gemm_tc_kernel<true, BF16W><<<grid1, kNumThreads, kSmemBytes, c.stream>>>(a, maps);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done(c, "gateup_tc");

  a.m0 = w->down;
  a.s0 = w->s_down;
  std::memset(&maps, 0, sizeof(maps));
  ok = (BF16W ? make_tmap_2d(&maps.c0, BF16, 2, x.down, uint64_t(c.E) * c.D, c.I, BK, 128, SW) &&
                    make_tmap_2d(&maps.cs0, BF16, 2, x.s_down, c.D, c.I, BK, 128, SW)
              : make_tmap_2d(&maps.c0, U32, 4, w->down.codes, uint64_t(c.E) * c.D, c.I / 8, 8, BN, NOSW) &&
                    make_tmap_2d(&maps.cs0, U32, 4, w->s_down.codes, c.D, c.I / 8, 8, BN, NOSW)) &&
       make_tmap_2d(&maps.a, BF16, 2, c.h, uint64_t(A + c.T), c.I, BK, kTileRows, SW);
  if (!ok) return cudaErrorInvalidValue;
  const int grid2 = std::max(1, std::min(num_sms(), c.max_blocks * (c.D / BN)));
  gemm_tc_kernel<false, BF16W><<<grid2, kNumThreads, kSmemBytes, c.stream>>>(a, maps);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  launch_done(c, "down_tc");
  return cast_y(c);
}

cudaError_t gemm_tc(const Ctx& c) { return c.wexp.gate ? gemm_tc_run<true>(c) : gemm_tc_run<false>(c); }

}  // namespace moe
