// Tensor-core grouped GEMMs of the prefill expert path with the dequantised
// weights in tensor memory ("Optimizing on-device inference for Apple
// Silicon", section "Dequantise weights during matrix multiplication": the
// 4-bit weights are expanded one small tile at a time on chip and never exist
// expanded in DRAM; section "Reduce intermediate and state traffic": gate/up
// fused with the gated activation, down fused with the routing weights, the
// shared expert and the un-permute).
//
// The MMA computes D[weight row, token] = W[128 x K] * X[N x K]^T:
//   A = 128 weight rows, dequantised by eight warps from registers straight
//       into a tensor-memory stage (tcgen05.st): no shared-memory round trip
//       for the expanded weights, and the MMA does not read them from shared
//       memory either;
//   B = the block's token rows (N <= 192, rounded up to 16), in shared memory
//       in the 128-byte-swizzled K-major layout: gathered from x with
//       cp.async (gate/up) or loaded by TMA from h (down);
//   D = fp32 in tensor memory, two 192-column buffers so the epilogue of one
//       tile overlaps the next tile's MMAs.
// Tensor memory (512 columns): accumulators 0..383, two A stages 384..511.
// A pipeline stage spans 128 of K (two quantisation groups), so the MMA warp
// issues eight MMAs per pair of barrier waits.
//
// gate/up tiles take 64 intermediate rows with the gate and up rows
// interleaved (lane 2i = gate row i, lane 2i+1 = up row i), so the epilogue
// pairs g and u with one shuffle; down tiles take 128 output columns.
//
// Warp roles (22 warps): 0 TMA for the packed codes, 1 TMEM allocator and MMA
// issuer, 2..5 the token operand (gate/up: cp.async gather of x rows, eight
// consecutive lanes per 128-byte row so every warp instruction covers four
// whole cache lines; down: 2-D TMA tiles of h), 6..13 dequantisation (two
// warps per TMEM lane quarter, one for each group of a stage), 14..21 epilogue
// (two warps per lane quarter, alternate 16-token column chunks).
// Every mbarrier wait is bounded; on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT, drains what it has in flight and exits.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int WM = 128;               // weight rows per tile (MMA M, TMEM lanes)
constexpr int WK = 64;                // one quantisation group
constexpr int kGroupsPerStage = 2;    // a pipeline stage spans 128 of K
constexpr uint32_t kCBytes = WM * WK / 2;               // 4 KB of codes
constexpr uint32_t kAGroupCols = WK / 2;                // 32 columns: one group's 64 bf16 per lane
constexpr uint32_t kAStageCols = kAGroupCols * kGroupsPerStage;
constexpr uint32_t kTmemCols = 512;
constexpr int kXposeStride = 36;  // floats per row of an epilogue transpose buffer (conflict-free float4 reads)
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpB0 = 2, kNumBWarps = 4, kWarpDq0 = 6;

// A launch shape of the kernel: the largest token block of a tile (MMA N),
// the dequantising warp sets (one per A stage in tensor memory: set p fills
// the stages t = p, p + SETS, ... and owns A stage p; four warps, one per
// TMEM lane quarter, each), the epilogue warps (EPIW / 4 per lane quarter)
// and the slots of the packed-code and token rings (the bytes in flight per SM).
// Tensor memory holds two accumulators of MAXN columns and SETS A stages.
template <int MAXN, int SETS, int EPIW, int CSLOTS, int BSLOTS, bool SBSMEM>
struct WtCfg {
  // SBSMEM: the TMA warp also copies each tile's scale and bias rows into a
  // two-slot ring in shared memory, ahead of use; otherwise the dequantising
  // warps load each stage's pair from global memory when they need it
  static constexpr int kSbSlots = SBSMEM ? 2 : 0;
  static constexpr uint32_t kSbBytes = 16384;  // one tile's rows: 8 K bytes, K <= 2048
  static constexpr int kMaxN = MAXN;
  static constexpr int kBStages = BSLOTS;  // token operand ring (shared memory)
  static constexpr int kCStages = CSLOTS;  // packed-code ring, one quantisation group per slot
  static constexpr int kAStages = SETS;
  static constexpr int kNumDqWarps = 4 * SETS;
  static constexpr int kNumEpiWarps = EPIW;
  static constexpr int kWarpEpi0 = kWarpDq0 + kNumDqWarps;
  static constexpr int kNumWarps = kWarpEpi0 + kNumEpiWarps;
  static constexpr int kNumThreads = kNumWarps * 32;
  static constexpr uint32_t kBHalf = kMaxN * WK * 2;             // one 128-byte-swizzled K block of 64
  static constexpr uint32_t kBBytes = kBHalf * kGroupsPerStage;
  static constexpr uint32_t kAccCols = kMaxN;                    // fp32 columns of one accumulator
  static constexpr uint32_t kAColBase = 2 * kAccCols;            // after the two accumulators
  static constexpr int kGatherPerThread = kMaxN * 8 / (kNumBWarps * 32);  // 16-byte chunks per thread per K block
  static constexpr int kEpiHalves = kNumEpiWarps / 4;            // epilogue warps per lane quarter
  static constexpr int kEpiStep = 16 * kEpiHalves;               // columns between a warp's 16-column chunks
  static constexpr int kEpiChunks = (kMaxN + kEpiStep - 1) / kEpiStep;
  static constexpr uint32_t kOffB = 0;
  static constexpr uint32_t kOffC = kOffB + kBStages * kBBytes;
  static constexpr uint32_t kOffXpose = kOffC + kCStages * kCBytes;  // down epilogue: [warp][16][36] floats
  static constexpr uint32_t kOffSb = kOffXpose + kNumEpiWarps * 16 * kXposeStride * 4;
  static constexpr uint32_t kOffBar = kOffSb + kSbSlots * kSbBytes;
  // bfull, bempty [kBStages]; afull, aempty [kAStages]; cfull, cempty [kCStages]; accf, acce [2]; drain; never;
  // sbfull, sbempty [kSbSlots]
  static constexpr uint32_t kNumBars = 2 * kBStages + 2 * kAStages + 2 * kCStages + 6 + 2 * kSbSlots;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr size_t kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static_assert(kAColBase + kAStages * kAStageCols <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kMaxN % 16 == 0 && (kMaxN * 8) % (kNumBWarps * 32) == 0, "whole gather chunks");
  static_assert(kCStages % (2 * SETS) == 0, "every code slot is read by one set");
  static_assert(kNumEpiWarps % 4 == 0, "epilogue warps cover the four lane quarters");
};
// 192-token blocks with two weight stages in flight (the default), and
// blocks of at most 64 tokens with four: small blocks leave tensor memory
// for more A stages, and their tiles are bound by the chain of dependent
// loads and dequantisation, not by the tensor pipe: their scale and bias rows
// come ahead of use through shared memory (at a stage of a few hundred
// cycles a global load per stage would be a DRAM round trip on the chain),
// and their code ring holds two stages per set, so that the next stage's
// codes are in flight while a set converts the current one.
using WtLarge = WtCfg<kWtBlockRows, 2, 8, 8, 3, false>;
using WtSmall = WtCfg<kWtSmallBlockRows, 4, 4, 16, 3, true>;

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrives on `bar` once every cp.async this thread has issued so far has
// landed; the barrier's expected count includes this arrival.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, descriptor version 1. Split in two 32-bit halves: the low
// half holds the start address (bits 0-13, in 16-byte units) and the leading
// byte offset; the high half the stride byte offset, the version bit and the
// swizzle mode, and is the same for every tile.
__device__ __forceinline__ uint32_t smem_desc_lo(uint32_t addr) { return ((addr & 0x3FFFFu) >> 4) | (1u << 16); }
constexpr uint32_t kSmemDescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_n(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(WM >> 4) << 24);
}

// One stage of 128 of K: eight K = 16 MMAs D (tensor memory) += A (tensor
// memory, columns a .. a+63) * B (shared memory: two 128-byte-swizzled K
// blocks of 64, the first with descriptor low half b_lo, the second kBHalf
// bytes further)^T, then commits that arrive on `bar_b` and `bar_a` (the two
// operand stages' release barriers) when they complete. The first MMA
// overwrites D when `accumulate` is 0. Executed by the whole, converged warp
// (the caller reconverges it first) so that every operand is warp-uniform and
// elect.sync picks the same lane every time: a commit tracks only the MMAs of
// the lane that executes it.
__device__ __forceinline__ void umma_stage(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t idesc, uint32_t accumulate,
                                           uint32_t bar_b, uint32_t bar_a, uint32_t b_half) {
  asm volatile(
      "{\n"
      " .reg .pred e, p, t;\n"
      " .reg .b32 a1, a2, a3, a4, a5, a6, a7, l1, l2, l3, l4, l5, l6, l7;\n"
      " .reg .b64 b0, b1, b2, b3, b4, b5, b6, b7;\n"
      " elect.sync _|e, 0xffffffff;\n"
      " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n"
      " add.u32 a4, %1, 32;\n add.u32 a5, %1, 40;\n add.u32 a6, %1, 48;\n add.u32 a7, %1, 56;\n"
      " add.u32 l1, %2, 2;\n add.u32 l2, %2, 4;\n add.u32 l3, %2, 6;\n"
      " add.u32 l4, %2, %8;\n add.u32 l5, l4, 2;\n add.u32 l6, l4, 4;\n add.u32 l7, l4, 6;\n"
      " mov.b64 b0, {%2, %3};\n mov.b64 b1, {l1, %3};\n mov.b64 b2, {l2, %3};\n mov.b64 b3, {l3, %3};\n"
      " mov.b64 b4, {l4, %3};\n mov.b64 b5, {l5, %3};\n mov.b64 b6, {l6, %3};\n mov.b64 b7, {l7, %3};\n"
      " setp.ne.b32 p, %5, 0;\n"
      " setp.eq.b32 t, %5, %5;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b0, %4, p;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %4, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %4, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %4, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %4, t;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n"
      "}" ::"r"(d),
      "r"(a), "r"(b_lo), "r"(kSmemDescHi), "r"(idesc), "r"(accumulate), "r"(bar_b), "r"(bar_a), "r"(b_half >> 4)
      : "memory");
}

// Commit by one elected lane of a converged warp (the same lane that issued
// the MMAs): `bar` receives one arrival when every MMA this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// The wait, with the registers of the outstanding load as operands: they are
// written asynchronously, so no use of them may be scheduled before this.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Byte offset of 16-byte chunk c of row r inside a 1024-aligned SW128 K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

struct WtArgs {
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

struct TileEntry {
  int g, p0, R;  // expert (E: the shared expert), first row, rows
};

struct WtMaps {
  CUtensorMap c0, c1;    // routed codes: gate, up (box 8 words x 64 rows) or down (box 8 x 128)
  CUtensorMap cs0, cs1;  // shared-expert codes
  CUtensorMap b;         // down only: h [T*k+T, I] (SW128, box 64 x kMaxN)
};

template <bool GATEUP, class C>
__global__ void __launch_bounds__(C::kNumThreads, 1) gemm_wt_kernel(const WtArgs args, const __grid_constant__ WtMaps maps) {
  constexpr int kMaxN = C::kMaxN, kAStages = C::kAStages, kNumDqWarps = C::kNumDqWarps;
  constexpr int kWarpEpi0 = C::kWarpEpi0, kNumEpiWarps = C::kNumEpiWarps, kEpiChunks = C::kEpiChunks;
  constexpr int kEpiStep = C::kEpiStep, kGatherPerThread = C::kGatherPerThread;
  constexpr uint32_t kBHalf = C::kBHalf, kBBytes = C::kBBytes, kAccCols = C::kAccCols, kAColBase = C::kAColBase;
  constexpr uint32_t kOffB = C::kOffB, kOffC = C::kOffC, kOffXpose = C::kOffXpose, kOffBar = C::kOffBar,
                     kOffMisc = C::kOffMisc;
  constexpr int kCStages = C::kCStages, kBStages = C::kBStages, kSbSlots = C::kSbSlots;
  constexpr int kSbRing = kSbSlots > 0 ? kSbSlots : 1;  // divisor for ring positions (unused when kSbSlots == 0)
  constexpr uint32_t kSbBytes = C::kSbBytes, kOffSb = C::kOffSb;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + kOffBar;
  auto bfull = [&](int s) { return bar0 + 8u * s; };
  auto bempty = [&](int s) { return bar0 + 8u * (kBStages + s); };
  auto afull = [&](int s) { return bar0 + 8u * (2 * kBStages + s); };
  auto aempty = [&](int s) { return bar0 + 8u * (2 * kBStages + kAStages + s); };
  auto cfull = [&](int s) { return bar0 + 8u * (2 * kBStages + 2 * kAStages + s); };
  auto cempty = [&](int s) { return bar0 + 8u * (2 * kBStages + 2 * kAStages + kCStages + s); };
  constexpr uint32_t kBarAcc = 2 * kBStages + 2 * kAStages + 2 * kCStages;
  auto accf = [&](int b) { return bar0 + 8u * (kBarAcc + b); };
  auto acce = [&](int b) { return bar0 + 8u * (kBarAcc + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (kBarAcc + 4);
  const uint32_t never_bar = bar0 + 8u * (kBarAcc + 5);  // test hook: nothing arrives here
  auto sbfull = [&](int s) { return bar0 + 8u * (kBarAcc + 6 + s); };
  auto sbempty = [&](int s) { return bar0 + 8u * (kBarAcc + 6 + kSbSlots + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WtArgs& a = args;
  const int NT = GATEUP ? a.I / 64 : a.D / WM;  // weight-row tiles per block-map entry
  const int K = GATEUP ? a.D : a.I;
  const int KS = K / WK;                   // quantisation groups per tile
  const int KT = KS / kGroupsPerStage;     // pipeline stages per tile
  const int A_rows = a.T * a.k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(bfull(s), GATEUP ? kNumBWarps * 32 : 1);
      mbar_init(bempty(s), 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(afull(s), 4);  // the four warps (one per lane quarter) of the set that owns the stage
      mbar_init(aempty(s), 1);
    }
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(cfull(s), 1);
      mbar_init(cempty(s), 4);  // the four warps of the set that reads the slot
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf(b), 1);
      mbar_init(acce(b), kNumEpiWarps);  // every epilogue warp drains its chunks
    }
    mbar_init(drain_bar, 1);
    mbar_init(never_bar, 1);
    for (int s = 0; s < kSbSlots; ++s) {
      mbar_init(sbfull(s), 1);
      mbar_init(sbempty(s), kNumDqWarps);  // every dequantising warp, after its last stage of the tile
    }
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
  // Launched as a programmatic dependent of the previous kernel: gate/up reads
  // the routing tables and the paired-order x, so every thread waits here for
  // that kernel; down reads only h from its predecessor (gate/up), so only the
  // thread that loads h waits (below), and the rest of its CTA sets up, loads
  // and dequantises its first weight stages during gate/up's last tiles.
  if (GATEUP) griddep_wait();
  griddep_launch();

  int nb = *a.n_blocks;
  if (nb > a.max_blocks || nb < 0) {
    if (threadIdx.x == 0) report(a.hdr, MOE_ERR_DEVICE_CHECK, 20);
    nb = 0;
  }
  const int n_tiles = nb * NT;

  // Block-map entries are loaded one tile ahead of use: every role issues
  // the loads of its next tile's entry when it starts a tile, so a new tile
  // does not begin with a global-memory round trip. An entry is checked when
  // its tile starts.
  auto entry_load = [&](int tile) {
    TileEntry e{0, 0, 0};
    if (tile < n_tiles) {
      const int b = tile / NT;
      e.g = a.blocks[3 * b];
      e.p0 = a.blocks[3 * b + 1];
      e.R = a.blocks[3 * b + 2];
    }
    return e;
  };
  auto entry_ok = [&](const TileEntry& e) {
    if (e.g < 0 || e.g > a.E || e.R < 1 || e.R > kMaxN || e.p0 < 0 || e.p0 + e.R > A_rows + a.T ||
        (e.g < a.E && e.p0 + e.R > A_rows)) {
      report(a.hdr, MOE_ERR_DEVICE_CHECK, 21);
      return false;
    }
    return true;
  };

  if (warp == kWarpTma) {
    // ---------------- TMA producer: codes (and h rows for down) ----------------
    if (lane == 0) {
      uint32_t it = 0, c_issued = 0, sb_issued = 0;
      bool ok = true;
      TileEntry nx = entry_load(blockIdx.x);
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const TileEntry e = nx;
        nx = entry_load(tile + gridDim.x);
        if (!entry_ok(e)) {
          *abort_flag = 1;
          break;
        }
        const int g = e.g, j = tile % NT;
        const bool sh = (g == a.E);
        const int ex = sh ? 0 : g;
        if (kSbSlots > 0) {
          // the tile's scale and bias rows: gate/up [gate s][gate b][up s][up b]
          // of 64 rows, down [s][b] of 128 rows, K / 64 bf16 per row
          const int ss = sb_issued % kSbRing;
          if (!(ok = mbar_wait(sbempty(ss), ((sb_issued / kSbRing) & 1u) ^ 1u, abort_flag, a.hdr))) break;
          const uint32_t sdst = base + kOffSb + ss * kSbBytes;
          const int G2 = K / 64;
          if (GATEUP) {
            const size_t row0 = size_t(ex) * a.I + j * 64;
            const uint32_t nb = 64u * G2 * 2;
            mbar_arrive_tx(sbfull(ss), 4 * nb);
            const moe_qmatrix& mg = sh ? a.s0 : a.m0;
            const moe_qmatrix& mu = sh ? a.s1 : a.m1;
            bulk_g2s(sdst, mg.scales + row0 * G2, nb, sbfull(ss));
            bulk_g2s(sdst + nb, mg.biases + row0 * G2, nb, sbfull(ss));
            bulk_g2s(sdst + 2 * nb, mu.scales + row0 * G2, nb, sbfull(ss));
            bulk_g2s(sdst + 3 * nb, mu.biases + row0 * G2, nb, sbfull(ss));
          } else {
            const size_t row0 = size_t(ex) * a.D + j * WM;
            const uint32_t nb = uint32_t(WM) * G2 * 2;
            mbar_arrive_tx(sbfull(ss), 2 * nb);
            const moe_qmatrix& md = sh ? a.s0 : a.m0;
            bulk_g2s(sdst, md.scales + row0 * G2, nb, sbfull(ss));
            bulk_g2s(sdst + nb, md.biases + row0 * G2, nb, sbfull(ss));
          }
          ++sb_issued;
        }
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int cs = it % kCStages;
          const uint32_t cph = (it / kCStages) & 1u;
          if (!(ok = mbar_wait(cempty(cs), cph ^ 1u, abort_flag, a.hdr))) break;
          const uint32_t cdst = base + kOffC + cs * kCBytes;
          mbar_arrive_tx(cfull(cs), kCBytes);
          if (GATEUP) {  // 64 gate rows, then the same 64 up rows
            const int row = ex * a.I + j * 64;
            tma_load_2d(cdst, sh ? &maps.cs0 : &maps.c0, ks * 8, row, cfull(cs));
            tma_load_2d(cdst + kCBytes / 2, sh ? &maps.cs1 : &maps.c1, ks * 8, row, cfull(cs));
          } else {
            tma_load_2d(cdst, sh ? &maps.cs0 : &maps.c0, ks * 8, ex * a.D + j * WM, cfull(cs));
          }
          c_issued = it + 1;
        }
      }
      // drain: every load this thread issued lands before the CTA exits
      for (uint32_t s = 0; s < uint32_t(kCStages); ++s)
        if (s < c_issued) {
          const uint32_t last = c_issued - 1 - ((c_issued - 1 - s) % kCStages);
          mbar_wait(cfull(s), (last / kCStages) & 1u, abort_flag, a.hdr, kWaitLimit, true);
        }
      for (uint32_t s = 0; s < uint32_t(kSbRing); ++s)
        if (s < sb_issued) {
          const uint32_t last = sb_issued - 1 - ((sb_issued - 1 - s) % kSbRing);
          mbar_wait(sbfull(s), (last / kSbRing) & 1u, abort_flag, a.hdr, kWaitLimit, true);
        }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer: the whole warp runs the loop, one lane issues ----------------
    // lane 0's wait result decides for the warp, so every branch stays uniform
    auto warp_wait = [&](uint32_t bar, uint32_t parity, bool draining) {
      const bool r = mbar_wait(bar, parity, abort_flag, a.hdr, kWaitLimit, draining);
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    uint32_t it = 0, tc = 0;
    bool ok = true;
    TileEntry nx = entry_load(blockIdx.x);
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
      const TileEntry e = nx;
      nx = entry_load(tile + gridDim.x);
      if (!entry_ok(e)) {
        *abort_flag = 1;
        break;
      }
      const int R = e.R;
      const uint32_t idesc = idesc_n((R + 15) & ~15);
      const int buf = tc & 1;
      if (!(ok = warp_wait(acce(buf), ((tc >> 1) & 1u) ^ 1u, false))) break;
      tc_fence_after();
      const uint32_t d = tmem + buf * kAccCols;
      for (int t = 0; t < KT; ++t, ++it) {
        const int s = it % kBStages, sa = it % kAStages;
        if (!(ok = warp_wait(bfull(s), (it / kBStages) & 1u, false))) break;
        if (!(ok = warp_wait(afull(sa), (it / kAStages) & 1u, false))) break;
        tc_fence_after();
        // the gathered tokens were written by cp.async (generic proxy): order them
        // before the tensor cores' (async proxy) reads
        if (GATEUP) fence_proxy_async();
        // the lanes left the barrier waits above at different times: reconverge
        // so that elect.sync picks lane 0, the lane of every earlier MMA
        __syncwarp();
        umma_stage(d, tmem + kAColBase + sa * kAStageCols, smem_desc_lo(base + kOffB + s * kBBytes), idesc,
                   t != 0 ? 1u : 0u, bempty(s), aempty(sa), kBHalf);
      }
      if (!ok) break;
      __syncwarp();
      umma_commit_warp(accf(buf));
    }
    __syncwarp();
    umma_commit_warp(drain_bar);  // all MMAs complete before tensor memory is released
    warp_wait(drain_bar, 0, true);
  } else if (warp >= kWarpB0 && warp < kWarpB0 + kNumBWarps) {
    // ---------------- the token operand (B) ----------------
    const int bt = threadIdx.x - kWarpB0 * 32;  // 0..127
    if (GATEUP) {
      // chunk m of this thread: row (bt + 128m) / 8, 16-byte chunk (bt + 128m) % 8.
      // The next tile's entry and its rows' perm entries are loaded while the
      // current tile's first stage is issued, so a new tile's gathers start
      // without waiting for two dependent global loads. The eight lanes that
      // share a row set split those loads (lane chunk c loads the rows of
      // chunks c, c + 8, ...) and exchange them by shuffles.
      constexpr int kRowRegs = (kGatherPerThread + 7) / 8;
      const int ch = bt & 7;
      TileEntry nx = entry_load(blockIdx.x);
      int nx_row[kRowRegs];  // routed: the perm entry of a row; shared: its token
      auto rows_load = [&](const TileEntry& ne) {
#pragma unroll
        for (int i = 0; i < kRowRegs; ++i) {
          const int m = ch + 8 * i;
          const int row = (bt >> 3) + 16 * m;
          const int rr = (m < kGatherPerThread && row < ne.R) ? row : 0;
          nx_row[i] = (ne.g == a.E) ? (ne.p0 + rr - A_rows) : a.perm[ne.p0 + rr];
        }
      };
      uint32_t it = 0;
      bool ok = blockIdx.x >= n_tiles || entry_ok(nx);
      if (ok && blockIdx.x < n_tiles) rows_load(nx);
      if (!ok) *abort_flag = 1;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const TileEntry e = nx;  // checked before its rows were loaded
        nx = entry_load(tile + gridDim.x);
        const bool sh = (e.g == a.E);
        const int R = e.R;
        const int n = (R + 15) & ~15;  // rows the MMA reads; R..n-1 repeat a valid row
        // byte offsets into x of this thread's chunks (x is under 4 GB)
        uint32_t src[kGatherPerThread];
#pragma unroll
        for (int m = 0; m < kGatherPerThread; ++m) {
          const int v = __shfl_sync(0xffffffffu, nx_row[m >> 3], (lane & 24) | (m & 7));
          int t = sh ? v : v / a.k;
          if (t < 0 || t >= a.T) {
            report(a.hdr, MOE_ERR_DEVICE_CHECK, 22);
            t = 0;
          }
          src[m] = uint32_t(t) * uint32_t(a.D * 2) + uint32_t(ch * 16);
        }
        const char* xbytes = reinterpret_cast<const char*>(a.x);
        // this thread copies chunk column bt & 7 of rows r0 + 16 m: in the
        // swizzled tile those land at sw0 + 2048 m (row & 7 is the same for all m)
        const int r0 = bt >> 3;
        const uint32_t sw0 = sw128(r0, bt & 7);
        uint32_t live = 0;  // bit m: row r0 + 16 m is read by the MMA
#pragma unroll
        for (int m = 0; m < kGatherPerThread; ++m)
          if (r0 + 16 * m < n) live |= 1u << m;
        for (int t = 0; t < KT; ++t, ++it) {
          const int s = it % kBStages;
          const uint32_t ph = (it / kBStages) & 1u;
          if (!(ok = mbar_wait(bempty(s), ph ^ 1u, abort_flag, a.hdr))) break;
          const uint32_t dst = base + kOffB + s * kBBytes + sw0;
          const int koff = t * kGroupsPerStage * 128;
#pragma unroll
          for (int hb = 0; hb < kGroupsPerStage; ++hb)
#pragma unroll
            for (int m = 0; m < kGatherPerThread; ++m)
              if (live & (1u << m)) cp_async16(dst + hb * kBHalf + 2048u * m, xbytes + src[m] + koff + hb * 128, 16u);
          cp_async_arrive_noinc(bfull(s));
          if (t == 0 && tile + int(gridDim.x) < n_tiles) {  // the next tile's rows
            if (entry_ok(nx)) {
              rows_load(nx);
            } else {
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
        }
      }
      cp_async_wait<0>();
    } else if (bt == 0) {
      // down: rows p0.. of h as one 2-D TMA tile per k-step, once gate/up is done
      griddep_wait();
      uint32_t it = 0, issued = 0;
      bool ok = true;
      TileEntry nx = entry_load(blockIdx.x);
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const TileEntry e = nx;
        nx = entry_load(tile + gridDim.x);
        if (!entry_ok(e)) {
          *abort_flag = 1;
          break;
        }
        const int p0 = e.p0;
        for (int t = 0; t < KT; ++t, ++it) {
          const int s = it % kBStages;
          const uint32_t ph = (it / kBStages) & 1u;
          if (!(ok = mbar_wait(bempty(s), ph ^ 1u, abort_flag, a.hdr))) break;
          mbar_arrive_tx(bfull(s), kBBytes);
          for (int hb = 0; hb < kGroupsPerStage; ++hb)
            tma_load_2d(base + kOffB + s * kBBytes + hb * kBHalf, &maps.b, (t * kGroupsPerStage + hb) * WK, p0,
                        bfull(s));
          issued = it + 1;
        }
      }
      for (uint32_t s = 0; s < uint32_t(kBStages); ++s)  // drain
        if (s < issued) {
          const uint32_t last = issued - 1 - ((issued - 1 - s) % kBStages);
          mbar_wait(bfull(s), (last / kBStages) & 1u, abort_flag, a.hdr, kWaitLimit, true);
        }
    }
  } else if (warp >= kWarpDq0 && warp < kWarpDq0 + kNumDqWarps) {
    // ---------------- dequantisation into the tensor-memory A stage ----------------
    // Four warps (one per TMEM lane quarter) fill the even stages, four the odd
    // ones: a warp converts both groups of its stage (all 128 codes of its
    // row), so each barrier wait, tensor-memory store wait and arrival is paid
    // once per stage, and consecutive stages are converted side by side.
    const int q = warp & 3;                          // TMEM lane quarter of this warp
    const int par = (warp - kWarpDq0) >> 2;          // the set: this warp fills stages par, par + kAStages, ...
    const int L = q * 32 + lane;                     // TMEM lane = weight row of the tile
    const int srow_stage = GATEUP ? ((L & 1) ? 64 + (L >> 1) : (L >> 1)) : L;  // row in the code stage
    uint32_t g0 = 0, t0 = 0, tcount = 0;  // groups, stages and tiles before this one
    bool ok = true;
    // only the expert of an entry is read here (one register held ahead);
    // the other roles check whole entries
    auto expert_of = [&](int tile) { return tile < n_tiles ? a.blocks[3 * (tile / NT)] : 0; };
    int nx_g = expert_of(blockIdx.x);
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, g0 += KS, t0 += KT, ++tcount) {
      const int g = nx_g, j = tile % NT;
      nx_g = expert_of(tile + gridDim.x);
      if (g < 0 || g > a.E) {
        report(a.hdr, MOE_ERR_DEVICE_CHECK, 21);
        *abort_flag = 1;
        break;
      }
      const bool sh = (g == a.E);
      const int ex = sh ? 0 : g;
      const uint16_t* srow;
      const uint16_t* brow;
      const int ss = int(tcount % kSbRing);
      if (kSbSlots > 0) {  // this row's pairs in the tile's shared-memory copy
        if (!(ok = mbar_wait(sbfull(ss), (tcount / kSbRing) & 1u, abort_flag, a.hdr))) break;
        const int G2 = K / 64;
        const uint16_t* sb = reinterpret_cast<const uint16_t*>(gbase + kOffSb + ss * kSbBytes);
        if (GATEUP) {
          srow = sb + ((L & 1) ? 128 * G2 : 0) + (L >> 1) * G2;
          brow = srow + 64 * G2;
        } else {
          srow = sb + L * G2;
          brow = srow + WM * G2;
        }
      } else {
        const moe_qmatrix& m = GATEUP ? ((L & 1) ? (sh ? a.s1 : a.m1) : (sh ? a.s0 : a.m0)) : (sh ? a.s0 : a.m0);
        const size_t row = GATEUP ? size_t(ex) * a.I + j * 64 + (L >> 1) : size_t(ex) * a.D + j * WM + L;
        srow = m.scales + row * (K / 64);
        brow = m.biases + row * (K / 64);
      }
      for (int t = par; t < KT && ok; t += kAStages) {
        const uint32_t is = t0 + t;
        const int s = is % kAStages;
        const uint32_t ph = (is / kAStages) & 1u;
        // the stage's two scales and two biases, one 32-bit load each (K / 64
        // is even and the arrays 16-byte aligned)
        const uint32_t sc2 = *reinterpret_cast<const uint32_t*>(srow + t * kGroupsPerStage);
        const uint32_t bi2 = *reinterpret_cast<const uint32_t*>(brow + t * kGroupsPerStage);
#pragma unroll 1
        for (int hb = 0; hb < kGroupsPerStage; ++hb) {
          const int ks = t * kGroupsPerStage + hb;
          const uint32_t ig = g0 + ks;
          const int cs = ig % kCStages;
          const uint32_t cph = (ig / kCStages) & 1u;
          const uint16_t sc = uint16_t(hb ? (sc2 >> 16) : (sc2 & 0xFFFFu));
          const uint16_t bi = uint16_t(hb ? (bi2 >> 16) : (bi2 & 0xFFFFu));
          if (!(ok = mbar_wait(cfull(cs), cph, abort_flag, a.hdr))) break;
          const uint8_t* crow = gbase + kOffC + cs * kCBytes + srow_stage * 32;
          const uint4 w0 = *reinterpret_cast<const uint4*>(crow);
          const uint4 w1 = *reinterpret_cast<const uint4*>(crow + 16);
          const __nv_bfloat162 s2 = __halves2bfloat162(__ushort_as_bfloat16(sc), __ushort_as_bfloat16(sc));
          const __nv_bfloat162 b2 = __halves2bfloat162(__ushort_as_bfloat16(bi), __ushort_as_bfloat16(bi));
          // gate/up: K in the paired order inside every group of eight (x was
          // permuted to match by the router); down: natural order (h)
          uint32_t o[32];
          if (GATEUP) {
            dq8_bf16_paired(w0.x, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 0));
            dq8_bf16_paired(w0.y, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 4));
            dq8_bf16_paired(w0.z, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 8));
            dq8_bf16_paired(w0.w, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 12));
            dq8_bf16_paired(w1.x, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 16));
            dq8_bf16_paired(w1.y, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 20));
            dq8_bf16_paired(w1.z, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 24));
            dq8_bf16_paired(w1.w, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 28));
          } else {
            dq8_bf16(w0.x, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 0));
            dq8_bf16(w0.y, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 4));
            dq8_bf16(w0.z, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 8));
            dq8_bf16(w0.w, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 12));
            dq8_bf16(w1.x, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 16));
            dq8_bf16(w1.y, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 20));
            dq8_bf16(w1.z, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 24));
            dq8_bf16(w1.w, s2, b2, *reinterpret_cast<uint32_t(*)[4]>(o + 28));
          }
          // the code stage goes back to the TMA only after every lane's reads
          // of it have returned: one instruction consumes all the words read
          // (a warp issues in order, so it waits for every lane's loads), and
          // the arrival depends on its result
          const uint32_t got = w0.x ^ w0.y ^ w0.z ^ w0.w ^ w1.x ^ w1.y ^ w1.z ^ w1.w;
          uint32_t zero;
          asm volatile("and.b32 %0, %1, 0;" : "=r"(zero) : "r"(got));
          __syncwarp();
          if (lane == int(zero)) mbar_arrive(cempty(cs));
          if (hb == 0) {
            if (!(ok = mbar_wait(aempty(s), ph ^ 1u, abort_flag, a.hdr))) break;
            tc_fence_after();  // the MMAs that read this A stage have completed
          }
          tmem_st32(tmem + (uint32_t(q * 32) << 16) + kAColBase + s * kAStageCols + hb * kAGroupCols, o);
          // tcgen05.st reads its source registers asynchronously: wait before
          // the next group's values overwrite them
          tmem_wait_st();
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull(s));
      }
      if (kSbSlots > 0) {  // the tile's scale and bias rows have been read
        __syncwarp();
        if (lane == 0) mbar_arrive(sbempty(ss));
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kNumEpiWarps) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int L = q * 32 + lane;                    // TMEM lane: weight row of the tile
    const int half = (warp - kWarpEpi0) >> 2;       // this warp takes 16-column chunks half, half + kEpiHalves, ...
    float* xb = reinterpret_cast<float*>(gbase + kOffXpose) + (warp - kWarpEpi0) * 16 * kXposeStride;
    uint32_t tc = 0;
    bool ok = true;
    TileEntry nx = entry_load(blockIdx.x);
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
      const TileEntry e = nx;
      nx = entry_load(tile + gridDim.x);
      if (!entry_ok(e)) {
        *abort_flag = 1;
        break;
      }
      const int g = e.g, p0 = e.p0, R = e.R, j = tile % NT;
      const int buf = tc & 1;
      const bool sh = (g == a.E);
      // down: this lane's token and routing weight for each of its chunks,
      // loaded before the accumulator is ready (perm, then topk_w)
      int tok[kEpiChunks];
      float wgt[kEpiChunks];
      if (!GATEUP) {
        int asg[kEpiChunks];
#pragma unroll
        for (int m = 0; m < kEpiChunks; ++m) {
          const int nn = half * 16 + kEpiStep * m + (lane >> 1);
          asg[m] = -1;
          tok[m] = 0;
          wgt[m] = 1.f;
          if (nn < R) {
            if (sh)
              tok[m] = p0 + nn - A_rows;
            else
              asg[m] = a.perm[p0 + nn];
          }
        }
#pragma unroll
        for (int m = 0; m < kEpiChunks; ++m)
          if (asg[m] >= 0) {
            tok[m] = asg[m] / a.k;
            wgt[m] = a.topk_w[asg[m]];
          }
      }
      if (a.epi_wait_limit > 0 && !(ok = mbar_wait(never_bar, 0, abort_flag, a.hdr, a.epi_wait_limit))) break;
      if (!(ok = mbar_wait(accf(buf), (tc >> 1) & 1u, abort_flag, a.hdr))) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + buf * kAccCols;
      // tensor-memory reads run one chunk ahead of the chunk being processed
      uint32_t va[16], vb[16];
      if (half * 16 < R) tmem_ld16(tbase + half * 16, va);
      tmem_wait_ld(va);
#pragma unroll
      for (int m = 0; m < kEpiChunks; ++m) {
        const int n0 = half * 16 + kEpiStep * m;
        if (n0 >= R) break;
        uint32_t(&v)[16] = (m & 1) ? vb : va;
        if (m + 1 < kEpiChunks && n0 + kEpiStep < R) tmem_ld16(tbase + n0 + kEpiStep, (m & 1) ? va : vb);
        if (GATEUP) {
          // lane 2i holds gate row i, lane 2i+1 up row i, for tokens n0..n0+15.
          // The pair swaps halves so that the even lane finishes the even
          // tokens and the odd lane the odd ones: each value computed once.
          const bool odd = lane & 1;
          float hv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float keep = __uint_as_float(odd ? v[2 * i + 1] : v[2 * i]);
            const float recv = __shfl_xor_sync(0xffffffffu, __uint_as_float(odd ? v[2 * i] : v[2 * i + 1]), 1);
            hv[i] = odd ? silu_mul(recv, keep) : silu_mul(keep, recv);
          }
          // lanes 4r and 4r+1 pack rows 2r, 2r+1 of their token parity
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float hn = __shfl_down_sync(0xffffffffu, hv[i], 2);
            const int nn = n0 + 2 * i + (odd ? 1 : 0);
            if ((lane & 2) == 0 && nn < R) {
              const uint32_t pk = uint32_t(f32_to_bf16(hv[i])) | (uint32_t(f32_to_bf16(hn)) << 16);
              *reinterpret_cast<uint32_t*>(a.h + size_t(p0 + nn) * a.I + j * 64 + (L >> 1)) = pk;
            }
          }
        } else {
          // transpose the warp's 32 columns x 16 tokens, then add them as
          // 16-byte reductions, eight lanes covering one token's 128-byte
          // line: each instruction touches four whole lines. Token c's index
          // and weight sit in lanes 2c and 2c+1.
#pragma unroll
          for (int c = 0; c < 16; ++c) xb[c * kXposeStride + lane] = __uint_as_float(v[c]);
          __syncwarp();
          const int quad = lane & 7;
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int c = (lane >> 3) + 4 * kq;
            const int tc_ = __shfl_sync(0xffffffffu, tok[m], 2 * c);
            const float w = __shfl_sync(0xffffffffu, wgt[m], 2 * c);
            if (n0 + c < R) {
              const float4 val = *reinterpret_cast<const float4*>(xb + c * kXposeStride + quad * 4);
              red_add_v4(a.y_acc + size_t(tc_) * a.D + j * WM + q * 32 + quad * 4, w * val.x, w * val.y, w * val.z,
                         w * val.w);
            }
          }
          __syncwarp();
        }
        if (m & 1)
          tmem_wait_ld(va);
        else
          tmem_wait_ld(vb);
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

// Both GEMMs of a layer with one launch shape C.
template <class C>
cudaError_t gemm_wt_run(const Ctx& c) {
  const moe_weights* w = c.w;
  if (c.BM < 1 || c.BM > C::kMaxN) return cudaErrorInvalidValue;  // a tile takes one block of <= kMaxN rows
  if (!c.xperm) return cudaErrorInvalidValue;  // gate/up gathers the paired-order x the router wrote
  if (!ensure_smem_limit(reinterpret_cast<const void*>(gemm_wt_kernel<true, C>), int(C::kSmemBytes)) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(gemm_wt_kernel<false, C>), int(C::kSmemBytes)))
    return cudaErrorInvalidValue;
  const int A = c.T * c.k;
  WtArgs a{c.xperm,  w->gate, w->up,   w->s_gate, w->s_up, c.blocks, c.n_blocks, c.perm, c.topk_w,
           c.h,      c.y_acc, c.hdr,   c.T,       c.D,     c.E,      c.k,        c.I,    c.max_blocks,
           (long long)c.opt.test_wait_cycles};
  WtMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const auto U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  bool ok = make_tmap_2d(&maps.c0, U32, 4, w->gate.codes, uint64_t(c.E) * c.I, c.D / 8, 8, 64, NOSW) &&
            make_tmap_2d(&maps.c1, U32, 4, w->up.codes, uint64_t(c.E) * c.I, c.D / 8, 8, 64, NOSW) &&
            make_tmap_2d(&maps.cs0, U32, 4, w->s_gate.codes, c.I, c.D / 8, 8, 64, NOSW) &&
            make_tmap_2d(&maps.cs1, U32, 4, w->s_up.codes, c.I, c.D / 8, 8, 64, NOSW);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t err = c.yacc_zeroed ? cudaSuccess : zero_yacc(c);
  if (err != cudaSuccess) return err;
  const int grid1 = std::max(1, std::min(num_sms(), c.max_blocks * (c.I / 64)));
  if ((err = launch_pdl(c, gemm_wt_kernel<true, C>, dim3(grid1), dim3(C::kNumThreads), C::kSmemBytes, a, maps)) !=
      cudaSuccess)
    return err;
  launch_done(c, "gateup_tc");

  a.m0 = w->down;
  a.s0 = w->s_down;
  std::memset(&maps, 0, sizeof(maps));
  ok = make_tmap_2d(&maps.c0, U32, 4, w->down.codes, uint64_t(c.E) * c.D, c.I / 8, 8, WM, NOSW) &&
       make_tmap_2d(&maps.cs0, U32, 4, w->s_down.codes, c.D, c.I / 8, 8, WM, NOSW) &&
       make_tmap_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.h, uint64_t(A + c.T), c.I, WK, C::kMaxN,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  const int grid2 = std::max(1, std::min(num_sms(), c.max_blocks * (c.D / WM)));
  if ((err = launch_pdl(c, gemm_wt_kernel<false, C>, dim3(grid2), dim3(C::kNumThreads), C::kSmemBytes, a, maps)) !=
      cudaSuccess)
    return err;
  launch_done(c, "down_tc");
  return cast_y(c);
}

// Pipeline stages of 128 of K per tile of each GEMM (D for gate/up, I for
// down) divide evenly among the warp sets, so that every A stage and every
// code slot is always filled by the same set (one set alone when a tile has
// a single stage): no parity wait can then run two phases ahead.
bool stages_fit_sets(const Ctx& c, int sets) {
  for (const int K : {c.D, c.I}) {
    const int kt = K / (WK * kGroupsPerStage);
    if (kt % sets != 0 && kt != 1) return false;
  }
  return true;
}

}  // namespace

bool gemm_wt_supported(const Ctx& c) {
  // the gather addresses x with 32-bit byte offsets
  return c.I % (WK * kGroupsPerStage) == 0 && c.D % WM == 0 && c.D % (WK * kGroupsPerStage) == 0 &&
         size_t(c.T) * c.D * 2 <= 0xFFFFFFFFu && stages_fit_sets(c, WtLarge::kAStages) && tmap_encoder_available();
}

bool gemm_wt_small_supported(const Ctx& c) {
  // a tile's scale and bias rows (8 K bytes for gate/up, 4 K for down) fit a
  // 16 KB slot, and their rows start 16-byte aligned (K % 512 == 0)
  return gemm_wt_supported(c) && stages_fit_sets(c, WtSmall::kAStages) && c.D % 512 == 0 && c.I % 512 == 0 &&
         8u * c.D <= WtSmall::kSbBytes && 4u * c.I <= WtSmall::kSbBytes;
}

cudaError_t gemm_wt(const Ctx& c) {
  if (c.BM <= WtSmall::kMaxN && gemm_wt_small_supported(c)) return gemm_wt_run<WtSmall>(c);
  return gemm_wt_run<WtLarge>(c);
}

}  // namespace moe
