// Internal interface between the translation units of the MoE library.
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

struct WsHeader;

// Chunk of tokens handled by one CTA of the top-k/histogram and scatter steps.
constexpr int kChunkTokens = 64;

// Rows per block-map entry consumed by the tensor-core GEMMs.
constexpr int kTcBlockRows = 128;  // weights dequantised into shared memory (MMA M = tokens)
constexpr int kWtBlockRows = 192;  // weights dequantised into tensor memory (MMA N = tokens)
constexpr int kWtSmallBlockRows = 64;  // the same with four weight stages in flight (small blocks)
constexpr int kMinBlockM = 16;      // smallest block size MOE_OPT_BLOCK_M accepts; sizes the block map

// Library options (moe_set_option). A call works on its own copy, taken
// once when the call starts, so that another thread's moe_set_option cannot
// change a call part-way.
struct Options {
  int gemv_max_rows = 4;  // the measured small-row sweep: the item kernel faster up to 4 rows, the grouped GEMM from 5
  int force_path = 0;
  int kernel_timing = 0;
  int gemm_impl = 0;
  int test_wait_cycles = 0;
  int block_m = 0;  // 0: the path's own block size
  int decode_fused = 1;
  int chunk_tokens = 8192;  // 0: one pass over all T
  int host_sync_routing = 0;
};
Options options_snapshot();

// Every expert's weights expanded to bf16 by a separate pass before the
// GEMMs (the unfused design, kept for comparison): [E][I][D] gate and up,
// [E][D][I] down, then the shared expert's three matrices, in one buffer.
struct ExpandedWeights {
  uint16_t* gate = nullptr;  // null: the kernels dequantise on chip
  uint16_t* up = nullptr;
  uint16_t* down = nullptr;
  uint16_t* s_gate = nullptr;
  uint16_t* s_up = nullptr;
  uint16_t* s_down = nullptr;
  size_t bytes = 0;
};
ExpandedWeights expanded_weights(const moe_weights* w, void* base);

// One call's resolved sizes and device pointers.
struct Ctx {
  Options opt;      // the call's options
  bool first_pass = true;  // first pass of its call: its first kernel clears the device status
  const moe_weights* w;
  int T, D, E, k, I;
  int BM;          // rows per block-map entry
  int max_blocks;  // capacity of the block map
  int n_chunks;    // ceil(T / kChunkTokens)
  const uint16_t* x;
  uint16_t* y;
  WsHeader* hdr;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* count;
  int32_t* off;
  int32_t* perm;
  int32_t* inv;
  int32_t* chunk;  // [n_chunks][E] per-chunk counts, then per-chunk bases
  int32_t* blocks;
  int32_t* n_blocks;
  uint16_t* h;
  float* y_acc;
  // x with every 8-element chunk in the paired order (dq8_bf16_paired), written
  // by the router for the gate/up GEMM of the tensor-memory path; null when no
  // kernel of the call reads it
  uint16_t* xperm = nullptr;
  uint16_t* xperm_area = nullptr;  // its place in the workspace
  cudaStream_t stream;
  bool yacc_zeroed = false;  // set when routing already cleared y_acc
  ExpandedWeights wexp;      // set: the separate expansion pass and bf16-weight GEMMs
  // x still arriving from the host on another stream: rows before
  // x_slice_end[i] are in place once x_ready[i] has completed (the last slice
  // ends at T). The router starts on each slice as it lands; every other
  // kernel runs after all of them. n_x_slices = 0: x is ready on `stream`.
  int n_x_slices = 0;
  const int* x_slice_end = nullptr;
  const cudaEvent_t* x_ready = nullptr;
};

// Makes `c.stream` wait until all of x has arrived (no-op without slices).
cudaError_t wait_x(const Ctx& c);
// Tokens whose router tiles fill exactly one wave of CTAs on this GPU (the
// unit in which x slices are sized, so that no router launch ends in a
// partial wave).
int router_wave_tokens(int E);

// Launches `kernel` on c.stream with programmatic stream serialisation: its
// CTAs may start while the stream's previous kernel finishes, and wait
// (griddep_wait in the kernel) before reading what that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(const Ctx& c, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Bookkeeping of launches: counts this library's kernels and, when kernel
// timing is on, records an event after each one.
void launch_done(const Ctx& c, const char* name);
void timing_begin(const Ctx& c);

// Routing: logits, top-k + weights + per-chunk histogram, scan + block map,
// scatter. Returns the first CUDA error. With yacc_zeroed given, the router
// kernel may also clear y_acc for the grouped GEMM that follows; then it sets
// *yacc_zeroed.
cudaError_t route(const Ctx& c, bool* yacc_zeroed = nullptr);

// Combine accumulator: zero before, bf16 cast after the down projection.
cudaError_t zero_yacc(const Ctx& c);
cudaError_t cast_y(const Ctx& c);

// Grouped-GEMM path (T above the GEMV threshold).
cudaError_t gemm_simt(const Ctx& c);
cudaError_t gemm_tc(const Ctx& c);
bool gemm_tc_supported(const Ctx& c);
// The separate pass: the weights of every expert with rows in this pass, and
// the shared expert's, to bf16 in c.wexp.
cudaError_t expand_weights(const Ctx& c);
cudaError_t gemm_wt(const Ctx& c);
bool gemm_wt_supported(const Ctx& c);
bool gemm_wt_small_supported(const Ctx& c);
int num_sms();

// 2-D TMA tensor map over a row-major [rows, cols] array (false if the
// driver's encoder is unavailable or rejects the map).
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t elem, const void* ptr, uint64_t rows,
                  uint64_t cols, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw,
                  CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
bool tmap_encoder_available();

// Decode GEMV path (a few rows).
cudaError_t gemv(const Ctx& c);
bool gemv_supported(const Ctx& c);
// One token: router logits, top-k, gate/up and down in one cooperative
// kernel (with the header counter zeroed on the stream first).
cudaError_t decode_fused(const Ctx& c);
bool decode_fused_supported(const Ctx& c);
// Two to eight rows: the same steps in one cooperative kernel that streams
// the union of the rows' experts through shared-memory rings.
cudaError_t decode_rows(const Ctx& c);
bool decode_rows_supported(const Ctx& c);
// 2..8 rows as items of the union's experts, one grid barrier (D <= 2048)
cudaError_t decode_items(const Ctx& c);
bool decode_items_supported(const Ctx& c);
// Router logits only, for up to 16 tokens.
// With xperm, it also writes the paired-order copy of x; with yacc, it clears
// the combine accumulator [T, D].
cudaError_t route_logits_small(const Ctx& c, uint16_t* xperm = nullptr, float* yacc = nullptr);

cudaError_t debug_dequant(const moe_qmatrix* m, int expert, int rows, int K, uint16_t* out,
                          cudaStream_t s);

// Host-side checks and sizes shared by the entry points.
constexpr int kMaxTokens = 1 << 20;
moe_status check_weights(const moe_weights* w);
// Tokens of one pass of a T-token call: T, or the chunk size when chunking
// is on and T is larger.
int pass_tokens(int T, const Options& opt);
// Workspace bytes of one pass over T tokens.
size_t pass_workspace_bytes(const moe_weights* w, int T);
// Starts this thread's launch count of a call at zero.
void reset_launch_count();

// The layer over T tokens as consecutive passes of at most `pass_tokens`
// tokens, all reusing one workspace laid out for a pass (the body of the
// workspace entry points). Counts the call's launches from zero. With
// `wexp` set, every pass takes the shared-memory tensor-core GEMM path with
// the separate expansion pass (see ExpandedWeights).
moe_status forward_passes(const moe_weights* w, const uint16_t* x, int T, uint16_t* y, void* workspace,
                          size_t workspace_bytes, void* stream, int pass_tokens, const Options& opt,
                          const ExpandedWeights* wexp = nullptr);

}  // namespace moe
