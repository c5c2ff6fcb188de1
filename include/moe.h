/* moe.h — C ABI of the GB300 4-bit mixture-of-experts FFN layer.
 *
 * The layer (from "Optimizing on-device inference for Apple Silicon",
 * Perplexity 2026, sections "Qwen creates three workload shapes",
 * "Dequantise weights during matrix multiplication", "Keep expert routing on
 * the GPU", "Optimise the single-row weight path" and "Reduce intermediate and
 * state traffic"):
 *
 *   logits[t,e] = x[t,:] . W_r[e,:] (+ bias[e])                     fp32
 *   top-k experts of each token (larger logit first, lower index on ties),
 *   weights w[t,j] = softmax over all E, renormalised over the k kept
 *   h = silu(x . dq(W_gate[e])^T) * (x . dq(W_up[e])^T)               bf16
 *   y[t] = sum_j w[t,j] * (h . dq(W_down[e_j])^T) + shared expert     bf16
 *
 * where dq(W)[n,kk] = scale[n,kk/64] * code[n,kk] + bias[n,kk/64]: 4-bit
 * codes, one bf16 scale and one bf16 bias per group of 64 weights along each
 * matrix's input axis.
 *
 * Conventions for every entry point:
 *   - Row-major arrays. bf16 values travel as their uint16_t bit patterns.
 *   - "device" pointers are CUDA device memory owned by the caller; the
 *     library never frees or retains them past the call (work is enqueued on
 *     the caller's stream and may still be running when the call returns).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Nothing throws across the ABI. Argument and shape errors are found on
 *     the host before anything is enqueued and return MOE_ERR_ARG /
 *     MOE_ERR_SHAPE / MOE_ERR_WORKSPACE. Launch failures return MOE_ERR_CUDA.
 *     Errors found by the kernels themselves (bounded waits that gave up,
 *     index checks) are recorded in a status word inside the workspace and
 *     reported by moe_get_device_status().
 *   - Not re-entrant on one workspace: two calls that overlap on the GPU must
 *     use distinct workspaces. Distinct workspaces and streams are
 *     independent. Options (moe_set_option) are process-wide; each call
 *     takes a copy of them when it starts, so a moe_set_option from another
 *     thread never changes a call part-way (it applies from the next call).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,            /* null pointer, bad option, negative T */
  MOE_ERR_SHAPE = 2,          /* D, I not multiples of 64; k, E out of range */
  MOE_ERR_WORKSPACE = 3,      /* workspace NULL, too small or not 256-byte aligned */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up */
  MOE_ERR_DEVICE_CHECK = 6    /* a device-side index/size check failed */
} moe_status;

/* One packed 4-bit matrix family of n_exp experts, each rows x K:
 *   codes  [n_exp, rows, K/8] uint32; code j (0..7) of word m is bits
 *          4j..4j+3 and holds element 8m+j of the row;
 *   scales [n_exp, rows, K/64] bf16, biases the same: group g of a row covers
 *          elements 64g..64g+63 (the matrix's input axis).
 * All three are device pointers, 16-byte aligned. */
typedef struct {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} moe_qmatrix;

/* The layer's weights (all device pointers, caller-owned).
 *   D hidden size, E routed experts, k experts kept per token, I expert
 *   intermediate size. Requirements: D % 64 == 0, I % 64 == 0 (one quant
 *   group is 64), 64 <= D <= 16384, 64 <= I <= 4096, 1 <= k <= E <= 1024,
 *   k <= 32.
 *   router_w    fp32 [E, D]
 *   router_bias fp32 [E] or NULL (added to the logits; NULL = no bias)
 *   gate, up    [E, I, D] (input axis D)      down   [E, D, I] (input axis I)
 *   s_gate, s_up [1, I, D]  s_down [1, D, I]   the shared expert, weight 1 */
typedef struct {
  int D, E, k, I;
  const float* router_w;
  const float* router_bias;
  moe_qmatrix gate, up, down;
  moe_qmatrix s_gate, s_up, s_down;
} moe_weights;

/* Device pointers into a workspace after moe_route()/moe_layer_forward(),
 * for inspection (tests, diagnostics). Valid until the workspace is reused.
 *   logits    fp32 [T, E]
 *   topk_idx  int32 [T, k]     topk_w fp32 [T, k]
 *   count     int32 [E]        off    int32 [E+1] exclusive scan of count
 *   perm      int32 [T*k]      row p of the permuted order holds assignment
 *                              a = t*k + j; inside an expert's segment rows
 *                              are in ascending a
 *   inv       int32 [T*k]      inv[perm[p]] = p
 *   blocks    int32 [max_blocks][3] = (group, first row, rows): for each
 *             expert in ascending order its segment cut into blocks of
 *             block_m rows (192 on the default tensor-core GEMM path, 128
 *             otherwise), then the shared expert as group E over rows
 *             T*k .. T*k+T-1 (token t at row T*k+t)
 *   n_blocks  int32 [1]        number of valid entries of blocks
 *   h         bf16 [T*k + T, I]  SwiGLU intermediate in the permuted order
 *                                (the shared expert's rows last)
 *   y_acc     fp32 [T, D]      the combine accumulator (GEMM path) */
typedef struct {
  int T, block_m, max_blocks;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* count;
  int32_t* off;
  int32_t* perm;
  int32_t* inv;
  int32_t* blocks;
  int32_t* n_blocks;
  uint16_t* h;
  float* y_acc;
} moe_route_view;

/* Options (process-wide). */
typedef enum {
  MOE_OPT_GEMV_MAX_ROWS = 1, /* T <= this runs the decode GEMV path (0..8; default 4:
                                on the D=2048, E=256, k=8, I=512 layer the one-launch
                                item kernel measured faster than the grouped GEMM at
                                2, 3 and 4 rows, and slower at 5 and 8) */
  MOE_OPT_FORCE_PATH = 2,    /* 0 auto by row count, 1 GEMV, 2 grouped GEMM */
  MOE_OPT_KERNEL_TIMING = 3, /* 1: record CUDA events around each kernel of
                                the next forwards (read with moe_kernel_times) */
  MOE_OPT_GEMM_IMPL = 4,     /* grouped GEMM used above the GEMV threshold:
                                0 tensor cores (tcgen05) with the dequantised weights
                                  in tensor memory (default),
                                1 CUDA cores (the comparison baseline),
                                2 tensor cores with the dequantised weights in
                                  shared memory */
  MOE_OPT_TEST_WAIT_CYCLES = 5, /* test hook: > 0 makes the tensor-core epilogue
                                first wait, for at most this many cycles, on a
                                barrier that nothing arrives on, so the
                                bounded-wait failure path (status
                                MOE_ERR_DEVICE_TIMEOUT, drain, clean exit) runs;
                                0 (the default) turns the hook off */
  MOE_OPT_BLOCK_M = 6,       /* rows per block-map entry (the grouped GEMMs' token
                                tile): 0 (default) uses the path's own size,
                                192 on the tensor-memory path and 128 on the
                                others; 16..192 in steps of 16 is clamped to
                                the path's size. The workspace always has
                                room for 16-row blocks. */
  MOE_OPT_DECODE_FUSED = 7,  /* 1 (default): a forward on the GEMV path (1 to 8
                                rows) runs the router logits, top-k, gate/up and
                                down in one cooperative kernel, when the device
                                can hold all its CTAs at once and the shape fits
                                its shared memory; 0: the separate routing and
                                GEMV kernels */
  MOE_OPT_CHUNK_TOKENS = 8,  /* prompt chunking ("Optimizing on-device inference
                                for Apple Silicon", "Bound temporary memory with
                                prompt chunking"): a forward with more tokens
                                than this runs as consecutive passes of at most
                                this many tokens that reuse one workspace, so
                                the workspace (and the host-entry staging) is
                                sized for one pass. Default 8192; 0 turns it
                                off (one pass over all T). Tokens are
                                independent, so the output does not change. Set
                                it before sizing the workspace. */
  MOE_OPT_HOST_SYNC_ROUTING = 9 /* 1: the host-scheduled routing variant ("Keep
                                expert routing on the GPU" describes it as the
                                design that section replaces): after routing,
                                each pass copies the expert block count to the
                                host and synchronises the stream before the
                                expert kernels are launched. The output is
                                unchanged; the call blocks. For measurement.
                                0 (default): no host synchronisation. */
} moe_option;

/* Bytes of workspace one call with T tokens needs (pure host; 0 on bad
 * arguments): the tables and buffers of one pass of min(T, chunk tokens)
 * tokens (MOE_OPT_CHUNK_TOKENS), so it stops growing at the chunk size. The
 * workspace also holds the device status word. The buffers are the routing
 * tables of "Keep expert routing on the GPU" (logits, top-k, counts, offsets,
 * permutation, block map), the intermediate of "Reduce intermediate and
 * state traffic" and the one-pass bound of "Bound temporary memory with
 * prompt chunking" ("Optimizing on-device inference for Apple Silicon"). */
size_t moe_workspace_size(const moe_weights* w, int T);

/* The whole layer on the GPU ("Optimizing on-device inference for Apple
 * Silicon": the routed and shared experts of "Qwen creates three workload
 * shapes", the routing of "Keep expert routing on the GPU", the fused
 * dequantising matrix kernels of "Dequantise weights during matrix
 * multiplication" for many rows and the single-row path of "Optimise the
 * single-row weight path" for few, with the row-count switch of "Why
 * continuous batching halved LLM throughput on an M2 Mac mini"): routing
 * (logits, top-k, weights, histogram, scan, scatter, block map), then either
 * the grouped-GEMM path or the decode GEMV path, then the combine into y.
 * Everything is enqueued on `stream` with no host synchronisation.
 * x: device bf16 [T, D]; y: device bf16 [T, D] (may not alias x); workspace:
 * device, >= moe_workspace_size(w, T) bytes, 256-byte aligned. T = 0 is a
 * no-op returning MOE_OK. */
moe_status moe_layer_forward(const moe_weights* w, const uint16_t* x, int T, uint16_t* y,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Same layer with HOST x and y: for each pass (chunk) copies its x rows into
 * the workspace, runs the layer, copies its y rows back; synchronises
 * `stream` before it returns. Page-locked host buffers make the copies
 * asynchronous DMA. The workspace must hold moe_workspace_size(w, T) +
 * moe_host_staging_size(w, T) (x and y staging for one pass).
 * The x rows of a pass go in as up to 16 slices on a copy stream of the
 * library's own, ordered after the work already on `stream`. A slice holds
 * the tokens of one or more whole waves of router CTAs on this GPU (608 at
 * E = 256 on 152 SMs). The router starts on each slice as it lands, so the
 * copy overlaps the router. The result is the same as with one copy. The
 * copy stream and its 17 events are created on the first call of each host
 * thread on each device and kept for the life of the process. When y_host is
 * page-locked memory this device can address (16-byte aligned), the layer's
 * last kernel writes y into it directly, with no staging and no copy back;
 * other host memory is staged and copied. */
size_t moe_host_staging_size(const moe_weights* w, int T);
moe_status moe_layer_forward_host(const moe_weights* w, const uint16_t* x_host, int T,
                                  uint16_t* y_host, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Routing only (the first five steps of the layer: the router and top-k of
 * "Qwen creates three workload shapes", then the histogram, scan, scatter and
 * block map of "Keep expert routing on the GPU", "Optimizing on-device
 * inference for Apple Silicon"), on `stream`, no host sync; fills `view`
 * with device pointers into the workspace. The tables are
 * the ones moe_layer_forward builds for the same T (same block_m). All T
 * tokens are routed in one pass: for T above the chunk size the workspace
 * must be sized with chunking off (MOE_OPT_CHUNK_TOKENS = 0), else the call
 * returns MOE_ERR_WORKSPACE. */
moe_status moe_route(const moe_weights* w, const uint16_t* x, int T, void* workspace,
                     size_t workspace_bytes, void* stream, moe_route_view* view);

/* Device pointers of the workspace arrays for T tokens without running
 * anything (e.g. to read h after moe_layer_forward). */
moe_status moe_workspace_view(const moe_weights* w, int T, void* workspace,
                              size_t workspace_bytes, moe_route_view* view);

/* Synchronises `stream`, then returns (and clears) the device status word of
 * `workspace`: MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_CHECK, the
 * first error any pass of the last call on that workspace recorded (a call
 * starts the word afresh; its later passes keep what earlier ones found). */
moe_status moe_get_device_status(void* workspace, void* stream);

moe_status moe_set_option(int option, int value);
int moe_get_option(int option);

/* With MOE_OPT_KERNEL_TIMING on, every forward records a CUDA event on its
 * stream before its first kernel and after each kernel. This call waits for
 * the last recorded event, then sums the device time of each kernel name over
 * all forwards since the previous call: up to `max` entries of (static name
 * string, total milliseconds, launches); *n gets the entry count. It then
 * forgets those events. */
moe_status moe_kernel_times(const char** names, float* total_ms, int* launches, int max, int* n);

/* Dequantises rows x K of expert `expert` of `m` into bf16 [rows, K] on the
 * device with the conversion the tensor-core GEMM uses (one round to nearest
 * even of scale*code + bias). A diagnostic of the weight format. */
moe_status moe_debug_dequant(const moe_qmatrix* m, int expert, int rows, int K, uint16_t* out,
                             void* stream);

/* The unfused design, for measuring what fusing dequantisation into the
 * GEMMs saves ("Optimizing on-device inference for Apple Silicon", section
 * "Dequantise weights during matrix multiplication", which compares a fused
 * kernel against a separate dequantisation pass plus GEMM). The layer as in
 * moe_layer_forward(), computed as: routing; a pass that expands the
 * weights of every expert that some row of the pass selected, and the
 * shared expert's, to bf16 in `wbuf` (each weight rounded once from
 * scale*code + bias, as the fused kernels round it); then the
 * shared-memory tensor-core grouped GEMMs reading those bf16 weights
 * through TMA. The output equals the fused shared-memory tensor-core path's
 * (MOE_OPT_GEMM_IMPL = 2) bit for bit.
 *   wbuf: device buffer of at least moe_expanded_weights_bytes(w) bytes,
 *   256-byte aligned, owned by the caller: [E][I][D] gate, [E][I][D] up,
 *   [E][D][I] down, then the shared expert's [I][D] gate, [I][D] up and
 *   [D][I] down, all bf16. Only selected experts' parts are written.
 *   workspace, x, y, stream, passes and T = 0: as for moe_layer_forward().
 *   Errors: MOE_ERR_ARG for a missing, unaligned or short wbuf or a shape
 *   the shared-memory GEMM does not take (I % 128 or D % 256 nonzero);
 *   otherwise as moe_layer_forward(). */
size_t moe_expanded_weights_bytes(const moe_weights* w);
moe_status moe_layer_forward_expanded(const moe_weights* w, const uint16_t* x, int T, uint16_t* y,
                                      void* workspace, size_t workspace_bytes, void* wbuf,
                                      size_t wbuf_bytes, void* stream);

/* Bytes of the library's fixed device scratch array used by
 * moe_layer_forward_static(). */
#define MOE_STATIC_SCRATCH_BYTES (8u << 20)

/* The whole layer, like moe_layer_forward(), but with no workspace argument:
 * its scratch memory is a fixed 8 MiB device array inside this library, so
 * the call allocates no device memory at all. (The source pages have no
 * counterpart; this serves callers that cannot allocate: loops that forbid
 * cudaMalloc after start-up because it can synchronise the device or fail on
 * fragmentation, and hosts that hand their plug-ins only input and output
 * buffers.)
 *   x, y, stream: as for moe_layer_forward(); the caller still owns them.
 *   T = 0 is a no-op returning MOE_OK; bad arguments are rejected on the
 *   host, before anything is enqueued, as for moe_layer_forward().
 *   Any T: the tokens run in consecutive passes of the largest count whose
 *   workspace fits MOE_STATIC_SCRATCH_BYTES (and no larger than the chunk
 *   size; for the D=2048, E=256, k=8, I=512 layer, 369 tokens). A layer whose
 *   single-token workspace does not fit returns MOE_ERR_WORKSPACE and
 *   enqueues nothing.
 *   The first call on each device looks up the array's device address (with
 *   that device current), so make that first call before any stream capture.
 *   Every call on a device shares the one array and leaves its contents
 *   behind; each call clears what must start at zero itself. Calls whose
 *   work overlaps on the GPU (unordered streams or host threads) race on the
 *   array: order them on one stream. The array occupies device memory on
 *   every GPU that loads the library, until the process exits. */
moe_status moe_layer_forward_static(const moe_weights* w, const uint16_t* x, int T, uint16_t* y,
                                    void* stream);

/* moe_get_device_status() for the scratch array of moe_layer_forward_static()
 * on the current device: synchronises `stream`, then returns and clears the
 * first device-side error any pass of the last static call recorded. */
moe_status moe_get_device_status_static(void* stream);

/* Number of this library's kernels the last forward call on this thread
 * launched (all of its passes). */
int moe_last_launch_count(void);

const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
