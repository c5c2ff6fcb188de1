// C ABI of the 4-bit MoE layer: argument checks, workspace layout, path
// selection and launch bookkeeping. Every step of the layer runs in this
// library's kernels on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kDefaultBlockM = 128;

Options g_opt;         // process-wide options, under g_opt_mu
std::mutex g_opt_mu;
std::mutex g_mu;       // kernel-timing marks

thread_local int t_launches = 0;

// Kernel timing: events recorded in stream order; consecutive pairs give
// each kernel's device time.
struct Mark {
  const char* name;  // nullptr = start of a forward
  cudaEvent_t ev;
};
std::vector<Mark> g_marks;
std::vector<cudaEvent_t> g_free_events;

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void mark(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t e = take_event();
  if (!e) return;
  cudaEventRecord(e, s);
  g_marks.push_back({name, e});
}

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

struct Layout {
  int BM, max_blocks, n_chunks;
  size_t logits, topk_idx, topk_w, count, off, perm, inv, chunk, blocks, n_blocks, h, y_acc, xperm, total;
};

Layout layout(const moe_weights* w, int T) {
  Layout L{};
  const size_t A = size_t(T) * w->k;
  L.BM = kDefaultBlockM;
  L.n_chunks = (T + kChunkTokens - 1) / kChunkTokens;
  // room for the smallest block size any path or option can use
  L.max_blocks = int(A / kMinBlockM + std::min<size_t>(w->E, A) + (T + kMinBlockM - 1) / kMinBlockM + 1);
  size_t o = sizeof(WsHeader);
  auto put = [&](size_t bytes) {
    const size_t at = o;
    o = al256(o + bytes);
    return at;
  };
  L.logits = put(size_t(T) * w->E * 4);
  L.topk_idx = put(A * 4);
  L.topk_w = put(A * 4);
  L.count = put(size_t(w->E) * 4);
  L.off = put(size_t(w->E + 1) * 4);
  L.perm = put(A * 4);
  L.inv = put(A * 4);
  L.chunk = put(size_t(L.n_chunks) * w->E * 4);
  L.blocks = put(size_t(L.max_blocks) * 3 * 4);
  L.n_blocks = put(4);
  L.h = put((A + T) * size_t(w->I) * 2);
  L.y_acc = put(size_t(T) * w->D * 4);
  L.xperm = put(size_t(T) * w->D * 2);
  L.total = o;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status check_qmat(const moe_qmatrix& m) {
  if (!m.codes || !m.scales || !m.biases) return MOE_ERR_ARG;
  if (!aligned16(m.codes) || !aligned16(m.scales) || !aligned16(m.biases)) return MOE_ERR_ARG;
  return MOE_OK;
}

}  // namespace

moe_status check_weights(const moe_weights* w) {
  if (!w) return MOE_ERR_ARG;
  if (w->D < 64 || w->D > 16384 || w->D % 64 || w->I < 64 || w->I > 4096 || w->I % 64) return MOE_ERR_SHAPE;
  if (w->k < 1 || w->k > 32 || w->E < w->k || w->E > 1024) return MOE_ERR_SHAPE;
  if (!w->router_w || !aligned16(w->router_w)) return MOE_ERR_ARG;
  const moe_qmatrix* ms[] = {&w->gate, &w->up, &w->down, &w->s_gate, &w->s_up, &w->s_down};
  for (const moe_qmatrix* m : ms)
    if (moe_status s = check_qmat(*m)) return s;
  return MOE_OK;
}

constexpr int kMaxT = kMaxTokens;

int pass_tokens(int T, const Options& o) { return (o.chunk_tokens > 0 && T > o.chunk_tokens) ? o.chunk_tokens : T; }

size_t pass_workspace_bytes(const moe_weights* w, int T) { return layout(w, T).total; }

void reset_launch_count() { t_launches = 0; }

namespace {

moe_status make_ctx(const moe_weights* w, const uint16_t* x, int T, uint16_t* y, void* ws, size_t ws_bytes,
                    void* stream, const Options& opt, Ctx* c) {
  if (moe_status s = check_weights(w)) return s;
  if (T < 0 || T > kMaxT) return MOE_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_WORKSPACE;
  const Layout L = layout(w, T);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  c->opt = opt;
  c->w = w;
  c->T = T;
  c->D = w->D;
  c->E = w->E;
  c->k = w->k;
  c->I = w->I;
  c->BM = L.BM;
  c->max_blocks = L.max_blocks;
  c->n_chunks = L.n_chunks;
  c->x = x;
  c->y = y;
  c->hdr = reinterpret_cast<WsHeader*>(base);
  c->logits = reinterpret_cast<float*>(base + L.logits);
  c->topk_idx = reinterpret_cast<int32_t*>(base + L.topk_idx);
  c->topk_w = reinterpret_cast<float*>(base + L.topk_w);
  c->count = reinterpret_cast<int32_t*>(base + L.count);
  c->off = reinterpret_cast<int32_t*>(base + L.off);
  c->perm = reinterpret_cast<int32_t*>(base + L.perm);
  c->inv = reinterpret_cast<int32_t*>(base + L.inv);
  c->chunk = reinterpret_cast<int32_t*>(base + L.chunk);
  c->blocks = reinterpret_cast<int32_t*>(base + L.blocks);
  c->n_blocks = reinterpret_cast<int32_t*>(base + L.n_blocks);
  c->h = reinterpret_cast<uint16_t*>(base + L.h);
  c->y_acc = reinterpret_cast<float*>(base + L.y_acc);
  c->xperm = nullptr;  // set by the path that reads it
  c->stream = static_cast<cudaStream_t>(stream);
  c->xperm_area = reinterpret_cast<uint16_t*>(base + L.xperm);
  return MOE_OK;
}

void fill_view(const Ctx& c, moe_route_view* v) {
  v->T = c.T;
  v->block_m = c.BM;
  v->max_blocks = c.max_blocks;
  v->logits = c.logits;
  v->topk_idx = c.topk_idx;
  v->topk_w = c.topk_w;
  v->count = c.count;
  v->off = c.off;
  v->perm = c.perm;
  v->inv = c.inv;
  v->blocks = c.blocks;
  v->n_blocks = c.n_blocks;
  v->h = c.h;
  v->y_acc = c.y_acc;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

enum class Path { DecodeFused, DecodeItems, DecodeRows, Gemv, GemmWt, GemmTc, GemmSimt };

// Chooses the expert path for this call and the block-map row count it
// consumes: 192 tokens per block for the tensor-core GEMM with weights in
// tensor memory, 128 for the others.
Path plan(Ctx& c) {
  const Options& o = c.opt;
  int path = o.force_path;
  if (path == 0) path = (c.T <= o.gemv_max_rows) ? 1 : 2;
  Path p;
  if (path == 1 && o.decode_fused && c.T == 1 && decode_fused_supported(c))
    p = Path::DecodeFused;
  else if (path == 1 && o.decode_fused && c.T > 1 && decode_items_supported(c))
    p = Path::DecodeItems;
  else if (path == 1 && o.decode_fused && c.T > 1 && decode_rows_supported(c))
    p = Path::DecodeRows;
  else if (path == 1 && gemv_supported(c))
    p = Path::Gemv;
  else if (o.gemm_impl == 0 && gemm_wt_supported(c))
    p = Path::GemmWt;
  else if (o.gemm_impl == 2 && gemm_tc_supported(c))
    p = Path::GemmTc;
  else
    p = Path::GemmSimt;
  int path_bm = (p == Path::GemmWt) ? kWtBlockRows : (p == Path::GemmTc) ? kTcBlockRows : kDefaultBlockM;
  // few rows per expert (at most 32 on average): the tensor-memory GEMM's
  // small-block shape, whose tiles keep four weight stages in flight
  if (p == Path::GemmWt && size_t(c.T) * c.k <= size_t(32) * c.E && gemm_wt_small_supported(c))
    path_bm = kWtSmallBlockRows;
  c.BM = o.block_m > 0 ? std::min(o.block_m, path_bm) : path_bm;
  return p;
}

}  // namespace

bool ensure_smem_limit(const void* func, int bytes) {
  struct Entry {
    const void* f;
    int dev;
    int bytes;
  };
  static std::vector<Entry> done;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : done)
    if (e.f == func && e.dev == dev && e.bytes >= bytes) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.push_back({func, dev, bytes});
  return true;
}

void launch_done(const Ctx& c, const char* name) {
  ++t_launches;
  if (c.opt.kernel_timing) mark(name, c.stream);
}

void timing_begin(const Ctx& c) {
  if (c.opt.kernel_timing) mark(nullptr, c.stream);
}

Options options_snapshot() {
  std::lock_guard<std::mutex> lk(g_opt_mu);
  return g_opt;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_weights* w, int T) {
  if (check_weights(w) != MOE_OK || T < 0 || T > kMaxT) return 0;
  return layout(w, pass_tokens(T, options_snapshot())).total;
}

size_t moe_host_staging_size(const moe_weights* w, int T) {
  if (check_weights(w) != MOE_OK || T < 0 || T > kMaxT) return 0;
  return 2 * al256(size_t(pass_tokens(T, options_snapshot())) * w->D * 2);
}

moe_status moe_route(const moe_weights* w, const uint16_t* x, int T, void* workspace, size_t workspace_bytes,
                     void* stream, moe_route_view* view) {
  Ctx c;
  if (moe_status s = make_ctx(w, x, T, nullptr, workspace, workspace_bytes, stream, options_snapshot(), &c))
    return s;
  if (T > 0 && (!x || !aligned16(x))) return MOE_ERR_ARG;
  t_launches = 0;
  plan(c);
  if (view) fill_view(c, view);
  if (T == 0) return MOE_OK;
  timing_begin(c);
  return cuda_status(route(c));
}

moe_status moe_workspace_view(const moe_weights* w, int T, void* workspace, size_t workspace_bytes,
                              moe_route_view* view) {
  Ctx c;
  if (!view) return MOE_ERR_ARG;
  if (moe_status s = make_ctx(w, nullptr, T, nullptr, workspace, workspace_bytes, nullptr, options_snapshot(), &c))
    return s;
  plan(c);
  fill_view(c, view);
  return MOE_OK;
}

// One pass of the layer over T tokens (T no larger than the workspace was
// laid out for). Adds its launches to the thread's count.
// With n_x_slices > 0, x arrives on another stream in slices (see Ctx).
// first_pass: the pass's first kernel starts the call's device status afresh
// (later passes keep what earlier ones recorded).
static moe_status forward_pass(const moe_weights* w, const uint16_t* x, int T, uint16_t* y, void* workspace,
                               size_t workspace_bytes, void* stream, const Options& opt, bool first_pass,
                               int n_x_slices = 0, const int* x_slice_end = nullptr,
                               const cudaEvent_t* x_ready = nullptr, const ExpandedWeights* wexp = nullptr) {
  Ctx c;
  if (moe_status s = make_ctx(w, x, T, y, workspace, workspace_bytes, stream, opt, &c)) return s;
  if (T == 0) return MOE_OK;
  c.first_pass = first_pass;
  c.n_x_slices = n_x_slices;
  c.x_slice_end = x_slice_end;
  c.x_ready = x_ready;
  Path path = plan(c);
  if (wexp) {  // the unfused form: always the shared-memory tensor-core GEMMs
    if (!gemm_tc_supported(c)) return MOE_ERR_ARG;
    path = Path::GemmTc;
    c.BM = c.opt.block_m > 0 ? std::min(c.opt.block_m, kTcBlockRows) : kTcBlockRows;
    c.wexp = *wexp;
  }
  if (path == Path::GemmWt) c.xperm = c.xperm_area;  // the router writes the paired-order x it gathers
  timing_begin(c);
  if (path == Path::DecodeFused || path == Path::DecodeItems || path == Path::DecodeRows) {  // routing included
    if (wait_x(c) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(path == Path::DecodeFused   ? decode_fused(c)
                       : path == Path::DecodeItems ? decode_items(c)
                                                   : decode_rows(c));
  }
  cudaError_t err = route(c, path == Path::Gemv ? nullptr : &c.yacc_zeroed);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  if (c.opt.host_sync_routing) {
    // the host-scheduled variant: the block count comes back to the host
    // before the expert kernels are launched (a stream synchronisation)
    static thread_local int* nb_host = nullptr;
    if (!nb_host && cudaMallocHost(&nb_host, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(nb_host, c.n_blocks, sizeof(int), cudaMemcpyDeviceToHost, c.stream) != cudaSuccess ||
        cudaStreamSynchronize(c.stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (*nb_host < 0 || *nb_host > c.max_blocks) return MOE_ERR_CUDA;
  }
  if (path == Path::Gemv) return cuda_status(gemv(c));
  if (c.wexp.gate && expand_weights(c) != cudaSuccess) return MOE_ERR_CUDA;
  if (path == Path::GemmWt) return cuda_status(gemm_wt(c));
  if (path == Path::GemmTc) return cuda_status(gemm_tc(c));
  return cuda_status(gemm_simt(c));
}

}  // extern "C"

moe_status moe::forward_passes(const moe_weights* w, const uint16_t* x, int T, uint16_t* y, void* workspace,
                               size_t workspace_bytes, void* stream, int step, const Options& opt,
                               const ExpandedWeights* wexp) {
  t_launches = 0;
  if (T == 0) return forward_pass(w, x, 0, y, workspace, workspace_bytes, stream, opt, true);  // checks the workspace
  if (!x || !y || !aligned16(x) || !aligned16(y) || x == y || step < 1) return MOE_ERR_ARG;
  for (int t0 = 0; t0 < T; t0 += step) {
    const int n = std::min(step, T - t0);
    const size_t at = size_t(t0) * w->D;
    if (moe_status s = forward_pass(w, x + at, n, y + at, workspace, workspace_bytes, stream, opt, t0 == 0, 0,
                                    nullptr, nullptr, wexp))
      return s;
  }
  return MOE_OK;
}

extern "C" {

// Prompt chunking ("Optimizing on-device inference for Apple Silicon",
// section "Bound temporary memory with prompt chunking"): T above the chunk
// size runs as consecutive passes over bounded token ranges on the caller's
// stream, all reusing one workspace sized for a single pass. Tokens are
// independent in this layer, so the output is the one pass's output.
moe_status moe_layer_forward(const moe_weights* w, const uint16_t* x, int T, uint16_t* y, void* workspace,
                             size_t workspace_bytes, void* stream) {
  const Options opt = options_snapshot();
  if (moe_status s = check_weights(w)) return s;
  if (T < 0 || T > kMaxT) return MOE_ERR_ARG;
  return forward_passes(w, x, T, y, workspace, workspace_bytes, stream, pass_tokens(T, opt), opt);
}

size_t moe_expanded_weights_bytes(const moe_weights* w) {
  if (check_weights(w) != MOE_OK) return 0;
  return expanded_weights(w, nullptr).bytes;
}

// The unfused design ("Optimizing on-device inference for Apple Silicon",
// section "Dequantise weights during matrix multiplication", which measures
// fusing the two): routing, a pass that expands the weights of every
// selected expert and of the shared expert to bf16 in `wbuf`, then grouped
// GEMMs that read those bf16 weights.
moe_status moe_layer_forward_expanded(const moe_weights* w, const uint16_t* x, int T, uint16_t* y, void* workspace,
                                      size_t workspace_bytes, void* wbuf, size_t wbuf_bytes, void* stream) {
  const Options opt = options_snapshot();
  if (moe_status s = check_weights(w)) return s;
  if (T < 0 || T > kMaxT) return MOE_ERR_ARG;
  const ExpandedWeights ex = expanded_weights(w, wbuf);
  if (T > 0 && (!wbuf || (reinterpret_cast<uintptr_t>(wbuf) & 255) != 0 || wbuf_bytes < ex.bytes)) return MOE_ERR_ARG;
  return forward_passes(w, x, T, y, workspace, workspace_bytes, stream, pass_tokens(T, opt), opt, &ex);
}

// The host entry point's copy stream and events, one set per thread and
// device, created on first use and kept for the life of the process.
constexpr int kHostSlices = 16;  // x goes in as up to this many slices
struct HostPipe {
  int device = -1;
  cudaStream_t copy = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t ready[kHostSlices] = {};
};

static HostPipe* host_pipe() {
  static thread_local HostPipe pipes[8];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  for (HostPipe& p : pipes) {
    if (p.device == dev) return &p;
    if (p.device >= 0) continue;
    if (cudaStreamCreateWithFlags(&p.copy, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    for (cudaEvent_t& e : p.ready)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    p.device = dev;
    return &p;
  }
  return nullptr;
}

moe_status moe_layer_forward_host(const moe_weights* w, const uint16_t* x_host, int T, uint16_t* y_host,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const Options opt = options_snapshot();
  if (check_weights(w) != MOE_OK) return check_weights(w);
  if (T < 0 || T > kMaxT) return MOE_ERR_ARG;
  t_launches = 0;
  if (T == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_ARG;
  // one pass's tokens are staged at a time: x in, the layer, y out
  const int step = pass_tokens(T, opt);
  const size_t need = layout(w, step).total, stage = al256(size_t(step) * w->D * 2);
  if (!workspace || workspace_bytes < need + 2 * stage) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(workspace);
  uint16_t* xd = reinterpret_cast<uint16_t*>(base + need);
  uint16_t* yd = reinterpret_cast<uint16_t*>(base + need + stage);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  HostPipe* hp = host_pipe();
  if (!hp) return MOE_ERR_CUDA;
  // page-locked y that this device can address is written by the layer's
  // last kernel directly (no staging, no copy back)
  uint16_t* y_direct = nullptr;
  {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, y_host) == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer &&
        aligned16(pa.devicePointer))
      y_direct = static_cast<uint16_t*>(pa.devicePointer);
    else
      cudaGetLastError();  // an unregistered pointer is not an error here
  }
  for (int t0 = 0; t0 < T; t0 += step) {
    const int n = std::min(step, T - t0);
    const size_t at = size_t(t0) * w->D;
    // x goes in on the copy stream, in slices, once the stream's earlier work
    // (which may still read the staging buffer) is done; the router starts
    // on each slice as it lands, and the copy overlaps it
    // slices of whole router waves, so each router launch fills the GPU
    const int wave = router_wave_tokens(w->E);
    const int per = wave * std::max(1, (n + kHostSlices * wave - 1) / (kHostSlices * wave));
    const int n_sl = (n + per - 1) / per;
    int end[kHostSlices];
    for (int i = 0; i < n_sl; ++i) end[i] = std::min(n, per * (i + 1));
    if (cudaEventRecord(hp->start, s) != cudaSuccess || cudaStreamWaitEvent(hp->copy, hp->start, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    for (int i = 0, r0 = 0; i < n_sl; r0 = end[i], ++i) {
      const size_t bytes = size_t(end[i] - r0) * w->D * 2;
      if (bytes && cudaMemcpyAsync(xd + size_t(r0) * w->D, x_host + at + size_t(r0) * w->D, bytes,
                                   cudaMemcpyHostToDevice, hp->copy) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (cudaEventRecord(hp->ready[i], hp->copy) != cudaSuccess) return MOE_ERR_CUDA;
    }
    moe_status st = forward_pass(w, xd, n, y_direct ? y_direct + at : yd, workspace, need, stream, opt, t0 == 0,
                                 n_sl, end, hp->ready);
    if (st != MOE_OK) {
      cudaStreamSynchronize(hp->copy);  // no copy into the workspace outlives the call
      return st;
    }
    if (!y_direct &&
        cudaMemcpyAsync(y_host + at, yd, size_t(n) * w->D * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_get_device_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (h.status != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpy(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return static_cast<moe_status>(h.status);
}

moe_status moe_set_option(int option, int value) {
  std::lock_guard<std::mutex> lk(g_opt_mu);
  switch (option) {
    case MOE_OPT_GEMV_MAX_ROWS:
      if (value < 0 || value > 8) return MOE_ERR_ARG;
      g_opt.gemv_max_rows = value;
      return MOE_OK;
    case MOE_OPT_FORCE_PATH:
      if (value < 0 || value > 2) return MOE_ERR_ARG;
      g_opt.force_path = value;
      return MOE_OK;
    case MOE_OPT_KERNEL_TIMING:
      if (value < 0 || value > 1) return MOE_ERR_ARG;
      g_opt.kernel_timing = value;
      return MOE_OK;
    case MOE_OPT_GEMM_IMPL:
      if (value < 0 || value > 2) return MOE_ERR_ARG;
      g_opt.gemm_impl = value;
      return MOE_OK;
    case MOE_OPT_DECODE_FUSED:
      if (value < 0 || value > 1) return MOE_ERR_ARG;
      g_opt.decode_fused = value;
      return MOE_OK;
    case MOE_OPT_BLOCK_M:
      if (value != 0 && (value < kMinBlockM || value > kWtBlockRows || value % 16 != 0)) return MOE_ERR_ARG;
      g_opt.block_m = value;
      return MOE_OK;
    case MOE_OPT_CHUNK_TOKENS:
      if (value < 0 || value > kMaxT) return MOE_ERR_ARG;
      g_opt.chunk_tokens = value;
      return MOE_OK;
    case MOE_OPT_HOST_SYNC_ROUTING:
      if (value < 0 || value > 1) return MOE_ERR_ARG;
      g_opt.host_sync_routing = value;
      return MOE_OK;
    case MOE_OPT_TEST_WAIT_CYCLES:
      if (value < 0) return MOE_ERR_ARG;
      g_opt.test_wait_cycles = value;
      return MOE_OK;
    default:
      return MOE_ERR_ARG;
  }
}

int moe_get_option(int option) {
  std::lock_guard<std::mutex> lk(g_opt_mu);
  switch (option) {
    case MOE_OPT_GEMV_MAX_ROWS: return g_opt.gemv_max_rows;
    case MOE_OPT_FORCE_PATH: return g_opt.force_path;
    case MOE_OPT_KERNEL_TIMING: return g_opt.kernel_timing;
    case MOE_OPT_GEMM_IMPL: return g_opt.gemm_impl;
    case MOE_OPT_TEST_WAIT_CYCLES: return g_opt.test_wait_cycles;
    case MOE_OPT_BLOCK_M: return g_opt.block_m;
    case MOE_OPT_DECODE_FUSED: return g_opt.decode_fused;
    case MOE_OPT_CHUNK_TOKENS: return g_opt.chunk_tokens;
    case MOE_OPT_HOST_SYNC_ROUTING: return g_opt.host_sync_routing;
    default: return -1;
  }
}

moe_status moe_kernel_times(const char** names, float* total_ms, int* launches, int max, int* n) {
  if (!n || max < 0 || (max > 0 && (!names || !total_ms || !launches))) return MOE_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  *n = 0;
  if (!g_marks.empty() && cudaEventSynchronize(g_marks.back().ev) != cudaSuccess) return MOE_ERR_CUDA;
  for (size_t i = 1; i < g_marks.size(); ++i) {
    if (!g_marks[i].name) continue;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_marks[i - 1].ev, g_marks[i].ev) != cudaSuccess) return MOE_ERR_CUDA;
    int slot = -1;
    for (int j = 0; j < *n; ++j)
      if (std::strcmp(names[j], g_marks[i].name) == 0) slot = j;
    if (slot < 0) {
      if (*n >= max) continue;
      slot = (*n)++;
      names[slot] = g_marks[i].name;
      total_ms[slot] = 0.f;
      launches[slot] = 0;
    }
    total_ms[slot] += ms;
    launches[slot] += 1;
  }
  for (const Mark& m : g_marks) g_free_events.push_back(m.ev);
  g_marks.clear();
  return MOE_OK;
}

moe_status moe_debug_dequant(const moe_qmatrix* m, int expert, int rows, int K, uint16_t* out, void* stream) {
  if (!m || !out || !m->codes || !m->scales || !m->biases) return MOE_ERR_ARG;
  if (expert < 0 || rows < 1 || K < 64 || K % 64) return MOE_ERR_SHAPE;
  return cuda_status(debug_dequant(m, expert, rows, K, out, static_cast<cudaStream_t>(stream)));
}

int moe_last_launch_count(void) { return t_launches; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

}  // extern "C"
