// CPU oracle for the 4-bit mixture-of-experts FFN layer.
//
// TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
// benchmark's CPU-baseline leg load this library. The product path never
// calls it, and it shares no code, header or table with the CUDA sources.
//
// It is the plain definition of the layer, slow on purpose: every weight is
// dequantised exactly in fp64, every dot product accumulates in fp64 in
// index order, one token at a time. Sources, all from "Optimizing on-device
// inference for Apple Silicon" (Perplexity, 2026) unless stated:
//   * 4-bit groupwise-affine weights, 64 weights per group sharing one bf16
//     scale and one bf16 bias: section "Dequantise weights during matrix
//     multiplication" (subsection of "Prefill").
//   * 256 routed experts scored by the router, 8 kept, plus one shared expert
//     that sees every token: section "Qwen creates three workload shapes".
//   * histogram -> exclusive prefix scan -> scatter into expert groups ->
//     block map of fixed-size blocks: section "Keep expert routing on the GPU".
//   * expert = two input projections with the gated activation, then the
//     output projection combined with the routing scores and the shared
//     expert's result: section "Reduce intermediate and state traffic".
//   * bytes per parameter bits/8 + 4/64: "Laya MLX Performance-Forschung",
//     section "Quantisierung".
//
// Readings where the pages are silent (each listed in the design notes):
//   R1 code j (0..7) of a uint32 word m is bits 4j..4j+3 and is element 8m+j.
//   R2 groups run along each matrix's input (reduction) axis: D for gate/up,
//      I for down. w[n][kk] = s[n][kk/64] * q[n][kk] + b[n][kk/64].
//   R3 router logits are fp32 in one fixed order (below), so that the top-k
//      decision, an integer, is taken identically by both implementations.
//   R4 top-k is taken on the logits: larger logit first, lower expert index
//      on ties. Weights: softmax over all E, renormalised over the k kept.
//      The pages are silent on non-finite logits: a NaN logit is ranked and
//      weighted as -inf, and -0 equals +0 (so the lower index wins).
//   R5 the shared expert has weight 1 and no gate.
//   R6 SwiGLU: h = silu(g) * u with silu(z) = z / (1 + exp(-z)).
//   R7 within an expert's segment rows are in ascending assignment index
//      a = t*k + j.
//
// Build: g++ -O2 -ffp-contract=off -std=c++17 -shared -fPIC (no -ffast-math).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

extern "C" {

typedef struct {
  const uint32_t* codes;   // [n_exp, rows, K/8]
  const uint16_t* scales;  // [n_exp, rows, K/64] bf16 bits
  const uint16_t* biases;  // [n_exp, rows, K/64] bf16 bits
} oracle_qmat;

typedef struct {
  int D, E, k, I;
  const float* router_w;     // [E, D]
  const float* router_bias;  // [E] or NULL
  oracle_qmat gate, up;      // [E, I, D]
  oracle_qmat down;          // [E, D, I]
  oracle_qmat s_gate, s_up;  // [1, I, D]
  oracle_qmat s_down;        // [1, D, I]
} oracle_layer;

}  // extern "C"

namespace {

float bf16_to_float(uint16_t h) {
  uint32_t u = uint32_t(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// 4-bit code of element kk of a packed row (reading R1).
int code_at(const uint32_t* row_words, int kk) {
  return int((row_words[kk / 8] >> (4 * (kk % 8))) & 0xFu);
}

// Dequantised weight of matrix m (rows x K per expert), expert ex, row n,
// column kk, exactly in fp64 (reading R2). s*q has at most 12 significant
// bits and adding b is exact in fp64 for these magnitudes.
double dq(const oracle_qmat& m, int rows, int K, int ex, int n, int kk) {
  const size_t row = size_t(ex) * rows + n;
  const uint32_t* words = m.codes + row * size_t(K / 8);
  const double s = bf16_to_float(m.scales[row * size_t(K / 64) + kk / 64]);
  const double b = bf16_to_float(m.biases[row * size_t(K / 64) + kk / 64]);
  return s * code_at(words, kk) + b;
}

// Router logit of token row xt for expert e (reading R3): 32 fp32 partial
// sums, partial l collecting elements 32c+l for c = 0,1,... with a fused
// multiply-add, then the pairwise tree l += l+16, l += l+8, ..., l += l+1,
// then + bias[e].
float router_logit(const oracle_layer& L, const uint16_t* xt, int e) {
  float acc[32];
  for (int l = 0; l < 32; ++l) acc[l] = 0.0f;
  const float* w = L.router_w + size_t(e) * L.D;
  for (int c = 0; c < L.D / 32; ++c)
    for (int l = 0; l < 32; ++l)
      acc[l] = std::fma(bf16_to_float(xt[32 * c + l]), w[32 * c + l], acc[l]);
  for (int off = 16; off >= 1; off /= 2)
    for (int l = 0; l < off; ++l) acc[l] = acc[l] + acc[l + off];
  float logit = acc[0];
  if (L.router_bias) logit = logit + L.router_bias[e];
  return logit;
}

// Value a logit is ranked and weighted by (reading R4): a NaN logit counts
// as -inf, so every logit has a place in one total order; -0 and +0 are the
// same value there (they compare equal), so the lower index goes first.
double rank_value(float v) { return std::isnan(v) ? -INFINITY : double(v); }

// Top-k of one token's E logits by (rank value desc, index asc), and the
// renormalised softmax weights (reading R4): softmax over all E, then each
// kept expert's probability divided by the sum over the k kept.
void topk_of_logits(const float* logits, int E, int k, int* idx, double* w) {
  std::vector<int> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return rank_value(logits[a]) > rank_value(logits[b]); });
  const double lmax = rank_value(logits[order[0]]);
  std::vector<double> p(E);
  double z = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = std::exp(rank_value(logits[e]) - lmax);
    z += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= z;  // softmax over all experts
  double kept = 0.0;
  for (int j = 0; j < k; ++j) {
    idx[j] = order[j];
    kept += p[order[j]];
  }
  for (int j = 0; j < k; ++j) w[j] = p[idx[j]] / kept;  // renormalise over the k
}

// Routing for one token: its logits, then their top-k and weights.
void route_token(const oracle_layer& L, const uint16_t* xt, float* logits, int* idx, double* w) {
  for (int e = 0; e < L.E; ++e) logits[e] = router_logit(L, xt, e);
  topk_of_logits(logits, L.E, L.k, idx, w);
}

// One SwiGLU expert on one token row, fp64 throughout (reading R6).
// gate/up are [I, D] rows of expert ex, down is [D, I].
void expert_ffn(const oracle_layer& L, const oracle_qmat& gate, const oracle_qmat& up,
                const oracle_qmat& down, int ex, const uint16_t* xt, double* h, double* y) {
  const int D = L.D, I = L.I;
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int d = 0; d < D; ++d) {
      const double xv = bf16_to_float(xt[d]);
      g += xv * dq(gate, I, D, ex, i, d);
      u += xv * dq(up, I, D, ex, i, d);
    }
    h[i] = g / (1.0 + std::exp(-g)) * u;
  }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += h[i] * dq(down, D, I, ex, d, i);
    y[d] = acc;
  }
}

template <class F>
void parallel_for(int n, int n_threads, F f) {
  if (n_threads <= 0) n_threads = int(std::max(1u, std::thread::hardware_concurrency()));
  n_threads = std::min(n_threads, std::max(n, 1));
  if (n_threads <= 1) {
    for (int i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int w = 0; w < n_threads; ++w)
    pool.emplace_back([&, w] {
      for (int i = w; i < n; i += n_threads) f(i);
    });
  for (auto& th : pool) th.join();
}

bool layer_ok(const oracle_layer* L) {
  return L && L->D > 0 && L->D % 64 == 0 && L->I > 0 && L->I % 64 == 0 && L->k >= 1 &&
         L->k <= L->E && L->router_w;
}

}  // namespace

extern "C" {

int oracle_threads_used(int n_threads) {
  if (n_threads <= 0) return int(std::max(1u, std::thread::hardware_concurrency()));
  return n_threads;
}

// Exact dequantisation of rows x K of one expert of a packed matrix.
int oracle_dequant(const oracle_qmat* m, int expert, int rows, int K, double* out) {
  if (!m || K % 64 != 0 || rows <= 0) return 1;
  for (int n = 0; n < rows; ++n)
    for (int kk = 0; kk < K; ++kk) out[size_t(n) * K + kk] = dq(*m, rows, K, expert, n, kk);
  return 0;
}

// Top-k and renormalised weights of one token's given logits [E] (reading
// R4; the router's own logits go through the same function).
int oracle_topk(const float* logits, int E, int k, int* topk_idx, double* topk_w) {
  if (!logits || E < 1 || k < 1 || k > E) return 1;
  topk_of_logits(logits, E, k, topk_idx, topk_w);
  return 0;
}

// Router for T tokens: logits [T, E] (optional), topk_idx [T, k], topk_w [T, k].
int oracle_route(const oracle_layer* L, const uint16_t* x, int T, float* logits, int* topk_idx,
                 double* topk_w, int n_threads) {
  if (!layer_ok(L) || T < 0) return 1;
  parallel_for(T, n_threads, [&](int t) {
    std::vector<float> lg(L->E);
    route_token(*L, x + size_t(t) * L->D, lg.data(), topk_idx + size_t(t) * L->k,
                topk_w + size_t(t) * L->k);
    if (logits) std::copy(lg.begin(), lg.end(), logits + size_t(t) * L->E);
  });
  return 0;
}

// Histogram, exclusive scan, scatter and block map (section "Keep expert
// routing on the GPU"). count [E], off [E+1], perm [T*k] (position ->
// assignment index a = t*k + j), inv [T*k] (assignment -> position),
// blocks [max_blocks][3] = (group, first position, rows). Routed groups come
// first in ascending expert order; the shared expert follows as group E,
// whose rows T*k .. T*k+T-1 are tokens 0..T-1. Returns the block count, or
// -1 if max_blocks is too small.
int oracle_route_tables(const int* topk_idx, int T, int k, int E, int BM, int* count, int* off,
                        int* perm, int* inv, int* blocks, int max_blocks) {
  if (T < 0 || k < 1 || E < k || BM < 1) return -1;
  const int A = T * k;
  for (int e = 0; e < E; ++e) count[e] = 0;
  for (int a = 0; a < A; ++a) count[topk_idx[a]] += 1;
  off[0] = 0;
  for (int e = 0; e < E; ++e) off[e + 1] = off[e] + count[e];
  std::vector<int> fill(E, 0);
  for (int a = 0; a < A; ++a) {  // ascending a: reading R7
    const int e = topk_idx[a];
    const int p = off[e] + fill[e]++;
    perm[p] = a;
    inv[a] = p;
  }
  int nb = 0;
  auto push = [&](int g, int first, int rows) {
    if (nb < max_blocks) {
      blocks[3 * nb + 0] = g;
      blocks[3 * nb + 1] = first;
      blocks[3 * nb + 2] = rows;
    }
    ++nb;
  };
  for (int e = 0; e < E; ++e)
    for (int r0 = 0; r0 < count[e]; r0 += BM) push(e, off[e] + r0, std::min(BM, count[e] - r0));
  for (int r0 = 0; r0 < T; r0 += BM) push(E, A + r0, std::min(BM, T - r0));
  return nb <= max_blocks ? nb : -1;
}

// Intermediate h[I] of one expert for one token row: expert in 0..E-1 for a
// routed expert, -1 for the shared expert.
int oracle_expert_h(const oracle_layer* L, int expert, const uint16_t* xt, double* h) {
  if (!layer_ok(L) || expert < -1 || expert >= L->E) return 1;
  std::vector<double> y(L->D);
  if (expert < 0)
    expert_ffn(*L, L->s_gate, L->s_up, L->s_down, 0, xt, h, y.data());
  else
    expert_ffn(*L, L->gate, L->up, L->down, expert, xt, h, y.data());
  return 0;
}

// The layer on a list of tokens: y[i] = sum_j w_j * FFN_{e_j}(x[t_i]) + FFN_shared(x[t_i]).
// tokens == NULL means all T tokens in order. y is fp64 [n_tokens, D].
int oracle_moe_forward(const oracle_layer* L, const uint16_t* x, int T, const int* tokens,
                       int n_tokens, double* y, int n_threads) {
  if (!layer_ok(L) || T < 0) return 1;
  if (!tokens) n_tokens = T;
  parallel_for(n_tokens, n_threads, [&](int i) {
    const int t = tokens ? tokens[i] : i;
    const uint16_t* xt = x + size_t(t) * L->D;
    std::vector<float> lg(L->E);
    std::vector<int> idx(L->k);
    std::vector<double> w(L->k), h(L->I), ye(L->D);
    route_token(*L, xt, lg.data(), idx.data(), w.data());
    double* yt = y + size_t(i) * L->D;
    for (int d = 0; d < L->D; ++d) yt[d] = 0.0;
    for (int j = 0; j < L->k; ++j) {
      expert_ffn(*L, L->gate, L->up, L->down, idx[j], xt, h.data(), ye.data());
      for (int d = 0; d < L->D; ++d) yt[d] += w[j] * ye[d];
    }
    expert_ffn(*L, L->s_gate, L->s_up, L->s_down, 0, xt, h.data(), ye.data());
    for (int d = 0; d < L->D; ++d) yt[d] += ye[d];  // shared expert, weight 1 (reading R5)
  });
  return 0;
}

// Brute-force twin: every expert on every token from fully dequantised
// matrices, each contribution multiplied by its top-k weight or by 0.
int oracle_moe_forward_dense_masked(const oracle_layer* L, const uint16_t* x, int T, double* y,
                                    int n_threads) {
  if (!layer_ok(L) || T < 0) return 1;
  const int D = L->D, I = L->I, E = L->E;
  std::vector<int> idx(size_t(T) * L->k);
  std::vector<double> w(size_t(T) * L->k);
  oracle_route(L, x, T, nullptr, idx.data(), w.data(), n_threads);
  std::vector<double> coef(size_t(T) * (E + 1), 0.0);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < L->k; ++j) coef[size_t(t) * (E + 1) + idx[size_t(t) * L->k + j]] = w[size_t(t) * L->k + j];
    coef[size_t(t) * (E + 1) + E] = 1.0;
  }
  for (size_t i = 0; i < size_t(T) * D; ++i) y[i] = 0.0;
  std::vector<double> wg(size_t(I) * D), wu(size_t(I) * D), wd(size_t(D) * I);
  for (int g = 0; g <= E; ++g) {
    const bool sh = (g == E);
    oracle_dequant(sh ? &L->s_gate : &L->gate, sh ? 0 : g, I, D, wg.data());
    oracle_dequant(sh ? &L->s_up : &L->up, sh ? 0 : g, I, D, wu.data());
    oracle_dequant(sh ? &L->s_down : &L->down, sh ? 0 : g, D, I, wd.data());
    parallel_for(T, n_threads, [&](int t) {
      std::vector<double> xt(D), h(I);
      for (int d = 0; d < D; ++d) xt[d] = bf16_to_float(x[size_t(t) * D + d]);
      for (int i = 0; i < I; ++i) {
        double a = 0.0, b = 0.0;
        for (int d = 0; d < D; ++d) {
          a += wg[size_t(i) * D + d] * xt[d];
          b += wu[size_t(i) * D + d] * xt[d];
        }
        h[i] = a / (1.0 + std::exp(-a)) * b;
      }
      const double c = coef[size_t(t) * (E + 1) + g];
      for (int d = 0; d < D; ++d) {
        double a = 0.0;
        for (int i = 0; i < I; ++i) a += wd[size_t(d) * I + i] * h[i];
        y[size_t(t) * D + d] += c * a;
      }
    });
  }
  return 0;
}

}  // extern "C"
