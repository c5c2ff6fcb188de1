// Tensor-core grouped GEMMs (tcgen05 + TMEM) for the prefill expert path, and
// the bf16 dequantisation diagnostic.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

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

}  // namespace

cudaError_t debug_dequant(const moe_qmatrix* m, int expert, int rows, int K, uint16_t* out, cudaStream_t s) {
  debug_dequant_kernel<<<256, 256, 0, s>>>(*m, expert, rows, K, out);
  return cudaGetLastError();
}

bool gemm_tc_supported(const Ctx&) { return false; }

cudaError_t gemm_tc(const Ctx&) { return cudaErrorNotSupported; }

}  // namespace moe
