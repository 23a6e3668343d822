// Elementwise gate activation rounded once to bf16: the gate factor of the
// gated RMSNorm (sigmoid, or silu(g) = g * sigmoid(g)), exposed on its own so
// that callers who apply the gate separately, and tests that enumerate all
// 65,536 bf16 gates, use the same device code as the fused kernel.  Likewise
// the two roundings of binary32 values the kernels use (to bf16, to E4M3), so
// that they can be checked over every binary32 bit pattern.
#include "common.cuh"
#include "kernels.h"

namespace fp8n {
namespace {

template <int ACT>
__global__ void __launch_bounds__(256) gate_act_kernel(const uint16_t* g, int64_t n, uint16_t* out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 2;
  for (int64_t i = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x); i < n; i += stride) {
    const uint32_t lo = g[i], hi = (i + 1 < n) ? g[i + 1] : 0u;
    const uint32_t r = act_bf16_pair(lo | (hi << 16), ACT);
    out[i] = (uint16_t)(r & 0xFFFFu);
    if (i + 1 < n) out[i + 1] = (uint16_t)(r >> 16);
  }
}

// out = bf16 (TO == 0) or E4M3 (TO == 1) of each binary32 value, a pair at a
// time through the kernels' packed conversions.
template <int TO>
__global__ void __launch_bounds__(256) convert_kernel(const float* in, int64_t n, void* out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 2;
  for (int64_t i = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x); i < n; i += stride) {
    const bool two = i + 1 < n;
    const float lo = in[i], hi = two ? in[i + 1] : 0.0f;
    if (TO == 0) {
      const uint32_t r = pack_bf16x2(lo, hi);
      uint16_t* o = static_cast<uint16_t*>(out);
      o[i] = (uint16_t)(r & 0xFFFFu);
      if (two) o[i + 1] = (uint16_t)(r >> 16);
    } else {
      const uint32_t r = e4m3x2(lo, hi);
      uint8_t* o = static_cast<uint8_t*>(out);
      o[i] = (uint8_t)(r & 0xFFu);
      if (two) o[i + 1] = (uint8_t)(r >> 8);
    }
  }
}

}  // namespace

cudaError_t launch_convert(const float* in, int64_t n, int to, void* out, cudaStream_t stream) {
  const int64_t pairs = (n + 1) / 2;
  int64_t grid = (pairs + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 16;
  if (grid > cap) grid = cap;
  if (to == 1)
    convert_kernel<1><<<(int)grid, 256, 0, stream>>>(in, n, out);
  else
    convert_kernel<0><<<(int)grid, 256, 0, stream>>>(in, n, out);
  return cudaGetLastError();
}

cudaError_t launch_gate_act(const uint16_t* g, int64_t n, int act, uint16_t* out,
                            cudaStream_t stream) {
  const int64_t pairs = (n + 1) / 2;
  int64_t grid = (pairs + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  if (act == kActSilu)
    gate_act_kernel<kActSilu><<<(int)grid, 256, 0, stream>>>(g, n, out);
  else
    gate_act_kernel<kActSigmoid><<<(int)grid, 256, 0, stream>>>(g, n, out);
  return cudaGetLastError();
}

}  // namespace fp8n
