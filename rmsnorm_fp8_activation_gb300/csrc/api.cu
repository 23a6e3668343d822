// C ABI of libfp8norm: argument validation on the host, then one launch on the
// caller's stream (see include/fp8norm.h for the contract of each call).
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fp8norm.h"
#include "kernels.h"

namespace {

thread_local int g_last_cuda_error = 0;

fp8n_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FP8N_OK;
  g_last_cuda_error = (int)e;
  return FP8N_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

namespace fp8n {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
  return n;
}

}  // namespace fp8n

extern "C" {

const char* fp8n_status_string(fp8n_status s) {
  switch (s) {
    case FP8N_OK: return "FP8N_OK";
    case FP8N_ERR_NULL: return "FP8N_ERR_NULL: a required pointer is NULL";
    case FP8N_ERR_SHAPE: return "FP8N_ERR_SHAPE: negative or inconsistent sizes or strides";
    case FP8N_ERR_MISALIGNED: return "FP8N_ERR_MISALIGNED: a pointer or stride breaks the 16-byte rule";
    case FP8N_ERR_UNSUPPORTED: return "FP8N_ERR_UNSUPPORTED: a size outside the supported range";
    case FP8N_ERR_BAD_SCALE: return "FP8N_ERR_BAD_SCALE: a descale is not finite and positive";
    case FP8N_ERR_CUDA: return "FP8N_ERR_CUDA: a CUDA runtime call failed";
  }
  return "unknown fp8n_status";
}

int fp8n_last_cuda_error(void) { return g_last_cuda_error; }

uint32_t fp8n_version(void) { return 0x000200u; }

// Shared validation of the per-token family: rows of T tokens, row length
// `row` = H*D elements; x (and gate when given) bf16 rows; outputs checked by
// the callers.
static fp8n_status check_rows(const void* x, int64_t x_stride, const void* gate,
                              int64_t gate_stride, bool with_gate, int64_t T, int64_t row) {
  if (x_stride < row || (with_gate && gate_stride < row)) return FP8N_ERR_SHAPE;
  if (T == 0) return FP8N_OK;
  if (!x || (with_gate && !gate)) return FP8N_ERR_NULL;
  if (!aligned16(x) || x_stride % 8 || (with_gate && (!aligned16(gate) || gate_stride % 8)))
    return FP8N_ERR_MISALIGNED;
  return FP8N_OK;
}

static bool bad_eps(float eps) { return !(eps >= 0.0f) || std::isinf(eps); }

static fp8n_status launch_tokens(const fp8n::GatedParams& p, fp8n_stream_t stream) {
  return cuda_status(fp8n::launch_gated(p, (cudaStream_t)stream));
}

fp8n_status fp8n_gated_rmsnorm_quant_token(const void* x, int64_t x_stride, const void* gate,
                                           int64_t gate_stride, const void* weight, int64_t T,
                                           int32_t H, int32_t D, float eps, fp8n_act act,
                                           void* out, int64_t out_stride, float* scale,
                                           uint32_t* status, fp8n_stream_t stream) {
  if (T < 0 || H < 1 || D < 1) return FP8N_ERR_SHAPE;
  if (act != FP8N_ACT_SIGMOID && act != FP8N_ACT_SILU) return FP8N_ERR_UNSUPPORTED;
  if (D % 8 != 0 || D > 8192 || (int64_t)H * D > 16384) return FP8N_ERR_UNSUPPORTED;
  if (bad_eps(eps)) return FP8N_ERR_UNSUPPORTED;
  const int64_t row = (int64_t)H * D;
  if (out_stride < row) return FP8N_ERR_SHAPE;
  fp8n_status s = check_rows(x, x_stride, gate, gate_stride, true, T, row);
  if (s != FP8N_OK || T == 0) return s;
  if (!weight || !out || !scale) return FP8N_ERR_NULL;
  if (!aligned16(weight) || !aligned16(out) || out_stride % 8 || ((uintptr_t)scale & 3u) ||
      ((uintptr_t)status & 3u))
    return FP8N_ERR_MISALIGNED;
  fp8n::GatedParams p = {};
  p.mode = fp8n::kModeNormQuant;
  p.x = (const uint16_t*)x;
  p.x_stride = x_stride;
  p.gate = (const uint16_t*)gate;
  p.gate_stride = gate_stride;
  p.weight = (const uint16_t*)weight;
  p.T = T;
  p.H = H;
  p.D = D;
  p.eps = eps;
  p.act = (int)act;
  p.out = (uint8_t*)out;
  p.out_stride = out_stride;
  p.scale = scale;
  p.status = status;
  return launch_tokens(p, stream);
}

fp8n_status fp8n_gated_rmsnorm_bf16(const void* x, int64_t x_stride, const void* gate,
                                    int64_t gate_stride, const void* weight, int64_t T, int32_t H,
                                    int32_t D, float eps, fp8n_act act, void* y, int64_t y_stride,
                                    uint32_t* status, fp8n_stream_t stream) {
  if (T < 0 || H < 1 || D < 1) return FP8N_ERR_SHAPE;
  if (act != FP8N_ACT_SIGMOID && act != FP8N_ACT_SILU) return FP8N_ERR_UNSUPPORTED;
  if (D % 8 != 0 || D > 8192 || (int64_t)H * D > 16384) return FP8N_ERR_UNSUPPORTED;
  if (bad_eps(eps)) return FP8N_ERR_UNSUPPORTED;
  const int64_t row = (int64_t)H * D;
  if (y_stride < row) return FP8N_ERR_SHAPE;
  fp8n_status s = check_rows(x, x_stride, gate, gate_stride, true, T, row);
  if (s != FP8N_OK || T == 0) return s;
  if (!weight || !y) return FP8N_ERR_NULL;
  if (!aligned16(weight) || !aligned16(y) || y_stride % 8 || ((uintptr_t)status & 3u))
    return FP8N_ERR_MISALIGNED;
  fp8n::GatedParams p = {};
  p.mode = fp8n::kModeNormOnly;
  p.x = (const uint16_t*)x;
  p.x_stride = x_stride;
  p.gate = (const uint16_t*)gate;
  p.gate_stride = gate_stride;
  p.weight = (const uint16_t*)weight;
  p.T = T;
  p.H = H;
  p.D = D;
  p.eps = eps;
  p.act = (int)act;
  p.y_out = (uint16_t*)y;
  p.y_stride = y_stride;
  p.status = status;
  return launch_tokens(p, stream);
}

// The gate product and the per-token quantisation without the norm, or the
// quantisation alone (gate == NULL path of the shared body below).
static fp8n_status token_quant(int mode, const void* x, int64_t x_stride, const void* gate,
                               int64_t gate_stride, int64_t T, int32_t N, int act, void* out,
                               int64_t out_stride, float* scale, uint32_t* status,
                               fp8n_stream_t stream) {
  if (T < 0 || N < 1) return FP8N_ERR_SHAPE;
  if (N % 8 != 0 || N > 16384) return FP8N_ERR_UNSUPPORTED;
  if (out_stride < N) return FP8N_ERR_SHAPE;
  const bool with_gate = mode == fp8n::kModeGateQuant;
  fp8n_status s = check_rows(x, x_stride, gate, gate_stride, with_gate, T, N);
  if (s != FP8N_OK || T == 0) return s;
  if (!out || !scale) return FP8N_ERR_NULL;
  if (!aligned16(out) || out_stride % 8 || ((uintptr_t)scale & 3u) || ((uintptr_t)status & 3u))
    return FP8N_ERR_MISALIGNED;
  fp8n::GatedParams p = {};
  p.mode = mode;
  p.x = (const uint16_t*)x;
  p.x_stride = x_stride;
  p.gate = (const uint16_t*)gate;
  p.gate_stride = gate_stride;
  p.T = T;
  p.H = 1;
  p.D = N;
  p.act = act;
  p.out = (uint8_t*)out;
  p.out_stride = out_stride;
  p.scale = scale;
  p.status = status;
  return launch_tokens(p, stream);
}

fp8n_status fp8n_gated_quant_token(const void* x, int64_t x_stride, const void* gate,
                                   int64_t gate_stride, int64_t T, int32_t N, fp8n_act act,
                                   void* out, int64_t out_stride, float* scale, uint32_t* status,
                                   fp8n_stream_t stream) {
  if (act != FP8N_ACT_SIGMOID && act != FP8N_ACT_SILU) return FP8N_ERR_UNSUPPORTED;
  return token_quant(fp8n::kModeGateQuant, x, x_stride, gate, gate_stride, T, N, (int)act, out,
                     out_stride, scale, status, stream);
}

fp8n_status fp8n_quant_token(const void* y, int64_t y_stride, int64_t T, int32_t N, void* out,
                             int64_t out_stride, float* scale, uint32_t* status,
                             fp8n_stream_t stream) {
  return token_quant(fp8n::kModeQuant, y, y_stride, nullptr, 0, T, N, 0, out, out_stride, scale,
                     status, stream);
}

fp8n_status fp8n_rmsnorm_quant_mx(const void* q, int64_t q_stride, const void* q_weight,
                                  int32_t Nq, const void* kv, int64_t kv_stride,
                                  const void* kv_weight, int32_t Nkv, int64_t M, float eps,
                                  void* q_out, int64_t q_out_stride, uint8_t* q_scale,
                                  int64_t q_scale_stride, void* kv_out, int64_t kv_out_stride,
                                  uint32_t* status, fp8n_stream_t stream) {
  if (M < 0 || Nq < 1 || Nkv < 0) return FP8N_ERR_SHAPE;
  if (Nq % 32 != 0 || Nq > 16384 || Nkv % 8 != 0 || Nkv > 16384) return FP8N_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f) || std::isinf(eps)) return FP8N_ERR_UNSUPPORTED;
  if (q_stride < Nq || q_out_stride < Nq || q_scale_stride < Nq / 32) return FP8N_ERR_SHAPE;
  if (Nkv > 0 && (kv_stride < Nkv || kv_out_stride < Nkv)) return FP8N_ERR_SHAPE;
  if (M == 0) return FP8N_OK;
  if (!q || !q_weight || !q_out || !q_scale) return FP8N_ERR_NULL;
  if (Nkv > 0 && (!kv || !kv_weight || !kv_out)) return FP8N_ERR_NULL;
  if (!aligned16(q) || !aligned16(q_weight) || !aligned16(q_out) || q_stride % 8 ||
      q_out_stride % 8 || ((uintptr_t)status & 3u))
    return FP8N_ERR_MISALIGNED;
  if (Nkv > 0 && (!aligned16(kv) || !aligned16(kv_weight) || !aligned16(kv_out) ||
                  kv_stride % 8 || kv_out_stride % 8))
    return FP8N_ERR_MISALIGNED;
  fp8n::MxParams p = {};
  p.q = (const uint16_t*)q;
  p.q_stride = q_stride;
  p.q_weight = (const uint16_t*)q_weight;
  p.Nq = Nq;
  p.kv = (const uint16_t*)kv;
  p.kv_stride = kv_stride;
  p.kv_weight = (const uint16_t*)kv_weight;
  p.Nkv = Nkv;
  p.M = M;
  p.eps = eps;
  p.q_out = (uint8_t*)q_out;
  p.q_out_stride = q_out_stride;
  p.q_scale = q_scale;
  p.q_scale_stride = q_scale_stride;
  p.kv_out = (uint16_t*)kv_out;
  p.kv_out_stride = kv_out_stride;
  p.status = status;
  return cuda_status(fp8n::launch_mx(p, (cudaStream_t)stream));
}

fp8n_status fp8n_rmsnorm_bf16(const void* x, int64_t x_stride, const void* weight, int64_t M,
                              int32_t N, float eps, void* y, int64_t y_stride, uint32_t* status,
                              fp8n_stream_t stream) {
  if (M < 0 || N < 1) return FP8N_ERR_SHAPE;
  if (N % 8 != 0 || N > 16384 || bad_eps(eps)) return FP8N_ERR_UNSUPPORTED;
  if (x_stride < N || y_stride < N) return FP8N_ERR_SHAPE;
  if (M == 0) return FP8N_OK;
  if (!x || !weight || !y) return FP8N_ERR_NULL;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y) || x_stride % 8 || y_stride % 8 ||
      ((uintptr_t)status & 3u))
    return FP8N_ERR_MISALIGNED;
  fp8n::MxParams p = {};  // no q columns: the kv path of (B) alone
  p.kv = (const uint16_t*)x;
  p.kv_stride = x_stride;
  p.kv_weight = (const uint16_t*)weight;
  p.Nkv = N;
  p.M = M;
  p.eps = eps;
  p.kv_out = (uint16_t*)y;
  p.kv_out_stride = y_stride;
  p.status = status;
  return cuda_status(fp8n::launch_mx(p, (cudaStream_t)stream));
}

fp8n_status fp8n_quant_mx(const void* y, int64_t y_stride, int64_t M, int32_t N, void* out,
                          int64_t out_stride, uint8_t* scale, int64_t scale_stride,
                          uint32_t* status, fp8n_stream_t stream) {
  if (M < 0 || N < 1) return FP8N_ERR_SHAPE;
  if (N % 32 != 0 || N > 16384) return FP8N_ERR_UNSUPPORTED;
  if (y_stride < N || out_stride < N || scale_stride < N / 32) return FP8N_ERR_SHAPE;
  if (M == 0) return FP8N_OK;
  if (!y || !out || !scale) return FP8N_ERR_NULL;
  if (!aligned16(y) || !aligned16(out) || y_stride % 8 || out_stride % 8 ||
      ((uintptr_t)status & 3u))
    return FP8N_ERR_MISALIGNED;
  fp8n::MxParams p = {};  // q taken as already normalised, no kv columns
  p.q = (const uint16_t*)y;
  p.q_stride = y_stride;
  p.Nq = N;
  p.M = M;
  p.q_out = (uint8_t*)out;
  p.q_out_stride = out_stride;
  p.q_scale = scale;
  p.q_scale_stride = scale_stride;
  p.q_prenorm = 1;
  p.status = status;
  return cuda_status(fp8n::launch_mx(p, (cudaStream_t)stream));
}

// Shared validation of the packed Q/K/V calls (descale pointers checked by
// the callers); fills the tensors of p.
static fp8n_status check_qkv(const void* q, const void* k, const void* v, int64_t qk_tok_stride,
                             int64_t qk_head_stride, int64_t v_tok_stride, int64_t v_head_stride,
                             int64_t T, int32_t H, int32_t Dqk, int32_t Dv, void* q_out,
                             void* k_out, void* v_out, fp8n::StaticParams* p) {
  if (T < 0 || H < 1 || Dqk < 1 || Dv < 1) return FP8N_ERR_SHAPE;
  if (Dqk % 8 || Dv % 8 || Dqk > 8192 || Dv > 8192 || H > fp8n::kMaxHeads)
    return FP8N_ERR_UNSUPPORTED;
  if (qk_head_stride < Dqk || v_head_stride < Dv || qk_tok_stride < 0 || v_tok_stride < 0)
    return FP8N_ERR_SHAPE;
  // one launch addresses every chunk with 32-bit indices
  const int64_t chunks = T * H * (int64_t)(2 * Dqk + Dv) / 8;
  if (chunks >= (int64_t)1 << 31) return FP8N_ERR_UNSUPPORTED;
  if (T == 0) return FP8N_OK;
  if (!q || !k || !v || !q_out || !k_out || !v_out) return FP8N_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(k_out) ||
      !aligned16(v_out) || qk_tok_stride % 8 || qk_head_stride % 8 || v_tok_stride % 8 ||
      v_head_stride % 8)
    return FP8N_ERR_MISALIGNED;
  const void* in[3] = {q, k, v};
  void* out[3] = {q_out, k_out, v_out};
  for (int i = 0; i < 3; ++i) {
    p->t[i].x = (const uint16_t*)in[i];
    p->t[i].tok_stride = i < 2 ? qk_tok_stride : v_tok_stride;
    p->t[i].head_stride = i < 2 ? qk_head_stride : v_head_stride;
    p->t[i].Dh = i < 2 ? Dqk : Dv;
    p->t[i].descale = nullptr;
    p->t[i].out = (uint8_t*)out[i];
  }
  p->T = T;
  p->H = H;
  p->status = nullptr;
  return FP8N_OK;
}

static bool misaligned4(const void* p) { return ((uintptr_t)p & 3u) != 0; }

fp8n_status fp8n_static_head_quant(const void* q, const void* k, const void* v,
                                   int64_t qk_tok_stride, int64_t qk_head_stride,
                                   int64_t v_tok_stride, int64_t v_head_stride, int64_t T,
                                   int32_t H, int32_t Dqk, int32_t Dv, const float* q_descale,
                                   const float* k_descale, const float* v_descale,
                                   const int32_t* cu_seqlens, int32_t num_seqs, void* q_out,
                                   void* k_out, void* v_out, uint32_t* status,
                                   fp8n_stream_t stream) {
  if (num_seqs < 0) return FP8N_ERR_SHAPE;
  fp8n::StaticParams p = {};
  fp8n_status s = check_qkv(q, k, v, qk_tok_stride, qk_head_stride, v_tok_stride, v_head_stride,
                            T, H, Dqk, Dv, q_out, k_out, v_out, &p);
  if (s != FP8N_OK || T == 0) return s;
  if (!q_descale || !k_descale || !v_descale) return FP8N_ERR_NULL;
  if (misaligned4(q_descale) || misaligned4(k_descale) || misaligned4(v_descale) ||
      misaligned4(status))
    return FP8N_ERR_MISALIGNED;
  if (misaligned4(cu_seqlens)) return FP8N_ERR_MISALIGNED;
  const float* d[3] = {q_descale, k_descale, v_descale};
  for (int i = 0; i < 3; ++i) p.t[i].descale = d[i];
  p.status = status;
  p.cu_seqlens = cu_seqlens;
  p.num_seqs = num_seqs;
  return cuda_status(fp8n::launch_static(p, (cudaStream_t)stream));
}

fp8n_status fp8n_dynamic_head_quant(const void* q, const void* k, const void* v,
                                    int64_t qk_tok_stride, int64_t qk_head_stride,
                                    int64_t v_tok_stride, int64_t v_head_stride, int64_t T,
                                    int32_t H, int32_t Dqk, int32_t Dv, uint32_t* workspace,
                                    float* q_descale, float* k_descale, float* v_descale,
                                    void* q_out, void* k_out, void* v_out, fp8n_stream_t stream) {
  fp8n::DynamicParams p = {};
  fp8n_status s = check_qkv(q, k, v, qk_tok_stride, qk_head_stride, v_tok_stride, v_head_stride,
                            T, H, Dqk, Dv, q_out, k_out, v_out, &p.s);
  if (s != FP8N_OK || T == 0) return s;
  if (!workspace || !q_descale || !k_descale || !v_descale) return FP8N_ERR_NULL;
  if (misaligned4(workspace) || misaligned4(q_descale) || misaligned4(k_descale) ||
      misaligned4(v_descale))
    return FP8N_ERR_MISALIGNED;
  p.descale_out[0] = q_descale;
  p.descale_out[1] = k_descale;
  p.descale_out[2] = v_descale;
  p.amax_bits = workspace;
  return cuda_status(fp8n::launch_dynamic(p, (cudaStream_t)stream));
}

}  // extern "C"

// ---- dynamic per-head quantisation without a caller workspace --------------
//
// The per-head maxima of fp8n_dynamic_head_quant_noalloc live in this
// file-scope device array instead of a caller buffer.  Every GPU that loads
// the library holds it (3 * 256 words, 3 KB) until the process exits.  Host
// code may not pass the array's name to a kernel (on the host it is only a
// stand-in for the device symbol): its device address is looked up once per
// device with cudaGetSymbolAddress and cached.
namespace {

constexpr int kNoAllocMaxHeads = 256;
// the kernels index the maxima up to 3 * H for every H the per-head calls take
static_assert(kNoAllocMaxHeads >= fp8n::kMaxHeads, "scratch smaller than the head range");
constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) uint32_t g_dynamic_scratch[3 * kNoAllocMaxHeads];

std::mutex g_scratch_mutex;
uint32_t* g_scratch_address[kNoAllocMaxDevices] = {};

// Device address of g_dynamic_scratch on the current device (looked up on
// the first call for that device).
fp8n_status noalloc_scratch(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kNoAllocMaxDevices) return FP8N_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_address[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_dynamic_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    g_scratch_address[dev] = static_cast<uint32_t*>(ptr);
  }
  *out = g_scratch_address[dev];
  return FP8N_OK;
}

}  // namespace

extern "C" {

fp8n_status fp8n_dynamic_head_quant_noalloc(const void* q, const void* k, const void* v,
                                            int64_t qk_tok_stride, int64_t qk_head_stride,
                                            int64_t v_tok_stride, int64_t v_head_stride,
                                            int64_t T, int32_t H, int32_t Dqk, int32_t Dv,
                                            float* q_descale, float* k_descale, float* v_descale,
                                            void* q_out, void* k_out, void* v_out,
                                            fp8n_stream_t stream) {
  if (H > kNoAllocMaxHeads) return FP8N_ERR_UNSUPPORTED;  // beyond the static scratch
  fp8n::DynamicParams p = {};
  fp8n_status s = check_qkv(q, k, v, qk_tok_stride, qk_head_stride, v_tok_stride, v_head_stride,
                            T, H, Dqk, Dv, q_out, k_out, v_out, &p.s);
  if (s != FP8N_OK || T == 0) return s;
  if (!q_descale || !k_descale || !v_descale) return FP8N_ERR_NULL;
  if (misaligned4(q_descale) || misaligned4(k_descale) || misaligned4(v_descale))
    return FP8N_ERR_MISALIGNED;
  uint32_t* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != FP8N_OK) return s;
  p.descale_out[0] = q_descale;
  p.descale_out[1] = k_descale;
  p.descale_out[2] = v_descale;
  p.amax_bits = scratch;  // zeroed on the stream by the launcher before use
  return cuda_status(fp8n::launch_dynamic(p, (cudaStream_t)stream));
}

fp8n_status fp8n_head_amax(const void* x, int64_t tok_stride, int64_t head_stride, int64_t T,
                           int32_t H, int32_t Dh, float* amax, fp8n_stream_t stream) {
  if (T < 0 || H < 1 || Dh < 1) return FP8N_ERR_SHAPE;
  if (Dh % 8 || Dh > 8192 || H > fp8n::kMaxHeads) return FP8N_ERR_UNSUPPORTED;
  if (head_stride < Dh || tok_stride < 0) return FP8N_ERR_SHAPE;
  if (T * H * (int64_t)Dh / 8 >= (int64_t)1 << 31) return FP8N_ERR_UNSUPPORTED;
  if (T == 0) return FP8N_OK;
  if (!x || !amax) return FP8N_ERR_NULL;
  if (!aligned16(x) || tok_stride % 8 || head_stride % 8 || misaligned4(amax))
    return FP8N_ERR_MISALIGNED;
  fp8n::AmaxParams p = {};
  p.x = (const uint16_t*)x;
  p.tok_stride = tok_stride;
  p.head_stride = head_stride;
  p.T = T;
  p.H = H;
  p.Dh = Dh;
  p.amax = amax;
  return cuda_status(fp8n::launch_head_amax(p, (cudaStream_t)stream));
}

// Shared validation of the inverse-RoPE calls; fills the input side of p.
static fp8n_status check_rope(const void* o, int64_t o_stride, int64_t T, int32_t H, int32_t D,
                              const int32_t* positions, const float* cos_sin,
                              int32_t num_positions, int32_t rope_off, int32_t rope_dim,
                              fp8n_rope_style style, uint32_t* status, fp8n::RopeParams* p) {
  if (T < 0 || H < 1 || D < 1 || rope_off < 0 || rope_dim < 0) return FP8N_ERR_SHAPE;
  if (style != FP8N_ROPE_HALF && style != FP8N_ROPE_INTERLEAVED) return FP8N_ERR_UNSUPPORTED;
  if (D % 32 || D > 8192 || rope_off % 8 || rope_dim % 16 || rope_off + rope_dim > D)
    return FP8N_ERR_UNSUPPORTED;
  // one launch addresses every MX block with 32-bit indices
  if (T * H * (int64_t)(D / 32) >= (int64_t)1 << 31) return FP8N_ERR_UNSUPPORTED;
  if (o_stride < (int64_t)H * D) return FP8N_ERR_SHAPE;
  if (rope_dim > 0 && num_positions < 1) return FP8N_ERR_SHAPE;
  if (T == 0) return FP8N_OK;
  if (!o || (rope_dim > 0 && (!positions || !cos_sin))) return FP8N_ERR_NULL;
  if (!aligned16(o) || o_stride % 8 || (rope_dim > 0 && (!aligned16(cos_sin) || misaligned4(positions))) ||
      misaligned4(status))
    return FP8N_ERR_MISALIGNED;
  p->o = (const uint16_t*)o;
  p->o_stride = o_stride;
  p->T = T;
  p->H = H;
  p->D = D;
  p->positions = positions;
  p->cos_sin = cos_sin;
  p->P = num_positions;
  p->rope_off = rope_off;
  p->R = rope_dim;
  p->interleaved = style == FP8N_ROPE_INTERLEAVED;
  p->status = status;
  return FP8N_OK;
}

fp8n_status fp8n_inv_rope_quant_mx(const void* o, int64_t o_stride, int64_t T, int32_t H,
                                   int32_t D, const int32_t* positions, const float* cos_sin,
                                   int32_t num_positions, int32_t rope_off, int32_t rope_dim,
                                   fp8n_rope_style style, void* out, int64_t out_stride,
                                   uint8_t* scale, int64_t scale_stride, uint32_t* status,
                                   fp8n_stream_t stream) {
  fp8n::RopeParams p = {};
  fp8n_status s = check_rope(o, o_stride, T, H, D, positions, cos_sin, num_positions, rope_off,
                             rope_dim, style, status, &p);
  if (s != FP8N_OK) return s;
  if (out_stride < (int64_t)H * D || scale_stride < (int64_t)H * (D / 32)) return FP8N_ERR_SHAPE;
  if (T == 0) return FP8N_OK;
  if (!out || !scale) return FP8N_ERR_NULL;
  if (!aligned16(out) || out_stride % 16) return FP8N_ERR_MISALIGNED;
  p.quant = 1;
  p.out = (uint8_t*)out;
  p.out_stride = out_stride;
  p.scale = scale;
  p.scale_stride = scale_stride;
  return cuda_status(fp8n::launch_inv_rope(p, (cudaStream_t)stream));
}

fp8n_status fp8n_inv_rope_bf16(const void* o, int64_t o_stride, int64_t T, int32_t H, int32_t D,
                               const int32_t* positions, const float* cos_sin,
                               int32_t num_positions, int32_t rope_off, int32_t rope_dim,
                               fp8n_rope_style style, void* y, int64_t y_stride, uint32_t* status,
                               fp8n_stream_t stream) {
  fp8n::RopeParams p = {};
  fp8n_status s = check_rope(o, o_stride, T, H, D, positions, cos_sin, num_positions, rope_off,
                             rope_dim, style, status, &p);
  if (s != FP8N_OK) return s;
  if (y_stride < (int64_t)H * D) return FP8N_ERR_SHAPE;
  if (T == 0) return FP8N_OK;
  if (!y) return FP8N_ERR_NULL;
  if (!aligned16(y) || y_stride % 8) return FP8N_ERR_MISALIGNED;
  p.quant = 0;
  p.y_out = (uint16_t*)y;
  p.y_stride = y_stride;
  return cuda_status(fp8n::launch_inv_rope(p, (cudaStream_t)stream));
}

fp8n_status fp8n_gate_act_bf16(const void* g, int64_t n, fp8n_act act, void* out,
                               fp8n_stream_t stream) {
  if (n < 0) return FP8N_ERR_SHAPE;
  if (act != FP8N_ACT_SIGMOID && act != FP8N_ACT_SILU) return FP8N_ERR_UNSUPPORTED;
  if (n == 0) return FP8N_OK;
  if (!g || !out) return FP8N_ERR_NULL;
  if (((uintptr_t)g & 1u) || ((uintptr_t)out & 1u)) return FP8N_ERR_MISALIGNED;
  return cuda_status(fp8n::launch_gate_act((const uint16_t*)g, n, (int)act, (uint16_t*)out,
                                           (cudaStream_t)stream));
}

fp8n_status fp8n_convert_f32(const float* in, int64_t n, fp8n_cvt to, void* out,
                             fp8n_stream_t stream) {
  if (n < 0) return FP8N_ERR_SHAPE;
  if (to != FP8N_CVT_BF16 && to != FP8N_CVT_E4M3) return FP8N_ERR_UNSUPPORTED;
  if (n == 0) return FP8N_OK;
  if (!in || !out) return FP8N_ERR_NULL;
  if (((uintptr_t)in & 3u) || (to == FP8N_CVT_BF16 && ((uintptr_t)out & 1u)))
    return FP8N_ERR_MISALIGNED;
  return cuda_status(fp8n::launch_convert(in, n, (int)to, out, (cudaStream_t)stream));
}

fp8n_status fp8n_check_descales(const float* descale, int32_t n, fp8n_stream_t stream) {
  if (n < 1 || n > 65536) return FP8N_ERR_SHAPE;
  if (!descale) return FP8N_ERR_NULL;
  if ((uintptr_t)descale & 3u) return FP8N_ERR_MISALIGNED;
  std::vector<float> h((size_t)n);
  cudaError_t e = cudaMemcpyAsync(h.data(), descale, sizeof(float) * (size_t)n,
                                  cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  for (float x : h)
    if (!(x > 0.0f) || std::isinf(x)) return FP8N_ERR_BAD_SCALE;
  return FP8N_OK;
}

}  // extern "C"
