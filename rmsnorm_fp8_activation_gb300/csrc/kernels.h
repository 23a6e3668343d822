// Launch parameters and host launchers of the libfp8norm kernels.  The C ABI
// in api.cu validates every argument before calling a launcher; launchers
// only choose the kernel variant and the grid, then enqueue one launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8n {

// Modes of the per-token kernels: (A) fused, and its steps on their own.
constexpr int kModeNormQuant = 0;  // gated per-head RMSNorm, then per-token FP8
constexpr int kModeGateQuant = 1;  // y = bf16(x * bf16(act(gate))), then per-token FP8
constexpr int kModeQuant = 2;      // per-token FP8 of the bf16 row x
constexpr int kModeNormOnly = 3;   // gated per-head RMSNorm to bf16 y

struct GatedParams {
  int mode;
  const uint16_t* x;
  int64_t x_stride;
  const uint16_t* gate;
  int64_t gate_stride;
  const uint16_t* weight;
  int64_t T;
  int H, D;
  float eps;
  int act;
  uint8_t* out;
  int64_t out_stride;
  float* scale;
  uint16_t* y_out;  // kModeNormOnly: bf16 [T, H*D]
  int64_t y_stride;
  uint32_t* status;
};

struct MxParams {
  const uint16_t* q;
  int64_t q_stride;
  const uint16_t* q_weight;
  int Nq;
  const uint16_t* kv;
  int64_t kv_stride;
  const uint16_t* kv_weight;
  int Nkv;
  int64_t M;
  float eps;
  uint8_t* q_out;
  int64_t q_out_stride;
  uint8_t* q_scale;
  int64_t q_scale_stride;
  uint16_t* kv_out;
  int64_t kv_out_stride;
  int q_prenorm;  // q is already normalised: MX-quantise it as given (no q_weight)
  uint32_t* status;
};

struct StaticTensor {
  const uint16_t* x;
  int64_t tok_stride, head_stride;
  int Dh;
  const float* descale;
  uint8_t* out;
};

struct StaticParams {
  StaticTensor t[3];  // Q, K, V
  int64_t T;
  int H;
  uint32_t* status;
  const int32_t* cu_seqlens;  // optional [num_seqs + 1], checked on the device
  int num_seqs;
};

// Dynamic per-head quantisation: the tensors of StaticParams with descale
// outputs instead of inputs (StaticTensor::descale is written), and a
// workspace of 3*H words that holds the per-head maxima between the passes.
struct DynamicParams {
  StaticParams s;
  float* descale_out[3];
  uint32_t* amax_bits;  // [3*H], overwritten
};

// Running per-head max |x| of one tensor: amax[h] = max(amax[h], max |x[:, h, :]|).
struct AmaxParams {
  const uint16_t* x;
  int64_t tok_stride, head_stride, T;
  int H, Dh;
  float* amax;
};

// Inverse RoPE of the o-projection input, then MXFP8 (or, without the
// quantisation, the rotated bf16 row).
struct RopeParams {
  const uint16_t* o;  // [T, H, D] bf16, token stride o_stride
  int64_t o_stride;
  int64_t T;
  int H, D;
  const int32_t* positions;  // [T]
  const float* cos_sin;      // [P, R]: cos of the R/2 pair angles, then their sin
  int P, rope_off, R;
  int interleaved;  // pairs (2i, 2i+1) of the span instead of (i, i + R/2)
  int quant;        // 1: codes and E8M0 scales; 0: the bf16 rows y_out
  uint8_t* out;     // [T, H*D] e4m3
  int64_t out_stride;
  uint8_t* scale;   // [T, H*D/32] E8M0
  int64_t scale_stride;
  uint16_t* y_out;  // [T, H*D] bf16
  int64_t y_stride;
  uint32_t* status;
};

// Largest head count of the per-head calls (per-head constants and maxima
// live in fixed arrays of this size).
constexpr int kMaxHeads = 256;

// Number of streaming multiprocessors of the current device (cached per device).
int sm_count();

cudaError_t launch_gated(const GatedParams& p, cudaStream_t stream);
cudaError_t launch_mx(const MxParams& p, cudaStream_t stream);
cudaError_t launch_static(const StaticParams& p, cudaStream_t stream);
cudaError_t launch_dynamic(const DynamicParams& p, cudaStream_t stream);
cudaError_t launch_head_amax(const AmaxParams& p, cudaStream_t stream);
cudaError_t launch_inv_rope(const RopeParams& p, cudaStream_t stream);
cudaError_t launch_convert(const float* in, int64_t n, int to, void* out, cudaStream_t stream);
cudaError_t launch_gate_act(const uint16_t* g, int64_t n, int act, uint16_t* out,
                            cudaStream_t stream);

// Spin limits of the pipeline waits (iterations of mbarrier.try_wait): the
// waits of the main loops, and the waits with which a CTA that gave up lets
// its copies still in flight land before it exits.  A test-only build sets
// FP8N_WAIT_LIMIT_MAIN=0, so that every main-loop wait gives up at once and
// the timeout path (status bit, drain, early exit) runs on real copies.
#ifndef FP8N_WAIT_LIMIT_MAIN
#define FP8N_WAIT_LIMIT_MAIN (1u << 22)
#endif
constexpr uint32_t kWaitLimitMain = FP8N_WAIT_LIMIT_MAIN;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kStatusBadDescale = 0x1u;
constexpr uint32_t kStatusTimeout = 0x2u;
constexpr uint32_t kStatusBadSeqlens = 0x4u;
constexpr uint32_t kStatusBadPosition = 0x8u;

}  // namespace fp8n
