// Launch parameters and host launchers of the libfp8norm kernels.  The C ABI
// in api.cu validates every argument before calling a launcher; launchers
// only choose the kernel variant and the grid, then enqueue one launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8n {

struct GatedParams {
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
};

// Number of streaming multiprocessors of the current device (cached per device).
int sm_count();

cudaError_t launch_gated(const GatedParams& p, cudaStream_t stream);
cudaError_t launch_mx(const MxParams& p, cudaStream_t stream);
cudaError_t launch_static(const StaticParams& p, cudaStream_t stream);
cudaError_t launch_gate_act(const uint16_t* g, int64_t n, int act, uint16_t* out,
                            cudaStream_t stream);

// Spin limit of every pipeline wait (iterations of mbarrier.try_wait).
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kStatusBadDescale = 0x1u;
constexpr uint32_t kStatusTimeout = 0x2u;

}  // namespace fp8n
