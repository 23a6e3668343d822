// (C) Static per-head FP8 quantisation of packed variable-length Q, K, V.
//
// Source: "[ROCm][MLA] Add guarded gfx942 FP8 context prefill" (vLLM PR
// 51551): calibrated static per-head descales replace the dynamic amax
// reductions, and one kernel quantises Q, K and V; descales must be finite
// and positive.  code = e4m3(RN32(x / descale[h])).
//
// GB300 design: an HBM stream (2 bytes in, 1 byte out per element).  The
// three tensors form one flat sequence of 16-byte input chunks (8 elements of
// one head); a persistent grid walks it with 16-byte loads, kUnroll chunks in
// flight per thread, and writes 8-byte code chunks to the contiguous outputs.
// Head indices come from a multiply-shift division (Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994).  The
// division itself is the IEEE quotient from the correctly rounded reciprocal
// of each descale (computed once per CTA) plus one FMA correction.
#include "common.cuh"
#include "kernels.h"

namespace fp8n {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kMaxHeads = 256;  // largest H taken (the API rejects more)

// n / d for 0 <= n < 2^31: q = (umulhi(n, m) + n) >> l with l = ceil(log2 d)
// and m = floor(2^32 (2^l - d) / d) + 1.
struct FastDiv {
  uint32_t d, m, l;
};

FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return {d, (uint32_t)m, l};
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(n, f.m) + n) >> f.l;
}

struct Flat {
  StaticTensor t[3];
  FastDiv cpr[3];     // chunks per (token, head) row
  FastDiv heads;      // H
  uint32_t end[3];    // cumulative chunk counts
  int H;
  uint32_t* status;
};

__global__ void __launch_bounds__(kThreads) static_head_kernel(const Flat f) {
  __shared__ float sd[3 * kMaxHeads], srd[3 * kMaxHeads];
  __shared__ uint32_t sbad[3 * kMaxHeads / 32];
  const int nh = 3 * f.H;
  for (int i = threadIdx.x; i < 3 * kMaxHeads / 32; i += blockDim.x) sbad[i] = 0;
  __syncthreads();
  bool any_bad = false;
  for (int i = threadIdx.x; i < nh; i += blockDim.x) {
    const float d = f.t[i / f.H].descale[i % f.H];
    const bool ok = (d > 0.0f) && (d <= 3.402823466e38f);  // finite and positive
    sd[i] = d;
    srd[i] = __frcp_rn(d);
    if (!ok) {
      atomicOr(&sbad[i >> 5], 1u << (i & 31));
      any_bad = true;
    }
  }
  if (any_bad && blockIdx.x == 0 && f.status) atomicOr(f.status, kStatusBadDescale);
  __syncthreads();

  const uint32_t total = f.end[2];
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < total;
       base += stride * kUnroll) {
    uint4 v[kUnroll];
    int hid[kUnroll];
    uint8_t* dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t c = base + u * stride;
      hid[u] = -1;
      if (c < total) {
        const int ti = c < f.end[0] ? 0 : (c < f.end[1] ? 1 : 2);
        const uint32_t cl = c - (ti ? f.end[ti - 1] : 0u);
        const uint32_t row = fdiv(cl, f.cpr[ti]);
        const uint32_t col = cl - row * f.cpr[ti].d;
        const uint32_t tok = fdiv(row, f.heads);
        const uint32_t h = row - tok * f.heads.d;
        const StaticTensor& T = f.t[ti];
        v[u] = __ldcs(reinterpret_cast<const uint4*>(T.x + (int64_t)tok * T.tok_stride +
                                                     (int64_t)h * T.head_stride + 8 * col));
        hid[u] = ti * f.H + (int)h;
        dst[u] = T.out + (size_t)cl * 8;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (hid[u] < 0) continue;
      const float d = sd[hid[u]], rd = srd[hid[u]];
      const bool bad = (sbad[hid[u] >> 5] >> (hid[u] & 31)) & 1u;
      const uint32_t* w = &v[u].x;
      uint32_t b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float q[2];
        const float x[2] = {bf16_lo(w[k]), bf16_hi(w[k])};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (bad) {
            q[i] = __fdiv_rn(x[i], d);  // any descale: the plain IEEE quotient
          } else {
            const float q0 = __fmul_rn(x[i], rd);
            const float qc = __fmaf_rn(__fmaf_rn(-q0, d, x[i]), rd, q0);
            // beyond 2^12 the code saturates anyway, and q0 also carries the
            // sign of zero and of underflowing quotients
            q[i] = (fabsf(q0) < 4096.0f && fabsf(q0) >= 0x1p-100f) ? qc : q0;
          }
        }
        b[k] = e4m3x2(q[0], q[1]);
      }
      __stcs(reinterpret_cast<uint2*>(dst[u]), make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16)));
    }
  }
}

}  // namespace

cudaError_t launch_static(const StaticParams& p, cudaStream_t stream) {
  Flat f;
  uint32_t acc = 0;
  for (int i = 0; i < 3; ++i) {
    f.t[i] = p.t[i];
    const uint32_t cpr = (uint32_t)(p.t[i].Dh / 8);
    f.cpr[i] = make_fastdiv(cpr);
    acc += (uint32_t)(p.T * p.H * (int64_t)cpr);
    f.end[i] = acc;
  }
  f.heads = make_fastdiv((uint32_t)p.H);
  f.H = p.H;
  f.status = p.status;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, static_head_kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int64_t need = ((int64_t)acc + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int grid = (int)(need < want ? need : want);
  static_head_kernel<<<grid, kThreads, 0, stream>>>(f);
  return cudaGetLastError();
}

}  // namespace fp8n
