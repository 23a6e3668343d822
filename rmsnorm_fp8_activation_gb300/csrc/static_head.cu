// (C) Static per-head FP8 quantisation of packed variable-length Q, K, V.
//
// Source: "[ROCm][MLA] Add guarded gfx942 FP8 context prefill" (vLLM PR
// 51551): calibrated static per-head descales replace the dynamic amax
// reductions, and one kernel quantises Q, K and V; descales must be finite
// and positive.  code = e4m3(RN32(x / descale[h])).
//
// GB300 design: an HBM stream (2 bytes in, 1 byte out per element).  Each
// tensor is a flat sequence of 16-byte input chunks (8 elements of one head);
// a persistent grid walks Q, then K, then V with 16-byte streaming loads,
// kUnroll chunks in flight per thread, and writes 8-byte code chunks to the
// contiguous outputs.
// Head indices come from a multiply-shift division (Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994).  The
// division itself is the IEEE quotient from the correctly rounded reciprocal
// of each descale (computed once per CTA) plus one FMA correction, on packed
// binary32 pairs.
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
  uint32_t n[3];      // chunks per tensor
  int H;
  uint32_t* status;
};

// Per-head constants: the descale d, -RN(1/d), the bf16 pair +-T with
// T = RU_bf16(512 d) (|x| above T saturates to 448 anyway, and clamping it
// keeps x * (1/d) finite), and whether d is finite and positive.
struct HeadConst {
  float d, nrd;
  uint32_t clamp2;
  uint32_t ok;
};

__device__ __forceinline__ uint32_t bf16x2_min_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// code pair of x / d for a bf16 pair x: the IEEE quotient from RN(1/d) and one
// FMA correction, arranged on -x (q0 = (-x)(-1/d), e = q0 d - x, q = q0 - e/d)
// so that signed zeros keep their sign.
__device__ __forceinline__ uint32_t quot_pair(uint32_t x, const HeadConst& hc) {
  if (!hc.ok) {  // any other descale: the plain IEEE quotient
    return e4m3x2(__fdiv_rn(bf16_lo(x), hc.d), __fdiv_rn(bf16_hi(x), hc.d));
  }
  x = bf16x2_max_nan(bf16x2_min_nan(x, hc.clamp2), hc.clamp2 | 0x80008000u);
  const f2_t nx = bf2_to_f2(x ^ 0x80008000u);
  const f2_t nrd = splat2(hc.nrd);
  const f2_t q0 = mul2(nx, nrd);
  const f2_t e = fma2(q0, splat2(hc.d), nx);
  return f2_to_e4m3x2(fma2(e, nrd, q0));
}

__global__ void __launch_bounds__(kThreads) static_head_kernel(const Flat f) {
  __shared__ HeadConst hcs[3 * kMaxHeads];
  const int nh = 3 * f.H;
  bool any_bad = false;
  for (int i = threadIdx.x; i < nh; i += blockDim.x) {
    const float d = f.t[i / f.H].descale[i % f.H];
    HeadConst hc;
    hc.d = d;
    hc.ok = (d > 0.0f) && (d <= 3.402823466e38f);  // finite and positive
    hc.nrd = -__frcp_rn(d);
    uint32_t b = __float_as_uint(__fmul_rn(d, 512.0f));
    if (b & 0xFFFFu) b += 0x10000u;                   // round up to bf16
    const uint32_t t = hc.ok ? (b >> 16) : 0x7F80u;   // inf: no clamp
    hc.clamp2 = t | (t << 16);
    hcs[i] = hc;
    any_bad |= !hc.ok;
  }
  if (any_bad && blockIdx.x == 0 && f.status) atomicOr(f.status, kStatusBadDescale);
  __syncthreads();

  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t first = blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 1
  for (int ti = 0; ti < 3; ++ti) {
    const StaticTensor T = f.t[ti];
    const FastDiv cpr = f.cpr[ti];
    const uint32_t n = f.n[ti];
    const HeadConst* hct = hcs + ti * f.H;
    for (uint32_t base = first; base < n; base += stride * kUnroll) {
      uint4 v[kUnroll];
      int hid[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = base + u * stride;
        hid[u] = -1;
        if (c < n) {
          const uint32_t row = fdiv(c, cpr);
          const uint32_t col = c - row * cpr.d;
          const uint32_t tok = fdiv(row, f.heads);
          const uint32_t h = row - tok * f.heads.d;
          v[u] = __ldcs(reinterpret_cast<const uint4*>(T.x + (int64_t)tok * T.tok_stride +
                                                       (int64_t)h * T.head_stride + 8 * col));
          hid[u] = (int)h;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (hid[u] < 0) continue;
        const HeadConst hc = hct[hid[u]];
        const uint32_t* w = &v[u].x;
        const uint2 o = make_uint2(quot_pair(w[0], hc) | (quot_pair(w[1], hc) << 16),
                                   quot_pair(w[2], hc) | (quot_pair(w[3], hc) << 16));
        __stcs(reinterpret_cast<uint2*>(T.out + (size_t)(base + u * stride) * 8), o);
      }
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
    f.n[i] = (uint32_t)(p.T * p.H * (int64_t)cpr);
    acc = f.n[i] > acc ? f.n[i] : acc;
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
