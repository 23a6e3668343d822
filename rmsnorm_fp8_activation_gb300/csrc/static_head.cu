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
// kUnroll (6) chunks in flight per thread, and writes 8-byte code chunks to the
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
constexpr int kUnroll = 6;

struct Flat {
  StaticTensor t[3];
  FastDiv cpr[3];     // chunks per (token, head) row
  FastDiv heads;      // H
  uint32_t n[3];      // chunks per tensor
  int H;
  int ntensors;       // tensors walked (the amax pass of a single tensor: 1)
  uint32_t* status;
  const int32_t* cu;  // optional sequence prefix sums [nseq + 1] (checked, not used)
  int nseq;
  int64_t T;
  int* amax_bits;     // dynamic variant: [3*H] per-head max |x| as float bits
  float* dout[3];     // dynamic variant: descale outputs
};

// Per-head constants: the descale d, -RN(1/d), the bf16 pair +-T with
// T = RU_bf16(512 d) (|x| above T saturates to 448 anyway, and clamping it
// keeps x * (1/d) finite), and which quotient path d takes: kFast for
// 2^-92 <= d <= 2^126, where 1/d is a normal binary32 and the FMA residual
// cannot underflow for any quotient that reaches a nonzero code
// (|x/d| >= 2^-11); kZero for the zero descale of an all-zero head in the
// dynamic variant (signed zero codes); kExact, the plain IEEE division, for
// every other d.
constexpr uint32_t kFast = 0, kExact = 1, kZero = 2;
struct HeadConst {
  float d, nrd;
  uint32_t clamp2;
  uint32_t path;
};

__device__ __forceinline__ HeadConst head_const(float d, bool dynamic) {
  HeadConst hc;
  hc.d = d;
  hc.path = (d >= 0x1p-92f && d <= 0x1p126f) ? kFast : (dynamic && d == 0.0f) ? kZero : kExact;
  hc.nrd = -__frcp_rn(d);
  uint32_t b = __float_as_uint(__fmul_rn(d, 512.0f));
  if (b & 0xFFFFu) b += 0x10000u;                            // round up to bf16
  const uint32_t t = hc.path == kFast ? (b >> 16) : 0x7F80u;  // inf: no clamp
  hc.clamp2 = t | (t << 16);
  return hc;
}

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
  if (hc.path != kFast) {
    if (hc.path == kZero) return (x >> 8 & 0x80u) | (x >> 16 & 0x8000u);  // the signs of x
    return e4m3x2(__fdiv_rn(bf16_lo(x), hc.d), __fdiv_rn(bf16_hi(x), hc.d));
  }
  x = bf16x2_max_nan(bf16x2_min_nan(x, hc.clamp2), hc.clamp2 | 0x80008000u);
  const f2_t nx = bf2_to_f2(x ^ 0x80008000u);
  const f2_t nrd = splat2(hc.nrd);
  const f2_t q0 = mul2(nx, nrd);
  const f2_t e = fma2(q0, splat2(hc.d), nx);
  return f2_to_e4m3x2(fma2(e, nrd, q0));
}

// DYN: the descales are RN32(amax / 448) of the per-head maxima that the
// amax pass left in f.amax_bits (float bits); block 0 also writes them out.
template <bool DYN>
__global__ void __launch_bounds__(kThreads) static_head_kernel(const Flat f) {
  __shared__ HeadConst hcs[3 * kMaxHeads];
  pdl_launch_dependents();  // programmatic dependent launch (see launch_pdl)
  pdl_wait();
  const int nh = 3 * f.H;
  bool any_bad = false;
  for (int i = threadIdx.x; i < nh; i += blockDim.x) {
    float d;
    if (DYN) {
      d = __fdiv_rn(__int_as_float(f.amax_bits[i]), 448.0f);
      if (blockIdx.x == 0) f.dout[i / f.H][i % f.H] = d;
    } else {
      d = f.t[i / f.H].descale[i % f.H];
      any_bad |= !((d > 0.0f) && (d <= 3.402823466e38f));  // not finite and positive
    }
    hcs[i] = head_const(d, DYN);
  }
  if (any_bad && blockIdx.x == 0 && f.status) atomicOr(f.status, kStatusBadDescale);
  // the packed batch's prefix sums, when given: cu[0] == 0, never decreasing,
  // cu[nseq] == T (block 0 only; the quantisation itself is elementwise)
  if (!DYN && blockIdx.x == 0 && f.cu && f.status) {
    bool bad = false;
    for (int i = threadIdx.x; i <= f.nseq; i += blockDim.x) {
      const int32_t c = f.cu[i];
      if (i == 0) bad |= c != 0;
      else bad |= c < f.cu[i - 1];
      if (i == f.nseq) bad |= (int64_t)c != f.T;
    }
    if (bad) atomicOr(f.status, kStatusBadSeqlens);
  }
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

// Per-head max |x| (the amax pass of the dynamic variant, and the running
// maxima of calibration).  bf16 magnitudes order like their bit patterns with
// the sign cleared, NaN above infinity above every finite value, so the max
// is an unsigned 16-bit max on packed pairs.  When the grid-stride S is a
// multiple of every tensor's chunks per token, each thread's chunks all sit
// in one head and its running max is folded into shared memory once per
// tensor; otherwise (UNIFORM false) it is folded whenever the head changes.
// Each block then takes its per-head maxima to f.amax_bits with one atomic
// max each (as ints: non-negative float bits order like the values).
template <bool UNIFORM>
__global__ void __launch_bounds__(kThreads) head_amax_kernel(const Flat f) {
  __shared__ int hmax[3 * kMaxHeads];
  pdl_launch_dependents();  // programmatic dependent launch (see launch_pdl)
  const int nh = f.ntensors * f.H;
  for (int i = threadIdx.x; i < nh; i += blockDim.x) hmax[i] = 0;
  pdl_wait();
  __syncthreads();
  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t first = blockIdx.x * blockDim.x + threadIdx.x;
  auto head_of = [&](uint32_t c, const FastDiv& cpr) {
    const uint32_t row = fdiv(c, cpr);
    return row - fdiv(row, f.heads) * f.heads.d;
  };
  auto fold = [&](int* slot, uint32_t m2) {
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    if (m) atomicMax(slot, (int)(m << 16));
  };
#pragma unroll 1
  for (int ti = 0; ti < f.ntensors; ++ti) {
    const StaticTensor T = f.t[ti];
    const FastDiv cpr = f.cpr[ti];
    const uint32_t n = f.n[ti];
    if (first >= n) continue;
    int* hm = hmax + ti * f.H;
    uint32_t cur = head_of(first, cpr), m2 = 0;
    for (uint32_t base = first; base < n; base += stride * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = base + u * stride;
        v[u] = make_uint4(0, 0, 0, 0);
        if (c < n) {
          const uint32_t row = fdiv(c, cpr);
          const uint32_t col = c - row * cpr.d;
          const uint32_t tok = fdiv(row, f.heads);
          const uint32_t h = row - tok * f.heads.d;
          v[u] = __ldcs(reinterpret_cast<const uint4*>(T.x + (int64_t)tok * T.tok_stride +
                                                       (int64_t)h * T.head_stride + 8 * col));
          if (!UNIFORM && h != cur) {
            fold(&hm[cur], m2);
            cur = h;
            m2 = 0;
          }
        }
        const uint32_t a = __vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu);
        const uint32_t b = __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, __vmaxu2(a, b));
      }
    }
    fold(&hm[cur], m2);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nh; i += blockDim.x)
    if (hmax[i]) atomicMax(&f.amax_bits[i], hmax[i]);
}

Flat make_flat(const StaticParams& p, uint32_t* max_chunks) {
  Flat f = {};
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
  f.ntensors = 3;
  f.status = p.status;
  f.cu = p.cu_seqlens;
  f.nseq = p.num_seqs;
  f.T = p.T;
  *max_chunks = acc;
  return f;
}

template <typename K>
cudaError_t persistent_grid(K kern, uint32_t max_chunks, int* grid) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int64_t need = ((int64_t)max_chunks + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  *grid = (int)(need < want ? need : want);
  return cudaSuccess;
}

uint64_t gcd64(uint64_t a, uint64_t b) {
  while (b) {
    const uint64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// The amax pass over f.ntensors tensors into f.amax_bits.  The grid is a
// multiple of the block count that makes the grid-stride a multiple of every
// tensor's chunks per token (the uniform case), when that multiple fits in
// the persistent grid.
cudaError_t launch_amax_pass(const Flat& f, uint32_t max_chunks, cudaStream_t stream) {
  int grid = 0;
  cudaError_t e = persistent_grid(head_amax_kernel<true>, max_chunks, &grid);
  if (e != cudaSuccess) return e;
  uint64_t L = 1;
  for (int i = 0; i < f.ntensors; ++i) {
    const uint64_t C = (uint64_t)f.heads.d * f.cpr[i].d;  // chunks per token
    L = L / gcd64(L, C) * C;
    if (L > (1u << 30)) break;
  }
  const uint64_t unit = L / gcd64(L, kThreads);  // blocks per uniform step
  int want = 0;
  e = persistent_grid(head_amax_kernel<true>, 0xFFFFFFFFu, &want);
  if (e != cudaSuccess) return e;
  if (unit <= (uint64_t)want) {
    const int g = (int)((uint64_t)want / unit * unit);
    return launch_pdl(head_amax_kernel<true>, g, kThreads, 0, stream, f);
  }
  return launch_pdl(head_amax_kernel<false>, grid, kThreads, 0, stream, f);
}

}  // namespace

cudaError_t launch_static(const StaticParams& p, cudaStream_t stream) {
  uint32_t chunks = 0;
  const Flat f = make_flat(p, &chunks);
  int grid = 0;
  cudaError_t e = persistent_grid(static_head_kernel<false>, chunks, &grid);
  if (e != cudaSuccess) return e;
  return launch_pdl(static_head_kernel<false>, grid, kThreads, 0, stream, f);
}

// Dynamic per-head quantisation: zero the maxima, the amax pass, then the
// quantisation pass with descales RN32(amax / 448) (two launches, no waits).
cudaError_t launch_dynamic(const DynamicParams& p, cudaStream_t stream) {
  uint32_t chunks = 0;
  Flat f = make_flat(p.s, &chunks);
  f.amax_bits = reinterpret_cast<int*>(p.amax_bits);
  for (int i = 0; i < 3; ++i) f.dout[i] = p.descale_out[i];
  f.status = nullptr;
  f.cu = nullptr;
  cudaError_t e = cudaMemsetAsync(p.amax_bits, 0, sizeof(uint32_t) * 3 * (size_t)p.s.H, stream);
  if (e != cudaSuccess) return e;
  e = launch_amax_pass(f, chunks, stream);
  if (e != cudaSuccess) return e;
  int grid = 0;
  e = persistent_grid(static_head_kernel<true>, chunks, &grid);
  if (e != cudaSuccess) return e;
  return launch_pdl(static_head_kernel<true>, grid, kThreads, 0, stream, f);
}

// Calibration: the running per-head maxima of one tensor, folded into amax.
cudaError_t launch_head_amax(const AmaxParams& p, cudaStream_t stream) {
  StaticParams s = {};
  for (int i = 0; i < 3; ++i) s.t[i] = {p.x, p.tok_stride, p.head_stride, p.Dh, nullptr, nullptr};
  s.T = p.T;
  s.H = p.H;
  uint32_t chunks = 0;
  Flat f = make_flat(s, &chunks);
  f.ntensors = 1;
  f.amax_bits = reinterpret_cast<int*>(p.amax);
  return launch_amax_pass(f, chunks, stream);
}

}  // namespace fp8n
