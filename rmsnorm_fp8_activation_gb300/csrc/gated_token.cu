// (A) Gated RMSNorm fused with per-token dynamic FP8 e4m3 quantisation.
//
// Source: "[ROCm][Kimi-K3] Fuse gated RMSNorm with per-token FP8 for KDA
// o_proj" (vLLM PR 54254): one kernel for the gated norm and the per-token
// amax quantisation; the torch reference helper rounds the normalised x to
// the activation dtype, multiplies by the weight in that dtype and by
// sigmoid(gate); the wrapper quantises the [t, heads*h] row with one scale.
//
// GB300 design: a persistent grid; each CTA walks tokens t = blockIdx.x,
// blockIdx.x + gridDim.x, ...  The x and gate rows of a token (one contiguous
// H*D bf16 span each) are staged into shared memory by cp.async.bulk copies
// that complete on an mbarrier, NSTAGE tokens ahead.  Thread j of the CTA owns
// 8*CPT consecutive elements of the row, so a head of D elements belongs to
// TPH = D/(8*CPT) neighbouring lanes: its sum of squares is a Kahan sum per
// thread and a double-float butterfly over those lanes.  y stays in registers
// as bf16 pairs; the row amax needs one CTA barrier per token, after which the
// stage is refilled and the codes are written with 8-byte stores.
//
// The same kernels, specialised at compile time, also run the steps of (A) on
// their own (the unfused pipeline): the gated norm to bf16 without the
// quantisation, and the per-token quantisation of a bf16 row with or without
// the gate product in front of it.
#include "common.cuh"
#include "kernels.h"

namespace fp8n {
namespace {

// What a compile-time mode computes: y from x alone (kModeQuant), from x and
// the gate (kModeGateQuant), or through the per-head norm (kModeNormQuant,
// kModeNormOnly); then codes and scales, or (kModeNormOnly) y itself.
template <int MODE>
struct ModeOf {
  static constexpr bool norm = MODE == kModeNormQuant || MODE == kModeNormOnly;
  static constexpr bool gate = MODE != kModeQuant;
  static constexpr bool quant = MODE != kModeNormOnly;
  static constexpr int nsrc = gate ? 2 : 1;  // rows staged per token
};

constexpr int kHeader = 1024;  // mbarriers at 0, amax partials at 64

// RN32(amax / 448) for amax >= 0: the Markstein sequence with the constant
// RN(1/448) gives the IEEE quotient for every finite bf16 amax (checked
// exhaustively on the host); infinities and NaN take the plain division.
__device__ __forceinline__ float scale_of(float amax) {
  if (!(amax <= 3.402823466e38f)) return __fdiv_rn(amax, 448.0f);
  return div_rn(amax, 448.0f, 1.0f / 448.0f);
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Slot of the thread's row segment read at step c: a rotation by j/(8/CPT)
// makes the eight 16-byte reads of each quarter-warp hit distinct bank groups.
template <int CPT>
__device__ __forceinline__ int slot_of(int c, int j) {
  return CPT == 1 ? 0 : (c + j / (8 / CPT)) % CPT;
}

// y pair = bf16(bf16(bf16(RN32(x*r)) * w) * ga) for one bf16 pair, where ga
// is the bf16 pair bf16(act(g)).
__device__ __forceinline__ uint32_t gated_pair(uint32_t xw, uint32_t ga, uint32_t ww, f2_t r2) {
  const uint32_t xn = f2_to_bf2(mul2(bf2_to_f2(xw), r2));
  return mul_bf16x2(mul_bf16x2(xn, ww), ga);
}

// Running max of |y| over bf16 pairs (NaN-propagating); acc stays >= 0.
__device__ __forceinline__ uint32_t amax_step(uint32_t acc, uint32_t y) {
  uint32_t d;
  asm("{\n .reg .b32 t;\n abs.bf16x2 t, %2;\n max.NaN.bf16x2 %0, %1, t;\n}\n"
      : "=r"(d) : "r"(acc), "r"(y));
  return d;
}

// Gate-activation table in shared memory: entry e (0 <= e < 8192) holds
// bf16(act(g)) for the bf16 gate with sign e >> 12 and magnitude bits
// kLutBase + (e & 0xFFF), i.e. every gate with 2^-15 <= |g| < 2^17.  Each CTA
// fills it once with act_bf16_pair (exact), so a lookup is the same value.
constexpr uint32_t kLutBase = 0x3800u;  // 2^-15
constexpr int kLutEntries = 8192;
constexpr int kLutBytes = 2 * kLutEntries;

template <int ACT>
__device__ __forceinline__ void lut_fill(uint32_t* lut32, int tid, int nthreads) {
  for (int w = tid; w < kLutEntries / 2; w += nthreads) {
    const uint32_t e0 = 2u * (uint32_t)w, e1 = e0 + 1u;
    const uint32_t g0 = ((e0 >> 12) << 15) | (kLutBase + (e0 & 0xFFFu));
    const uint32_t g1 = ((e1 >> 12) << 15) | (kLutBase + (e1 & 0xFFFu));
    lut32[w] = act_bf16_pair(g0 | (g1 << 16), ACT);
  }
}

// bf16(act()) of a chunk of four gate pairs through the table.  With
// d = |g| - base per half, both halves of every pair are in range when no
// d has a bit in 0xF000 (a magnitude below the base borrows into those bits);
// then 2d | (sign bits moved to bit 13) is the pair of byte offsets.  A chunk
// with any lane out of range takes the arithmetic path for all its pairs.
template <int ACT>
__device__ __forceinline__ void lut_chunk(const uint8_t* lut, const uint32_t g[4], uint32_t ga[4]) {
  uint32_t d[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) d[k] = (g[k] & 0x7FFF7FFFu) - (kLutBase | (kLutBase << 16));
  if ((d[0] | d[1] | d[2] | d[3]) & 0xF000F000u) {
#pragma unroll
    for (int k = 0; k < 4; ++k) ga[k] = act_bf16_pair(g[k], ACT);
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t off = (d[k] * 2u) | ((g[k] >> 2) & 0x20002000u);
    const uint32_t v0 = *reinterpret_cast<const uint16_t*>(lut + (off & 0xFFFFu));
    const uint32_t v1 = *reinterpret_cast<const uint16_t*>(lut + (off >> 16));
    ga[k] = __byte_perm(v0, v1, 0x5410);
  }
}

// Token quantiser: code = e4m3(RN32(y / scale)), from the correctly rounded
// reciprocal and one FMA correction on packed pairs.  It is arranged on -y
// (q0 = (-y)*(-1/s), e = q0*s - y, q = q0 - e/s) so that the signs of zero
// quotients survive.  A zero scale gives signed zero codes.  The correction is
// exact while the residual e does not underflow, which holds for every
// quotient that can reach a nonzero code (|q| >= 2^-11) once s >= 2^-60;
// smaller scales (|y| tiny) first multiply y and the scale by 2^64, an exact
// rescaling that keeps the quotient.
struct TokenQuant {
  f2_t s2, nrs2;
  bool zero, tiny;
  __device__ __forceinline__ TokenQuant(float s) {
    zero = (s == 0.0f);
    tiny = (s > 0.0f) && (s < 0x1p-60f);
    const float sc = tiny ? __fmul_rn(s, 0x1p64f) : s;
    s2 = splat2(sc);
    nrs2 = splat2(-__frcp_rn(sc));
  }
  template <bool TINY>
  __device__ __forceinline__ uint32_t pair(uint32_t y) const {
    if (zero) return f2_to_e4m3x2(bf2_to_f2(y));
    f2_t ny = neg_bf2_to_f2(y);
    if (TINY) ny = mul2(ny, splat2(0x1p64f));
    const f2_t q0 = mul2(ny, nrs2);
    const f2_t e = fma2(q0, s2, ny);
    return f2_to_e4m3x2(fma2(e, nrs2, q0));
  }
  template <bool TINY>
  __device__ __forceinline__ uint2 chunk(const uint32_t y[4]) const {
    return make_uint2(pair<TINY>(y[0]) | (pair<TINY>(y[1]) << 16),
                      pair<TINY>(y[2]) | (pair<TINY>(y[3]) << 16));
  }
};

// The exact mean square of the heads flagged in a warp (D a power of two):
// from the heads' sums of squares in 128-bit integers, or, for a head whose
// exponents span too much for that, in double-double (every lane sums its
// `count` chunks at p, the TPH lanes of a head combine), from which a flagged
// lane steps ms to RN32(S / D).  Called by the whole warp.
static __device__ __noinline__ float head_ms_exact(const uint4* p, int count, int tph, int D,
                                                   float ms, bool flagged) {
  int log2d = 0;
  while ((1 << log2d) < D) ++log2d;
  float mi = ms;
  const bool ok = head_ms_int(p, 1, count, tph, log2d, &mi);
  if (!__any_sync(0xFFFFFFFFu, flagged && !ok)) return flagged ? mi : ms;
  dd Sd = sumsq_dd(p, 1, count);
  for (int m = 1; m < tph; m <<= 1) Sd = dd_add(Sd, shfl_xor_dd(Sd, m));
  if (!flagged) return ms;
  return ok ? mi : ms_resolve(Sd, (float)D, ms);
}

// Sum of squares of a head in the staged layout, from the thread's segment
// xs (CPT 16-byte chunks, read in the rotated order): two Sum2 chains (even
// and odd chunks) per thread, so that each running sum takes at most 8
// additions, then the butterfly over the head's TPH lanes.
template <int CPT, int TPH>
__device__ __forceinline__ df head_sum(const uint8_t* xs, int tid, bool active) {
  sumsq2 acc[2];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const uint4 xv = active ? *reinterpret_cast<const uint4*>(xs + 16 * slot_of<CPT>(c, tid))
                            : make_uint4(0, 0, 0, 0);
    const uint32_t* xw = &xv.x;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[c & 1].add_sq(xw[k]);
  }
  df S = CPT > 1 ? df_add(acc[0].value(), acc[1].value()) : acc[0].value();
#pragma unroll
  for (int m = 1; m < TPH; m <<= 1) S = df_add(S, shfl_xor_df(S, m));
  return S;
}

// Relative error bound of head_sum.
template <int CPT, int TPH>
__host__ __device__ __forceinline__ float head_sum_rel_err() {
  int lg = 0;
  while ((1 << lg) < TPH) ++lg;
  return sumsq_rel_err(4 * ((CPT + 1) / 2), 3 + lg);
}

// The fused quantisation's head sum: the same layout with one Kahan-
// compensated chain per thread (two packed lanes; four operations per pair
// instead of Sum2's eight).  It is not an exact sum: in rare heads (a large
// square after a smaller running sum, or compensation bits below a term's
// precision) RN32(S / D) comes out one binary32 ulp off, which moves a code by
// one step at most, rarely (about one code in 10^7 on the benchmark data);
// that is the reduction-order budget of the per-token codes, and it keeps this
// kernel at the HBM roofline.
template <int CPT, int TPH>
__device__ __forceinline__ df head_sum_fast(const uint8_t* xs, int tid, bool active) {
  kahan2 acc;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const uint4 xv = active ? *reinterpret_cast<const uint4*>(xs + 16 * slot_of<CPT>(c, tid))
                            : make_uint4(0, 0, 0, 0);
    const uint32_t* xw = &xv.x;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc.add_sq(xw[k]);
  }
  df S = acc.value();
#pragma unroll
  for (int m = 1; m < TPH; m <<= 1) S = df_add(S, shfl_xor_df(S, m));
  return S;
}

// Whether head_sum's double-float S is the exact sum of squares of the head
// (sum_is_exact over the head's elements).  Heads of bf16 data often sum
// exactly to a binary32 tie; this settles them without the double-double
// sum.  Called by the whole warp.
template <int CPT, int TPH>
__device__ __forceinline__ bool head_sum_exact(const uint8_t* xs, bool active, float Sh) {
  uint32_t emin = 255u;
  if (active) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(xs + 16 * c);
      emin = emin_pair(emin_pair(emin_pair(emin_pair(emin, v.x), v.y), v.z), v.w);
    }
  }
#pragma unroll
  for (int m = 1; m < TPH; m <<= 1) emin = min(emin, __shfl_xor_sync(0xFFFFFFFFu, emin, m));
  return sum_is_exact(emin, Sh, 4 * ((CPT + 1) / 2));
}


template <int MODE, int ACT, int CPT, int TPH, bool LUT>
__global__ void __launch_bounds__(512) gated_token_tma(const GatedParams p, int nstage) {
  using M = ModeOf<MODE>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int row = p.H * p.D;
  const uint32_t row_bytes = 2u * (uint32_t)row;
  const uint32_t stage_bytes = M::nsrc * row_bytes;
  const int nthr = row / (8 * CPT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const bool active = tid < nthr;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* red = reinterpret_cast<uint32_t*>(smem + 64);  // per-warp amax bits
  uint8_t* lut = smem + kHeader;  // at a fixed offset: its base folds into the loads
  uint16_t* wsm = reinterpret_cast<uint16_t*>(smem + kHeader + (LUT ? kLutBytes : 0));  // weight [D]
  uint8_t* stages = smem + kHeader + (LUT ? kLutBytes : 0) + (M::norm ? 2 * p.D : 0);

  auto issue = [&](int s, int64_t t) {
    uint32_t bar = smem_u32(&bars[s]);
    uint32_t dst = smem_u32(stages + (size_t)s * stage_bytes);
    mbar_expect_tx(bar, stage_bytes);
    bulk_g2s(dst, p.x + t * p.x_stride, row_bytes, bar);
    if (M::gate) bulk_g2s(dst + row_bytes, p.gate + t * p.gate_stride, row_bytes, bar);
  };
  // programmatic dependent launch: the next kernel of the stream may start its
  // launch now (it waits for this one to finish before it touches memory), and
  // this one touches global memory only once the previous kernel is done
  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) mbar_init(smem_u32(&bars[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();
  // the first rows are requested before anything else, so that their copies
  // overlap the weight load and the table fill
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
      if (t < p.T) issue(s, t);
    }
  }
  if (M::norm)
    for (int i = tid; i < p.D / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(wsm)[i] = reinterpret_cast<const uint4*>(p.weight)[i];
  for (int i = tid; i < 64; i += blockDim.x) red[i] = 0u;  // both halves of the warp maxima
  __syncthreads();
  if (LUT) {  // filled while the first rows are in flight
    lut_fill<ACT>(reinterpret_cast<uint32_t*>(lut), tid, blockDim.x);
    __syncthreads();
  }

  const int seg = tid * 8 * CPT;  // first element of the thread's segment
  // an idle thread (past the row) reads segment 0 and is masked out of the
  // token maximum and the stores, so that no read needs a test
  const int rseg = active ? seg : 0;
  const uint16_t* wseg = wsm + (rseg % p.D);
  const float inv_d = 1.0f / (float)p.D;  // exact: D is a power of two here
  // error bound of a head's sum relative to S, plus the squares below 2^-126
  // that binary32 rounds (at most 2^-150 each)
  const float rel_err = head_sum_rel_err<CPT, TPH>();
  const float sq_floor = (float)p.D * 0x1p-149f;

  int it = 0;
  bool timeout = false;
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, ++it) {
    const int s = it % nstage;
    if (!mbar_wait(smem_u32(&bars[s]), (uint32_t)(it / nstage) & 1u, kWaitLimitMain)) timeout = true;
    const uint8_t* sx = stages + (size_t)s * stage_bytes + (size_t)rseg * 2;
    const uint8_t* sg = sx + row_bytes;

    // pass 1: the head's sum of squares (x is read again in pass 2) and ms =
    // RN32(S / D).  The quantisation takes the fast compensated sum.  The bf16
    // output of the gated norm takes the exact one: Sum2, then RN32(S) is
    // decided when it is the same at both ends of S's error interval (RN is
    // monotone; the probes' own roundings are far below err; S.h == 0 means
    // every square is at most 2^-150, and then so is S / D: its rounding is
    // 0), else a certified-exact sum needs nothing more, else the integer
    // path.  The lanes of a head agree on S, so a head is flagged as a whole.
    float ms = 0.0f;
    if (M::norm && M::quant) {
      const df S = head_sum_fast<CPT, TPH>(sx, tid, true);
      ms = __fmul_rn(__fadd_rn(S.h, S.l), inv_d);
    } else if (M::norm) {
      df S = head_sum<CPT, TPH>(sx, tid, true);
      const float err = __fmaf_rn(S.h, rel_err, sq_floor);
      bool unsure = S.h != 0.0f &&
                    __fadd_rn(S.h, __fadd_rn(S.l, err)) != __fadd_rn(S.h, __fsub_rn(S.l, err));
      ms = __fmul_rn(__fadd_rn(S.h, S.l), inv_d);
      if (__any_sync(0xFFFFFFFFu, unsure)) {
        const bool exact = head_sum_exact<CPT, TPH>(sx, active, S.h);  // every lane: shuffles
        unsure = unsure && !exact;
        if (__any_sync(0xFFFFFFFFu, unsure))
          ms = head_ms_exact(reinterpret_cast<const uint4*>(sx), active ? CPT : 0, TPH, p.D, ms, unsure);
      }
    }

    // pass 2: y (= bf16(bf16(bf16(x r) w) act(g)) through the norm), kept as bf16 pairs
    const f2_t r2 = splat2(M::norm ? rms_factor(ms, p.eps) : 1.0f);
    uint32_t y[CPT][4];
    uint32_t am2 = 0;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int off = 16 * slot_of<CPT>(c, tid);
      const uint4 xv = *reinterpret_cast<const uint4*>(sx + off);
      const uint4 gv = M::gate ? *reinterpret_cast<const uint4*>(sg + off) : make_uint4(0, 0, 0, 0);
      const uint32_t *xw = &xv.x, *gw = &gv.x;
      uint32_t ga[4];
      if (M::gate) {
        if (LUT) {
          lut_chunk<ACT>(lut, gw, ga);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) ga[k] = act_bf16_pair(gw[k], ACT);
        }
      }
      if (M::norm) {
        const uint4 wv = *reinterpret_cast<const uint4*>(wseg + 8 * slot_of<CPT>(c, tid));
        const uint32_t* ww = &wv.x;
#pragma unroll
        for (int k = 0; k < 4; ++k) y[c][k] = gated_pair(xw[k], ga[k], ww[k], r2);
      } else if (M::gate) {
#pragma unroll
        for (int k = 0; k < 4; ++k) y[c][k] = mul_bf16x2(xw[k], ga[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) y[c][k] = xw[k];
      }
      if (M::quant) {
#pragma unroll
        for (int k = 0; k < 4; ++k) am2 = amax_step(am2, y[c][k]);
      }
    }
    if (!active) am2 = 0u;  // an idle lane's y is not part of the row
    // the token amax as bf16 bits: non-negative bf16 values (NaN above
    // infinity) order as unsigned integers, so one warp reduction takes it
    uint32_t* redb = red + (it & 1) * 32;
    if (M::quant) {
      const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, max(am2 & 0xFFFFu, am2 >> 16));
      redb[warp] = wmax;  // (every lane stores the same value)
    }
    // every thread is done with stage s and has published its warp's amax; a
    // wait that gave up in any thread stops the whole CTA (thread 0 drains)
    if (__syncthreads_or(timeout)) {
      timeout = true;
      break;
    }
    if (tid == 0) {
      const int64_t tn = t + (int64_t)nstage * gridDim.x;
      if (tn < p.T) {
        // the threads' reads of stage s come before the copy that overwrites it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(s, tn);
      }
    }
    if (!M::quant) {
      if (active) {
        uint16_t* yrow = p.y_out + t * p.y_stride + seg;
#pragma unroll
        for (int c = 0; c < CPT; ++c)
          *reinterpret_cast<uint4*>(yrow + 8 * slot_of<CPT>(c, tid)) =
              make_uint4(y[c][0], y[c][1], y[c][2], y[c][3]);
      }
      continue;
    }
    uint32_t tbits = 0u;  // the slots past the last warp hold 0
    for (int w = 0; w < nwarps; w += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(redb + w);
      tbits = max(max(tbits, v.x), max(v.y, max(v.z, v.w)));
    }
    // (max.NaN makes a NaN amax the canonical NaN)
    const float scale = scale_of(fmax_nan(__uint_as_float(tbits << 16), 0.0f));
    if (tid == 0) p.scale[t] = scale;
    if (active) {
      const TokenQuant tq(scale);
      uint8_t* orow = p.out + t * p.out_stride + seg;
      if (!tq.tiny) {
#pragma unroll
        for (int c = 0; c < CPT; ++c)
          *reinterpret_cast<uint2*>(orow + 8 * slot_of<CPT>(c, tid)) = tq.chunk<false>(y[c]);
      } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c)
          *reinterpret_cast<uint2*>(orow + 8 * slot_of<CPT>(c, tid)) = tq.chunk<true>(y[c]);
      }
    }
  }

  if (timeout && tid == 0) {
    if (p.status) atomicOr(p.status, kStatusTimeout);
    // let copies still in flight land before the CTA's shared memory goes away
    for (int i = it; i < it + nstage; ++i) {
      const int64_t ti = blockIdx.x + (int64_t)i * gridDim.x;
      if (ti < p.T) mbar_wait(smem_u32(&bars[i % nstage]), (uint32_t)(i / nstage) & 1u, kWaitLimit);
    }
  }
}

// One token of the generic path (any D that is a multiple of 8; the CTA
// works on the token together): chunk sums of squares, per-head mean squares
// (exact: a head its double-float sum cannot decide is summed again in
// double-double), then y and the amax, then y again and the codes (or,
// without the quantisation, y itself).  Shared memory: the chunk sums, the
// head factors and the warp maxima.
template <int MODE, int ACT>
__device__ __forceinline__ void generic_token(const GatedParams& p, int64_t t, uint8_t* smem) {
  using M = ModeOf<MODE>;
  const int row = p.H * p.D, nch = row / 8, cph = p.D / 8;
  df* part = reinterpret_cast<df*>(smem);
  float* rf = reinterpret_cast<float*>(smem + (size_t)nch * sizeof(df));
  float* red = rf + p.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const float n = (float)p.D;
  const uint16_t* xrow = p.x + t * p.x_stride;
  const uint16_t* grow = p.gate + t * p.gate_stride;
  if (M::norm) {
    for (int c = tid; c < nch; c += blockDim.x) {
      const uint4 v = *reinterpret_cast<const uint4*>(xrow + 8 * c);
      sumsq2 acc;
      const uint32_t* w = &v.x;
#pragma unroll
      for (int k = 0; k < 4; ++k) acc.add_sq(w[k]);
      part[c] = acc.value();
    }
    __syncthreads();
    for (int h = warp; h < p.H; h += nwarps) {  // warp-uniform: one head per warp
      df S = {0.0f, 0.0f};
      for (int c = lane; c < cph; c += 32) S = df_add(S, part[h * cph + c]);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) S = df_add(S, shfl_xor_df(S, m));
      float ms = mean_from_sum(S, n, 0.0f, false);
      const float err = __fmaf_rn(S.h, sumsq_rel_err(4, (cph + 31) / 32 + 6), n * 0x1p-149f);
      const bool unsure = ms_uncertain(S, n, ms, err);
      if (__any_sync(0xFFFFFFFFu, unsure)) {
        const int cnt = lane < cph ? (cph - lane + 31) / 32 : 0;
        dd Sd = sumsq_dd(reinterpret_cast<const uint4*>(xrow + (size_t)h * p.D) + lane, 32, cnt);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) Sd = dd_add(Sd, shfl_xor_dd(Sd, m));
        if (unsure) ms = ms_resolve(Sd, n, ms);
      }
      if (lane == 0) rf[h] = rms_factor(ms, p.eps);
    }
    __syncthreads();
  }

  auto y_chunk = [&](int c, uint32_t y[4]) {
    const uint4 xv = *reinterpret_cast<const uint4*>(xrow + 8 * c);
    const uint32_t* xw = &xv.x;
    if (!M::gate) {
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = xw[k];
      return;
    }
    const uint4 gv = *reinterpret_cast<const uint4*>(grow + 8 * c);
    const uint32_t* gw = &gv.x;
    if (M::norm) {
      const uint4 wv = *reinterpret_cast<const uint4*>(p.weight + 8 * (c % cph));
      const f2_t r2 = splat2(rf[c / cph]);
      const uint32_t* ww = &wv.x;
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = gated_pair(xw[k], act_bf16_pair(gw[k], ACT), ww[k], r2);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = mul_bf16x2(xw[k], act_bf16_pair(gw[k], ACT));
    }
  };

  if (!M::quant) {
    uint16_t* yrow = p.y_out + t * p.y_stride;
    for (int c = tid; c < nch; c += blockDim.x) {
      uint32_t y[4];
      y_chunk(c, y);
      *reinterpret_cast<uint4*>(yrow + 8 * c) = make_uint4(y[0], y[1], y[2], y[3]);
    }
    __syncthreads();  // part / rf are reused by the next token
    return;
  }

  uint32_t am2 = 0;
  for (int c = tid; c < nch; c += blockDim.x) {
    uint32_t y[4];
    y_chunk(c, y);
#pragma unroll
    for (int k = 0; k < 4; ++k) am2 = amax_step(am2, y[k]);
  }
  float amax = fmax_nan(bf16_lo(am2), bf16_hi(am2));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmax_nan(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  float tam = red[0];
  for (int w = 1; w < nwarps; ++w) tam = fmax_nan(tam, red[w]);
  const float scale = scale_of(tam);
  const TokenQuant tq(scale);
  if (tid == 0) p.scale[t] = scale;
  uint8_t* orow = p.out + t * p.out_stride;
  for (int c = tid; c < nch; c += blockDim.x) {
    uint32_t y[4];
    y_chunk(c, y);
    *reinterpret_cast<uint2*>(orow + 8 * c) = tq.tiny ? tq.chunk<true>(y) : tq.chunk<false>(y);
  }
  __syncthreads();  // part / rf / red are reused by the next token
}

// Head sizes and row lengths the staged kernel does not take: one CTA per
// token at a time, rows strided over a persistent grid.
template <int MODE, int ACT>
__global__ void __launch_bounds__(256) gated_token_generic(const GatedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_launch_dependents();  // programmatic dependent launch (see launch_pdl)
  pdl_wait();
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) generic_token<MODE, ACT>(p, t, smem);
}

// Rows of 16 KB or more per stage get one stage per CTA, so that four CTAs
// fit on an SM and the loads of the others overlap each CTA's compute (its own
// next row also lands while it quantises); shorter rows get two stages.  The
// gate table is used when each CTA walks enough tokens to pay for filling it.
// The grid is the SM count times the CTAs that fit.
template <int MODE, int ACT, int CPT, int TPH, bool LUT>
cudaError_t launch_tma_v(const GatedParams& p, cudaStream_t stream) {
  using M = ModeOf<MODE>;
  auto kern = gated_token_tma<MODE, ACT, CPT, TPH, LUT>;
  const int row = p.H * p.D;
  const int nthr = row / (8 * CPT);
  const int block = (nthr + 31) / 32 * 32;
  const size_t stage_bytes = 2u * M::nsrc * (size_t)row;
  const int nstage = stage_bytes >= 32 * 1024 ? 1 : 2;
  const size_t smem =
      kHeader + (M::norm ? 2 * (size_t)p.D : 0) + (LUT ? kLutBytes : 0) + nstage * stage_bytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, block, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int grid = (int)(p.T < want ? p.T : want);
  return launch_pdl(kern, grid, block, smem, stream, p, nstage);
}

template <int MODE, int ACT, int CPT, int TPH>
cudaError_t launch_tma(const GatedParams& p, cudaStream_t stream) {
  if (ModeOf<MODE>::gate) {
    // filling the table costs about as much as 8192 activations computed in
    // the arithmetic path; it pays when each CTA evaluates twice that many
    const int64_t per_cta = p.T / ((int64_t)sm_count() * 4);
    if (per_cta * p.H * p.D >= 2 * kLutEntries)
      return launch_tma_v<MODE, ACT, CPT, TPH, true>(p, stream);
  }
  return launch_tma_v<MODE, ACT, CPT, TPH, false>(p, stream);
}

// Shared memory of the generic path: chunk sums, head factors, warp maxima.
inline size_t generic_smem(const GatedParams& p) {
  return (size_t)(p.H * p.D / 8) * sizeof(df) + (size_t)p.H * 4 + 32 * 4;
}


template <int MODE, int ACT>
cudaError_t launch_generic(const GatedParams& p, cudaStream_t stream) {
  auto kern = gated_token_generic<MODE, ACT>;
  const size_t smem = generic_smem(p);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int grid = (int)(p.T < want ? p.T : want);
  return launch_pdl(kern, grid, 256, smem, stream, p);
}

template <int MODE, int ACT>
cudaError_t dispatch(const GatedParams& p, cudaStream_t stream) {
  const int row = p.H * p.D;
  if (!ModeOf<MODE>::norm) {
    // no per-head reduction: the staged kernel takes any row of whole
    // 32-element chunks (four per thread) that fits one CTA and a stage
    if (row % 32 == 0 && row / 32 <= 512 && 2 * ModeOf<MODE>::nsrc * row <= 64 * 1024)
      return launch_tma<MODE, ACT, 4, 1>(p, stream);
    return launch_generic<MODE, ACT>(p, stream);
  }
  // staged kernel: D/8 a power of two, a head spans at most a warp, the row
  // fits one CTA and a stage fits shared memory.  A batch that gives each CTA
  // at most one token (decode) spreads a D = 128 head over 16 lanes of one
  // chunk each instead of 4 lanes of four: shorter chains per thread, the
  // same arithmetic.
  int cpt = p.D >= 32 ? 4 : p.D / 8;
  if (p.D == 128 && p.T <= sm_count() && row / 8 <= 512) cpt = 1;
  const int tph = p.D / (8 * cpt);
  const bool pow2 = (p.D & (p.D - 1)) == 0;
  if (pow2 && tph >= 1 && tph <= 32 && row / (8 * cpt) <= 512 && 4 * row <= 64 * 1024) {
    switch (cpt * 100 + tph) {
      case 101: return launch_tma<MODE, ACT, 1, 1>(p, stream);
      case 116: return launch_tma<MODE, ACT, 1, 16>(p, stream);
      case 201: return launch_tma<MODE, ACT, 2, 1>(p, stream);
      case 401: return launch_tma<MODE, ACT, 4, 1>(p, stream);
      case 402: return launch_tma<MODE, ACT, 4, 2>(p, stream);
      case 404: return launch_tma<MODE, ACT, 4, 4>(p, stream);
      case 408: return launch_tma<MODE, ACT, 4, 8>(p, stream);
      case 416: return launch_tma<MODE, ACT, 4, 16>(p, stream);
      case 432: return launch_tma<MODE, ACT, 4, 32>(p, stream);
      default: break;
    }
  }
  return launch_generic<MODE, ACT>(p, stream);
}

template <int MODE>
cudaError_t dispatch_act(const GatedParams& p, cudaStream_t stream) {
  return p.act == kActSilu ? dispatch<MODE, kActSilu>(p, stream)
                           : dispatch<MODE, kActSigmoid>(p, stream);
}

}  // namespace

cudaError_t launch_gated(const GatedParams& p, cudaStream_t stream) {
  switch (p.mode) {
    case kModeNormQuant: return dispatch_act<kModeNormQuant>(p, stream);
    case kModeGateQuant: return dispatch_act<kModeGateQuant>(p, stream);
    case kModeQuant: return dispatch<kModeQuant, kActSigmoid>(p, stream);
    case kModeNormOnly: return dispatch_act<kModeNormOnly>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp8n
