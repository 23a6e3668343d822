// (B) Fused q/kv RMSNorm: q leaves as MXFP8 (E4M3 elements, one E8M0 scale
// per 32 consecutive elements, scales row-major), kv as normalised bf16.
//
// Source: "[ROCm][Perf] FP8 o-projection for DeepSeek-V4.1-Flash MLA on AMD
// MI355X" (vLLM PR 57081), third commit message: one producer normalises q
// and kv and emits q as MXFP8 with row-major E8M0 scales, so the two q
// consumers read the same quantised tensor.  Block scale rule: OCP
// Microscaling Formats v1.0 section 5, X = 2^(floor(log2 amax) - 8) for E4M3.
//
// GB300 design: one warp per row, rows strided over a persistent grid.  Lane
// l owns the 16-byte chunks l, l+32, l+64, ... of the q row and of the kv row
// (coalesced 512-byte steps), kept in registers between the two passes (sum
// of squares, then normalise + quantise).  An MX block is four consecutive
// chunks, i.e. four neighbouring lanes of one step, so its amax takes two
// xor-shuffles.  Rows longer than eight steps are read twice instead.
//
// The same kernels run the two steps of (B) on their own: with no q columns,
// the row RMSNorm to bf16 (the kv path); with q_prenorm set, the MX
// quantisation of an already normalised bf16 q.
#include "common.cuh"
#include "kernels.h"

namespace fp8n {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// bf16(bf16(RN32(x * r)) * w) for a chunk of 8 (4 pairs).
__device__ __forceinline__ uint32_t norm_pair(uint32_t x, uint32_t w, f2_t r2) {
  return mul_bf16x2(f2_to_bf2(mul2(bf2_to_f2(x), r2)), w);
}
__device__ __forceinline__ void norm_chunk(const uint4& xv, const uint4& wv, f2_t r2, uint32_t y[4]) {
  y[0] = norm_pair(xv.x, wv.x, r2);
  y[1] = norm_pair(xv.y, wv.y, r2);
  y[2] = norm_pair(xv.z, wv.z, r2);
  y[3] = norm_pair(xv.w, wv.w, r2);
}
__device__ __forceinline__ uint4 norm_chunk4(const uint4& xv, const uint4& wv, f2_t r2) {
  return make_uint4(norm_pair(xv.x, wv.x, r2), norm_pair(xv.y, wv.y, r2), norm_pair(xv.z, wv.z, r2),
                    norm_pair(xv.w, wv.w, r2));
}

// E8M0 exponent e (scale 2^e) of a block whose amax has bf16 bits A (>= 0):
// floor(log2 A) - 8 clamped to [-127, 127]; -127 for a zero block; the code
// 0xFF (returned as e = 128) for NaN or infinity.
__device__ __forceinline__ int mx_exponent(uint32_t A) {
  if (A >= 0x7F80u) return 128;
  if (A == 0u) return -127;
  const uint32_t ef = A >> 7;
  const int E = ef ? (int)ef - 127 : -133 + (31 - __clz((int)(A & 0x7Fu)));
  const int e = E - 8;
  return e < -127 ? -127 : e;  // E <= 127, so e <= 119
}

// ms = RN32(S / n) of one row from its double-float sum of squares S
// (reduced over the warp, so every lane holds it and the flag is the same on
// every lane), and whether S may not decide that rounding (then
// row_ms_exact settles it).
__device__ __forceinline__ float row_ms(df S, int n, bool n_pow2, int steps, bool* unsure) {
  const float nf = (float)n;
  const float ms = mean_from_sum(S, nf, 1.0f / nf, n_pow2);
  *unsure = ms_uncertain(S, nf, ms, __fmaf_rn(S.h, sumsq_rel_err(4 * steps, 6), nf * 0x1p-149f));
  return ms;
}

// The exact ms of a row whose double-float sum S could not decide it: when
// S is itself exact (sum_is_exact over the row's elements; lane l holds
// chunks l, l + 32, ...) in binary32, else from the chunks summed in
// double-double over the warp.  Called by all lanes of the warp together.
static __device__ __noinline__ float row_ms_exact(const uint4* row, int n, df S, int steps, float ms,
                                                  int lane) {
  const int ch = n / 8;
  const int cnt = lane < ch ? (ch - lane + 31) / 32 : 0;
  uint32_t emin = 255u;
  for (int i = 0; i < cnt; ++i) {
    const uint4 v = row[lane + 32 * i];
    emin = emin_pair(emin_pair(emin_pair(emin_pair(emin, v.x), v.y), v.z), v.w);
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) emin = min(emin, __shfl_xor_sync(0xFFFFFFFFu, emin, s));
  if (sum_is_exact(emin, S.h, 4 * steps)) return ms_resolve_exact(S, (float)n, ms);
  dd Sd = sumsq_dd(row + lane, 32, cnt);
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) Sd = dd_add(Sd, shfl_xor_dd(Sd, s));
  return ms_resolve(Sd, (float)n, ms);
}

// QS / KS: 512-byte steps of the q / kv row held in registers between the two
// passes (0: the row is read again in the second pass).
template <int QS, int KS>
__global__ void __launch_bounds__(kWarps * 32, (QS + KS >= 8) ? 2 : 3) rmsnorm_mx_kernel(const MxParams p) {
  constexpr bool RESIDENT = QS > 0;
  pdl_launch_dependents();  // programmatic dependent launch (see launch_pdl)
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int qch = p.Nq / 8, kch = p.Nkv / 8;
  const int qsteps = (qch + 31) / 32, ksteps = (kch + 31) / 32;
  const bool q_pow2 = (p.Nq & (p.Nq - 1)) == 0, k_pow2 = (p.Nkv & (p.Nkv - 1)) == 0;
  const bool q_norm = qch > 0 && !p.q_prenorm;

  for (int64_t m = gwarp; m < p.M; m += nwarps) {
    const uint16_t* qrow = p.q + m * p.q_stride;
    const uint16_t* krow = p.kv + m * p.kv_stride;
    constexpr int QR = QS > 0 ? QS : 1, KR = KS > 0 ? KS : 1;
    uint4 qr[QR], kr[KR];
    sumsq2 aq, ak;
    if (RESIDENT) {
#pragma unroll
      for (int j = 0; j < QR; ++j) {
        const int c = 32 * j + lane;
        qr[j] = make_uint4(0, 0, 0, 0);
        if (c < qch) qr[j] = *reinterpret_cast<const uint4*>(qrow + 8 * c);
      }
#pragma unroll
      for (int j = 0; j < KR; ++j) {
        const int c = 32 * j + lane;
        kr[j] = make_uint4(0, 0, 0, 0);
        if (c < kch) kr[j] = *reinterpret_cast<const uint4*>(krow + 8 * c);
      }
      if (!p.q_prenorm) {
#pragma unroll
        for (int j = 0; j < QR; ++j) {
          const uint32_t* qw = &qr[j].x;
#pragma unroll
          for (int k = 0; k < 4; ++k) aq.add_sq(qw[k]);
        }
      }
#pragma unroll
      for (int j = 0; j < KR; ++j) {
        const uint32_t* kw = &kr[j].x;
#pragma unroll
        for (int k = 0; k < 4; ++k) ak.add_sq(kw[k]);
      }
    } else {
      for (int c = lane; c < (p.q_prenorm ? 0 : qch); c += 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + 8 * c);
        const uint32_t* w = &v.x;
#pragma unroll
        for (int k = 0; k < 4; ++k) aq.add_sq(w[k]);
      }
      for (int c = lane; c < kch; c += 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(krow + 8 * c);
        const uint32_t* w = &v.x;
#pragma unroll
        for (int k = 0; k < 4; ++k) ak.add_sq(w[k]);
      }
    }
    df Sq = aq.value(), Sk = ak.value();
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
      Sq = df_add(Sq, shfl_xor_df(Sq, s));
      Sk = df_add(Sk, shfl_xor_df(Sk, s));
    }
    bool uq = false, uk = false;
    float msq = q_norm ? row_ms(Sq, p.Nq, q_pow2, qsteps, &uq) : 0.0f;
    float msk = kch ? row_ms(Sk, p.Nkv, k_pow2, ksteps, &uk) : 0.0f;
    if (uq) msq = row_ms_exact(reinterpret_cast<const uint4*>(qrow), p.Nq, Sq, qsteps, msq, lane);  // rare
    if (uk) msk = row_ms_exact(reinterpret_cast<const uint4*>(krow), p.Nkv, Sk, ksteps, msk, lane);
    const f2_t rq = splat2(q_norm ? rms_factor(msq, p.eps) : 0.0f);
    const f2_t rk = splat2(kch ? rms_factor(msk, p.eps) : 0.0f);

    uint8_t* qo = p.q_out + m * p.q_out_stride;
    uint8_t* so = p.q_scale + m * p.q_scale_stride;
    uint16_t* ko = p.kv_out + m * p.kv_out_stride;
    // one 512-byte step of q: normalise, MX-quantise (all lanes take part in
    // the block shuffles; lanes past the row end carry zeros)
    auto q_step = [&](int j, const uint4& xv) {
      const int c = 32 * j + lane;
      uint32_t y[4];
      if (p.q_prenorm) {
        y[0] = xv.x, y[1] = xv.y, y[2] = xv.z, y[3] = xv.w;
      } else {
        uint4 wv = make_uint4(0, 0, 0, 0);
        if (c < qch) wv = *reinterpret_cast<const uint4*>(p.q_weight + 8 * c);
        norm_chunk(xv, wv, rq, y);
      }
      uint32_t am = absmax_bf16x2(absmax_bf16x2(y[0], y[1]), absmax_bf16x2(y[2], y[3]));
      am = absmax_bf16x2(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      am = absmax_bf16x2(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
      const uint32_t A = __float_as_uint(fmax_nan(bf16_lo(am), bf16_hi(am))) >> 16;
      const int e = mx_exponent(A);
      if (c < qch) {
        if ((lane & 3) == 0) so[c >> 2] = (uint8_t)(e + 127);
        uint2 o;
        if (e == 128) {
          o = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else {
          const float sc = pow2i(-e);  // exact power-of-two scaling
          uint32_t b[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            b[k] = e4m3x2(__fmul_rn(bf16_lo(y[k]), sc), __fmul_rn(bf16_hi(y[k]), sc));
          o = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
        }
        *reinterpret_cast<uint2*>(qo + 8 * c) = o;
      }
    };
    auto kv_step = [&](int j, const uint4& xv) {
      const int c = 32 * j + lane;
      if (c >= kch) return;
      const uint4 wv = *reinterpret_cast<const uint4*>(p.kv_weight + 8 * c);
      *reinterpret_cast<uint4*>(ko + 8 * c) = norm_chunk4(xv, wv, rk);
    };
    auto run_row = [&]() {
      if (RESIDENT) {
#pragma unroll
        for (int j = 0; j < QR; ++j)
          if (j < qsteps) q_step(j, qr[j]);
#pragma unroll
        for (int j = 0; j < KR; ++j)
          if (j < ksteps) kv_step(j, kr[j]);
      } else {
        for (int j = 0; j < qsteps; ++j) {
          const int c = 32 * j + lane;
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (c < qch) xv = *reinterpret_cast<const uint4*>(qrow + 8 * c);
          q_step(j, xv);
        }
        for (int j = 0; j < ksteps; ++j) {
          const int c = 32 * j + lane;
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (c < kch) xv = *reinterpret_cast<const uint4*>(krow + 8 * c);
          kv_step(j, xv);
        }
      }
    };
    run_row();
  }
}

// Largest magnitude of four bf16 pairs as bf16 bits, over the four lanes of an
// MX block (lanes 4b..4b+3); NaN-propagating.
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t y) {  // acc >= 0
  uint32_t d;
  asm("{\n .reg .b32 t;\n abs.bf16x2 t, %2;\n max.NaN.bf16x2 %0, %1, t;\n}\n"
      : "=r"(d) : "r"(acc), "r"(y));
  return d;
}
__device__ __forceinline__ uint32_t block_amax_bits(const uint32_t y[4]) {
  uint32_t m = absmax2(absmax2(absmax2(absmax2(0u, y[0]), y[1]), y[2]), y[3]);
  m = absmax2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = absmax2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  return __float_as_uint(fmax_nan(bf16_lo(m), bf16_hi(m))) >> 16;
}

// Staged variant for rows that fit two per-warp slots: each warp owns two
// shared-memory slots (q row then kv row) filled by cp.async.bulk on its own
// mbarriers, and starts the copy of its next-but-one row as soon as a slot is
// consumed, so row loads overlap the arithmetic of the row before.  Lane l
// reads chunks l, l+32, ... of the slot (consecutive 16-byte words: no bank
// conflicts) in both passes.
constexpr int kSlots = 2;
constexpr int kStagedMaxWarps = 32;
// mbarriers of every warp (8 bytes per slot), ahead of the row slots
constexpr int kStagedHeader = kStagedMaxWarps * kSlots * 8;
static_assert(kStagedHeader % 128 == 0, "row slots start 128-byte aligned");

__global__ void __launch_bounds__(kStagedMaxWarps * 32) rmsnorm_mx_tma(const MxParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_launch_dependents();  // programmatic dependent launch (see launch_pdl)
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const int64_t gwarp = (int64_t)blockIdx.x * wpb + warp;
  const int64_t nwarps = (int64_t)gridDim.x * wpb;
  const int qch = p.Nq / 8, kch = p.Nkv / 8;
  const uint32_t qbytes = 2u * (uint32_t)p.Nq, kbytes = 2u * (uint32_t)p.Nkv;
  const uint32_t slot_bytes = qbytes + kbytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * kSlots;
  const uint4* wq = reinterpret_cast<const uint4*>(smem + kStagedHeader);  // weights, once per CTA
  const uint4* wk = wq + qch;
  uint8_t* slots = smem + kStagedHeader + slot_bytes + (size_t)warp * kSlots * slot_bytes;
  const bool q_pow2 = (p.Nq & (p.Nq - 1)) == 0, k_pow2 = (p.Nkv & (p.Nkv - 1)) == 0;
  for (int i = threadIdx.x; i < qch + kch; i += blockDim.x) {
    if (i >= qch)
      const_cast<uint4*>(wq)[i] = reinterpret_cast<const uint4*>(p.kv_weight)[i - qch];
    else if (!p.q_prenorm)
      const_cast<uint4*>(wq)[i] = reinterpret_cast<const uint4*>(p.q_weight)[i];
  }
  __syncthreads();

  if (lane == 0) {
    for (int s = 0; s < kSlots; ++s) mbar_init(smem_u32(&bars[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();
  auto issue = [&](int s, int64_t m) {
    const uint32_t bar = smem_u32(&bars[s]);
    const uint32_t dst = smem_u32(slots + (size_t)s * slot_bytes);
    mbar_expect_tx(bar, slot_bytes);
    if (qbytes) bulk_g2s(dst, p.q + m * p.q_stride, qbytes, bar);
    if (kbytes) bulk_g2s(dst + qbytes, p.kv + m * p.kv_stride, kbytes, bar);
  };
  if (lane == 0)
    for (int s = 0; s < kSlots; ++s) {
      const int64_t m = gwarp + s * nwarps;
      if (m < p.M) issue(s, m);
    }

  int it = 0;
  bool timeout = false;
  for (int64_t m = gwarp; m < p.M; m += nwarps, ++it) {
    const int s = it % kSlots;
    if (!mbar_wait(smem_u32(&bars[s]), (uint32_t)(it / kSlots) & 1u, kWaitLimitMain)) timeout = true;
    if (__any_sync(0xFFFFFFFFu, timeout)) {  // the whole warp stops (lane 0 drains)
      timeout = true;
      break;
    }
    const uint4* sq = reinterpret_cast<const uint4*>(slots + (size_t)s * slot_bytes);
    const uint4* sk = reinterpret_cast<const uint4*>(slots + (size_t)s * slot_bytes + qbytes);
    sumsq2 aq, ak;
    for (int c = lane; c < (p.q_prenorm ? 0 : qch); c += 32) {
      const uint4 v = sq[c];
      const uint32_t* w = &v.x;
#pragma unroll
      for (int k = 0; k < 4; ++k) aq.add_sq(w[k]);
    }
    for (int c = lane; c < kch; c += 32) {
      const uint4 v = sk[c];
      const uint32_t* w = &v.x;
#pragma unroll
      for (int k = 0; k < 4; ++k) ak.add_sq(w[k]);
    }
    df Sq = aq.value(), Sk = ak.value();
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      Sq = df_add(Sq, shfl_xor_df(Sq, o));
      Sk = df_add(Sk, shfl_xor_df(Sk, o));
    }
    const int qsteps = (qch + 31) / 32;
    const bool q_norm = qch > 0 && !p.q_prenorm;
    bool uq = false, uk = false;
    float msq = q_norm ? row_ms(Sq, p.Nq, q_pow2, qsteps, &uq) : 0.0f;
    float msk = kch ? row_ms(Sk, p.Nkv, k_pow2, (kch + 31) / 32, &uk) : 0.0f;
    if (uq) msq = row_ms_exact(sq, p.Nq, Sq, qsteps, msq, lane);  // rare; uq, uk are warp-uniform
    if (uk) msk = row_ms_exact(sk, p.Nkv, Sk, (kch + 31) / 32, msk, lane);
    const f2_t rq = splat2(q_norm ? rms_factor(msq, p.eps) : 0.0f);
    const f2_t rk = splat2(kch ? rms_factor(msk, p.eps) : 0.0f);
    uint8_t* qo = p.q_out + m * p.q_out_stride;
    uint8_t* so = p.q_scale + m * p.q_scale_stride;
    uint16_t* ko = p.kv_out + m * p.kv_out_stride;
    auto run_row = [&]() {
      for (int j = 0; j < qsteps; ++j) {  // warp-uniform: every lane takes part in the shuffles
        const int c = 32 * j + lane;
        uint4 xv = make_uint4(0, 0, 0, 0), wv = xv;
        if (c < qch) {
          xv = sq[c];
          if (!p.q_prenorm) wv = wq[c];
        }
        uint32_t y[4];
        if (p.q_prenorm) {
          y[0] = xv.x, y[1] = xv.y, y[2] = xv.z, y[3] = xv.w;
        } else {
          norm_chunk(xv, wv, rq, y);
        }
        const uint32_t code = mx_code(block_amax_bits(y));
        if (c < qch) {
          if ((lane & 3) == 0) so[c >> 2] = (uint8_t)code;
          uint2 o;
          if (code == 0xFFu) {
            o = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
          } else {
            const f2_t sc = splat2(pow2i(127 - (int)code));  // 2^-e, exact scaling
            uint32_t b[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) b[k] = f2_to_e4m3x2(mul2(bf2_to_f2(y[k]), sc));
            o = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
          }
          *reinterpret_cast<uint2*>(qo + 8 * c) = o;
        }
      }
      for (int c = lane; c < kch; c += 32)
        *reinterpret_cast<uint4*>(ko + 8 * c) = norm_chunk4(sk[c], wk[c], rk);
    };
    run_row();
    __syncwarp();  // every lane is done with slot s
    if (lane == 0) {
      const int64_t mn = m + kSlots * nwarps;
      if (mn < p.M) issue(s, mn);
    }
  }
  if (timeout && lane == 0) {
    if (p.status) atomicOr(p.status, kStatusTimeout);
    for (int i = it; i < it + kSlots; ++i) {
      const int64_t mi = gwarp + (int64_t)i * nwarps;
      if (mi < p.M) mbar_wait(smem_u32(&bars[i % kSlots]), (uint32_t)(i / kSlots) & 1u, kWaitLimit);
    }
  }
}

// ---- rows in per-warp slots, one lane per half MX block -------------------
//
// The fused q/kv producer for rows of at most kRowsMaxQRounds x 512 q and
// kRowsMaxKRounds x 256 kv elements.  One CTA per SM; warp w of the grid walks
// rows w, w + W, w + 2W, ... (W = warps in the grid) through two shared-memory
// slots of its own, each filled by cp.async.bulk copies on its own mbarrier:
// a warp requests its first row before anything else and each next row as
// soon as the current one has landed, so one row is in flight while one is
// computed.  (Requesting every row of an SM at the start made each warp's
// first row arrive anywhere in the whole read window, and the warps then
// waited and computed in lock-step.)  The weights arrive by one more bulk copy
// on a CTA-wide mbarrier, so no warp waits at a block barrier for global
// memory.
//
// Lane layout.  q round j: lane l owns the sixteen elements of half-block
// hb = 32j + l (chunks 2hb and 2hb + 1), so an MX block is the lane pair
// (l, l ^ 1): its amax is the lane's running |max| over eight bf16 pairs and
// one xor-shuffle, and both lanes store the E8M0 code.  The two chunks are
// read in a rotated order (lanes with bit 2 set take the odd one first) so
// that the eight 16-byte reads of a quarter-warp hit distinct bank groups.
// kv round j: lane l owns chunk 32j + l.  The sums of squares of q and kv are
// reduced over the warp together, as pairs of packed double-floats.
constexpr int kRowsMaxQRounds = 4;
constexpr int kRowsMaxKRounds = 4;
constexpr int kRowsMaxWarps = 28;
constexpr int kRowsMaxSlots = 2;
// the weights' mbarrier, then every warp's slot mbarriers
constexpr int kRowsHeader = 16 + kRowsMaxWarps * kRowsMaxSlots * 8;
static_assert(kRowsHeader % 16 == 0, "weights and slots start 16-byte aligned");

// Two double-floats side by side (the q and kv sums of squares): the
// arithmetic of df_add, lane by lane, in packed binary32.
struct df2 {
  f2_t h, l;
};
__device__ __forceinline__ df2 df2_add(df2 a, df2 b) {
  const f2_t s = add2(a.h, b.h);
  const f2_t bb = sub2(s, a.h);
  const f2_t e = add2(sub2(a.h, sub2(s, bb)), sub2(b.h, bb));
  const f2_t t = add2(e, add2(a.l, b.l));
  const f2_t h = add2(s, t);
  return {h, sub2(t, sub2(h, s))};
}
__device__ __forceinline__ df2 shfl_xor_df2(df2 v, int lane_mask) {
  return {__shfl_xor_sync(0xFFFFFFFFu, v.h, lane_mask), __shfl_xor_sync(0xFFFFFFFFu, v.l, lane_mask)};
}

// RN32(S / n) as row_ms takes it, without a division: q = RN(S.h * RN(1/n)) is
// within an ulp of S.h / n, so the remainder S.h - q n is exact (n <= 2^14)
// and one correction gives the nearest binary32 of S / n except within about
// 2^-46 S of a rounding boundary, which the uncertainty test flags.  k: the
// additions of each running sum behind S.
// Both forms are evaluated and one is selected, so that lanes working on rows
// of different lengths do not diverge.
__device__ __forceinline__ float row_ms_k(df S, int n, float inv_n, bool n_pow2, int k,
                                          bool* unsure) {
  const float nf = (float)n;
  const float ms_pow2 = __fmul_rn(__fadd_rn(S.h, S.l), inv_n);
  const float q = __fmul_rn(S.h, inv_n);
  const float rem = __fmaf_rn(-q, nf, S.h);
  const float ms = n_pow2 ? ms_pow2 : __fadd_rn(q, __fmul_rn(__fadd_rn(rem, S.l), inv_n));
  *unsure = ms_uncertain(S, nf, ms, __fmaf_rn(S.h, sumsq_rel_err(k, 6), nf * 0x1p-149f));
  return ms;
}

// FULL: the rows fill every round (Nq = 512 QR, Nkv = 256 KR), so no lane
// needs a bounds test.
template <int QR, int KR, bool FULL>
__global__ void __launch_bounds__(kRowsMaxWarps * 32, 1) rmsnorm_mx_rows(const MxParams p, int nslot) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const int64_t gwarp = (int64_t)blockIdx.x * wpb + warp;
  const int64_t nwarps = (int64_t)gridDim.x * wpb;
  const int qch = p.Nq / 8, kch = p.Nkv / 8, nhb = p.Nq / 16;
  const uint32_t qbytes = 2u * (uint32_t)p.Nq, kbytes = 2u * (uint32_t)p.Nkv;
  const uint32_t slot_bytes = qbytes + kbytes;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 16) + warp * kRowsMaxSlots;
  const uint4* wq = reinterpret_cast<const uint4*>(smem + kRowsHeader);  // weights, once per CTA
  const uint4* wk = wq + qch;
  uint8_t* slots = smem + kRowsHeader + slot_bytes + (size_t)warp * nslot * slot_bytes;

  auto issue = [&](int s, int64_t m) {
    const uint32_t bar = smem_u32(&bars[s]);
    const uint32_t dst = smem_u32(slots + (size_t)s * slot_bytes);
    mbar_expect_tx(bar, slot_bytes);
    bulk_g2s(dst, p.q + m * p.q_stride, qbytes, bar);
    if (kbytes) bulk_g2s(dst + qbytes, p.kv + m * p.kv_stride, kbytes, bar);
  };
  // programmatic dependent launch (see launch_pdl): shared-memory set-up may
  // overlap the previous kernel; global memory only after pdl_wait
  pdl_launch_dependents();
  if (lane == 0) {
    for (int s = 0; s < nslot; ++s) mbar_init(smem_u32(&bars[s]), 1);
    if (warp == 0) mbar_init(smem_u32(wbar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();
  if (lane == 0) {
    // one row up front: the first rows of all warps (half the bytes of two each)
    // land sooner, and every later row is requested as its predecessor lands
    if (gwarp < p.M) issue(0, gwarp);
    if (warp == 0) {
      const uint32_t bar = smem_u32(wbar), dst = smem_u32(smem + kRowsHeader);
      mbar_expect_tx(bar, slot_bytes);
      bulk_g2s(dst, p.q_weight, qbytes, bar);
      if (kbytes) bulk_g2s(dst + qbytes, p.kv_weight, kbytes, bar);
    }
  }
  __syncthreads();  // every mbarrier is initialised

  const int rot = (lane >> 2) & 1;
  const bool q_pow2 = (p.Nq & (p.Nq - 1)) == 0, k_pow2 = (p.Nkv & (p.Nkv - 1)) == 0;
  const float inv_nq = 1.0f / (float)p.Nq, inv_nk = KR ? 1.0f / (float)p.Nkv : 0.0f;
  bool timeout = gwarp < p.M && !mbar_wait(smem_u32(wbar), 0u, kWaitLimitMain);
  int it = 0;
  for (int64_t m = gwarp; m < p.M; m += nwarps, ++it) {
    const int s = it % nslot;
    if (!timeout && !mbar_wait(smem_u32(&bars[s]), (uint32_t)(it / nslot) & 1u, kWaitLimitMain))
      timeout = true;
    if (__any_sync(0xFFFFFFFFu, timeout)) {  // the whole warp stops (lane 0 drains)
      timeout = true;
      break;
    }
    // the next row goes into the other slot, which held the row before this one
    // (done: every lane passed the __syncwarp that ended its iteration)
    if (lane == 0 && m + nwarps < p.M) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue((it + 1) % nslot, m + nwarps);
    }
    const uint4* sq = reinterpret_cast<const uint4*>(slots + (size_t)s * slot_bytes);
    const uint4* sk = sq + qch;
    // pass 1: Sum2 of the squares (one running sum pair for q, one for kv),
    // then both double-floats reduced over the warp together
    sumsq2 aq, ak;
#pragma unroll
    for (int j = 0; j < QR; ++j) {
      const int hb = 32 * j + lane;
      uint4 a = make_uint4(0, 0, 0, 0), b = a, c = a;
      if (FULL || hb < nhb) {
        a = sq[2 * hb + rot];
        b = sq[2 * hb + 1 - rot];
      }
      if (KR && j < KR && (FULL || 32 * j + lane < kch)) c = sk[32 * j + lane];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        aq.add_sq((&a.x)[k]);
        aq.add_sq((&b.x)[k]);
        if (KR && j < KR) ak.add_sq((&c.x)[k]);
      }
    }
#pragma unroll
    for (int j = QR; j < KR; ++j) {
      uint4 c = make_uint4(0, 0, 0, 0);
      if (FULL || 32 * j + lane < kch) c = sk[32 * j + lane];
#pragma unroll
      for (int k = 0; k < 4; ++k) ak.add_sq((&c.x)[k]);
    }
    const df vq = aq.value(), vk = ak.value();
    df2 S = {f2(vq.h, vk.h), f2(vq.l, vk.l)};
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) S = df2_add(S, shfl_xor_df2(S, o));
    // the scalar tail once for both rows: q's mean square and factor in the
    // even lanes, kv's in the odd lanes, then broadcast from lanes 0 and 1
    const float2 sh = unf2(S.h), sl = unf2(S.l);
    const df Sq = {sh.x, sl.x}, Sk = {sh.y, sl.y};
    const bool odd = KR && (lane & 1);
    bool u = false;
    const float ms = row_ms_k(odd ? Sk : Sq, odd ? p.Nkv : p.Nq, odd ? inv_nk : inv_nq,
                              odd ? k_pow2 : q_pow2, odd ? 4 * KR : 8 * QR, &u);
    const uint32_t unsure = __ballot_sync(0xFFFFFFFFu, u);
    float msq = __shfl_sync(0xFFFFFFFFu, ms, 0);
    float msk = KR ? __shfl_sync(0xFFFFFFFFu, ms, 1) : 0.0f;
    if (unsure & 1u) msq = row_ms_exact(sq, p.Nq, Sq, 2 * QR, msq, lane);  // rare; warp-uniform
    if (KR && (unsure & 2u)) msk = row_ms_exact(sk, p.Nkv, Sk, KR, msk, lane);
    const float r = rms_factor(odd ? msk : msq, p.eps);
    const f2_t rq = splat2(__shfl_sync(0xFFFFFFFFu, r, 0));
    const f2_t rk = splat2(KR ? __shfl_sync(0xFFFFFFFFu, r, 1) : 0.0f);

    // pass 2: q -> MXFP8, kv -> bf16, read from the slot again
    uint8_t* qo = p.q_out + m * p.q_out_stride;
    uint8_t* so = p.q_scale + m * p.q_scale_stride;
#pragma unroll
    for (int j = 0; j < QR; ++j) {
      if (!FULL && 32 * j >= nhb) break;  // warp-uniform
      const int hb = 32 * j + lane;
      const bool ok = FULL || hb < nhb;
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0, w0 = x0, w1 = x0;
      if (ok) {
        x0 = sq[2 * hb + rot];
        x1 = sq[2 * hb + 1 - rot];
        w0 = wq[2 * hb + rot];
        w1 = wq[2 * hb + 1 - rot];
      }
      uint32_t y[8];
      norm_chunk(x0, w0, rq, y);
      norm_chunk(x1, w1, rq, y + 4);
      uint32_t am = absmax8(y, y + 4);
      am = max_nan_bf16x2(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      const uint32_t mag = am;
      const uint32_t code = mx_code(max(mag & 0xFFFFu, mag >> 16));
      if (ok) {
        so[hb >> 1] = (uint8_t)code;  // both lanes of the block store the same byte
        uint32_t o[4];
        if (code == 0xFFu) {
          o[0] = o[1] = o[2] = o[3] = 0x7F7F7F7Fu;
        } else {
          const uint32_t sb = (254u - code) << 7;  // bf16 bits of 2^-e (normal: code <= 246)
          const uint32_t s2 = sb | (sb << 16);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            o[k] = scaled_e4m3_pair(y[2 * k], s2) | (scaled_e4m3_pair(y[2 * k + 1], s2) << 16);
        }
        *reinterpret_cast<uint2*>(qo + 8 * (2 * hb + rot)) = make_uint2(o[0], o[1]);
        *reinterpret_cast<uint2*>(qo + 8 * (2 * hb + 1 - rot)) = make_uint2(o[2], o[3]);
      }
    }
    uint16_t* ko = p.kv_out + m * p.kv_out_stride;
#pragma unroll
    for (int j = 0; j < KR; ++j) {
      const int c = 32 * j + lane;
      if (FULL || c < kch) *reinterpret_cast<uint4*>(ko + 8 * c) = norm_chunk4(sk[c], wk[c], rk);
    }
    __syncwarp();  // every lane is done with slot s before it is refilled
  }
  if (timeout && lane == 0) {
    // the row whose wait gave up is the only one in flight
    if (p.status) atomicOr(p.status, kStatusTimeout);
    if (gwarp + (int64_t)it * nwarps < p.M)
      mbar_wait(smem_u32(&bars[it % nslot]), (uint32_t)(it / nslot) & 1u, kWaitLimit);
  }
  // the weights' copy has landed before the CTA's shared memory goes away
  if (threadIdx.x == 0) mbar_wait(smem_u32(wbar), 0u, kWaitLimit);
}

// One CTA per SM with two row slots per warp and as many warps (up to
// kRowsMaxWarps) as shared memory holds; a batch smaller than the grid spreads
// its rows over more SMs with fewer warps each.
#ifndef FP8N_ROWS_WARPS
#define FP8N_ROWS_WARPS kRowsMaxWarps
#endif
template <int QR, int KR, bool FULL>
cudaError_t launch_rows_v(const MxParams& p, cudaStream_t stream) {
  auto kern = rmsnorm_mx_rows<QR, KR, FULL>;
  const size_t slot = 2 * (size_t)(p.Nq + p.Nkv);
  const size_t budget = 227 * 1024 - 1024 - kRowsHeader - slot;  // less the weights
  const int nslot = kRowsMaxSlots;
  int w = (int)(budget / ((size_t)nslot * slot));
  if (w > FP8N_ROWS_WARPS) w = FP8N_ROWS_WARPS;
  const int sms = sm_count();
  const int64_t per_sm = (p.M + sms - 1) / sms;
  if (per_sm < w) w = (int)(per_sm < 1 ? 1 : per_sm);
  const size_t smem = kRowsHeader + slot + (size_t)w * nslot * slot;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t need = (p.M + w - 1) / w;
  const int grid = (int)(need < sms ? need : sms);
  return launch_pdl(kern, grid, w * 32, smem, stream, p, nslot);
}

template <int QR, int KR>
cudaError_t launch_rows_f(const MxParams& p, cudaStream_t stream) {
  if (p.Nq == 512 * QR && p.Nkv == 256 * KR) return launch_rows_v<QR, KR, true>(p, stream);
  return launch_rows_v<QR, KR, false>(p, stream);
}

template <int QR>
cudaError_t launch_rows_q(const MxParams& p, int kr, cudaStream_t stream) {
  switch (kr) {
    case 0: return launch_rows_f<QR, 0>(p, stream);
    case 1: return launch_rows_f<QR, 1>(p, stream);
    case 2: return launch_rows_f<QR, 2>(p, stream);
    default: return launch_rows_f<QR, 4>(p, stream);
  }
}

// Warps per CTA: the count (up to 32) whose CTAs pack the most warps into an
// SM's shared memory (two row slots per warp); a row per warp-slot pair keeps
// the slowest warp at as few rows as the SM count allows.
cudaError_t launch_staged(const MxParams& p, cudaStream_t stream) {
  const size_t per_warp = (size_t)kSlots * 2 * (size_t)(p.Nq + p.Nkv);
  const size_t budget = 227 * 1024;
  int best_w = 8, best_total = 0;
  const size_t wbytes = 2 * (size_t)(p.Nq + p.Nkv);  // the weights, once per CTA
  for (int w = 4; w <= kStagedMaxWarps; ++w) {
    const size_t cta = kStagedHeader + wbytes + w * per_warp + 1024;  // + the per-CTA reservation
    const int ctas = (int)(budget / cta);
    const int total = ctas * w > 64 ? 64 / w * w : ctas * w;  // 64 warps per SM at most
    if (total > best_total) { best_total = total; best_w = w; }
  }
  const size_t smem = kStagedHeader + wbytes + (size_t)best_w * per_warp;
  cudaError_t e =
      cudaFuncSetAttribute(rmsnorm_mx_tma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_mx_tma, best_w * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int64_t need = (p.M + best_w - 1) / best_w;
  const int grid = (int)(need < want ? need : want);
  return launch_pdl(rmsnorm_mx_tma, grid, best_w * 32, smem, stream, p);
}

template <int QS, int KS>
cudaError_t launch_variant(const MxParams& p, cudaStream_t stream) {
  auto kern = rmsnorm_mx_kernel<QS, KS>;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int64_t need = (p.M + kWarps - 1) / kWarps;
  const int grid = (int)(need < want ? need : want);
  return launch_pdl(kern, grid, kWarps * 32, 0, stream, p);
}

}  // namespace

// Variant: the staged kernel for rows up to 3072 elements, else the smallest
// register-resident (q steps, kv steps) pair that holds the rows, else the
// two-pass kernel.
cudaError_t launch_mx(const MxParams& p, cudaStream_t stream) {
  // the fused producer with rows that fit the register-resident kernel
  const int qr = (p.Nq + 511) / 512, kr = (p.Nkv + 255) / 256;
  if (!p.q_prenorm && p.Nq > 0 && qr <= kRowsMaxQRounds && kr <= kRowsMaxKRounds) {
    switch (qr) {
      case 1: return launch_rows_q<1>(p, kr, stream);
      case 2: return launch_rows_q<2>(p, kr, stream);
      case 3: return launch_rows_q<3>(p, kr, stream);
      default: return launch_rows_q<4>(p, kr, stream);
    }
  }
  // rows of up to 3072 elements (q + kv): the staged kernel, 96 KB per CTA at most
  if (p.Nq + p.Nkv <= 3072) return launch_staged(p, stream);
  const int qs = (p.Nq / 8 + 31) / 32, ks = (p.Nkv / 8 + 31) / 32;
  if (ks <= 2) {
    if (qs <= 2) return launch_variant<2, 2>(p, stream);
    if (qs <= 4) return launch_variant<4, 2>(p, stream);
    if (qs <= 6) return launch_variant<6, 2>(p, stream);
    if (qs <= 8) return launch_variant<8, 2>(p, stream);
  } else if (ks <= 8 && qs <= 8) {
    return launch_variant<8, 8>(p, stream);
  }
  return launch_variant<0, 0>(p, stream);
}

}  // namespace fp8n
