/*
 * CPU oracle for the normalize-then-quantize path: TEST INFRASTRUCTURE ONLY.
 * See fp8norm_oracle.h for the sources cited as [GATED], [MX], [STATIC],
 * [OCP8] and [OCPMX].  Build flags: -O2 -ffp-contract=off, no fast-math, so
 * that every float expression below is exactly one IEEE binary32 operation.
 */
#include "fp8norm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ===================================================================== */
/* bfloat16                                                               */
/* ===================================================================== */

/* Exact value of a bf16 bit pattern: the top half of a binary32. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* bf16(v): round-to-nearest-even of a real value (given as a double) to
 * bfloat16.  Quantum 2^(E-7) for a normal result with leading exponent E,
 * 2^-133 below the normal range (gradual underflow); results whose rounded
 * magnitude reaches 2^128 become infinity; NaN becomes the quiet NaN 0x7FC0. */
uint16_t oracle_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e2;
  frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): leading exponent E = e2 - 1 */
  int E = e2 - 1;
  int qexp = (E < -126) ? -133 : E - 7;
  double n = rint(ldexp(a, -qexp)); /* ties to even (default rounding mode) */
  double r = ldexp(n, qexp);
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ===================================================================== */
/* OCP E4M3 ("fn"): bias 7, no infinities, 0x7F/0xFF NaN, max 448        */
/* ===================================================================== */

double oracle_e4m3_to_double(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* subnormal: m * 2^-9 */
  else
    mag = ldexp((double)(8 + m), e - 10); /* 1.m * 2^(e-7) */
  return s ? -mag : mag;
}

/* e4m3(v): saturating round-to-nearest-even [OCP8].  NaN -> 0x7F; |v| at or
 * above 448 (infinities included) -> +-448 (0x7E / 0xFE); otherwise the
 * nearest E4M3 value with ties to the even mantissa; the sign of zero and of
 * results that round to zero is kept. */
uint8_t oracle_e4m3_from_float(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  int qexp = (E < -6) ? -9 : E - 3; /* quantum of the binade (or subnormal) */
  double n = rint(ldexp(a, -qexp));
  double r = ldexp(n, qexp); /* r <= 448 because a < 448 */
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return sign | (uint8_t)n; /* subnormal code m */
  frexp(r, &e2);
  int Er = e2 - 1;                                  /* -6 .. 8 */
  int m = (int)ldexp(r, 3 - Er) - 8;                /* 3-bit mantissa */
  return sign | (uint8_t)(((Er + 7) << 3) | m);
}

/* ===================================================================== */
/* Activation of the gate, rounded once to bf16                          */
/* ===================================================================== */

/* [GATED] review thread: the gate enters through torch.sigmoid and the
 * product is formed in the activation dtype.  Reading: the gate factor is the
 * correctly rounded bf16 of the real function.  sigmoid(g) = 1/(1+e^-g);
 * silu(g) = g * sigmoid(g) (the silu gate is not on the pages; it is placed
 * where the sigmoid is).  Evaluated in double, whose error (a few units in
 * 2^-53) is far below the bf16 rounding quantum.  Limits are used at the
 * infinities: sigmoid(+inf) = 1, sigmoid(-inf) = 0, silu(+inf) = +inf,
 * silu(-inf) = -0.  NaN stays NaN. */
/* bf16 of hi + lo where lo is a tiny correction (|lo| < one double ulp of
 * hi): hi decides, except when hi is exactly halfway between two bf16
 * values, where the sign of lo breaks the tie. */
static uint16_t bf16_from_pair(double hi, double lo) {
  if (lo != 0.0 && hi != 0.0 && isfinite(hi)) {
    int e2;
    frexp(fabs(hi), &e2);
    int E = e2 - 1;
    int qexp = (E < -126) ? -133 : E - 7;
    double n = ldexp(hi, -qexp);
    double fl = floor(n);
    if (n - fl == 0.5) /* a zero result keeps the sign of hi + lo, i.e. of hi */
      return oracle_bf16_from_double(copysign(ldexp(lo > 0 ? fl + 1.0 : fl, qexp), hi));
  }
  return oracle_bf16_from_double(hi);
}

uint16_t oracle_act_bf16(uint16_t g, int act) {
  double x = oracle_bf16_to_double(g);
  if (isnan(x)) return 0x7FC0;
  if (isinf(x)) {
    if (act == ORACLE_ACT_SIGMOID) return x > 0 ? 0x3F80 : 0x0000;
    return x > 0 ? 0x7F80 : 0x8000;
  }
  /* Tiny gates: silu(x) = x/2 + x^2/4 - x^4/48 + ...  Here x/2 can be exactly
   * a bf16 tie (x a subnormal with odd mantissa), and only the x^2/4 term,
   * which a double evaluation of x * sigmoid(x) loses, says which way to
   * round.  Both terms are exact in double; the next one is 2^-60 smaller. */
  if (act == ORACLE_ACT_SILU && fabs(x) < 0x1p-30) return bf16_from_pair(x / 2.0, x * x / 4.0);
  double sig = 1.0 / (1.0 + exp(-x));
  double v = (act == ORACLE_ACT_SIGMOID) ? sig : x * sig;
  return oracle_bf16_from_double(v);
}

void oracle_bf16_from_float_n(const float* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_double((double)v[i]);
}

void oracle_e4m3_from_float_n(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_float(v[i]);
}

void oracle_act_bf16_n(const uint16_t* g, int64_t n, int act, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_act_bf16(g[i], act);
}

/* ===================================================================== */
/* Mean of squares, exact sum then one binary32 rounding                  */
/* ===================================================================== */

/* The pages do not show how the per-head (or per-row) mean square is
 * accumulated.  Reading: ms = RN32(sum(x^2) / n) with the sum exact, so the
 * result does not depend on any summation order.  Every bf16 value is
 * x = M * 2^k with an integer 0 <= M < 256 and -133 <= k <= 120, hence
 * x^2 * 2^266 = M^2 * 2^(2k + 266) is an integer below 2^522: the squares are
 * added exactly into a 640-bit fixed-point accumulator, the total is divided
 * by n with a long division, and the quotient is rounded to binary32 from its
 * leading bits plus a sticky bit. */
#define OR_LIMBS 22
float oracle_mean_square_bf16(const uint16_t* x, int64_t n) {
  uint32_t acc[OR_LIMBS];
  memset(acc, 0, sizeof acc);
  int saw_nan = 0, saw_inf = 0;
  for (int64_t i = 0; i < n; ++i) {
    uint16_t b = x[i] & 0x7FFF;
    uint32_t ef = b >> 7, mf = b & 0x7F;
    if (ef == 0xFF) {
      if (mf) saw_nan = 1; else saw_inf = 1;
      continue;
    }
    if (b == 0) continue;
    uint32_t M = ef ? (128 + mf) : mf;
    int k = ef ? (int)ef - 134 : -133;
    int s = 2 * k + 266; /* 0 .. 506 */
    uint64_t add = (uint64_t)(M * M) << (s % 32);
    int limb = s / 32;
    while (add) { /* add with carry propagation, limb by limb */
      uint64_t t = (uint64_t)acc[limb] + (add & 0xFFFFFFFFu);
      acc[limb] = (uint32_t)t;
      add = (add >> 32) + (t >> 32);
      ++limb;
    }
  }
  if (saw_nan) return NAN;
  if (saw_inf) return INFINITY;
  /* B = acc * 2^64 (two extra low limbs), Q = floor(B / n), R = B mod n. */
  uint32_t B[OR_LIMBS + 2], Q[OR_LIMBS + 2];
  B[0] = 0;
  B[1] = 0;
  for (int i = 0; i < OR_LIMBS; ++i) B[i + 2] = acc[i];
  uint64_t rem = 0;
  int top = -1;
  for (int i = OR_LIMBS + 1; i >= 0; --i) {
    uint64_t cur = (rem << 32) | B[i];
    Q[i] = (uint32_t)(cur / (uint64_t)n);
    rem = cur % (uint64_t)n;
    if (top < 0 && Q[i]) top = i;
  }
  if (top < 0) return 0.0f; /* all squares were zero */
  int p = top * 32 + 31;
  while (!((Q[p / 32] >> (p % 32)) & 1u)) --p; /* leading bit of Q */
  /* value = (Q + R/n) * 2^-330.  Keep 24 bits, or fewer below 2^-126 where
   * the binary32 quantum is 2^-149, i.e. bit 181 of Q. */
  int shift = p - 23;
  if (shift < 181) shift = 181;
#define QBIT(j) ((j) >= 0 ? ((Q[(j) / 32] >> ((j) % 32)) & 1u) : 0u)
  uint64_t mant = 0;
  for (int j = p; j >= shift; --j) mant = (mant << 1) | QBIT(j);
  uint32_t round_bit = QBIT(shift - 1);
  int sticky = rem != 0;
  for (int j = shift - 2; j >= 0 && !sticky; --j) sticky = QBIT(j) != 0;
#undef QBIT
  if (round_bit && (sticky || (mant & 1u))) ++mant;
  return (float)ldexp((double)mant, shift - 330);
}

/* r = 1 / sqrt(ms + eps) with each step one IEEE binary32 operation:
 * v = RN32(ms + eps), s = RN32(sqrt v), r = RN32(1 / s). */
float oracle_rms_factor(float ms, float eps) {
  float v = ms + eps;
  float s = sqrtf(v);
  return 1.0f / s;
}

/* bf16(bf16(RN32(x * r)) * w): the normalised value rounded to the
 * activation dtype, times the weight in that dtype (a bf16 x bf16 product is
 * exact in double, then rounded once). */
static uint16_t norm_times_weight(uint16_t xb, float r, uint16_t wb) {
  float xn = (float)oracle_bf16_to_double(xb) * r;
  uint16_t xnb = oracle_bf16_from_double((double)xn);
  return oracle_bf16_from_double(oracle_bf16_to_double(xnb) * oracle_bf16_to_double(wb));
}

/* ===================================================================== */
/* Operation (A)                                                          */
/* ===================================================================== */

/* [GATED]: per head, RMS over D; times the weight; times act(gate); then the
 * whole token row [H*D] is quantised with one scale: amax = max |y|,
 * scale = RN32(amax / 448) (448 = largest finite E4M3), code =
 * e4m3(RN32(y / scale)).  A token whose amax is zero gets scale 0 and codes
 * that are zeros carrying the sign of y (no epsilon floor on the scale). */
/* Per-token quantisation of a bf16 row y[n] ([GATED] wrapper: one scale over
 * the whole [heads*h] row).  Also the standalone per-token quant applied to an
 * already-normalised row in the same page's decode path. */
void oracle_quant_row(const uint16_t* y, int64_t n, uint8_t* out, float* scale_out) {
  double amax = 0.0;
  int any_nan = 0;
  for (int64_t i = 0; i < n; ++i) {
    double a = fabs(oracle_bf16_to_double(y[i]));
    if (isnan(a)) any_nan = 1;
    else if (a > amax) amax = a;
  }
  float famax = any_nan ? NAN : (float)amax; /* exact: amax is a bf16 value */
  float scale = famax / 448.0f;
  *scale_out = scale;
  for (int64_t i = 0; i < n; ++i) {
    float yv = (float)oracle_bf16_to_double(y[i]);
    if (famax == 0.0f)
      out[i] = (y[i] & 0x8000) ? 0x80 : 0x00;
    else
      out[i] = oracle_e4m3_from_float(yv / scale);
  }
}

/* y = bf16(bf16(bf16(RN32(x * r)) * w) * bf16(act(g))) for one token, heads of D.
 * ms_given: NULL, or the mean square of each head to use in place of the exact
 * one (a diagnostic input; see oracle_gated_rmsnorm_quant_one_ms). */
static void gated_rmsnorm_row_ms(const uint16_t* x_tok, const uint16_t* gate_tok,
                                 const uint16_t* weight, int32_t H, int32_t D, float eps, int act,
                                 const float* ms_given, uint16_t* y_tok) {
  for (int32_t h = 0; h < H; ++h) {
    const uint16_t* xh = x_tok + (int64_t)h * D;
    const uint16_t* gh = gate_tok + (int64_t)h * D;
    float ms = ms_given ? ms_given[h] : oracle_mean_square_bf16(xh, D);
    float r = oracle_rms_factor(ms, eps);
    for (int32_t d = 0; d < D; ++d) {
      uint16_t u = norm_times_weight(xh[d], r, weight[d]);
      uint16_t g = oracle_act_bf16(gh[d], act);
      y_tok[(int64_t)h * D + d] =
          oracle_bf16_from_double(oracle_bf16_to_double(u) * oracle_bf16_to_double(g));
    }
  }
}

void oracle_gated_rmsnorm_row(const uint16_t* x_tok, const uint16_t* gate_tok,
                              const uint16_t* weight, int32_t H, int32_t D, float eps, int act,
                              uint16_t* y_tok) {
  gated_rmsnorm_row_ms(x_tok, gate_tok, weight, H, D, eps, act, NULL, y_tok);
}

/* (A) on one token with each head's mean square given instead of computed.
 * Not part of the definition: the parity checks call it with a head's exact
 * ms moved by a unit or two in the last place, to tell whether a token on
 * which the fused kernel differs is explained by that head's summation
 * order alone (every other step unchanged). */
void oracle_gated_rmsnorm_quant_one_ms(const uint16_t* x_tok, const uint16_t* gate_tok,
                                       const uint16_t* weight, int32_t H, int32_t D, float eps,
                                       int act, const float* ms, uint16_t* y_tok,
                                       uint8_t* out_tok, float* scale_tok) {
  gated_rmsnorm_row_ms(x_tok, gate_tok, weight, H, D, eps, act, ms, y_tok);
  oracle_quant_row(y_tok, (int64_t)H * D, out_tok, scale_tok);
}

void oracle_gated_rmsnorm_quant_one(const uint16_t* x_tok, const uint16_t* gate_tok,
                                    const uint16_t* weight, int32_t H, int32_t D,
                                    float eps, int act, uint16_t* y_tok,
                                    uint8_t* out_tok, float* scale_tok) {
  oracle_gated_rmsnorm_row(x_tok, gate_tok, weight, H, D, eps, act, y_tok);
  oracle_quant_row(y_tok, (int64_t)H * D, out_tok, scale_tok);
}

void oracle_gated_rmsnorm_quant_token(const uint16_t* x, int64_t x_stride,
                                      const uint16_t* gate, int64_t gate_stride,
                                      const uint16_t* weight, int64_t T, int32_t H,
                                      int32_t D, float eps, int act, uint8_t* out,
                                      int64_t out_stride, float* scale) {
  int64_t n = (int64_t)H * D;
  uint16_t* y = (uint16_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(uint16_t));
  for (int64_t t = 0; t < T; ++t)
    oracle_gated_rmsnorm_quant_one(x + t * x_stride, gate + t * gate_stride, weight, H, D,
                                   eps, act, y, out + t * out_stride, scale + t);
  free(y);
}

/* Gated per-token quant without the norm: y = bf16(x * bf16(act(g))), then the
 * per-token quantisation.  The gate product in the activation dtype follows
 * [GATED]'s helper; the sigmoid-mul + per-token FP8 epilogue of the MLA o_proj
 * named on that page is this map with the sigmoid. */
void oracle_gated_quant_row(const uint16_t* x, const uint16_t* gate, int64_t n, int act,
                            uint16_t* y, uint8_t* out, float* scale) {
  for (int64_t i = 0; i < n; ++i)
    y[i] = oracle_bf16_from_double(oracle_bf16_to_double(x[i]) *
                                   oracle_bf16_to_double(oracle_act_bf16(gate[i], act)));
  oracle_quant_row(y, n, out, scale);
}

/* ===================================================================== */
/* Operation (B)                                                          */
/* ===================================================================== */

/* [OCPMX]: the shared scale of a block is 2^(floor(log2 amax) - 8) for E4M3
 * elements, stored as the E8M0 code e + 127 with e clamped to [-127, 127].
 * A zero block gets e = -127 (code 0); a block whose amax is NaN or infinite
 * gets the E8M0 NaN code 0xFF. */
uint8_t oracle_e8m0_code(uint16_t amax_bits) {
  double A = fabs(oracle_bf16_to_double(amax_bits));
  if (isnan(A) || isinf(A)) return 0xFF;
  if (A == 0.0) return 0;
  int e2;
  frexp(A, &e2);
  int e = (e2 - 1) - 8; /* floor(log2 A) - 8, exact for every binary value */
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return (uint8_t)(e + 127);
}

/* Normalised bf16 row: bf16(bf16(RN32(x * r)) * w), r from the full row. */
void oracle_rmsnorm_row(const uint16_t* x, const uint16_t* w, int32_t n, float eps,
                        uint16_t* y) {
  float r = oracle_rms_factor(oracle_mean_square_bf16(x, n), eps);
  for (int32_t j = 0; j < n; ++j) y[j] = norm_times_weight(x[j], r, w[j]);
}

/* [MX] third commit message: one producer normalises q and kv; q leaves as
 * MXFP8 (E4M3 elements, one E8M0 scale per 32 consecutive elements, scales
 * row-major [M, Nq/32]); kv leaves as the normalised bf16.  The MX quantiser
 * consumes the bf16 normalised q, as the unfused steps would.  Elements are
 * e4m3(yq * 2^-e), the power-of-two scaling being exact. */
void oracle_rmsnorm_quant_mx(const uint16_t* q, int64_t q_stride, const uint16_t* q_weight,
                             int32_t Nq, const uint16_t* kv, int64_t kv_stride,
                             const uint16_t* kv_weight, int32_t Nkv, int64_t M, float eps,
                             uint8_t* q_out, int64_t q_out_stride, uint8_t* q_scale,
                             int64_t q_scale_stride, uint16_t* kv_out,
                             int64_t kv_out_stride) {
  uint16_t* yq = (uint16_t*)malloc((size_t)(Nq > 0 ? Nq : 1) * sizeof(uint16_t));
  for (int64_t m = 0; m < M; ++m) {
    if (Nq > 0) oracle_rmsnorm_row(q + m * q_stride, q_weight, Nq, eps, yq);
    if (Nkv > 0) oracle_rmsnorm_row(kv + m * kv_stride, kv_weight, Nkv, eps, kv_out + m * kv_out_stride);
    oracle_quant_mx_row(yq, Nq, q_out + m * q_out_stride, q_scale + m * q_scale_stride);
  }
  free(yq);
}

/* MX quantisation of one bf16 row of n (a multiple of 32) values: per block of
 * 32, the E8M0 code of its amax and the E4M3 codes of the scaled elements. */
void oracle_quant_mx_row(const uint16_t* yq, int32_t n, uint8_t* codes, uint8_t* scales) {
  {
    for (int32_t b = 0; b < n / 32; ++b) {
      const uint16_t* blk = yq + 32 * b;
      uint16_t amax_bits = 0;
      double amax = 0.0;
      int bad = 0;
      for (int j = 0; j < 32; ++j) {
        double a = fabs(oracle_bf16_to_double(blk[j]));
        if (isnan(a) || isinf(a)) bad = 1;
        else if (a > amax) { amax = a; amax_bits = blk[j] & 0x7FFF; }
      }
      uint8_t code = bad ? 0xFF : oracle_e8m0_code(amax_bits);
      scales[b] = code;
      uint8_t* o = codes + 32 * b;
      for (int j = 0; j < 32; ++j) {
        if (code == 0xFF) { o[j] = 0x7F; continue; }
        double scaled = ldexp(oracle_bf16_to_double(blk[j]), -((int)code - 127));
        /* Exact unless the scaled value falls below 2^-126, where it is far
         * below half the smallest E4M3 step and encodes to a signed zero. */
        o[j] = oracle_e4m3_from_float((float)scaled);
      }
    }
  }
}

/* ===================================================================== */
/* Inverse RoPE, then MXFP8 (the o-projection input)                      */
/* ===================================================================== */

/* [MX] first commit message: the FP8 o-projection input comes from a fused
 * inverse-RoPE + FP8 quantiser feeding an MX-scaled a8w8 GEMM; second commit
 * message: the layer holds a pre-computed FP32 cos/sin cache (4096
 * positions).  Reading: positions index rows of the cache [P, R] (cos of the
 * R/2 pair angles, then their sin); the rotated span of each head is
 * [rope_off, rope_off + R); pair i is (rope_off + i, rope_off + R/2 + i)
 * (rotate-half) or (rope_off + 2i, rope_off + 2i + 1) (interleaved); the
 * inverse rotation of a pair (x1, x2) by its angle is
 *   y1 = x1 cos + x2 sin,  y2 = x2 cos - x1 sin,
 * each product and sum one IEEE binary32 operation, rounded to bf16 (the
 * model dtype); the other elements pass unchanged.  The MXFP8 quantiser of
 * operation (B) then takes the bf16 row [H*D]. */
void oracle_inv_rope_row(const uint16_t* o_tok, int32_t H, int32_t D, int32_t rope_off,
                         int32_t R, int interleaved, const float* cs, uint16_t* y_tok) {
  int32_t half = R / 2;
  for (int64_t j = 0; j < (int64_t)H * D; ++j) y_tok[j] = o_tok[j];
  for (int32_t h = 0; h < H; ++h) {
    const uint16_t* x = o_tok + (int64_t)h * D;
    uint16_t* y = y_tok + (int64_t)h * D;
    for (int32_t i = 0; i < half; ++i) {
      int32_t j1 = interleaved ? rope_off + 2 * i : rope_off + i;
      int32_t j2 = interleaved ? rope_off + 2 * i + 1 : rope_off + half + i;
      float x1 = (float)oracle_bf16_to_double(x[j1]);
      float x2 = (float)oracle_bf16_to_double(x[j2]);
      float c = cs[i], s = cs[half + i];
      float a = x1 * c, b = x2 * s;
      float y1 = a + b;
      float d = x2 * c, e = x1 * s;
      float y2 = d - e;
      y[j1] = oracle_bf16_from_double((double)y1);
      y[j2] = oracle_bf16_from_double((double)y2);
    }
  }
}

void oracle_inv_rope_quant_mx(const uint16_t* o, int64_t o_stride, int64_t T, int32_t H,
                              int32_t D, const int32_t* positions, const float* cos_sin,
                              int32_t rope_off, int32_t R, int interleaved, uint8_t* out,
                              int64_t out_stride, uint8_t* scale, int64_t scale_stride) {
  int64_t n = (int64_t)H * D;
  uint16_t* y = (uint16_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(uint16_t));
  for (int64_t t = 0; t < T; ++t) {
    oracle_inv_rope_row(o + t * o_stride, H, D, rope_off, R, interleaved,
                        cos_sin + (int64_t)positions[t] * R, y);
    oracle_quant_mx_row(y, (int32_t)n, out + t * out_stride, scale + t * scale_stride);
  }
  free(y);
}

/* ===================================================================== */
/* Operation (C)                                                          */
/* ===================================================================== */

/* [STATIC]: each head of Q, K or V is divided by its calibrated descale and
 * cast to FP8: code = e4m3(RN32(x / descale[h])).  The descale is used as
 * given (validating it is the caller's job); varlen packing only stacks the
 * sequences along T, so the map is elementwise over the packed tensor. */
void oracle_static_head_quant(const uint16_t* x, int64_t tok_stride, int64_t head_stride,
                              int64_t T, int32_t H, int32_t Dh, const float* descale,
                              uint8_t* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int32_t h = 0; h < H; ++h)
      for (int32_t d = 0; d < Dh; ++d) {
        float xv = (float)oracle_bf16_to_double(x[t * tok_stride + h * head_stride + d]);
        out[(t * H + h) * Dh + d] = oracle_e4m3_from_float(xv / descale[h]);
      }
}

/* Running per-head maximum of |x| over all tokens and d ([STATIC]: the layer
 * collects Q/K/V maxima in calibration mode; the dynamic path these static
 * scales replace reduces the same maxima on every step).  amax[h] is updated
 * in place: amax[h] = max(amax[h], max |x[:, h, :]|); NaN propagates. */
void oracle_head_amax(const uint16_t* x, int64_t tok_stride, int64_t head_stride, int64_t T,
                      int32_t H, int32_t Dh, float* amax) {
  for (int32_t h = 0; h < H; ++h) {
    double m = (double)amax[h];
    int nan = isnan(m);
    for (int64_t t = 0; t < T; ++t)
      for (int32_t d = 0; d < Dh; ++d) {
        double a = fabs(oracle_bf16_to_double(x[t * tok_stride + h * head_stride + d]));
        if (isnan(a)) nan = 1;
        else if (a > m) m = a;
      }
    amax[h] = nan ? NAN : (float)m;
  }
}

/* Dynamic per-head quant: descale[h] = RN32(amax[h] / 448) from this tensor's
 * own maxima, then the static map with those descales; a head whose amax is 0
 * gets descale 0 and signed zero codes (the zero-token rule of the per-token
 * quantiser, applied per head). */
void oracle_dynamic_head_quant(const uint16_t* x, int64_t tok_stride, int64_t head_stride,
                               int64_t T, int32_t H, int32_t Dh, float* descale, uint8_t* out) {
  for (int32_t h = 0; h < H; ++h) descale[h] = 0.0f;
  oracle_head_amax(x, tok_stride, head_stride, T, H, Dh, descale);
  for (int32_t h = 0; h < H; ++h) descale[h] = descale[h] / 448.0f;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t h = 0; h < H; ++h)
      for (int32_t d = 0; d < Dh; ++d) {
        uint16_t b = x[t * tok_stride + h * head_stride + d];
        float xv = (float)oracle_bf16_to_double(b);
        out[(t * H + h) * Dh + d] = descale[h] == 0.0f ? ((b & 0x8000) ? 0x80 : 0x00)
                                                       : oracle_e4m3_from_float(xv / descale[h]);
      }
}
