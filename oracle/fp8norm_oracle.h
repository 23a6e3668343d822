/*
 * CPU oracle for the normalize-then-quantize path: TEST INFRASTRUCTURE ONLY.
 *
 * This header and fp8norm_oracle.c are a plain, slow, single-threaded C11
 * restatement of what the three operations compute, written so that a reader
 * can check every rounding step against its source by eye.  Only the tests,
 * the package's smoke check and the benchmark's CPU-baseline leg may load it;
 * the product library never links, includes or calls it, and it shares no
 * code, header, table or constant with the CUDA sources.
 *
 * Sources (web pages, by title and section):
 *   [GATED]  "[ROCm][Kimi-K3] Fuse gated RMSNorm with per-token FP8 for KDA
 *            o_proj" (vLLM PR 54254): Purpose; Tests (fused result checked
 *            against sequential gated RMSNorm + per-token amax, scale exact,
 *            dequant atol/rtol 1e-3); review thread on the torch reference
 *            helper (xn rounded to the activation dtype, times the weight in
 *            that dtype, times the sigmoid of the gate) and on the wrapper
 *            (t, heads, h unpacked from x; fp8_max from finfo of the quant
 *            dtype; result reshaped to [t, heads*h]).
 *   [MX]     "[ROCm][Perf] FP8 o-projection for DeepSeek-V4.1-Flash MLA on
 *            AMD MI355X" (vLLM PR 57081): third commit message (fused q/kv
 *            RMSNorm producer, q emitted as MXFP8 with row-major E8M0 scales,
 *            bitwise identical to the unfused path); description (ue8m0
 *            scale format, 32-wide blocks).
 *   [STATIC] "[ROCm][MLA] Add guarded gfx942 FP8 context prefill" (vLLM PR
 *            51551): Summary and "What this PR does" (static per-head Q/K/V
 *            scales from a calibrated artifact, finite positive descales,
 *            one-kernel static quantizer, 12 heads, D192 Q/K, D128 V).
 *   [OCP8]   OCP 8-bit Floating Point Specification (OFP8) rev 1.0, E4M3.
 *   [OCPMX]  OCP Microscaling Formats (MX) v1.0, section 5 (scale
 *            X = 2^(floor(log2 amax) - emax_elem), emax_elem = 8 for E4M3).
 *
 * Numeric conventions (all fixed here, see the .c file for each step):
 *   bf16 values are passed as their uint16 bit patterns, e4m3 as uint8,
 *   E8M0 as uint8.  "RN32(v)" is IEEE binary32 round-to-nearest-even,
 *   "bf16(v)" is round-to-nearest-even to bfloat16 (8 significant bits,
 *   binary32 exponent range, gradual underflow, overflow to infinity),
 *   "e4m3(v)" is saturating round-to-nearest-even to OCP E4M3 ("fn").
 */
#ifndef FP8NORM_ORACLE_H
#define FP8NORM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_ACT_SIGMOID = 0, ORACLE_ACT_SILU = 1 };

/* ---- codecs ---------------------------------------------------------- */
double   oracle_bf16_to_double(uint16_t b);
uint16_t oracle_bf16_from_double(double v);
double   oracle_e4m3_to_double(uint8_t c);
uint8_t  oracle_e4m3_from_float(float v);

/* bf16(act(g)): the real sigmoid or silu of a bf16 gate, rounded once. */
uint16_t oracle_act_bf16(uint16_t g, int act);

/* Element-wise array forms of the codecs above (plain loops). */
void oracle_bf16_from_float_n(const float* v, int64_t n, uint16_t* out);
void oracle_e4m3_from_float_n(const float* v, int64_t n, uint8_t* out);
void oracle_act_bf16_n(const uint16_t* g, int64_t n, int act, uint16_t* out);

/* RN32( (sum_i x_i^2) / n ) with the sum taken exactly; n >= 1, n < 2^31. */
float oracle_mean_square_bf16(const uint16_t* x, int64_t n);

/* Reciprocal RMS factor r = RN32(1 / RN32(sqrt(RN32(ms + eps)))). */
float oracle_rms_factor(float ms, float eps);

/* ---- operation (A): gated RMSNorm + per-token dynamic FP8 -------------- */
/* x, gate: [T, H, D] bf16, token stride x_stride / gate_stride (elements),
 * heads contiguous within a token; weight: [D] bf16 shared by all heads.
 * out: [T, H*D] e4m3 with token stride out_stride; scale: [T] fp32. */
void oracle_gated_rmsnorm_quant_token(const uint16_t* x, int64_t x_stride,
                                      const uint16_t* gate, int64_t gate_stride,
                                      const uint16_t* weight, int64_t T, int32_t H,
                                      int32_t D, float eps, int act, uint8_t* out,
                                      int64_t out_stride, float* scale);

/* Same operation for a single token t, writing only y (bf16 bits, [H*D]),
 * the codes and the scale of that token.  Used for sampled checks. */
void oracle_gated_rmsnorm_quant_one(const uint16_t* x_tok, const uint16_t* gate_tok,
                                    const uint16_t* weight, int32_t H, int32_t D,
                                    float eps, int act, uint16_t* y_tok,
                                    uint8_t* out_tok, float* scale_tok);

/* The same with the mean square of each head taken from ms[H] instead of
 * computed (a diagnostic for classifying mismatches by summation order). */
void oracle_gated_rmsnorm_quant_one_ms(const uint16_t* x_tok, const uint16_t* gate_tok,
                                       const uint16_t* weight, int32_t H, int32_t D, float eps,
                                       int act, const float* ms, uint16_t* y_tok,
                                       uint8_t* out_tok, float* scale_tok);

/* ---- the steps of (A), each on its own --------------------------------- */
/* Per-token quantisation of one bf16 row y[n]: scale = RN32(max|y| / 448),
 * codes e4m3(RN32(y / scale)); a zero row gets scale 0 and signed zeros. */
void oracle_quant_row(const uint16_t* y, int64_t n, uint8_t* out, float* scale);
/* (A) without the quantisation: y [H*D] bf16 for one token. */
void oracle_gated_rmsnorm_row(const uint16_t* x_tok, const uint16_t* gate_tok,
                              const uint16_t* weight, int32_t H, int32_t D, float eps, int act,
                              uint16_t* y_tok);
/* Gate product without the norm, then the per-token quantisation:
 * y = bf16(x * bf16(act(gate))) over n values. */
void oracle_gated_quant_row(const uint16_t* x, const uint16_t* gate, int64_t n, int act,
                            uint16_t* y, uint8_t* out, float* scale);

/* ---- operation (B): fused q/kv RMSNorm, q -> MXFP8, kv -> bf16 ---------- */
/* q: [M, Nq] bf16 (row stride q_stride), kv: [M, Nkv] bf16 (kv_stride);
 * Nq % 32 == 0.  q_out: e4m3 [M, Nq]; q_scale: E8M0 [M, Nq/32] row-major;
 * kv_out: bf16 [M, Nkv]. */
void oracle_rmsnorm_quant_mx(const uint16_t* q, int64_t q_stride, const uint16_t* q_weight,
                             int32_t Nq, const uint16_t* kv, int64_t kv_stride,
                             const uint16_t* kv_weight, int32_t Nkv, int64_t M, float eps,
                             uint8_t* q_out, int64_t q_out_stride, uint8_t* q_scale,
                             int64_t q_scale_stride, uint16_t* kv_out,
                             int64_t kv_out_stride);

/* The steps of (B): one normalised bf16 row, and the MX quantisation of a
 * bf16 row (n a multiple of 32; codes [n], E8M0 scales [n/32]). */
void oracle_rmsnorm_row(const uint16_t* x, const uint16_t* w, int32_t n, float eps, uint16_t* y);
void oracle_quant_mx_row(const uint16_t* yq, int32_t n, uint8_t* codes, uint8_t* scales);

/* E8M0 code of a block whose largest magnitude is the bf16 value `amax`. */
uint8_t oracle_e8m0_code(uint16_t amax_bits);

/* ---- inverse RoPE, then MXFP8 (the o-projection input) ------------------ */
/* One token: y = o with each head's span [rope_off, rope_off + R) rotated back
 * by the angles whose cos/sin are cs[0 .. R/2) / cs[R/2 .. R); pairs
 * (i, i + R/2) of the span, or (2i, 2i + 1) when interleaved. */
void oracle_inv_rope_row(const uint16_t* o_tok, int32_t H, int32_t D, int32_t rope_off,
                         int32_t R, int interleaved, const float* cs, uint16_t* y_tok);
/* o: [T, H, D] bf16 (token stride o_stride); positions [T] index the cache
 * cos_sin [P, R]; out: e4m3 [T, H*D]; scale: E8M0 [T, H*D/32] row-major. */
void oracle_inv_rope_quant_mx(const uint16_t* o, int64_t o_stride, int64_t T, int32_t H,
                              int32_t D, const int32_t* positions, const float* cos_sin,
                              int32_t rope_off, int32_t R, int interleaved, uint8_t* out,
                              int64_t out_stride, uint8_t* scale, int64_t scale_stride);

/* ---- operation (C): static per-head FP8 quant of packed Q/K/V ---------- */
/* One tensor: x [T, H, Dh] bf16 with (tok_stride, head_stride) in elements,
 * descale [H] fp32; out [T, H, Dh] e4m3 contiguous. */
void oracle_static_head_quant(const uint16_t* x, int64_t tok_stride, int64_t head_stride,
                              int64_t T, int32_t H, int32_t Dh, const float* descale,
                              uint8_t* out);

/* ---- dynamic per-head quant (what the static scales replace) ----------- */
/* amax[h] = max(amax[h], max over t, d of |x[t, h, d]|), NaN-propagating. */
void oracle_head_amax(const uint16_t* x, int64_t tok_stride, int64_t head_stride, int64_t T,
                      int32_t H, int32_t Dh, float* amax);
/* descale[h] = RN32(amax_h / 448) of this tensor, then codes as in (C); a zero
 * head gets descale 0 and signed zero codes. */
void oracle_dynamic_head_quant(const uint16_t* x, int64_t tok_stride, int64_t head_stride,
                               int64_t T, int32_t H, int32_t Dh, float* descale, uint8_t* out);

#ifdef __cplusplus
}
#endif
#endif
