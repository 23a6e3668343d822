/*
 * libfp8norm: row-wise normalize-then-quantize for GB300 (sm_103a).
 *
 * C ABI.  Every operation takes caller-owned DEVICE pointers, plain sizes and
 * strides (in elements), and the caller's cudaStream_t; it validates its
 * arguments on the host, enqueues its work on that stream (one kernel; the
 * dynamic per-head quantisation: a memset and two kernels) and returns
 * without synchronising, so the calls can be captured in a CUDA graph.
 * The operations allocate no memory and keep no state between calls.
 *
 * Element encodings: bf16 inputs/outputs are bfloat16 bit patterns (uint16);
 * e4m3 outputs are OCP FP8 E4M3 ("fn": bias 7, max 448, NaN 0x7F/0xFF, no
 * infinities); E8M0 scales are OCP MX exponent codes (value 2^(code - 127),
 * 0xFF = NaN).  "RN32" is IEEE binary32 round-to-nearest-even, "bf16()"
 * round-to-nearest-even to bfloat16, "e4m3()" saturating round-to-nearest-even
 * to E4M3 (|v| >= 448 -> +-448, sign of zero kept).
 *
 * Alignment: every tensor pointer must be 16-byte aligned; bf16 row strides
 * must be multiples of 8 elements (16-byte rows) and e4m3 row strides
 * multiples of 8 bytes (the kernels move 16-byte input and 8-byte output
 * chunks); see each call.
 *
 * Errors: a nonzero fp8n_status is returned and nothing is enqueued when an
 * argument is invalid.  FP8N_ERR_CUDA means a CUDA call failed; the CUDA error
 * code is then available from fp8n_last_cuda_error() on the calling thread.
 * A zero-sized problem (T == 0, M == 0) returns FP8N_OK without a launch.
 *
 * Optional device status word (uint32_t*, may be NULL): kernels OR bits into
 * it and never clear it: FP8N_STATUS_BAD_DESCALE (a descale that is not finite
 * and positive was used), FP8N_STATUS_PIPELINE_TIMEOUT (a pipeline wait gave
 * up after its iteration limit; the outputs of that launch are incomplete),
 * FP8N_STATUS_BAD_SEQLENS (the sequence prefix sums given to
 * fp8n_static_head_quant are not a valid partition of the T tokens),
 * FP8N_STATUS_BAD_POSITION (a token position outside the cos/sin cache was
 * clamped into it by the inverse-RoPE calls).
 */
#ifndef FP8NORM_H
#define FP8NORM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8n_stream_t; /* the same type as cudaStream_t */

typedef enum {
  FP8N_OK = 0,
  FP8N_ERR_NULL = 1,        /* a required pointer is NULL */
  FP8N_ERR_SHAPE = 2,       /* negative or inconsistent sizes / strides */
  FP8N_ERR_MISALIGNED = 3,  /* a pointer or stride breaks the 16-byte rule */
  FP8N_ERR_UNSUPPORTED = 4, /* a size outside the supported range */
  FP8N_ERR_BAD_SCALE = 5,   /* fp8n_check_descales found a bad descale */
  FP8N_ERR_CUDA = 6         /* a CUDA runtime call failed */
} fp8n_status;

typedef enum { FP8N_ACT_SIGMOID = 0, FP8N_ACT_SILU = 1 } fp8n_act;

/* Pairing of the rotated dims in a head's RoPE span [rope_off, rope_off + R):
 * (rope_off + i, rope_off + R/2 + i) or (rope_off + 2i, rope_off + 2i + 1). */
typedef enum { FP8N_ROPE_HALF = 0, FP8N_ROPE_INTERLEAVED = 1 } fp8n_rope_style;

#define FP8N_STATUS_BAD_DESCALE 0x1u
#define FP8N_STATUS_PIPELINE_TIMEOUT 0x2u
#define FP8N_STATUS_BAD_SEQLENS 0x4u
#define FP8N_STATUS_BAD_POSITION 0x8u

/* Human-readable name of a status code (static storage). */
const char* fp8n_status_string(fp8n_status s);

/* cudaError_t of the last FP8N_ERR_CUDA returned on this thread (0 if none). */
int fp8n_last_cuda_error(void);

/* Library version as 0xMMmmpp. */
uint32_t fp8n_version(void);

/*
 * (A) Gated RMSNorm fused with per-token dynamic FP8 quantisation.
 *
 * Source: "[ROCm][Kimi-K3] Fuse gated RMSNorm with per-token FP8 for KDA
 * o_proj" (vLLM PR 54254): Purpose (one kernel for gated RMSNorm and per-token
 * amax FP8 ahead of the o_proj GEMM); Tests (checked against sequential gated
 * RMSNorm + per-token amax); review thread on the torch reference helper and
 * the wrapper.
 *
 * For each token t and head h (per-head RMS over D):
 *   ms  = RN32(sum_d x[t,h,d]^2 / D)          (sum exact, order independent)
 *   r   = RN32(1 / RN32(sqrt(RN32(ms + eps))))
 *   y   = bf16( bf16(bf16(RN32(x * r)) * w[d]) * bf16(act(gate[t,h,d])) )
 * act is sigmoid or silu(g) = g * sigmoid(g), correctly rounded to bf16.
 * Per token (one scale over all H*D values):
 *   scale[t] = RN32(max|y| / 448);  out[t, h*D + d] = e4m3(RN32(y / scale[t]))
 * A token with max|y| == 0 gets scale 0 and zero codes carrying the sign of y.
 * The fused kernel sums the squares with a compensated (not exact) sum: in
 * rare heads its ms is one binary32 ulp off the exact one, which can move a
 * code by one step (the reduction-order budget of the codes).  The step
 * functions below take the exact mean square.
 *
 * x, gate : bf16 [T, H, D]; heads contiguous inside a token; token strides
 *           x_stride / gate_stride (elements, multiples of 8, >= H*D).
 * weight  : bf16 [D], shared by all heads.
 * out     : e4m3 [T, H*D], token stride out_stride (bytes = elements,
 *           multiple of 8, >= H*D).
 * scale   : fp32 [T].
 * Limits  : D a multiple of 8, 8 <= D <= 8192, H >= 1, H*D <= 16384,
 *           eps finite and >= 0; otherwise FP8N_ERR_UNSUPPORTED / _SHAPE.
 */
fp8n_status fp8n_gated_rmsnorm_quant_token(const void* x, int64_t x_stride, const void* gate,
                                           int64_t gate_stride, const void* weight, int64_t T,
                                           int32_t H, int32_t D, float eps, fp8n_act act,
                                           void* out, int64_t out_stride, float* scale,
                                           uint32_t* status, fp8n_stream_t stream);

/*
 * The steps of (A) on their own: the unfused pipeline that (A) replaces, and
 * the standalone per-token quantiser that other producers feed.
 *
 * Source: "[ROCm][Kimi-K3] Fuse gated RMSNorm with per-token FP8 for KDA
 * o_proj" (vLLM PR 54254): Purpose (gated RMSNorm followed by a standalone
 * dynamic per-token FP8 quant in the linear; the fused-decode output is
 * quantised by the per-token quantiser alone) and Profile, "Unfused" (the
 * gated norm and the per-token quant as two launches, 8.5 us against 4.2 us
 * fused); the cross-referenced "[ROCm][Kimi-K3] Fuse MLA sigmoid-mul with
 * per-token FP8 for o_proj" (PR 55043, title only) for the gate product
 * followed by the per-token quant.  Every rounding is the one of (A), with
 * the exact mean square, so fp8n_quant_token(fp8n_gated_rmsnorm_bf16(...))
 * is (A)'s definition bit for bit (the fused call is within its code
 * tolerance of it).
 */

/* y[t, h*D + d] = the bf16 y of (A), written out instead of quantised.
 * x, gate, weight, limits: as (A).  y: bf16 [T, H*D], token stride y_stride
 * (elements, multiple of 8, >= H*D). */
fp8n_status fp8n_gated_rmsnorm_bf16(const void* x, int64_t x_stride, const void* gate,
                                    int64_t gate_stride, const void* weight, int64_t T, int32_t H,
                                    int32_t D, float eps, fp8n_act act, void* y, int64_t y_stride,
                                    uint32_t* status, fp8n_stream_t stream);

/* Per-token FP8 of bf16 rows: scale[t] = RN32(max_n |y[t,n]| / 448),
 * out[t, n] = e4m3(RN32(y[t,n] / scale[t])) (zero rows: scale 0, signed zero
 * codes).  y: bf16 [T, N], token stride y_stride (elements, multiple of 8);
 * out: e4m3 [T, N], out_stride (bytes, multiple of 8); scale: fp32 [T].
 * Limits: N a multiple of 8 with 8 <= N <= 16384. */
fp8n_status fp8n_quant_token(const void* y, int64_t y_stride, int64_t T, int32_t N, void* out,
                             int64_t out_stride, float* scale, uint32_t* status,
                             fp8n_stream_t stream);

/* Gate product then per-token FP8: y = bf16(x * bf16(act(gate))) per element
 * of a token row of N values (no norm), then the quantisation of
 * fp8n_quant_token.  x, gate: bf16 [T, N] with token strides (elements,
 * multiples of 8); out, scale, limits: as fp8n_quant_token. */
fp8n_status fp8n_gated_quant_token(const void* x, int64_t x_stride, const void* gate,
                                   int64_t gate_stride, int64_t T, int32_t N, fp8n_act act,
                                   void* out, int64_t out_stride, float* scale, uint32_t* status,
                                   fp8n_stream_t stream);

/*
 * (B) Fused q/kv RMSNorm: q leaves as MXFP8, kv as normalised bf16.
 *
 * Source: "[ROCm][Perf] FP8 o-projection for DeepSeek-V4.1-Flash MLA on AMD
 * MI355X" (vLLM PR 57081), third commit message (one producer normalises q and
 * kv, emits q as MXFP8 with row-major E8M0 scales, bitwise identical to the
 * unfused steps); OCP Microscaling Formats v1.0 section 5 (block scale
 * 2^(floor(log2 amax) - 8) for E4M3 elements).
 *
 * Per row m:  yq = bf16(bf16(RN32(q * r_q)) * q_weight), r_q over the whole q
 * row as in (A); per 32-column block b of yq:
 *   e = clamp(floor(log2 max|yq_b|) - 8, -127, 127)  (e = -127 if the block is 0)
 *   q_scale[m, b] = e + 127;  q_out[m, 32b + j] = e4m3(yq * 2^-e)
 * kv_out[m, :] = bf16(bf16(RN32(kv * r_kv)) * kv_weight).
 *
 * q     : bf16 [M, Nq], row stride q_stride (elements, multiple of 8).
 * kv    : bf16 [M, Nkv], row stride kv_stride (elements, multiple of 8); may be
 *         NULL when Nkv == 0.
 * q_out : e4m3 [M, Nq], row stride q_out_stride (bytes, multiple of 8).
 * q_scale: E8M0 uint8 [M, Nq/32] row-major, row stride q_scale_stride (bytes).
 * kv_out: bf16 [M, Nkv], row stride kv_out_stride (elements, multiple of 8).
 * Limits: Nq a multiple of 32 with 32 <= Nq <= 16384; Nkv a multiple of 8 with
 *         0 <= Nkv <= 16384.
 */
fp8n_status fp8n_rmsnorm_quant_mx(const void* q, int64_t q_stride, const void* q_weight,
                                  int32_t Nq, const void* kv, int64_t kv_stride,
                                  const void* kv_weight, int32_t Nkv, int64_t M, float eps,
                                  void* q_out, int64_t q_out_stride, uint8_t* q_scale,
                                  int64_t q_scale_stride, void* kv_out, int64_t kv_out_stride,
                                  uint32_t* status, fp8n_stream_t stream);

/*
 * The two steps of (B) on their own.  Source: "[ROCm][Perf] FP8 o-projection
 * for DeepSeek-V4.1-Flash MLA on AMD MI355X" (vLLM PR 57081), third commit
 * message: the fused producer is bitwise identical to the unfused path, a
 * row RMSNorm to bf16 followed by the MXFP8 quantisation of q.  Hence
 * fp8n_quant_mx(fp8n_rmsnorm_bf16(q)) equals the q outputs of
 * fp8n_rmsnorm_quant_mx, and fp8n_rmsnorm_bf16(kv) its kv output.
 */

/* y[m, :] = bf16(bf16(RN32(x * r)) * weight), r over the whole row as in (B).
 * x: bf16 [M, N], row stride x_stride; weight: bf16 [N]; y: bf16 [M, N], row
 * stride y_stride (elements, multiples of 8).  Limits: N a multiple of 8 with
 * 8 <= N <= 16384, eps finite and >= 0. */
fp8n_status fp8n_rmsnorm_bf16(const void* x, int64_t x_stride, const void* weight, int64_t M,
                              int32_t N, float eps, void* y, int64_t y_stride, uint32_t* status,
                              fp8n_stream_t stream);

/* MXFP8 of bf16 rows as given (the block rule of (B) without the norm):
 * scale[m, b] = E8M0 code of block b of y[m, :], out = e4m3(y * 2^-e).
 * y: bf16 [M, N] (row stride multiple of 8); out: e4m3 [M, N] (row stride
 * bytes, multiple of 8); scale: uint8 [M, N/32], row stride scale_stride.
 * Limits: N a multiple of 32 with 32 <= N <= 16384. */
fp8n_status fp8n_quant_mx(const void* y, int64_t y_stride, int64_t M, int32_t N, void* out,
                          int64_t out_stride, uint8_t* scale, int64_t scale_stride,
                          uint32_t* status, fp8n_stream_t stream);

/*
 * Inverse RoPE of the o-projection input, then MXFP8.
 *
 * Source: "[ROCm][Perf] FP8 o-projection for DeepSeek-V4.1-Flash MLA on AMD
 * MI355X" (vLLM PR 57081): first commit message (a fused inverse-RoPE + FP8
 * quantiser feeds the MX-scaled a8w8 o-projection GEMM) and second commit
 * message (the layer holds a pre-computed FP32 cos/sin cache of 4096
 * positions).  The pages give neither the rotation convention nor the cache
 * layout; both are arguments here.
 *
 * Per token t, with cache row cs = cos_sin[positions[t]] (cos of the R/2
 * pair angles, then their sin), every head's span [rope_off, rope_off + R)
 * is rotated back pair by pair (pair i as fp8n_rope_style says):
 *   y1 = bf16(RN32(RN32(x1 * cs[i]) + RN32(x2 * cs[R/2 + i])))
 *   y2 = bf16(RN32(RN32(x2 * cs[i]) - RN32(x1 * cs[R/2 + i])))
 * other elements pass unchanged; the bf16 row [H*D] is then quantised as the
 * q part of fp8n_rmsnorm_quant_mx: per 32 consecutive elements
 *   e = clamp(floor(log2 max|y|) - 8, -127, 127), scale = e + 127,
 *   out = e4m3(y * 2^-e).
 * fp8n_quant_mx(fp8n_inv_rope_bf16(...)) equals this call bit for bit.
 *
 * o        : bf16 [T, H, D], heads contiguous, token stride o_stride
 *            (elements, multiple of 8, >= H*D).
 * positions: int32 [T] device, each in [0, num_positions); a position
 *            outside is clamped into the cache and sets
 *            FP8N_STATUS_BAD_POSITION (when status is not NULL).
 * cos_sin  : fp32 [num_positions, rope_dim] device, 16-byte aligned.
 * out      : e4m3 [T, H*D], token stride out_stride (bytes, multiple of 16).
 * scale    : E8M0 uint8 [T, H*D/32] row-major, token stride scale_stride.
 * Limits   : D a multiple of 32 in [32, 8192]; rope_off a multiple of 8;
 *            rope_dim a multiple of 16 (0: no rotation, only the MXFP8);
 *            rope_off + rope_dim <= D; fewer than 2^31 MX blocks in all.
 */
fp8n_status fp8n_inv_rope_quant_mx(const void* o, int64_t o_stride, int64_t T, int32_t H,
                                   int32_t D, const int32_t* positions, const float* cos_sin,
                                   int32_t num_positions, int32_t rope_off, int32_t rope_dim,
                                   fp8n_rope_style style, void* out, int64_t out_stride,
                                   uint8_t* scale, int64_t scale_stride, uint32_t* status,
                                   fp8n_stream_t stream);

/* The inverse-RoPE step alone: y[t, :] = the rotated bf16 row above.
 * y: bf16 [T, H*D], token stride y_stride (elements, multiple of 8).  Other
 * arguments and limits: as fp8n_inv_rope_quant_mx. */
fp8n_status fp8n_inv_rope_bf16(const void* o, int64_t o_stride, int64_t T, int32_t H, int32_t D,
                               const int32_t* positions, const float* cos_sin,
                               int32_t num_positions, int32_t rope_off, int32_t rope_dim,
                               fp8n_rope_style style, void* y, int64_t y_stride, uint32_t* status,
                               fp8n_stream_t stream);

/*
 * (C) Static per-head FP8 quantisation of packed variable-length Q, K, V.
 *
 * Source: "[ROCm][MLA] Add guarded gfx942 FP8 context prefill" (vLLM PR
 * 51551): Summary and "What this PR does" (static per-head Q/K/V scales from a
 * calibrated artifact replace dynamic amax reductions; a one-kernel static
 * quantizer; finite positive descales; 12 heads, D192 Q/K, D128 V).
 *
 *   q_out[t,h,d] = e4m3(RN32(q[t,h,d] / q_descale[h]))  and likewise for k, v,
 * all three tensors in one launch.
 *
 * q, k     : bf16 [T, H, Dqk] with token stride qk_tok_stride and head stride
 *            qk_head_stride (elements, multiples of 8); the d axis contiguous.
 * v        : bf16 [T, H, Dv] with v_tok_stride, v_head_stride.
 * descales : fp32 [H] each, device memory.  A descale that is not finite and
 *            positive is still applied as an IEEE division and sets
 *            FP8N_STATUS_BAD_DESCALE in *status (when status is not NULL).
 * cu_seqlens: optional int32 [num_seqs + 1] device prefix sums of the packed
 *            sequences (NULL allowed; 4-byte aligned).  The map is elementwise,
 *            so the codes do not depend on it; when it and status are both
 *            given, the kernel checks on the device (no host synchronisation)
 *            that cu_seqlens[0] == 0, that the sums never decrease and that
 *            cu_seqlens[num_seqs] == T, and sets FP8N_STATUS_BAD_SEQLENS in
 *            *status otherwise.
 * outputs  : e4m3, contiguous [T, H, Dqk] / [T, H, Dv].
 * Limits   : Dqk, Dv multiples of 8 in [8, 8192]; 1 <= H <= 256; fewer than
 *            2^31 16-byte chunks in Q, K and V together.
 */
fp8n_status fp8n_static_head_quant(const void* q, const void* k, const void* v,
                                   int64_t qk_tok_stride, int64_t qk_head_stride,
                                   int64_t v_tok_stride, int64_t v_head_stride, int64_t T,
                                   int32_t H, int32_t Dqk, int32_t Dv, const float* q_descale,
                                   const float* k_descale, const float* v_descale,
                                   const int32_t* cu_seqlens, int32_t num_seqs, void* q_out,
                                   void* k_out, void* v_out, uint32_t* status,
                                   fp8n_stream_t stream);

/*
 * Dynamic per-head FP8 quantisation of packed Q, K, V: the path that the
 * static quantiser (C) replaces, and the producer of (C)'s descales.
 *
 * Source: "[ROCm][MLA] Add guarded gfx942 FP8 context prefill" (vLLM PR
 * 51551): Summary (static per-head scales remove the dynamic amax
 * reductions) and the commit messages (dynamic per-head reductions cost work
 * on every long-context prefill step; dynamic FP8 stays available).
 *
 * For each tensor X in (Q, K, V) and head h:
 *   descale_X[h] = RN32(max_{t,d} |X[t,h,d]| / 448)
 *   X_out[t,h,d] = e4m3(RN32(X[t,h,d] / descale_X[h]))
 * A head whose values are all zero gets descale 0 and zero codes carrying the
 * sign of x; a NaN anywhere in a head makes its descale NaN and its codes
 * NaN.  Tensors, strides, outputs and limits: as (C).
 * workspace: device uint32 [3*H], 4-byte aligned, owned by the caller; the
 *            call zeroes it on the stream and leaves the per-head maxima in it
 *            (as binary32 bit patterns); calls that share it must not overlap.
 * q/k/v_descale: fp32 [H] device outputs.
 * Work enqueued: a memset of the workspace, the max pass, the quantise pass.
 */
fp8n_status fp8n_dynamic_head_quant(const void* q, const void* k, const void* v,
                                    int64_t qk_tok_stride, int64_t qk_head_stride,
                                    int64_t v_tok_stride, int64_t v_head_stride, int64_t T,
                                    int32_t H, int32_t Dqk, int32_t Dv, uint32_t* workspace,
                                    float* q_descale, float* k_descale, float* v_descale,
                                    void* q_out, void* k_out, void* v_out, fp8n_stream_t stream);

/*
 * fp8n_dynamic_head_quant without a workspace argument: the same computation
 * and outputs, for callers that cannot allocate device memory, such as code
 * embedded in a host application that owns all device memory through its
 * own fixed pool (allocating outside it breaks the host's memory accounting),
 * or code on a latency-critical path where cudaMalloc would synchronise the
 * device.  This entry point has no counterpart in the paper.
 *
 * The per-head maxima are kept in a static device array of the library
 * (3 * 256 words, 3 KB, held by every GPU that loads the library until the
 * process exits).  The first call on each device looks up that array's
 * device address (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture.  The cached address belongs to the device's
 * primary context (the one the CUDA runtime uses): call this entry point
 * with that context current, and not after cudaDeviceReset (which ends the
 * context and with it the array) unless the library is loaded anew.  The call allocates nothing and zeroes the
 * array on `stream` before using it.  All calls share the one array: two
 * calls whose work overlaps on the GPU (different streams, or the same array
 * in use by an earlier call not yet finished on another stream) race and
 * may produce wrong descales; order them on one stream or with events.
 * Limits as fp8n_dynamic_head_quant; H above 256 is rejected with
 * FP8N_ERR_UNSUPPORTED.
 */
fp8n_status fp8n_dynamic_head_quant_noalloc(const void* q, const void* k, const void* v,
                                            int64_t qk_tok_stride, int64_t qk_head_stride,
                                            int64_t v_tok_stride, int64_t v_head_stride,
                                            int64_t T, int32_t H, int32_t Dqk, int32_t Dv,
                                            float* q_descale, float* k_descale, float* v_descale,
                                            void* q_out, void* k_out, void* v_out,
                                            fp8n_stream_t stream);

/*
 * Calibration: running per-head maxima of one packed tensor,
 *   amax[h] = max(amax[h], max_{t,d} |x[t,h,d]|),
 * as collected after warm-up to build (C)'s descales.  Source: "[ROCm][MLA]
 * Add guarded gfx942 FP8 context prefill" (vLLM PR 51551), "What this PR
 * does" (layer-owned Q/K/V maxima collected after warmup in calibration
 * mode).  x: bf16 [T, H, Dh] with token and head strides (elements, multiples
 * of 8); amax: fp32 [H] device, in/out, entries >= +0 on entry (start from
 * zeros); a NaN in x makes its head's entry NaN.  Limits: Dh a multiple of 8
 * in [8, 8192], 1 <= H <= 256.
 */
fp8n_status fp8n_head_amax(const void* x, int64_t tok_stride, int64_t head_stride, int64_t T,
                           int32_t H, int32_t Dh, float* amax, fp8n_stream_t stream);

/*
 * Gate activation alone: out[i] = bf16(act(g[i])), act = sigmoid or
 * silu(g) = g * sigmoid(g), correctly rounded (nearest-even of the real
 * function; limits at +-inf, NaN stays NaN).  This is the gate factor of (A),
 * computed by the same device code; the source is the torch reference helper
 * in "[ROCm][Kimi-K3] Fuse gated RMSNorm with per-token FP8 for KDA o_proj"
 * (the gate enters through torch.sigmoid in the activation dtype).
 * g, out: bf16 [n], 2-byte aligned device pointers; n >= 0.
 */
fp8n_status fp8n_gate_act_bf16(const void* g, int64_t n, fp8n_act act, void* out,
                               fp8n_stream_t stream);

/* Target of fp8n_convert_f32. */
typedef enum { FP8N_CVT_BF16 = 0, FP8N_CVT_E4M3 = 1 } fp8n_cvt;

/*
 * The two roundings of binary32 values that every operation above ends with,
 * alone: out[i] = bf16(in[i]) (nearest-even, 2 bytes each; NaN stays NaN) or
 * out[i] = e4m3(in[i]) (OCP E4M3 "fn": saturating nearest-even, |v| above 448
 * and infinities to +-448, NaN to 0x7F/0xFF, signed zeros kept; 1 byte each),
 * by the same device conversions the kernels use.  Sources: the torch
 * reference helper in "[ROCm][Kimi-K3] Fuse gated RMSNorm with per-token FP8
 * for KDA o_proj" (values rounded to the bf16 activation dtype; codes in the
 * e4m3 format whose largest value 448 is the quantiser's fp8 maximum) and the
 * OCP 8-bit floating point specification (OFP8) for E4M3.
 * in: fp32 [n], 4-byte aligned device pointer; out: [n] bf16 (2-byte aligned)
 * or uint8; n >= 0; FP8N_ERR_UNSUPPORTED for another target.
 */
fp8n_status fp8n_convert_f32(const float* in, int64_t n, fp8n_cvt to, void* out,
                             fp8n_stream_t stream);

/*
 * Synchronous helper: reads n fp32 descales from device memory (through a
 * host copy on `stream`, which it synchronises) and returns
 * FP8N_ERR_BAD_SCALE unless every one is finite and > 0.  Source: the
 * static-scale validation in "[ROCm][MLA] Add guarded gfx942 FP8 context
 * prefill" (finite positive descales are checked before use; missing or
 * incompatible scales fail instead of falling back).  Not for use inside a
 * stream capture.  1 <= n <= 65536.
 */
fp8n_status fp8n_check_descales(const float* descale, int32_t n, fp8n_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
