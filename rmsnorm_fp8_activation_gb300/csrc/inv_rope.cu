// Inverse RoPE of the o-projection input, then MXFP8.
//
// Source: "[ROCm][Perf] FP8 o-projection for DeepSeek-V4.1-Flash MLA on AMD
// MI355X" (vLLM PR 57081): first commit message (a fused inverse-RoPE + FP8
// quantiser feeds the MX-scaled a8w8 o-projection GEMM) and second commit
// message (the layer holds a pre-computed FP32 cos/sin cache of 4096
// positions).  Per token t with position p: every head's span
// [rope_off, rope_off + R) is rotated back pair by pair with the cache row p,
//   y1 = x1 cos + x2 sin,  y2 = x2 cos - x1 sin
// (each product and sum one binary32 operation), rounded to bf16, and the bf16
// row [H*D] is quantised to MXFP8 by the block rule of the fused q/kv
// producer: E8M0 code floor(log2 amax) - 8 + 127 per 32 elements, element
// codes e4m3(y * 2^-e).
//
// GB300 design: an HBM stream.  Work units are half MX blocks (two adjacent
// 16-byte chunks of one head); a warp takes 64 units at a time (lane l: units
// l and l + 32, read-only loads), the blocks of a head that meet the RoPE span
// and the others in two separate loops, so that the rotation is warp-uniform
// work.  The span starts on a chunk and holds whole chunks, so a chunk is
// rotated or passed through as a whole; with rotate-half pairs a chunk's
// partner lies R/2 elements away in the same head (another lane reads it too,
// so it comes from L1), with interleaved pairs it is the chunk itself.  The
// rotation takes binary32 products and sums through the rounding intrinsics
// (never contracted into a fused multiply-add).  An MX block is two
// neighbouring lanes: the largest magnitude over the lane's eight bf16 pairs
// and one xor-shuffle give its amax.
#include "common.cuh"
#include "kernels.h"

namespace fp8n {
namespace {

constexpr int kRopeThreads = 256;

// Work units are half MX blocks (two adjacent 16-byte chunks).  The blocks of
// a head that meet the RoPE span ("rope blocks", [rb0, rb0 + nrb)) and the
// others ("pure blocks") are walked by two separate loops, so that the
// rotation is warp-uniform work.
struct RopeIdx {
  FastDiv heads;     // H
  FastDiv pure_hb;   // half-blocks of the pure blocks of a head
  FastDiv rope_hb;   // half-blocks of the rope blocks of a head
  uint32_t rb0_hb;   // first rope half-block of a head
  uint32_t rope_n;   // rope half-blocks of a head (0 without a span)
  uint32_t n_pure, n_rope;  // units of each kind in the launch
};

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// RN32(RN32(x c) + RN32(w s)), each step its own binary32 operation.  The
// rounding intrinsics are never contracted into a fused multiply-add (packed
// f32x2 multiplies followed by packed adds were: the compiler fused them,
// which rounds once where the definition rounds twice).
__device__ __forceinline__ float rot1(float x, float c, float w, float s) {
  return __fadd_rn(__fmul_rn(x, c), __fmul_rn(w, s));
}

// y pair = bf16 pair of (x c + w s) for bf16 pairs x, w and binary32 pairs
// (c0, c1), (s0, s1).  Both halves of a rotation take this form:
// y1 = x1 c + x2 s, and y2 = x2 c - x1 s = x2 c + (-x1) s, since negating a
// product's factor negates the rounded product and a + (-b) is a - b, signs of
// zero included.
__device__ __forceinline__ uint32_t rot_pair(uint32_t x, uint32_t w, float c0, float c1, float s0,
                                             float s1) {
  return pack_bf16x2(rot1(bf16_lo(x), c0, bf16_lo(w), s0), rot1(bf16_hi(x), c1, bf16_hi(w), s1));
}

// Interleaved pairs (2k, 2k+1) of a chunk, with the angles cc, ss of its four
// pairs: (x1, x2) -> (x1 c + x2 s, x2 c + (-x1) s).
__device__ __forceinline__ void rot_interleaved(uint4& v, float4 cc, float4 ss) {
  uint32_t* w = &v.x;
  const float cv[4] = {cc.x, cc.y, cc.z, cc.w}, sv[4] = {ss.x, ss.y, ss.z, ss.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t swapped = __byte_perm(w[k], 0, 0x1032) ^ 0x80000000u;  // (x2, -x1)
    w[k] = rot_pair(w[k], swapped, cv[k], cv[k], sv[k], sv[k]);
  }
}

// Rotate-half pairs of a chunk with its partner chunk pv (already negated for
// a chunk of the second half) and the angles of its eight pairs.
__device__ __forceinline__ void rot_half(uint4& v, const uint4& pv, float4 c0, float4 c1, float4 s0,
                                         float4 s1) {
  uint32_t* w = &v.x;
  const uint32_t* pw = &pv.x;
  const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = rot_pair(w[k], pw[k], cv[2 * k], cv[2 * k + 1], sv[2 * k], sv[2 * k + 1]);
}

__device__ __forceinline__ uint4 negate_bf16x8(uint4 v) {
  return make_uint4(v.x ^ 0x80008000u, v.y ^ 0x80008000u, v.z ^ 0x80008000u, v.w ^ 0x80008000u);
}

// The chunk v (head-local elements j0 .. j0 + 7 of token t's head at src)
// rotated back; j0 lies in the span.
template <bool INTERLEAVED>
__device__ __forceinline__ void rotate_chunk(const RopeParams& p, const uint16_t* src, int j0,
                                             uint32_t t, uint4& v, bool& bad) {
  const int half = p.R / 2;
  int pos = __ldg(p.positions + t);
  if (pos < 0 || pos >= p.P) {  // outside the cache: flagged, clamped to stay in bounds
    bad = true;
    pos = pos < 0 ? 0 : p.P - 1;
  }
  const float* cs = p.cos_sin + (int64_t)pos * p.R;
  if (INTERLEAVED) {  // pair index i0 + k
    const int i0 = (j0 - p.rope_off) / 2;
    rot_interleaved(v, __ldg(reinterpret_cast<const float4*>(cs + i0)),
                    __ldg(reinterpret_cast<const float4*>(cs + half + i0)));
    return;
  }
  // rotate-half: the partner chunk lies R/2 elements away in the same head; a
  // chunk of the second half takes its partner negated
  const bool first = j0 < p.rope_off + half;
  const int i0 = j0 - p.rope_off - (first ? 0 : half);
  uint4 pv = ldg16(src + (first ? j0 + half : j0 - half));
  if (!first) pv = negate_bf16x8(pv);
  const float4* c4 = reinterpret_cast<const float4*>(cs + i0);
  const float4* s4 = reinterpret_cast<const float4*>(cs + half + i0);
  rot_half(v, pv, __ldg(c4), __ldg(c4 + 1), __ldg(s4), __ldg(s4 + 1));
}

// The MXFP8 codes of a half block (lane pair = MX block; called by the whole
// warp) and its E8M0 byte; both lanes of a block store the same byte.
__device__ __forceinline__ uint4 mx_half_block(const uint4& v0, const uint4& v1, bool ok,
                                               uint8_t* scale_at) {
  uint32_t am = absmax8(&v0.x, &v1.x);
  am = max_nan_bf16x2(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
  const uint32_t code = mx_code(max(am & 0xFFFFu, am >> 16));
  if (ok) *scale_at = (uint8_t)code;
  if (code == 0xFFu) return make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const uint32_t sb = (254u - code) << 7;  // bf16 bits of 2^-e (normal: code <= 246)
  const uint32_t s2 = sb | (sb << 16);
  const uint32_t* a = &v0.x;
  const uint32_t* b = &v1.x;
  return make_uint4(scaled_e4m3_pair(a[0], s2) | (scaled_e4m3_pair(a[1], s2) << 16),
                    scaled_e4m3_pair(a[2], s2) | (scaled_e4m3_pair(a[3], s2) << 16),
                    scaled_e4m3_pair(b[0], s2) | (scaled_e4m3_pair(b[1], s2) << 16),
                    scaled_e4m3_pair(b[2], s2) | (scaled_e4m3_pair(b[3], s2) << 16));
}

// One loop over units of one kind: a warp takes 64 units at a time, lane l
// units l and l + 32 (two adjacent chunks each: an MX block is the lane pair
// (l, l ^ 1), its amax one xor-shuffle away).  Consecutive lanes hold
// consecutive half-blocks of a head's pure (or rope) blocks, so the loads of
// a warp are runs of contiguous bytes.
template <bool QUANT, bool INTERLEAVED, bool ROT>
__device__ __forceinline__ void unit_loop(const RopeParams& p, const RopeIdx& ix, bool& bad) {
  constexpr int kSteps = 2;
  const int lane = threadIdx.x & 31;
  const uint32_t n = ROT ? ix.n_rope : ix.n_pure;
  const FastDiv& per_head = ROT ? ix.rope_hb : ix.pure_hb;
  const uint32_t rs0 = (uint32_t)p.rope_off / 8, rs1 = (uint32_t)(p.rope_off + p.R) / 8;
  const uint32_t warps = gridDim.x * (blockDim.x >> 5);
  for (uint32_t base = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * (32 * kSteps);
       base < n; base += warps * (32 * kSteps)) {
    uint4 v[kSteps][2];
    uint32_t tk[kSteps], hk[kSteps], bk[kSteps];  // token, head, half-block in the head
#pragma unroll
    for (int j = 0; j < kSteps; ++j) {
      const uint32_t u = base + 32 * j + lane;
      v[j][0] = v[j][1] = make_uint4(0, 0, 0, 0);
      tk[j] = hk[j] = bk[j] = 0;
      if (u < n) {
        const uint32_t th = fdiv(u, per_head);
        const uint32_t k = u - th * per_head.d;
        const uint32_t t = fdiv(th, ix.heads);
        tk[j] = t, hk[j] = th - t * ix.heads.d;
        bk[j] = ROT ? ix.rb0_hb + k : (k < ix.rb0_hb ? k : k + ix.rope_n);
        const uint16_t* src = p.o + (int64_t)t * p.o_stride + (int64_t)hk[j] * p.D + 16 * bk[j];
        v[j][0] = ldg16(src);
        v[j][1] = ldg16(src + 8);
      }
    }
    if (ROT) {
#pragma unroll
      for (int j = 0; j < kSteps; ++j) {
        if (base + 32 * j + lane >= n) continue;
        const uint16_t* head = p.o + (int64_t)tk[j] * p.o_stride + (int64_t)hk[j] * p.D;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t c = 2 * bk[j] + k;  // chunk in the head
          if (c >= rs0 && c < rs1) rotate_chunk<INTERLEAVED>(p, head, 8 * (int)c, tk[j], v[j][k], bad);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kSteps; ++j) {
      const bool ok = base + 32 * j + lane < n;
      const int64_t col = (int64_t)hk[j] * p.D + 16 * bk[j];  // first element in the row
      if (!QUANT) {
        if (ok) {
          uint16_t* dst = p.y_out + (int64_t)tk[j] * p.y_stride + col;
          *reinterpret_cast<uint4*>(dst) = v[j][0];
          *reinterpret_cast<uint4*>(dst + 8) = v[j][1];
        }
        continue;
      }
      const uint4 o = mx_half_block(v[j][0], v[j][1], ok,
                                    p.scale + (int64_t)tk[j] * p.scale_stride + (col >> 5));
      if (ok) *reinterpret_cast<uint4*>(p.out + (int64_t)tk[j] * p.out_stride + col) = o;
    }
  }
}

template <bool QUANT, bool INTERLEAVED>
__global__ void __launch_bounds__(kRopeThreads, 4) inv_rope_kernel(const RopeParams p, const RopeIdx ix) {
  pdl_launch_dependents();  // programmatic dependent launch (see launch_pdl)
  pdl_wait();
  bool bad = false;
  unit_loop<QUANT, INTERLEAVED, false>(p, ix, bad);
  unit_loop<QUANT, INTERLEAVED, true>(p, ix, bad);
  if (bad && p.status) atomicOr(p.status, kStatusBadPosition);
}

template <bool QUANT, bool INTERLEAVED>
cudaError_t launch_v(const RopeParams& p, const RopeIdx& ix, cudaStream_t stream) {
  auto kern = inv_rope_kernel<QUANT, INTERLEAVED>;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRopeThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t units = (int64_t)ix.n_pure + ix.n_rope;
  const int64_t want = (int64_t)sm_count() * per_sm;
  const int64_t need = (units + 2 * kRopeThreads - 1) / (2 * kRopeThreads);  // 2 units a lane
  const int grid = (int)(need < want ? need : want);
  return launch_pdl(kern, grid, kRopeThreads, 0, stream, p, ix);
}

}  // namespace

cudaError_t launch_inv_rope(const RopeParams& p, cudaStream_t stream) {
  const uint32_t bph = (uint32_t)p.D / 32;  // MX blocks per head
  const uint32_t rb0 = p.R ? (uint32_t)p.rope_off / 32 : 0;
  const uint32_t rb1 = p.R ? ((uint32_t)(p.rope_off + p.R) + 31) / 32 : 0;
  const uint32_t pure = 2 * (bph - (rb1 - rb0)), rope = 2 * (rb1 - rb0);
  const uint32_t th = (uint32_t)p.T * (uint32_t)p.H;
  RopeIdx ix;
  ix.heads = make_fastdiv((uint32_t)p.H);
  ix.pure_hb = make_fastdiv(pure ? pure : 1);
  ix.rope_hb = make_fastdiv(rope ? rope : 1);
  ix.rb0_hb = 2 * rb0;
  ix.rope_n = rope;
  ix.n_pure = th * pure;
  ix.n_rope = th * rope;
  if (p.quant)
    return p.interleaved ? launch_v<true, true>(p, ix, stream) : launch_v<true, false>(p, ix, stream);
  return p.interleaved ? launch_v<false, true>(p, ix, stream) : launch_v<false, false>(p, ix, stream);
}

}  // namespace fp8n
