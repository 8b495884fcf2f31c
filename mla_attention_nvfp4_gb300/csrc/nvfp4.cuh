// NVFP4 device codecs shared by the cache-write kernel, the prefill
// epilogue and the quantise-rows hook.
//
// NVFP4: e2m1 codes, one e4m3 block scale per 16 elements, fp32 global scale
// gs (dequantisation direction).  Source: "Add NVFP4/FP8 Q/K/P/V + 2:4
// attention quantization for MLA (vLLM TRITON_MLA) - #2244", PR description,
// "Contract notes" (block 1x16 along the contraction axis, E4M3 block scale,
// global amax/(6*448)).
//
// Two evaluations of the block scale and codes:
//  * correctly rounded (block_scale_rn, encode8_rn; the cache write): the
//    definition in IEEE float32 arithmetic, divisions included,
//        s_raw = (amax16 / 6) / gs,   sb = e4m3 RNE-satfinite(s_raw),
//        S     = e4m3(sb) * gs,       code = e2m1 RNE-satfinite(x / S)
//    (all codes 0 when S is 0).  Each division a / b is computed from the
//    correctly rounded reciprocal y = 1/b: q0 = a * y, r = a - q0 * b
//    (exact, one fma), q = q0 + r * y (one fma), which is the correctly
//    rounded quotient (Markstein's theorem for round-to-nearest division
//    from a correctly rounded reciprocal): bit-identical to float32
//    division, at two fmas per element;
//  * reciprocal form (block_scale, encode8; the prefill epilogue and the
//    quantise-rows hook): s_raw = amax16 * (1 / (6 gs)), q = x * (1 / S),
//    each quotient within 1.5 ulp of the correctly rounded one, so a code or
//    scale byte differs from it only when that quotient lies within 1.5 ulp
//    of a rounding midpoint.  The epilogue's quantisation sits on the
//    prefill's critical path (it holds the output accumulator), where the
//    two fmas per element measured 7 % of the prefill.
// A global scale outside [2^-100, 2^100] is invalid (codes and scales 0).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mla {

// 2 x f32 -> e2m1x2 byte; `lo` goes to bits 0..3, `hi` to bits 4..7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// 8 x f32 -> 8 e2m1 codes in one 32-bit word, element i in nibble i.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// f32 -> e4m3 byte, round to nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t cvt_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// 2 x f32 -> 2 e4m3 bytes (lo in bits 0..7).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// e4m3 byte -> f32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two e4m3 bytes (lo in bits 0..7) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_pair(uint32_t two_bytes) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return h2;
}

__device__ __forceinline__ bool scale_ok(float gs) {
  return gs >= 7.888609052210118e-31f && gs <= 1.2676506002282294e30f;  // [2^-100, 2^100]
}

// a / b rounded to nearest even, given y = 1 / b rounded to nearest even
// and a quotient that cannot overflow.
__device__ __forceinline__ float div_rn(float a, float b, float y) {
  const float q0 = __fmul_rn(a, y);
  return __fmaf_rn(__fmaf_rn(-q0, b, a), y, q0);
}

// Per-tensor factors of the raw block scale: 1 / gs (correctly rounded
// form) and 1 / (6 gs) (reciprocal form), each rounded to nearest.
__device__ __forceinline__ float inv_scale(float gs) { return __frcp_rn(gs); }
__device__ __forceinline__ float scale_factor(float gs) { return __frcp_rn(__fmul_rn(6.0f, gs)); }

// Correctly rounded block scale from the block's amax (exact in any
// reduction order) and inv_gs = inv_scale(gs).  Returns the scale byte sb
// and sets S = e4m3(sb) * gs and R = 1 / S (rounded to nearest), or R = 0
// when S is 0 (the block then encodes as all-zero codes).  `bounded` tells
// whether every |x| / S of the block is at most ~6.4 (the scale did not
// saturate), so that the codes' quotients cannot overflow.
__device__ __forceinline__ uint32_t block_scale_rn(float amax, float inv_gs, float gs, float& R, float& S,
                                                   bool& bounded) {
  const float sixth = 0.16666667163372040f;  // 1/6 rounded to nearest float32
  const float q6 = div_rn(amax, 6.0f, sixth);
  const float s0 = __fmul_rn(q6, inv_gs);
  const float s_raw = isfinite(s0) ? div_rn(q6, gs, inv_gs) : s0;
  const uint32_t sb = cvt_e4m3(s_raw);
  bounded = s_raw <= 448.0f;
  S = __fmul_rn(e4m3_to_f32(sb), gs);
  R = (S > 0.f) ? __frcp_rn(S) : 0.f;
  return sb;
}

// Eight correctly rounded codes of x / S (element i in nibble i); all zero
// when R == 0.  An unbounded block (saturated scale) keeps the reciprocal
// products, which the conversion saturates the same way.
__device__ __forceinline__ uint32_t encode8_rn(const float* x, float R, float S, bool bounded) {
  if (R == 0.f) return 0u;
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = bounded ? div_rn(x[i], S, R) : __fmul_rn(x[i], R);
  return cvt_e2m1x8(q);
}

// Reciprocal-form block scale from the block's amax and k = scale_factor(gs):
// returns sb and sets R = 1 / S, or R = 0 when S is 0.
__device__ __forceinline__ uint32_t block_scale(float amax, float k, float gs, float& R) {
  const uint32_t sb = cvt_e4m3(__fmul_rn(amax, k));
  const float S = __fmul_rn(e4m3_to_f32(sb), gs);
  R = (S > 0.f) ? __frcp_rn(S) : 0.f;
  return sb;
}

// Eight reciprocal-form codes of x * R (element i in nibble i); all zero
// when R == 0.
__device__ __forceinline__ uint32_t encode8(const float* x, float R) {
  if (R == 0.f) return 0u;
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(x[i], R);
  return cvt_e2m1x8(q);
}

__device__ __forceinline__ float amax8(const float* x) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
  return a;
}

// Byte offset of scale (m, k) in the 128x4-swizzled scale-factor buffer of a
// [M, K] scale matrix: 512-byte tiles of 128 rows x 4 columns, ordered
// row-major over (m/128, k/4), with (m%32)*16 + ((m%128)/32)*4 + k%4 inside.
// Source: "feat: MLA prefill NVFP4 fused output - #8", PR description (the
// 128x4-swizzled block-scale layout consumed by NVFP4 GEMMs).
__device__ __forceinline__ int64_t sf_offset(int64_t m, int64_t k, int64_t k_tiles) {
  return ((m >> 7) * k_tiles + (k >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (k & 3);
}

__device__ __forceinline__ void flag_error(uint32_t* error_word, uint32_t bits) {
  if (error_word != nullptr) atomicOr(error_word, bits);
}

// bf16x2 (packed in a u32) -> two floats
__device__ __forceinline__ void bf16x2_to_f32(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xFFFF0000u);
}

}  // namespace mla
