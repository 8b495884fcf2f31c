// NVFP4 device codecs shared by the cache-write kernel, the prefill
// epilogue and the quantise-rows hook.
//
// NVFP4: e2m1 codes, one e4m3 block scale per 16 elements, fp32 global scale
// gs (dequantisation direction).  Source: "Add NVFP4/FP8 Q/K/P/V + 2:4
// attention quantization for MLA (vLLM TRITON_MLA) - #2244", PR description,
// "Contract notes" (block 1x16 along the contraction axis, E4M3 block scale,
// global amax/(6*448)).
//
// Float32 operation order of one block (every op IEEE round-to-nearest, no
// contraction; reciprocals instead of divisions, as NVFP4 quantisers
// usually do):
//     k     = 1 / (6 * gs)                       once per tensor
//     s_raw = amax16 * k
//     sb    = e4m3 RNE-satfinite(s_raw)
//     S     = e4m3(sb) * gs
//     code  = e2m1 RNE-satfinite(x * (1 / S)), all codes 0 when S is 0
// A global scale outside [2^-100, 2^100] is invalid (codes and scales 0).
// The conversions use the sm_100-family cvt instructions, which round to
// nearest even and clamp to the largest finite value (448, 6).
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

__device__ __forceinline__ bool scale_ok(float gs) {
  return gs >= 7.888609052210118e-31f && gs <= 1.2676506002282294e30f;  // [2^-100, 2^100]
}

// k = 1 / (6 * gs): the per-tensor factor of the raw block scale.
__device__ __forceinline__ float scale_factor(float gs) { return __frcp_rn(__fmul_rn(6.0f, gs)); }

// Block scale from the block's amax (amax is exact in any reduction order)
// and k = scale_factor(gs).  Returns the scale byte sb and sets R = 1 / S
// with S = e4m3(sb) * gs, or R = 0 when S is 0 (the block then encodes as
// all-zero codes).
__device__ __forceinline__ uint32_t block_scale(float amax, float k, float gs, float& R) {
  const uint32_t sb = cvt_e4m3(__fmul_rn(amax, k));
  const float S = __fmul_rn(e4m3_to_f32(sb), gs);
  R = (S > 0.f) ? __frcp_rn(S) : 0.f;
  return sb;
}

// Eight codes of x * R (element i in nibble i); all zero when R == 0.
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
