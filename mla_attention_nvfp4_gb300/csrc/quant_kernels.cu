// Elementwise NVFP4 kernels: latent cache write, the quantise-rows hook and
// the global-scale reduction.  All three are HBM-bound: no tensor cores,
// 16-byte vector loads, one pass over the input.
#include <cuda_runtime.h>

#include <atomic>

#include "launch.h"
#include "nvfp4.cuh"

namespace mla {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void unpack8_bf16(const uint4& v, float* f) {
  bf16x2_to_f32(v.x, f[0], f[1]);
  bf16x2_to_f32(v.y, f[2], f[3]);
  bf16x2_to_f32(v.z, f[4], f[5]);
  bf16x2_to_f32(v.w, f[6], f[7]);
}

// ---------------------------------------------------------------------------
// Cache write.  One warp per token.  Lane l loads latent elements [8l, 8l+8)
// and [256+8l, 256+8l+8) with two fully coalesced 512-byte warp loads; the
// block of 16 is shared by lanes 2j and 2j+1, whose amax is combined with one
// shuffle.  Record stores: 2 x 128 B of codes, 32 B of scales, the RoPE part
// and the 16-byte zero pad.
// Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
// TRITON_MLA) - #2244", second commit message (quantise at cache-write
// time); "nvfp4 MLA KV cache + per-layer outer-scale + fp8-RoPE KV-cell
// (sm120) - #33", review of api.py (432 / 368-byte records).
// ---------------------------------------------------------------------------
template <bool kFp8Rope>
__global__ void __launch_bounds__(256) cache_write_kernel(
    const __nv_bfloat16* __restrict__ kv_c, int64_t kv_stride, const __nv_bfloat16* __restrict__ k_pe,
    int64_t pe_stride, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
    uint8_t* __restrict__ cache, int64_t num_slots, const float* __restrict__ gs_ptr,
    uint32_t* error_word) {
  constexpr int kRecord = kFp8Rope ? 368 : 432;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float gs = *gs_ptr;
  const bool gs_valid = scale_ok(gs);
  const float inv_gs = inv_scale(gs);
  if (!gs_valid && warp == 0 && lane == 0) flag_error(error_word, MLA_DEVERR_SCALE);

  // Quantise one token's record from its loaded row, latent and rope parts.
  auto emit = [&](int64_t t, int64_t slot, const uint4& va, const uint4& vb, const uint4& vr) {
    if (slot < 0) return;
    if (slot >= num_slots) {
      if (lane == 0) flag_error(error_word, MLA_DEVERR_BOUNDS);
      return;
    }
    float xa[8], xb[8];
    unpack8_bf16(va, xa);
    unpack8_bf16(vb, xb);
    float am_a = amax8(xa), am_b = amax8(xb);
    am_a = fmaxf(am_a, __shfl_xor_sync(0xffffffffu, am_a, 1));
    am_b = fmaxf(am_b, __shfl_xor_sync(0xffffffffu, am_b, 1));
    uint32_t code_a = 0, code_b = 0, sb_a = 0, sb_b = 0;
    if (gs_valid) {
      float Ra, Rb, Sa, Sb;
      bool ba, bb;
      sb_a = block_scale_rn(am_a, inv_gs, gs, Ra, Sa, ba);
      sb_b = block_scale_rn(am_b, inv_gs, gs, Rb, Sb, bb);
      code_a = encode8_rn(xa, Ra, Sa, ba);
      code_b = encode8_rn(xb, Rb, Sb, bb);
    }
    uint8_t* rec = cache + slot * kRecord;
    reinterpret_cast<uint32_t*>(rec)[lane] = code_a;        // bytes [4l, 4l+4)
    reinterpret_cast<uint32_t*>(rec + 128)[lane] = code_b;  // bytes [128+4l, ...)
    if ((lane & 1) == 0) {
      rec[256 + (lane >> 1)] = static_cast<uint8_t>(sb_a);
      rec[256 + 16 + (lane >> 1)] = static_cast<uint8_t>(sb_b);
    }
    if (lane < 8) {
      if constexpr (kFp8Rope) {
        float r[8];
        unpack8_bf16(vr, r);
        const uint32_t w0 = cvt_e4m3x2(r[0], r[1]) | (cvt_e4m3x2(r[2], r[3]) << 16);
        const uint32_t w1 = cvt_e4m3x2(r[4], r[5]) | (cvt_e4m3x2(r[6], r[7]) << 16);
        reinterpret_cast<uint2*>(rec + 288)[lane] = make_uint2(w0, w1);
      } else {
        reinterpret_cast<uint4*>(rec + 288)[lane] = vr;
      }
    } else if (lane == 8) {
      *reinterpret_cast<uint4*>(rec + kRecord - 16) = make_uint4(0, 0, 0, 0);
    }
  };
  // Two tokens per iteration, both tokens' loads issued before either is
  // quantised: twice the bytes in flight per warp.
  for (int64_t t0 = warp; t0 < num_tokens; t0 += 2 * n_warps) {
    const int64_t t1 = t0 + n_warps;
    const bool has1 = t1 < num_tokens;
    const int64_t slot0 = slot_mapping[t0];
    const int64_t slot1 = has1 ? slot_mapping[t1] : -1;
    const __nv_bfloat16* row0 = kv_c + t0 * kv_stride;
    const uint4 va0 = ldg_stream(row0 + 8 * lane);
    const uint4 vb0 = ldg_stream(row0 + 256 + 8 * lane);
    uint4 vr0 = make_uint4(0, 0, 0, 0), va1 = vr0, vb1 = vr0, vr1 = vr0;
    if (lane < 8) vr0 = ldg_stream(k_pe + t0 * pe_stride + 8 * lane);
    if (has1) {
      const __nv_bfloat16* row1 = kv_c + t1 * kv_stride;
      va1 = ldg_stream(row1 + 8 * lane);
      vb1 = ldg_stream(row1 + 256 + 8 * lane);
      if (lane < 8) vr1 = ldg_stream(k_pe + t1 * pe_stride + 8 * lane);
    }
    emit(t0, slot0, va0, vb0, vr0);
    if (has1) emit(t1, slot1, va1, vb1, vr1);
  }
}

int launch_cache_write(const void* kv_c, int64_t kv_stride, const void* k_pe, int64_t pe_stride,
                       const int64_t* slot_mapping, int64_t num_tokens, uint8_t* cache,
                       int64_t num_slots, int record_bytes, const float* gs,
                       uint32_t* error_word, cudaStream_t stream, int num_sms) {
  if (num_tokens == 0) return MLA_OK;
  // One wave: as many blocks as fit on the SMs at once, each warp looping
  // over its tokens (a grid of many short-lived blocks measured ~10 % slower
  // on the 262,144-token write).
  const bool fp8 = record_bytes == 368;
  const void* kernel = fp8 ? reinterpret_cast<const void*>(cache_write_kernel<true>)
                           : reinterpret_cast<const void*>(cache_write_kernel<false>);
  static std::atomic<int> resident[2];  // blocks per SM, by record width
  int per_sm = resident[fp8].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (const int st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0)))
      return st;
    if (per_sm < 1) per_sm = 1;
    resident[fp8].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t want = (num_tokens + 7) / 8;  // 8 warps per block, one token each
  const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
  const int grid = static_cast<int>(want < cap ? want : cap);
  auto kv = static_cast<const __nv_bfloat16*>(kv_c);
  auto pe = static_cast<const __nv_bfloat16*>(k_pe);
  if (fp8)
    cache_write_kernel<true><<<grid, 256, 0, stream>>>(kv, kv_stride, pe, pe_stride, slot_mapping,
                                                       num_tokens, cache, num_slots, gs, error_word);
  else
    cache_write_kernel<false><<<grid, 256, 0, stream>>>(kv, kv_stride, pe, pe_stride, slot_mapping,
                                                        num_tokens, cache, num_slots, gs, error_word);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Gather of a cached context chunk: the records of the given slots read back
// as bf16 latent (x_hat = e2m1 * e4m3 * gs, rounded once to bf16) and k_pe.
// One warp per token; lane l dequantises latent block l (16 features, its 8
// code bytes and scale byte) and writes 32 bytes, the warp a 1 KB row.
// Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA ..." -
// #2244, second commit message (cached-context prefill chunks gather from
// the quantised paged cache).
// ---------------------------------------------------------------------------

// bf16 nearest (ties to even) to the exact product a * b (a with at most 8
// significant bits, b any float32): hi = a * b rounded to float32, lo its
// exact error (one fma); only when hi sits exactly halfway between two bf16
// values does lo decide the direction.
__device__ __forceinline__ uint32_t bf16_of_product(float a, float b) {
  const float hi = __fmul_rn(a, b);
  const float lo = __fmaf_rn(a, b, -hi);
  const uint32_t u = __float_as_uint(hi);
  if ((u & 0xFFFFu) == 0x8000u && lo != 0.f) return ((lo > 0.f) == (hi > 0.f)) ? (u >> 16) + 1u : (u >> 16);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

template <bool kFp8Rope>
__global__ void __launch_bounds__(256) gather_latent_kernel(const uint8_t* __restrict__ cache, int64_t num_slots,
                                                            const float* __restrict__ gs_ptr,
                                                            const int64_t* __restrict__ slots, int64_t n,
                                                            __nv_bfloat16* __restrict__ kv_c,
                                                            __nv_bfloat16* __restrict__ k_pe, uint32_t* error_word) {
  constexpr int kRecord = kFp8Rope ? 368 : 432;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float gs = *gs_ptr;
  if (!scale_ok(gs) && warp == 0 && lane == 0) flag_error(error_word, MLA_DEVERR_SCALE);
  for (int64_t t = warp; t < n; t += n_warps) {
    const int64_t slot = slots[t];
    const bool ok = slot >= 0 && slot < num_slots;
    if (slot >= num_slots && lane == 0) flag_error(error_word, MLA_DEVERR_BOUNDS);
    uint4 out0 = make_uint4(0, 0, 0, 0), out1 = out0, rope = out0;
    if (ok) {
      const uint8_t* rec = cache + slot * kRecord;
      const uint2 codes = *reinterpret_cast<const uint2*>(rec + 8 * lane);
      const float s = e4m3_to_f32(rec[256 + lane]);
      uint32_t w[8];
      const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // features 2i, 2i+1 of the block: one code byte
        const uint32_t byte = (cw[i >> 2] >> (8 * (i & 3))) & 0xFFu;
        uint32_t h2;
        asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h2) : "r"(byte));
        const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
        const float c0 = __low2float(hv) * s, c1 = __high2float(hv) * s;  // exact: <= 7 significant bits
        w[i] = bf16_of_product(c0, gs) | (bf16_of_product(c1, gs) << 16);
      }
      out0 = make_uint4(w[0], w[1], w[2], w[3]);
      out1 = make_uint4(w[4], w[5], w[6], w[7]);
      if (lane < 8) {
        if constexpr (kFp8Rope) {  // 8 e4m3 values -> bf16 (exact)
          const uint2 e = *reinterpret_cast<const uint2*>(rec + 288 + 8 * lane);
          const uint32_t ew[2] = {e.x, e.y};
          uint32_t r[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t two = (ew[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
            const uint32_t hf = e4m3x2_to_f16x2_pair(two);
            const __half2 hv = *reinterpret_cast<const __half2*>(&hf);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__low2float(hv), __high2float(hv));
            r[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          rope = make_uint4(r[0], r[1], r[2], r[3]);
        } else {
          rope = *reinterpret_cast<const uint4*>(rec + 288 + 16 * lane);
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(kv_c + t * 512 + 16 * lane);
    dst[0] = out0;
    dst[1] = out1;
    if (lane < 8) reinterpret_cast<uint4*>(k_pe + t * 64)[lane] = rope;
  }
}

int launch_gather_latent(const uint8_t* cache, int64_t num_slots, int record_bytes, const float* gs,
                         const int64_t* slots, int64_t n, void* kv_c, void* k_pe, uint32_t* error_word,
                         cudaStream_t stream, int num_sms) {
  if (n == 0) return MLA_OK;
  const int64_t want = (n + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  auto kv = static_cast<__nv_bfloat16*>(kv_c);
  auto pe = static_cast<__nv_bfloat16*>(k_pe);
  if (record_bytes == 368)
    gather_latent_kernel<true><<<grid, 256, 0, stream>>>(cache, num_slots, gs, slots, n, kv, pe, error_word);
  else
    gather_latent_kernel<false><<<grid, 256, 0, stream>>>(cache, num_slots, gs, slots, n, kv, pe, error_word);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Merge of partial prefill results (e.g. a context chunk's and the new
// tokens' causal attention) by their natural-log LSE, written as the fused
// NVFP4 output: O = sum_i exp(lse_i - LSE) O_i (each O_i normalised), then
// the prefill epilogue's quantiser, codes at [t, h*64 + d/2] and the scales
// 128x4-swizzled; LSE = ln sum_i exp(lse_i).  Thread = one block of 16
// features of one (token, head); padding rows of the scale buffer get zeros.
// Source: "#2244", first commit message (natural-log LSE for chunked-context
// merging); "feat: MLA prefill NVFP4 fused output - #8" (the fused output).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) merge_fused_out_kernel(const float* __restrict__ o_parts,
                                                              const float* __restrict__ lse_parts, int parts,
                                                              int64_t T, int H, const float* __restrict__ gs_ptr,
                                                              uint8_t* __restrict__ codes,
                                                              uint8_t* __restrict__ scales, float* __restrict__ lse,
                                                              uint32_t* error_word) {
  const int64_t K = static_cast<int64_t>(H) * 8;  // scale columns
  const int64_t Kp = (K + 3) & ~int64_t(3);
  const int64_t Tp = (T + 127) & ~int64_t(127);
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= Tp * Kp) return;
  const int64_t t = idx / Kp, kc = idx % Kp;
  const float gs = *gs_ptr;
  const bool gs_valid = scale_ok(gs);
  if (!gs_valid && idx == 0) flag_error(error_word, MLA_DEVERR_SCALE);
  uint32_t sb = 0;
  if (t < T && kc < K) {
    const int h = static_cast<int>(kc >> 3), blk = static_cast<int>(kc & 7);
    float m = -INFINITY;
    for (int i = 0; i < parts; ++i) m = fmaxf(m, lse_parts[(static_cast<int64_t>(i) * H + h) * T + t]);
    float v[16], tot = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = 0.f;
    if (m != -INFINITY) {
      for (int i = 0; i < parts; ++i) {
        const float l = lse_parts[(static_cast<int64_t>(i) * H + h) * T + t];
        if (l == -INFINITY) continue;
        const float wgt = expf(l - m);
        tot += wgt;
        const float4* src = reinterpret_cast<const float4*>(o_parts + ((static_cast<int64_t>(i) * T + t) * H + h) * 128 + 16 * blk);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = src[q];
          v[4 * q] = fmaf(wgt, f.x, v[4 * q]);
          v[4 * q + 1] = fmaf(wgt, f.y, v[4 * q + 1]);
          v[4 * q + 2] = fmaf(wgt, f.z, v[4 * q + 2]);
          v[4 * q + 3] = fmaf(wgt, f.w, v[4 * q + 3]);
        }
      }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= inv;
    uint32_t lo = 0, hi = 0;
    if (gs_valid) {
      float R;
      sb = block_scale(fmaxf(amax8(v), amax8(v + 8)), scale_factor(gs), gs, R);
      lo = encode8(v, R);
      hi = encode8(v + 8, R);
    }
    *reinterpret_cast<uint2*>(codes + t * (K * 8) + kc * 8) = make_uint2(lo, hi);
    if (lse != nullptr && blk == 0) lse[static_cast<int64_t>(h) * T + t] = tot > 0.f ? m + logf(tot) : -INFINITY;
  }
  scales[sf_offset(t, kc, Kp / 4)] = static_cast<uint8_t>(sb);
}

int launch_merge_fused_out(const float* o_parts, const float* lse_parts, int parts, int64_t T, int H,
                           const float* gs, uint8_t* codes, uint8_t* scales, float* lse, uint32_t* error_word,
                           cudaStream_t stream) {
  const int64_t Kp = (static_cast<int64_t>(H) * 8 + 3) / 4 * 4;
  const int64_t n = (T + 127) / 128 * 128 * Kp;
  if (n == 0) return MLA_OK;
  const int64_t grid = (n + 255) / 256;
  if (grid > 0x7FFFFFFF) return MLA_ERR_INVALID_ARG;
  merge_fused_out_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(o_parts, lse_parts, parts, T, H, gs, codes,
                                                                          scales, lse, error_word);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Quantise rows (fp32 [M, N] -> packed codes + swizzled scales).  One thread
// per scale slot of the padded [Mp, Kp] scale matrix: real slots quantise a
// block of 16, padding slots write a zero scale byte.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quantize_rows_kernel(const float* __restrict__ x, int64_t M,
                                                            int64_t N, const float* __restrict__ gs_ptr,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales,
                                                            uint32_t* error_word) {
  const int64_t K = N / 16;
  const int64_t Kp = (K + 3) & ~int64_t(3);
  const int64_t Mp = (M + 127) & ~int64_t(127);
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= Mp * Kp) return;
  const int64_t m = idx / Kp, k = idx % Kp;
  const float gs = *gs_ptr;
  const bool gs_valid = scale_ok(gs);
  const float kf = scale_factor(gs);
  if (!gs_valid && idx == 0) flag_error(error_word, MLA_DEVERR_SCALE);
  uint32_t sb = 0;
  if (m < M && k < K) {
    const float4* src = reinterpret_cast<const float4*>(x + m * N + k * 16);
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = src[i];
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
    uint32_t lo = 0, hi = 0;
    if (gs_valid) {
      float R;
      sb = block_scale(fmaxf(amax8(v), amax8(v + 8)), kf, gs, R);
      lo = encode8(v, R);
      hi = encode8(v + 8, R);
    }
    *reinterpret_cast<uint2*>(codes + m * (N / 2) + k * 8) = make_uint2(lo, hi);
  }
  scales[sf_offset(m, k, Kp / 4)] = static_cast<uint8_t>(sb);
}

// ---------------------------------------------------------------------------
// Fake quantisation of the prefill operands: each operand quantised once to
// NVFP4 along the axis its product contracts and written back as the exact
// f16 value code * e4m3 scale (the global scale left out, applied by the
// attention to the fp32 results).  Q and K: blocks of 16 of the 192
// features of a (token, head) row; V: blocks of 16 tokens of a (head,
// feature) column counted from the sequence's first token, the last block
// of a sequence ragged.  Correctly rounded quotients (the cache write's
// quantiser).  code * scale has at most 6 significant bits and lies in
// [2^-10, 2688], so it is exact in f16.
// Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
// TRITON_MLA) - #2244", first commit message (fused Q/K/P/V fake quant in
// the prefill) and PR description ("Contract notes": NVFP4 1x16 along the
// contraction axis, e4m3 block scale, amax/(6*448)).
// ---------------------------------------------------------------------------
// 16 values -> 8 f16x2 words of code * scale (element 2i low in word i).
__device__ __forceinline__ void qdq16_f16(const float* x, bool gs_valid, float inv_gs, float gs, uint32_t* w) {
  uint32_t c0 = 0, c1 = 0, sb = 0;
  if (gs_valid) {
    float R, S;
    bool bounded;
    sb = block_scale_rn(fmaxf(amax8(x), amax8(x + 8)), inv_gs, gs, R, S, bounded);
    c0 = encode8_rn(x, R, S, bounded);
    c1 = encode8_rn(x + 8, R, S, bounded);
  }
  const uint32_t s2 = e4m3x2_to_f16x2_pair(sb | (sb << 8));
  const __half2 sh = *reinterpret_cast<const __half2*>(&s2);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = ((i < 4 ? c0 : c1) >> (8 * (i & 3))) & 0xFFu;
    uint32_t h2;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h2) : "r"(byte));
    const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), sh);
    w[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// Q and K (blockIdx.y selects): thread = one block of 16 features.
__global__ void __launch_bounds__(256) qdq_features_kernel(const __nv_bfloat16* __restrict__ q, int64_t q_st,
                                                           int64_t q_sh, const __nv_bfloat16* __restrict__ k,
                                                           int64_t k_st, int64_t k_sh, int64_t T, int H,
                                                           const float* __restrict__ gs_q,
                                                           const float* __restrict__ gs_k, __half* __restrict__ q_out,
                                                           __half* __restrict__ k_out, uint32_t* error_word) {
  const bool is_k = blockIdx.y != 0;
  const __nv_bfloat16* x = is_k ? k : q;
  const int64_t st = is_k ? k_st : q_st, sh = is_k ? k_sh : q_sh;
  __half* out = is_k ? k_out : q_out;
  const float gs = is_k ? *gs_k : *gs_q;
  const bool gs_valid = scale_ok(gs);
  const float inv_gs = inv_scale(gs);
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (!gs_valid && idx == 0) flag_error(error_word, MLA_DEVERR_SCALE);
  if (idx >= T * H * 12) return;
  const int64_t row = idx / 12, b = idx % 12;
  const int64_t t = row / H, h = row % H;
  const uint4* src = reinterpret_cast<const uint4*>(x + t * st + h * sh + 16 * b);
  float f[16];
  unpack8_bf16(src[0], f);
  unpack8_bf16(src[1], f + 8);
  uint32_t w[8];
  qdq16_f16(f, gs_valid, inv_gs, gs, w);
  uint4* dst = reinterpret_cast<uint4*>(out + row * 192 + 16 * b);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// V: CTA = (block of 16 tokens, sequence); thread = two features of one head
// over the block's tokens.
__global__ void __launch_bounds__(256) qdq_tokens_kernel(const __nv_bfloat16* __restrict__ v, int64_t v_st,
                                                         int64_t v_sh, const int32_t* __restrict__ cu, int64_t T,
                                                         int H, const float* __restrict__ gs_v,
                                                         __half* __restrict__ v_out, uint32_t* error_word) {
  const int seq = blockIdx.y;
  const int a = cu[seq], e = cu[seq + 1];
  const float gs = *gs_v;
  const bool gs_valid = scale_ok(gs);
  const float inv_gs = inv_scale(gs);
  if (!gs_valid && blockIdx.x == 0 && seq == 0 && threadIdx.x == 0) flag_error(error_word, MLA_DEVERR_SCALE);
  if (a < 0 || e > T || a > e) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(error_word, MLA_DEVERR_BOUNDS);
    return;
  }
  const int64_t t0 = a + 16 * static_cast<int64_t>(blockIdx.x);
  const int64_t rem = e - t0;
  const int n = rem < 16 ? static_cast<int>(rem) : 16;
  if (n <= 0) return;
  for (int pr = threadIdx.x; pr < H * 64; pr += blockDim.x) {
    const int h = pr >> 6, d = 2 * (pr & 63);
    float c0[16], c1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t u = 0;
      if (i < n) u = *reinterpret_cast<const uint32_t*>(v + (t0 + i) * v_st + h * v_sh + d);
      bf16x2_to_f32(u, c0[i], c1[i]);
    }
    uint32_t w0[8], w1[8];
    qdq16_f16(c0, gs_valid, inv_gs, gs, w0);
    qdq16_f16(c1, gs_valid, inv_gs, gs, w1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // token i: (feature d, feature d+1) from the two columns' halves i
      const uint32_t pair = __byte_perm(w0[i >> 1], w1[i >> 1], (i & 1) ? 0x7632 : 0x5410);
      if (i < n) *reinterpret_cast<uint32_t*>(v_out + ((t0 + i) * H + h) * 128 + d) = pair;
    }
  }
}

int launch_qdq_operands(const QdqArgs& a, cudaStream_t stream) {
  const int64_t blocks = a.total * a.num_heads * 12;
  if (blocks > 0) {
    const dim3 grid(static_cast<unsigned>((blocks + 255) / 256), 2);
    qdq_features_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), a.q_st, a.q_sh, static_cast<const __nv_bfloat16*>(a.k), a.k_st,
        a.k_sh, a.total, a.num_heads, a.gs_q, a.gs_k, static_cast<__half*>(a.q_out), static_cast<__half*>(a.k_out),
        a.error_word);
  }
  if (a.num_seqs > 0 && a.max_seqlen > 0) {
    const dim3 grid(static_cast<unsigned>((a.max_seqlen + 15) / 16), static_cast<unsigned>(a.num_seqs));
    qdq_tokens_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(a.v), a.v_st, a.v_sh, a.cu_seqlens,
                                                a.total, a.num_heads, a.gs_v, static_cast<__half*>(a.v_out),
                                                a.error_word);
  }
  return launch_status();
}

int launch_quantize_rows(const float* x, int64_t M, int64_t N, const float* gs, uint8_t* codes,
                         uint8_t* scales, uint32_t* error_word, cudaStream_t stream) {
  const int64_t K = N / 16;
  const int64_t total = ((M + 127) / 128 * 128) * ((K + 3) / 4 * 4);
  if (total == 0) return MLA_OK;
  const int64_t grid = (total + 255) / 256;
  if (grid > 0x7fffffff) return MLA_ERR_INVALID_ARG;
  quantize_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(x, M, N, gs, codes, scales,
                                                                         error_word);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Global scale: gs = fp32(amax|x| / 2688).  Pass 1 reduces |x| into the
// output word as an unsigned integer (non-negative floats order like their
// bit patterns); pass 2 turns the maximum into the scale in place.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t n,
                                                   uint32_t* __restrict__ out_bits) {
  float m = 0.f;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n8 = n / 8;
  for (int64_t i = tid; i < n8; i += stride) {
    float f[8];
    unpack8_bf16(ldg_stream(x + 8 * i), f);
    m = fmaxf(m, amax8(f));
  }
  for (int64_t i = n8 * 8 + tid; i < n; i += stride) m = fmaxf(m, fabsf(__bfloat162float(x[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int i = 1; i < 8; ++i) b = fmaxf(b, red[i]);
    atomicMax(out_bits, __float_as_uint(b));
  }
}

__global__ void finalize_scale_kernel(float* gs) {
  const float amax = __uint_as_float(*reinterpret_cast<uint32_t*>(gs));
  *gs = __fdiv_rn(amax, 2688.0f);
}

int launch_global_scale(const void* x, int64_t n, float* gs, cudaStream_t stream, int num_sms) {
  if (const int st = cuda_status(cudaMemsetAsync(gs, 0, sizeof(float), stream))) return st;
  const int64_t want = (n / 8 + 255) / 256 + 1;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  amax_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), n,
                                        reinterpret_cast<uint32_t*>(gs));
  finalize_scale_kernel<<<1, 1, 0, stream>>>(gs);
  return launch_status();
}

}  // namespace mla
