// Causal varlen MLA prefill (q/k dim 192, v dim 128) whose epilogue writes
// NVFP4: packed e2m1 codes plus e4m3 block scales in the 128x4-swizzled
// layout, so no standalone quantisation pass runs.
//
// Source: "feat: MLA prefill NVFP4 fused output - #8" (PR description and
// the review of the float4_e2m1fn_x2 output view); "Add NVFP4/FP8 Q/K/P/V +
// 2:4 attention quantization for MLA (vLLM TRITON_MLA) - #2244", first
// commit message (varlen prefill, asymmetric 192/128 head dims, natural-log
// LSE).
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "nvfp4.cuh"

namespace mla {
namespace {

constexpr int kDqk = 192, kDv = 128;
constexpr int kBM = 64, kBN = 64, kThreads = 256;
constexpr int kQS = kDqk + 1, kVS = kDv + 1, kPS = kBN + 1;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct PrefillParams {
  const __nv_bfloat16 *q, *k, *v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const int32_t* cu;
  int64_t total;
  int num_heads;
  float scale_log2;
  const float* gs;
  uint8_t* codes;
  uint8_t* scales;
  float* lse;
  uint32_t* error_word;
};

// One CTA = (64-row query tile, head, sequence).  fp32 tiles in shared
// memory, CUDA-core products, NVFP4 epilogue.
__global__ void __launch_bounds__(kThreads) prefill_kernel(PrefillParams p) {
  extern __shared__ float smem[];
  float* q_s = smem;                 // [64][193], reused for O in the epilogue
  float* k_s = q_s + kBM * kQS;      // [64][193]
  float* v_s = k_s + kBN * kQS;      // [64][129]
  float* p_s = v_s + kBN * kVS;      // [64][65]
  __shared__ float alpha_s[kBM];
  __shared__ float l_s[kBM], m_s[kBM];

  const int tile = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int tid = threadIdx.x;
  const int64_t K_cols = static_cast<int64_t>(p.num_heads) * 8;
  const int64_t k_tiles = (K_cols + 3) / 4;

  // padding rows [total, roundup(total,128)) of this head's 8 scale columns
  if (tile == 0 && seq == 0) {
    const int64_t Mp = (p.total + 127) / 128 * 128;
    for (int64_t i = tid; i < (Mp - p.total) * 8; i += kThreads)
      p.scales[sf_offset(p.total + i / 8, static_cast<int64_t>(h) * 8 + i % 8, k_tiles)] = 0;
  }

  const int seq_begin = p.cu[seq], seq_end = p.cu[seq + 1];
  const int n = seq_end - seq_begin;
  const int row0 = tile * kBM;
  if (n <= 0 || row0 >= n || seq_begin < 0 || seq_end > p.total) {
    if ((seq_begin < 0 || seq_end > p.total || n < 0) && tid == 0 && tile == 0 && h == 0)
      flag_error(p.error_word, MLA_DEVERR_BOUNDS);
    return;
  }
  const float gs = *p.gs;
  const bool gs_valid = scale_ok(gs);
  if (!gs_valid && tid == 0 && tile == 0 && h == 0 && seq == 0) flag_error(p.error_word, MLA_DEVERR_SCALE);
  const int rows = min(kBM, n - row0);

  for (int i = tid; i < kBM * kDqk; i += kThreads) {
    const int r = i / kDqk, d = i % kDqk;
    q_s[r * kQS + d] = (r < rows) ? __bfloat162float(p.q[(seq_begin + row0 + r) * p.q_st + h * p.q_sh + d]) : 0.f;
  }
  if (tid < kBM) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }

  const int rg = tid / 16, kg = tid % 16;  // scores: rows 4rg..4rg+3, keys kg + 16i
  const int pr = tid / 4, pf = tid % 4;    // PV: row pr, features pf + 4i
  float o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = 0.f;

  const int last_key = row0 + rows - 1;
  const int n_kv = last_key / kBN + 1;
  for (int kt = 0; kt < n_kv; ++kt) {
    const int key0 = kt * kBN;
    __syncthreads();
    for (int i = tid; i < kBN * kDqk; i += kThreads) {
      const int j = i / kDqk, d = i % kDqk;
      k_s[j * kQS + d] = (key0 + j < n) ? __bfloat162float(p.k[(seq_begin + key0 + j) * p.k_st + h * p.k_sh + d]) : 0.f;
    }
    for (int i = tid; i < kBN * kDv; i += kThreads) {
      const int j = i / kDv, d = i % kDv;
      v_s[j * kVS + d] = (key0 + j < n) ? __bfloat162float(p.v[(seq_begin + key0 + j) * p.v_st + h * p.v_sh + d]) : 0.f;
    }
    __syncthreads();

    float s[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[a][c] = 0.f;
    for (int d = 0; d < kDqk; ++d) {
      float qv[4], kv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qv[a] = q_s[(4 * rg + a) * kQS + d];
#pragma unroll
      for (int c = 0; c < 4; ++c) kv[c] = k_s[(kg + 16 * c) * kQS + d];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[a][c] = fmaf(qv[a], kv[c], s[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * rg + a;
      const int qi = row0 + r;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kj = key0 + kg + 16 * c;
        s[a][c] = (kj <= qi && r < rows) ? s[a][c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[a][c]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = m_s[r];
      const float m_new = fmaxf(m_old, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float pv = exp2f(s[a][c] - m_use);
        p_s[r * kPS + kg + 16 * c] = pv;
        ls += pv;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      __syncwarp();
      if (kg == 0) {
        const float alpha = exp2f(m_old - m_use);
        alpha_s[r] = alpha;
        l_s[r] = l_s[r] * alpha + ls;
        m_s[r] = m_new;
      }
    }
    __syncthreads();
    const float alpha = alpha_s[pr];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= alpha;
    for (int j = 0; j < kBN; ++j) {
      const float pj = p_s[pr * kPS + j];
      const float* vr = v_s + j * kVS + pf;
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = fmaf(pj, vr[4 * i], o[i]);
    }
  }

  // epilogue: normalise, stage O in smem, quantise blocks of 16 per row
  __syncthreads();
  float* o_s = q_s;  // [64][129]
  {
    const float l = l_s[pr];
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) o_s[pr * kVS + pf + 4 * i] = o[i] * inv;
  }
  __syncthreads();
  {
    const int r = tid / 4, part = tid % 4;  // features [32 part, 32 part + 32)
    if (r < rows) {
      const int64_t m = seq_begin + row0 + r;
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = o_s[r * kVS + 32 * part + i];
      uint32_t w[4] = {0, 0, 0, 0}, sb0 = 0, sb1 = 0;
      if (gs_valid) {
        float S0, S1;
        sb0 = block_scale(fmaxf(amax8(x), amax8(x + 8)), gs, S0);
        sb1 = block_scale(fmaxf(amax8(x + 16), amax8(x + 24)), gs, S1);
        w[0] = encode8(x, S0);
        w[1] = encode8(x + 8, S0);
        w[2] = encode8(x + 16, S1);
        w[3] = encode8(x + 24, S1);
      }
      *reinterpret_cast<uint4*>(p.codes + m * (static_cast<int64_t>(p.num_heads) * 64) + h * 64 + part * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
      const int64_t kcol = static_cast<int64_t>(h) * 8 + part * 2;
      p.scales[sf_offset(m, kcol, k_tiles)] = static_cast<uint8_t>(sb0);
      p.scales[sf_offset(m, kcol + 1, k_tiles)] = static_cast<uint8_t>(sb1);
      if (p.lse != nullptr && part == 0) {
        const float l = l_s[r];
        p.lse[static_cast<int64_t>(h) * p.total + m] = l > 0.f ? (m_s[r] + log2f(l)) * kLn2 : -INFINITY;
      }
    }
  }
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream, int /*num_sms*/) {
  PrefillParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.q_st = a.q_st; p.q_sh = a.q_sh; p.k_st = a.k_st; p.k_sh = a.k_sh; p.v_st = a.v_st; p.v_sh = a.v_sh;
  p.cu = a.cu_seqlens;
  p.total = a.total_tokens;
  p.num_heads = a.num_heads;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.gs = a.gs;
  p.codes = a.out_codes;
  p.scales = a.out_scales;
  p.lse = a.lse;
  p.error_word = a.error_word;
  const size_t smem = (kBM * kQS + kBN * kQS + kBN * kVS + kBM * kPS) * sizeof(float);
  if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MLA_ERR_LAUNCH;
  dim3 grid((a.max_seqlen + kBM - 1) / kBM, a.num_heads, a.num_seqs);
  if (grid.x > 0x7fffffffu || grid.y > 65535u || grid.z > 65535u) return MLA_ERR_INVALID_ARG;
  prefill_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH;
}

}  // namespace mla
