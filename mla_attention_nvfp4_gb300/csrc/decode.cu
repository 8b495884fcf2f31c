// Absorbed MLA decode over the NVFP4 latent cache, split along the keys,
// merged by natural-log LSE.
//
// Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
// TRITON_MLA) - #2244", first commit message (split-K absorbed decode over
// the paged latent cache with grouped query heads; natural-log LSE for
// merging) and third commit message (the write-once latent is both K and V);
// "nvfp4 MLA KV cache + per-layer outer-scale + fp8-RoPE KV-cell (sm120) -
// #33" (sparse top-k decode, bf16 Q, per-layer outer scale restored on read).
//
// scores s_j = softmax_scale * (q_lat . x_hat_j + q_pe . rope_j),
// x_hat = e2m1(code) * e4m3(scale) * gs; out = sum_j softmax(s)_j x_hat_j.
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "nvfp4.cuh"

namespace mla {
namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kTile = 32;        // keys per tile
constexpr int kThreads = 256;
constexpr int kKStride = 577;    // padded row of the fp32 key tile in smem
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  const float v = mag[c & 7u];
  return (c & 8u) ? -v : v;
}

struct DecodeParams {
  const __nv_bfloat16* q;
  int batch, num_heads;
  const uint8_t* cache;
  int64_t num_slots;
  const int32_t* page_table;
  int64_t pt_stride;
  int page_size;
  const int32_t* seq_lens;
  const int32_t* topk;
  int topk_n;
  float scale_log2;  // softmax_scale * log2(e)
  const float* gs;
  float* part_o;     // [batch, splits, heads, 512]
  float* part_lse;   // [batch, splits, heads]
  int splits;
  uint32_t* error_word;
};

// Slot of key position t of sequence b, or -1 for padding / out of range.
__device__ __forceinline__ int64_t key_slot(const DecodeParams& p, int b, int t, bool& bad) {
  int64_t slot;
  if (p.topk != nullptr) {
    slot = p.topk[static_cast<int64_t>(b) * p.topk_n + t];
  } else {
    if (t / p.page_size >= p.pt_stride) {  // sequence longer than its page-table row
      bad = true;
      return -1;
    }
    const int page = p.page_table[static_cast<int64_t>(b) * p.pt_stride + t / p.page_size];
    slot = (page < 0) ? -1 : static_cast<int64_t>(page) * p.page_size + t % p.page_size;
    if (page < 0) bad = true;
  }
  if (slot >= p.num_slots) {
    bad = true;
    slot = -1;
  }
  return slot;
}

// One CTA = (split, batch b, group of 16 heads).  The key tile is
// dequantised to fp32 in shared memory, scores and PV run on CUDA cores.
template <int kRecord>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeParams p) {
  extern __shared__ float smem[];
  float* q_s = smem;                                // [16][576]
  float* k_s = q_s + kHeadsPerCta * 576;            // [32][577]
  float* p_s = k_s + kTile * kKStride;              // [16][32]
  __shared__ int valid_s[kTile];

  const int split = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * kHeadsPerCta;
  const int tid = threadIdx.x;
  const float gs = *p.gs;
  const int n_keys = (p.topk != nullptr) ? p.topk_n : p.seq_lens[b];
  const int n_tiles = (n_keys + kTile - 1) / kTile;
  const int per = (n_tiles + p.splits - 1) / p.splits;
  const int t_begin = split * per, t_end = min(n_tiles, t_begin + per);

  // q (bf16) -> fp32 smem; heads past num_heads are zero rows
  for (int i = tid; i < kHeadsPerCta * 576; i += kThreads) {
    const int h = h0 + i / 576;
    q_s[i] = (h < p.num_heads)
                 ? __bfloat162float(p.q[(static_cast<int64_t>(b) * p.num_heads + h) * 576 + i % 576])
                 : 0.f;
  }

  const int hh = tid / 16;   // head within the group for scores and PV
  const int lane16 = tid % 16;
  float o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  for (int tile = t_begin; tile < t_end; ++tile) {
    __syncthreads();  // previous tile fully consumed
    // dequantise: 8 threads per key, thread covers 64 latent + 8 rope dims
    {
      const int j = tid / 8, part = tid % 8;
      const int t = tile * kTile + j;
      bool bad = false;
      int64_t slot = -1;
      if (t < n_keys) slot = key_slot(p, b, t, bad);
      if (bad && part == 0) flag_error(p.error_word, MLA_DEVERR_BOUNDS);
      float* dst = k_s + j * kKStride;
      if (slot >= 0) {
        const uint8_t* rec = p.cache + slot * kRecord;
        const uint4 c0 = *reinterpret_cast<const uint4*>(rec + 32 * part);
        const uint4 c1 = *reinterpret_cast<const uint4*>(rec + 32 * part + 16);
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(rec + 256 + 4 * part);
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float s = e4m3_to_f32((sc >> (8 * (w / 2))) & 0xFFu) * gs;
#pragma unroll
          for (int n = 0; n < 8; ++n) dst[64 * part + 8 * w + n] = e2m1_value(words[w] >> (4 * n)) * s;
        }
        if constexpr (kRecord == 432) {
          const uint4 r = *reinterpret_cast<const uint4*>(rec + 288 + 16 * part);
          float f[8];
          bf16x2_to_f32(r.x, f[0], f[1]);
          bf16x2_to_f32(r.y, f[2], f[3]);
          bf16x2_to_f32(r.z, f[4], f[5]);
          bf16x2_to_f32(r.w, f[6], f[7]);
#pragma unroll
          for (int n = 0; n < 8; ++n) dst[512 + 8 * part + n] = f[n];
        } else {
          const uint2 r = *reinterpret_cast<const uint2*>(rec + 288 + 8 * part);
#pragma unroll
          for (int n = 0; n < 8; ++n)
            dst[512 + 8 * part + n] = e4m3_to_f32(((n < 4 ? r.x : r.y) >> (8 * (n % 4))) & 0xFFu);
        }
      } else {
        for (int n = 0; n < 64; ++n) dst[64 * part + n] = 0.f;
        for (int n = 0; n < 8; ++n) dst[512 + 8 * part + n] = 0.f;
      }
      if (part == 0) valid_s[j] = slot >= 0;
    }
    __syncthreads();

    // scores: thread (head hh, keys lane16 and lane16+16)
    float s0 = 0.f, s1 = 0.f;
    {
      const float* qh = q_s + hh * 576;
      const float* k0 = k_s + lane16 * kKStride;
      const float* k1 = k_s + (lane16 + 16) * kKStride;
#pragma unroll 8
      for (int d = 0; d < 576; ++d) {
        const float qd = qh[d];
        s0 = fmaf(qd, k0[d], s0);
        s1 = fmaf(qd, k1[d], s1);
      }
    }
    s0 = valid_s[lane16] ? s0 * p.scale_log2 : -INFINITY;
    s1 = valid_s[lane16 + 16] ? s1 * p.scale_log2 : -INFINITY;
    float mt = fmaxf(s0, s1);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    const float m_new = fmaxf(m_run, mt);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float p0 = exp2f(s0 - m_use), p1 = exp2f(s1 - m_use);
    float ls = p0 + p1;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    const float alpha = exp2f(m_run - m_use);
    l_run = l_run * alpha + ls;
    m_run = m_new;
    p_s[hh * kTile + lane16] = p0;
    p_s[hh * kTile + lane16 + 16] = p1;
    __syncthreads();

    // PV: thread (head hh) owns features lane16 + 16 i
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= alpha;
    for (int j = 0; j < kTile; ++j) {
      const float pj = p_s[hh * kTile + j];
      const float* v = k_s + j * kKStride + lane16;
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = fmaf(pj, v[16 * i], o[i]);
    }
  }

  const int h = h0 + hh;
  if (h < p.num_heads) {
    const int64_t row = (static_cast<int64_t>(b) * p.splits + split) * p.num_heads + h;
    const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
    float* dst = p.part_o + row * 512 + lane16;
#pragma unroll
    for (int i = 0; i < 32; ++i) dst[16 * i] = o[i] * inv;
    if (lane16 == 0)
      p.part_lse[row] = (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
  }
}

// Merge the per-split partials of one (batch, head): LSE = ln sum exp(lse_i),
// out = sum exp(lse_i - LSE) o_i.
__global__ void __launch_bounds__(128) decode_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse,
                                                           int splits, int num_heads,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int b = blockIdx.x / num_heads, h = blockIdx.x % num_heads;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s)
    m = fmaxf(m, part_lse[(static_cast<int64_t>(b) * splits + s) * num_heads + h]);
  float tot = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (m != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const int64_t row = (static_cast<int64_t>(b) * splits + s) * num_heads + h;
      const float l = part_lse[row];
      if (l == -INFINITY) continue;
      const float w = expf(l - m);
      tot += w;
      const float4 v = reinterpret_cast<const float4*>(part_o + row * 512)[threadIdx.x];
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  __nv_bfloat16* o = out + (static_cast<int64_t>(b) * num_heads + h) * 512 + 4 * threadIdx.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = __float2bfloat16_rn(acc[i] * inv);
  if (lse != nullptr && threadIdx.x == 0)
    lse[static_cast<int64_t>(b) * num_heads + h] = (tot > 0.f) ? m + logf(tot) : -INFINITY;
}

}  // namespace

size_t decode_workspace_bytes(int batch, int num_heads, int num_splits) {
  const size_t rows = static_cast<size_t>(batch) * num_splits * num_heads;
  const size_t o_bytes = rows * 512 * sizeof(float);
  const size_t l_bytes = (rows * sizeof(float) + 255) / 256 * 256;
  return o_bytes + l_bytes;
}

int decode_default_splits(int batch, int num_heads, int num_sms) {
  const int groups = (num_heads + kHeadsPerCta - 1) / kHeadsPerCta;
  const int ctas = batch * groups;
  int s = (2 * num_sms + ctas - 1) / ctas;
  return s < 1 ? 1 : (s > 64 ? 64 : s);
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream, int /*num_sms*/) {
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.batch = a.batch;
  p.num_heads = a.num_heads;
  p.cache = a.cache;
  p.num_slots = a.num_slots;
  p.page_table = a.page_table;
  p.pt_stride = a.page_table_stride;
  p.page_size = a.page_size;
  p.seq_lens = a.seq_lens;
  p.topk = a.topk_indices;
  p.topk_n = a.topk;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.gs = a.gs;
  p.splits = a.num_splits;
  p.error_word = a.error_word;
  const size_t rows = static_cast<size_t>(a.batch) * a.num_splits * a.num_heads;
  p.part_o = static_cast<float*>(a.workspace);
  p.part_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + rows * 512 * sizeof(float));

  const size_t smem = (kHeadsPerCta * 576 + kTile * kKStride + kHeadsPerCta * kTile) * sizeof(float);
  dim3 grid(a.num_splits, a.batch, (a.num_heads + kHeadsPerCta - 1) / kHeadsPerCta);
  if (a.record_bytes == 432) {
    if (cudaFuncSetAttribute(decode_split_kernel<432>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MLA_ERR_LAUNCH;
    decode_split_kernel<432><<<grid, kThreads, smem, stream>>>(p);
  } else {
    if (cudaFuncSetAttribute(decode_split_kernel<368>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MLA_ERR_LAUNCH;
    decode_split_kernel<368><<<grid, kThreads, smem, stream>>>(p);
  }
  if (cudaGetLastError() != cudaSuccess) return MLA_ERR_LAUNCH;
  decode_merge_kernel<<<a.batch * a.num_heads, 128, 0, stream>>>(
      p.part_o, p.part_lse, a.num_splits, a.num_heads, static_cast<__nv_bfloat16*>(a.out), a.lse);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH;
}

}  // namespace mla
