// Absorbed MLA decode over the NVFP4 latent cache on tcgen05 tensor cores,
// split along the keys and merged by natural-log LSE.
//
// Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
// TRITON_MLA) - #2244", first commit message (split-K absorbed decode over
// the paged latent cache with grouped query heads; natural-log LSE for
// merging chunks) and third commit message (the write-once latent is both
// operands: V is the latent, with K's feature-axis quantisation); "nvfp4 MLA
// KV cache + per-layer outer-scale + fp8-RoPE KV-cell (sm120) - #33" (sparse
// top-k decode, bf16 Q staged unquantised, per-layer outer scale restored on
// read).
//
//   s_j = softmax_scale * (q_lat . x_hat_j + q_pe . rope_j),
//   x_hat = e2m1(code) * e4m3(scale) * gs,   out = sum_j softmax(s)_j x_hat_j.
//
// The global scale gs is folded out of the tensor-core operands: the key
// tile holds c*s (exact in f16) and k_pe (bf16), the query tile holds
// [sigma*q_lat (f16), sigma*q_pe/gs (bf16)] with sigma a per-head power of
// two keeping sigma*q_lat inside the f16 range, the product is multiplied by
// softmax_scale*gs/sigma, and the output by gs.
//
// Work unit = (sequence b, split, group of up to 128 heads), run by a
// cluster of two CTAs.  CTA r owns latent features [256r, 256r+256) and RoPE
// features [32r, 32r+32): it stages and dequantises only its half of every
// record, keeps its half of Q in TMEM, computes a partial score tile over
// its 288 dims, and accumulates its 256-column half of O.  The partial score
// tiles (128 heads x 32 keys, fp32) are exchanged through distributed shared
// memory, so both CTAs run the same softmax on the full scores.  This keeps
// the 128 x 512 fp32 output within one SM's 512 TMEM columns per CTA and
// does no tensor-core work twice.
//
// Warp roles per CTA (320 threads):
//   warp 0      producer: slot ids, cp.async of the CTA's record halves
//               into a 4-stage raw ring (16-byte chunks).
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S_j  = Q_half . K_j^T   M=128 N=32 K=288, Q from TMEM
//                 O   += P_j . V_j        M=128 N=256 K=32, P from TMEM,
//                                         V = the latent tile read MN-major
//   warps 2..5  dequantise raw records into 128-byte-swizzled tiles: latent
//               c*s in f16 (one cvt + one multiply per pair), RoPE in bf16.
//   warps 6..9  Q staging, partial-score exchange, online softmax, O
//               correction and the partial-output epilogue; thread = head.
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "nvfp4.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTok = 32;           // keys per tile
constexpr int kHeads = 128;        // heads per work unit (MMA M)
constexpr int kThreads = 320;
constexpr int kRawStride = 224;    // bytes per key in the raw ring (208 used)
constexpr int kRawStages = 6;
constexpr int kKvStages = 3;
constexpr int kXchBufs = 4;
constexpr uint32_t kRawBytes = kTok * kRawStride;         // 7168
constexpr uint32_t kKvBlock = kTok * 128;                 // one 64-feature column block
constexpr uint32_t kKvBytes = 5 * kKvBlock;               // 4 latent blocks + RoPE block
constexpr uint32_t kXchBytes = kHeads * kTok * 4;         // 16384
constexpr uint32_t kSmKv = 0;
constexpr uint32_t kSmRaw = kSmKv + kKvStages * kKvBytes;
constexpr uint32_t kSmXch = kSmRaw + kRawStages * kRawBytes;
constexpr uint32_t kSmBytes = kSmXch + kXchBufs * kXchBytes;
constexpr uint32_t kSmAlloc = kSmBytes + 1024;
static_assert(kSmAlloc <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t kTQ = 0;                  // Q half: 288 bf16 = 144 columns
__host__ __device__ constexpr uint32_t col_s(int buf) { return 160u + 32u * buf; }  // scores, 32 cols
__host__ __device__ constexpr uint32_t col_p(int buf) { return 224u + 16u * buf; }  // P bf16 pairs, 16 cols
constexpr uint32_t kTO = 256;                // O half, 256 columns

// Latent products run on f16 operands (c*s is exact in f16; Q is scaled per
// row by a power of two so that it cannot overflow f16); the RoPE K-steps
// run as separate bf16 MMAs into the same accumulator.
constexpr uint32_t kIdescQKLat = idesc_f16_f32(128, kTok, false, false);
constexpr uint32_t kIdescQKRope = idesc_bf16_f32(128, kTok, false, false);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 256, false, true);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

struct Params {
  const __nv_bfloat16* q;
  int batch, num_heads;
  const uint8_t* cache;
  int64_t num_slots;
  int record_bytes;
  const int32_t* page_table;
  int64_t pt_stride;
  int page_size;
  const int32_t* seq_lens;
  const int32_t* topk;
  int topk_n;
  float softmax_scale;
  const float* gs;
  float* part_o;    // [batch, splits, heads, 512]
  float* part_lse;  // [batch, splits, heads]
  int splits;
  uint32_t* error_word;
};

struct alignas(8) Barriers {
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  uint64_t kv_full[kKvStages], kv_empty[kKvStages];
  uint64_t q_ready;
  uint64_t s_full[2], s_free[2];
  uint64_t xch_full[kXchBufs];
  uint64_t p_full[2], pv_done[2];
  uint64_t o_full;
};

// Key addressing in two halves so that the index load can be issued tiles
// ahead of its use: load_index() performs one unconditional, in-bounds load
// (the page-table entry or the top-k index of key position t, clamped into
// its row); key_slot() then turns that value into a slot id, or -1 for
// padding / positions past the sequence, and notes out-of-range ids.
__device__ __forceinline__ int32_t load_index(const Params& p, int b, int t) {
  if (p.topk != nullptr) {
    const int tc = min(max(t, 0), max(p.topk_n - 1, 0));
    return p.topk[static_cast<int64_t>(b) * p.topk_n + tc];
  }
  const int pi = min(max(t, 0) / p.page_size, static_cast<int>(p.pt_stride) - 1);
  return p.page_table[static_cast<int64_t>(b) * p.pt_stride + pi];
}

__device__ __forceinline__ int64_t key_slot(const Params& p, int32_t idx, int t, int n_keys, bool& bad) {
  if (t >= n_keys) return -1;
  int64_t slot;
  if (p.topk != nullptr) {
    if (idx < 0) return -1;  // padding entry
    slot = idx;
  } else {
    if (t / p.page_size >= p.pt_stride || idx < 0) {
      bad = true;
      return -1;
    }
    slot = static_cast<int64_t>(idx) * p.page_size + t % p.page_size;
  }
  if (slot >= p.num_slots) {
    bad = true;
    return -1;
  }
  return slot;
}

__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t in = static_cast<uint16_t>(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a), y = *reinterpret_cast<__half2*>(&b);
  __half2 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

// f16x2 -> bf16x2; exact for e4m3 values (4 significant bits).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  const __half2 x = *reinterpret_cast<const __half2*>(&h);
  const float2 f = __half22float2(x);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

template <int kRecord>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) decode_tc_kernel(Params p) {
  constexpr bool kFp8Rope = (kRecord == 368);
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ uint32_t raw_mask[kRawStages];  // valid keys of each raw stage

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int split = blockIdx.x >> 1, b = blockIdx.y, hg = blockIdx.z;
  const int n_keys = (p.topk != nullptr) ? p.topk_n : max(0, p.seq_lens[b]);
  const int n_tiles_all = (n_keys + kTok - 1) / kTok;
  const int per = (n_tiles_all + p.splits - 1) / p.splits;
  const int tile0 = split * per;
  const int nt = max(0, min(n_tiles_all, tile0 + per) - tile0);
  uint32_t* err = p.error_word;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = smem + kSmKv;
  uint8_t* sRaw = smem + kSmRaw;
  uint8_t* sXch = smem + kSmXch;

  if (threadIdx.x == 0) {
    abort_s = 0;
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(&bars.raw_full[i], 33);  // 32 cp.async arrivals + the mask writer
      mbar_init(&bars.raw_empty[i], 128);
    }
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&bars.kv_full[i], 128);
      mbar_init(&bars.kv_empty[i], 1);
    }
    mbar_init(&bars.q_ready, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], 128);
      mbar_init(&bars.p_full[i], 128);
      mbar_init(&bars.pv_done[i], 1);
    }
    for (int i = 0; i < kXchBufs; ++i) mbar_init(&bars.xch_full[i], 1);
    mbar_init(&bars.o_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote store
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Index loads run two tiles ahead of their use.
    bool bad = false;
    int32_t idx_a = nt > 0 ? load_index(p, b, tile0 * kTok + lane) : -1;
    int32_t idx_b = nt > 1 ? load_index(p, b, (tile0 + 1) * kTok + lane) : -1;
    for (int j = 0; j < nt; ++j) {
      const int st = j % kRawStages;
      const uint32_t ph = (j / kRawStages) & 1;
      const int32_t idx = idx_a;
      idx_a = idx_b;
      if (j + 2 < nt) idx_b = load_index(p, b, (tile0 + j + 2) * kTok + lane);
      const int64_t slot = key_slot(p, idx, (tile0 + j) * kTok + lane, n_keys, bad);
      if (!mbar_wait(&bars.raw_empty[st], ph ^ 1, err, &abort_s)) break;
      const unsigned vmask = __ballot_sync(0xffffffffu, slot >= 0);
      if (slot >= 0) {
        const uint8_t* rec = p.cache + slot * kRecord;
        uint8_t* dst = sRaw + st * kRawBytes + lane * kRawStride;
#pragma unroll
        for (int i = 0; i < 8; ++i) cp_async16(dst + 16 * i, rec + 128 * rank + 16 * i);
        cp_async16(dst + 128, rec + 256 + 16 * rank);
        if constexpr (kFp8Rope) {
#pragma unroll
          for (int i = 0; i < 2; ++i) cp_async16(dst + 144 + 16 * i, rec + 288 + 32 * rank + 16 * i);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) cp_async16(dst + 144 + 16 * i, rec + 288 + 64 * rank + 16 * i);
        }
      }
      cp_async_arrive(&bars.raw_full[st]);
      if (lane == 0) {
        raw_mask[st] = vmask;
        mbar_arrive(&bars.raw_full[st]);
      }
    }
    if (bad && rank == 0) flag_error(err, MLA_DEVERR_BOUNDS);
    cp_async_wait_all();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && nt > 0) {
      const uint32_t kv_addr = smem_u32(sKV);
      bool ok = mbar_wait(&bars.q_ready, 0, err, &abort_s);
      tc_fence_after();
      auto issue_pv = [&](int i) -> bool {
        const int pb = i & 1;
        if (!mbar_wait(&bars.p_full[pb], (i >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t vbase = kv_addr + (i % kKvStages) * kKvBytes;
#pragma unroll
        for (int kk = 0; kk < kTok / 16; ++kk) {
          const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, kKvBlock, 1024);
          mma_ts(tmem + kTO, tmem + col_p(pb) + kk * 8, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars.kv_empty[i % kKvStages]);
        mma_commit(&bars.pv_done[pb]);
        return true;
      };
      // QK runs two tiles ahead of PV: S(i+2) is computed while the softmax
      // works on tile i.
      auto issue_qk = [&](int j) -> bool {
        const int ks = j % kKvStages;
        const int sb = j & 1;
        if (!mbar_wait(&bars.kv_full[ks], (j / kKvStages) & 1, err, &abort_s)) return false;
        if (j >= 2 && !mbar_wait(&bars.s_free[sb], ((j - 2) >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t kbase = kv_addr + ks * kKvBytes;
#pragma unroll
        for (int kk = 0; kk < 18; ++kk) {
          const uint64_t bd = smem_desc_sw128(kbase + (kk >> 2) * kKvBlock + (kk & 3) * 32, 0, 1024);
          mma_ts(tmem + col_s(sb), tmem + kTQ + kk * 8, bd, kk < 16 ? kIdescQKLat : kIdescQKRope, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full[sb]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && nt > 1) ok = issue_qk(1);
      for (int i = 0; ok && i < nt; ++i) {
        if (i + 2 < nt && !issue_qk(i + 2)) {
          ok = false;
          break;
        }
        if (!issue_pv(i)) ok = false;
      }
      mma_commit(&bars.o_full);
      mbar_wait(&bars.o_full, 0, err, nullptr);  // every MMA retired
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------- dequantise
    const int dt = threadIdx.x - 64;
    const int tok = dt >> 2, part = dt & 3;
    for (int j = 0; j < nt; ++j) {
      const int st = j % kRawStages, ks = j % kKvStages;
      if (!mbar_wait(&bars.raw_full[st], (j / kRawStages) & 1, err, &abort_s)) break;
      if (!mbar_wait(&bars.kv_empty[ks], ((j / kKvStages) & 1) ^ 1, err, &abort_s)) break;
      const bool valid = (raw_mask[st] >> tok) & 1u;
      uint8_t* kv = sKV + ks * kKvBytes;
      const uint32_t sw = tok & 7;
      uint4 outv[8];
      uint4 rope_out = make_uint4(0, 0, 0, 0);
      if (valid) {
        const uint8_t* raw = sRaw + st * kRawBytes + tok * kRawStride;
        const uint4 c0 = *reinterpret_cast<const uint4*>(raw + 32 * part);
        const uint4 c1 = *reinterpret_cast<const uint4*>(raw + 32 * part + 16);
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(raw + 128 + 4 * part);
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const uint32_t sbyte = (sc >> (8 * blk)) & 0xFFu;
          const uint32_t s2 = e4m3x2_to_f16x2(sbyte | (sbyte << 8));
#pragma unroll
          for (int hw = 0; hw < 2; ++hw) {  // 8 codes per word
            uint32_t h[4];
            e2m1x8_to_f16x8(words[2 * blk + hw], h);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = hmul2_u32(h[i], s2);  // c*s, exact in f16
            outv[2 * blk + hw] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        if constexpr (kFp8Rope) {
          const uint2 r = *reinterpret_cast<const uint2*>(raw + 144 + 8 * part);
          uint32_t o[4];
          o[0] = f16x2_to_bf16x2(e4m3x2_to_f16x2(r.x & 0xFFFFu));
          o[1] = f16x2_to_bf16x2(e4m3x2_to_f16x2(r.x >> 16));
          o[2] = f16x2_to_bf16x2(e4m3x2_to_f16x2(r.y & 0xFFFFu));
          o[3] = f16x2_to_bf16x2(e4m3x2_to_f16x2(r.y >> 16));
          rope_out = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          rope_out = *reinterpret_cast<const uint4*>(raw + 144 + 16 * part);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) outv[i] = make_uint4(0, 0, 0, 0);
      }
      // latent features [64 part, 64 part + 64): column block `part`, 8 chunks
      uint8_t* row = kv + part * kKvBlock + tok * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(row + ((c ^ sw) << 4)) = outv[c];
      // RoPE features [8 part, 8 part + 8) of this CTA's 32: column block 4
      *reinterpret_cast<uint4*>(kv + 4 * kKvBlock + tok * 128 + ((part ^ sw) << 4)) = rope_out;
      fence_async_smem();
      mbar_arrive(&bars.kv_full[ks]);
      mbar_arrive(&bars.raw_empty[st]);
    }
  } else {
    // ------------------------------------------- softmax and epilogue
    const int quad = warp & 3;
    const int hr = quad * 32 + lane;  // head row within the group
    const int head = hg * kHeads + hr;
    const bool head_ok = head < p.num_heads;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float gs = *p.gs;
    const bool gs_ok = scale_ok(gs);
    float score_scale = p.softmax_scale * gs * kLog2e;
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    if (nt > 0) {
      // Q half -> TMEM: [sigma*q_lat[256r : 256r+256] as f16 pairs,
      //                  sigma*q_pe[32r : 32r+32]/gs as bf16 pairs]
      const __nv_bfloat16* qrow = p.q + (static_cast<int64_t>(b) * p.num_heads + head) * 576;
      const float inv_gs = gs_ok ? 1.f / gs : 0.f;
      float qmax = 0.f;  // over the whole latent row, so both CTAs pick the same sigma
      if (head_ok) {
#pragma unroll 4
        for (int i = 0; i < 64; ++i) {
          const uint4 w = reinterpret_cast<const uint4*>(qrow)[i];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float lo, hi;
            bf16x2_to_f32(ws[k], lo, hi);
            qmax = fmaxf(qmax, fmaxf(fabsf(lo), fabsf(hi)));
          }
        }
      }
      // sigma = 2^-a with sigma*qmax < 2^16 (f16 max 65504)
      const int qexp = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFFu) - 127;
      const int a_sh = max(0, min(qexp - 14, 100));
      const float sigma = __uint_as_float(static_cast<uint32_t>(127 - a_sh) << 23);
      score_scale *= __uint_as_float(static_cast<uint32_t>(127 + a_sh) << 23);
#pragma unroll
      for (int c = 0; c < 144; c += 16) {
        uint32_t v[16];
        if (head_ok) {
          if (c < 128) {
            const uint4* src = reinterpret_cast<const uint4*>(qrow + 256 * rank + 2 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 w = src[i];
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float lo, hi;
                bf16x2_to_f32(ws[k], lo, hi);
                __half2 h2 = __floats2half2_rn(lo * sigma, hi * sigma);
                v[4 * i + k] = *reinterpret_cast<uint32_t*>(&h2);
              }
            }
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(qrow + 512 + 32 * rank);
            const float f = inv_gs * sigma;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 w = src[i];
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float lo, hi;
                bf16x2_to_f32(ws[k], lo, hi);
                v[4 * i + k] = pack_bf16(lo * f, hi * f);
              }
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0u;
        }
        tmem_st16(tmem + lane_off + kTQ + c, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.q_ready);

      const uint32_t xch_local = smem_u32(sXch);
      const uint32_t xch_peer = map_peer(xch_local, peer);
      const uint32_t swz = hr & 7;
      // fetch(j): read this CTA's partial scores of tile j from TMEM, free
      // the S buffer, send them to the peer and note which keys are valid.
      auto fetch = [&](int j, float (&s)[kTok], int32_t& idx) -> bool {
        const int sb = j & 1;
        const int xb = j % kXchBufs;
        if (hr == 0) mbar_expect_tx(&bars.xch_full[xb], kXchBytes);
        idx = load_index(p, b, (tile0 + j) * kTok + lane);  // consumed two steps later
        if (!mbar_wait(&bars.s_full[sb], (j >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        uint32_t v0[16], v1[16];
        tmem_ld16(tmem + lane_off + col_s(sb), v0);
        tmem_ld16(tmem + lane_off + col_s(sb) + 16, v1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars.s_free[sb]);
        const uint32_t dst = xch_peer + xb * kXchBytes + hr * 128;
        const uint32_t rbar = map_peer(smem_u32(&bars.xch_full[xb]), peer);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_async_v4(dst + ((static_cast<uint32_t>(i) ^ swz) << 4),
                      make_uint4(v0[4 * i], v0[4 * i + 1], v0[4 * i + 2], v0[4 * i + 3]), rbar);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_async_v4(dst + ((static_cast<uint32_t>(i + 4) ^ swz) << 4),
                      make_uint4(v1[4 * i], v1[4 * i + 1], v1[4 * i + 2], v1[4 * i + 3]), rbar);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          s[i] = __uint_as_float(v0[i]);
          s[16 + i] = __uint_as_float(v1[i]);
        }
        return true;
      };

      // step(j): combine tile j with the peer's partial, online softmax, P(j)
      // into TMEM; then fetch tile j+2 into the same registers.
      auto step = [&](int j, float (&s)[kTok], int32_t& idx) -> bool {
        const int pb = j & 1;
        const int xb = j % kXchBufs;
        bool bad = false;
        const unsigned valid = __ballot_sync(0xffffffffu, key_slot(p, idx, (tile0 + j) * kTok + lane, n_keys, bad) >= 0);
        if (!mbar_wait(&bars.xch_full[xb], (j / kXchBufs) & 1, err, &abort_s)) return false;
        const uint8_t* src = sXch + xb * kXchBytes + hr * 128;
        float x[kTok];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 f = *reinterpret_cast<const float4*>(src + ((static_cast<uint32_t>(i) ^ swz) << 4));
          x[4 * i] = s[4 * i] + f.x;
          x[4 * i + 1] = s[4 * i + 1] + f.y;
          x[4 * i + 2] = s[4 * i + 2] + f.z;
          x[4 * i + 3] = s[4 * i + 3] + f.w;
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (valid == 0xffffffffu) {
#pragma unroll
          for (int c = 0; c < kTok; ++c) {
            x[c] *= score_scale;
            mq[c & 3] = fmaxf(mq[c & 3], x[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kTok; ++c) {
            x[c] = ((valid >> c) & 1u) ? x[c] * score_scale : -INFINITY;
            mq[c & 3] = fmaxf(mq[c & 3], x[c]);
          }
        }
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        float m_use = m_run, alpha = 1.f;
        const bool raise = mx > m_run + kRescaleThreshold;
        if (raise) {
          m_use = mx;
          alpha = ex2_approx(m_run - mx);
        }
        // P(j) reuses the buffer PV(j-2) read; an O rescale needs PV(j-1) retired
        if (j >= 2 && !mbar_wait(&bars.pv_done[pb], ((j - 2) >> 1) & 1, err, &abort_s)) return false;
        if (__any_sync(0xffffffffu, raise && j > 0)) {
          if (!mbar_wait(&bars.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err, &abort_s)) return false;
          tc_fence_after();
#pragma unroll 4
          for (int c = 0; c < 256; c += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_off + kTO + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st16(tmem + lane_off + kTO + c, v);
          }
          tmem_st_wait();
        }
        m_run = m_use;
        const float m_ref = (m_use == -INFINITY) ? 0.f : m_use;  // no valid key so far
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(x[2 * i] - m_ref), p1 = ex2_approx(x[2 * i + 1] - m_ref);
          ls[i & 3] += p0 + p1;
          __half2 h2 = __floats2half2_rn(p0, p1);  // P <= 2^8 (lazy reference), f16 operand
          pv[i] = *reinterpret_cast<uint32_t*>(&h2);
        }
        l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
        tc_fence_after();
        tmem_st16(tmem + lane_off + col_p(pb), pv);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.p_full[pb]);
        if (j + 2 < nt) return fetch(j + 2, s, idx);
        return true;
      };

      float s_a[kTok], s_b[kTok];
      int32_t idx_a = -1, idx_b = -1;
      ok = fetch(0, s_a, idx_a);
      if (ok && nt > 1) ok = fetch(1, s_b, idx_b);
      for (int j = 0; ok && j < nt; j += 2) {
        ok = step(j, s_a, idx_a);
        if (ok && j + 1 < nt) ok = step(j + 1, s_b, idx_b);
      }
      if (ok) ok = mbar_wait(&bars.o_full, 0, err, &abort_s);
    }
    // partial output of this split: O half / l (scaled by gs), lse.  TMEM
    // loads are warp-collective, so every lane loads; only stores depend on
    // the head.
    const bool live = __all_sync(0xffffffffu, ok) && nt > 0;
    const bool have = live && l_run > 0.f;
    const float f = have ? gs / l_run : 0.f;
    const int64_t row = (static_cast<int64_t>(b) * p.splits + split) * p.num_heads + head;
    float4* dst = reinterpret_cast<float4*>(p.part_o + row * 512 + 256 * rank);
    if (live) tc_fence_after();
#pragma unroll 2
    for (int c = 0; c < 256; c += 16) {
      uint32_t v[16];
      if (live) {
        tmem_ld16(tmem + lane_off + kTO + c, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0u;
      }
      if (head_ok) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[c / 4 + i] = make_float4(__uint_as_float(v[4 * i]) * f, __uint_as_float(v[4 * i + 1]) * f,
                                       __uint_as_float(v[4 * i + 2]) * f, __uint_as_float(v[4 * i + 3]) * f);
      }
    }
    if (head_ok && rank == 0) p.part_lse[row] = have ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still address it
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
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
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(o) = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
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
  const int groups = (num_heads + kHeads - 1) / kHeads;
  const int pairs = num_sms / 2;
  const int units = batch * groups;
  int s = pairs / (units > 0 ? units : 1);
  return s < 1 ? 1 : (s > 64 ? 64 : s);
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream, int /*num_sms*/) {
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.batch = a.batch;
  p.num_heads = a.num_heads;
  p.cache = a.cache;
  p.num_slots = a.num_slots;
  p.record_bytes = a.record_bytes;
  p.page_table = a.page_table;
  p.pt_stride = a.page_table_stride;
  p.page_size = a.page_size;
  p.seq_lens = a.seq_lens;
  p.topk = a.topk_indices;
  p.topk_n = a.topk;
  p.softmax_scale = a.softmax_scale;
  p.gs = a.gs;
  p.splits = a.num_splits;
  p.error_word = a.error_word;
  const size_t rows = static_cast<size_t>(a.batch) * a.num_splits * a.num_heads;
  p.part_o = static_cast<float*>(a.workspace);
  p.part_lse = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + rows * 512 * sizeof(float));

  dim3 grid(2 * a.num_splits, a.batch, (a.num_heads + kHeads - 1) / kHeads);
  if (grid.y > 65535u || grid.z > 65535u) return MLA_ERR_INVALID_ARG;
  if (a.record_bytes == 432) {
    if (const int st = cuda_status(cudaFuncSetAttribute(decode_tc_kernel<432>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmAlloc)))) return st;
    decode_tc_kernel<432><<<grid, kThreads, kSmAlloc, stream>>>(p);
  } else {
    if (const int st = cuda_status(cudaFuncSetAttribute(decode_tc_kernel<368>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmAlloc)))) return st;
    decode_tc_kernel<368><<<grid, kThreads, kSmAlloc, stream>>>(p);
  }
  if (const int st = launch_status()) return st;
  decode_merge_kernel<<<a.batch * a.num_heads, 128, 0, stream>>>(
      p.part_o, p.part_lse, a.num_splits, a.num_heads, static_cast<__nv_bfloat16*>(a.out), a.lse);
  return launch_status();
}

}  // namespace mla
