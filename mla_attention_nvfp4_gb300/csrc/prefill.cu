// Causal varlen MLA prefill (q/k head dim 192, v head dim 128) on tcgen05
// tensor cores, whose epilogue writes NVFP4 directly: packed e2m1 codes plus
// e4m3 block scales in the 128x4-swizzled layout, so no standalone
// quantisation pass runs.
//
// Source: "feat: MLA prefill NVFP4 fused output - #8" (PR description: FA
// writes the packed e2m1 output, the global scale and the swizzled e4m3
// block-scale buffer consumed by the NVFP4 GEMMs; review of the
// float4_e2m1fn_x2 output view [-1, H, v_head_dim/2]); "Add NVFP4/FP8
// Q/K/P/V + 2:4 attention quantization for MLA (vLLM TRITON_MLA) - #2244",
// first commit message (varlen prefill with asymmetric 192/128 head dims,
// natural-log LSE).
//
// One CTA = one 128-row query tile of one (sequence, head).  Warp roles:
//   warp 0      TMA producer: Q once, then K/V tiles of 128 keys into a
//               two-stage ring (128-byte swizzled, K-major rows).
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S_j = Q K_j^T       M=128 N=128 K=192, A and B from smem
//                 O  += P_j V_j       M=128 N=128 K=128, A (P) from TMEM,
//                                     B = V tile read MN-major
//   warps 2..9  softmax, O correction and epilogue: two warpgroups, each
//               thread one query row and one half (64 columns) of S and O.
// TMEM columns: S double buffer [0,128) [128,256); O [256,384).  P_j (bf16)
// overwrites the first 64 columns of its S buffer after the row is read.
// The running max is only raised when a row's max grows by more than 8
// (log2 units), so O is rarely rescaled; P stays <= 2^8, exact enough in
// bf16, and numerator and denominator share the same reference.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "nvfp4.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 128, kDqk = 192, kDv = 128;
constexpr int kThreads = 320;
constexpr uint32_t kQBytes = kBM * kDqk * 2;  // 49152
constexpr uint32_t kKBytes = kBN * kDqk * 2;  // 49152
constexpr uint32_t kVBytes = kBN * kDv * 2;   // 32768
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = kSmemQ + kQBytes;
constexpr uint32_t kSmemV = kSmemK + 2 * kKBytes;
constexpr uint32_t kSmemBytes = kSmemV + 2 * kVBytes;  // 212992
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;      // + alignment slack
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 256
static_assert(kSmemAlloc <= 232448, "shared memory budget");

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);

struct Params {
  const int32_t* cu;
  int num_seqs;
  int64_t total;
  int num_heads;
  int q_tiles;  // grid.x
  float scale_log2;
  const float* gs;
  uint8_t* codes;
  uint8_t* scales;
  float* lse;
  uint32_t* error_word;
};

struct alignas(8) Barriers {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_full;
  uint64_t red[2], red_l;  // the two softmax groups exchanging row maxima / sums
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ float red_s[2][2][kBM];  // per-group row maxima, double-buffered by tile parity
  __shared__ float red_l[2][kBM];     // per-group row sums

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, seq = blockIdx.z;
  const int tile = p.q_tiles - 1 - static_cast<int>(blockIdx.x);  // heavy (late) tiles first
  const int64_t k_tiles_sf = (static_cast<int64_t>(p.num_heads) * 8 + 3) / 4;

  // rows [total, roundup(total,128)) of this head's scale columns are zero
  if (blockIdx.x == 0 && seq == 0) {
    const int64_t Mp = (p.total + 127) / 128 * 128;
    for (int64_t i = threadIdx.x; i < (Mp - p.total) * 8; i += kThreads)
      p.scales[sf_offset(p.total + i / 8, static_cast<int64_t>(h) * 8 + i % 8, k_tiles_sf)] = 0;
  }
  const int seq_begin = p.cu[seq], seq_end = p.cu[seq + 1];
  const int n = seq_end - seq_begin;
  if (seq_begin < 0 || seq_end > p.total || n < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) flag_error(p.error_word, MLA_DEVERR_BOUNDS);
    return;
  }
  const int row0 = tile * kBM;
  if (row0 >= n) return;
  const int n_kv = (min(n, row0 + kBM) - 1) / kBN + 1;  // causal: keys < row0 + 128
  const float gs = *p.gs;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kSmemQ;
  uint8_t* sK = smem + kSmemK;
  uint8_t* sV = smem + kSmemV;

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], 256);
    }
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.o_full, 1);
    mbar_init(&bars.red[0], 256);
    mbar_init(&bars.red[1], 256);
    mbar_init(&bars.red_l, 256);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tS0 = tmem, tS1 = tmem + 128;
  const uint32_t tO = tmem + 256;
  uint32_t* err = p.error_word;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const int tok0 = seq_begin + row0;
      mbar_expect_tx(&bars.q_full, kQBytes);
      for (int cb = 0; cb < 3; ++cb) tma_load_3d(sQ + cb * 16384, &tm_q, cb * 64, h, tok0, &bars.q_full);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        const int key0 = seq_begin + j * kBN;
        if (!mbar_wait(&bars.k_empty[s], ph ^ 1, err, &abort_s)) break;
        mbar_expect_tx(&bars.k_full[s], kKBytes);
        for (int cb = 0; cb < 3; ++cb)
          tma_load_3d(sK + s * kKBytes + cb * 16384, &tm_k, cb * 64, h, key0, &bars.k_full[s]);
        if (!mbar_wait(&bars.v_empty[s], ph ^ 1, err, &abort_s)) break;
        mbar_expect_tx(&bars.v_full[s], kVBytes);
        for (int cb = 0; cb < 2; ++cb)
          tma_load_3d(sV + s * kVBytes + cb * 16384, &tm_v, cb * 64, h, key0, &bars.v_full[s]);
      }
      // every copy issued has landed before the CTA can exit
      mbar_wait(&bars.q_full, 0, err, nullptr);
      for (int jj = max(0, j - 2); jj < j; ++jj) {
        mbar_wait(&bars.k_full[jj & 1], (jj >> 1) & 1, err, nullptr);
        mbar_wait(&bars.v_full[jj & 1], (jj >> 1) & 1, err, nullptr);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      // Descriptors are built once; a K-step only adds its byte offset >> 4
      // to the start-address field (addresses stay below 256 KB, no carry).
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      const uint64_t dq = smem_desc_sw128(q_addr, 0, 1024);
      const uint64_t dk0 = smem_desc_sw128(k_addr, 0, 1024), dk1 = smem_desc_sw128(k_addr + kKBytes, 0, 1024);
      const uint64_t dv0 = smem_desc_sw128(v_addr, 16384, 1024), dv1 = smem_desc_sw128(v_addr + kVBytes, 16384, 1024);
      bool ok = mbar_wait(&bars.q_full, 0, err, &abort_s);
      auto issue_pv = [&](int i) -> bool {
        const int b = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(&bars.p_full[b], ph, err, &abort_s)) return false;
        if (!mbar_wait(&bars.v_full[b], ph, err, &abort_s)) return false;
        tc_fence_after();
        const uint64_t vd = b ? dv1 : dv0;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tO, (b ? tS1 : tS0) + kk * 8, vd + ((kk * 2048) >> 4), kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.v_empty[b]);
        mma_commit(&bars.pv_done);
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&bars.k_full[s], ph, err, &abort_s)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = s ? dk1 : dk0;
#pragma unroll
        for (int kk = 0; kk < kDqk / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(s ? tS1 : tS0, dq + off, kd + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full[s]);
        mma_commit(&bars.k_empty[s]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n_kv - 1);
      mma_commit(&bars.o_full);
      mbar_wait(&bars.o_full, 0, err, nullptr);  // all MMAs retired
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    // Two warpgroups share each row: group g handles score columns
    // [64g, 64g+64) and output columns [64g, 64g+64).  Row maxima and sums
    // are combined through shared memory.
    const int g = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int qi = row0 + r;         // query index within the sequence
    const int c0 = 64 * g;           // first score / output column of this group
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait(&bars.s_full[b], ph, err, &abort_s)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[64];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t v[16];
        tmem_ld16((b ? tS1 : tS0) + lane_off + c0 + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[c + i] = __uint_as_float(v[i]);
      }
      tmem_ld_wait();
      // max of the raw scores (scale_log2 > 0); the scale is applied inside
      // the exponent below
      const int key0 = j * kBN + c0;
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (key0 + 63 > qi) {  // diagonal tile: mask keys after the query
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          x[c] = (key0 + c <= qi) ? x[c] : -INFINITY;
          mq[c & 3] = fmaxf(mq[c & 3], x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) mq[c & 3] = fmaxf(mq[c & 3], x[c]);
      }
      // row max over both halves (also orders every S read before any P write)
      red_s[b][g][r] = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
      mbar_arrive(&bars.red[b]);
      if (!mbar_wait(&bars.red[b], ph, err, &abort_s)) {
        ok = false;
        break;
      }
      const float mx = fmaxf(red_s[b][0][r], red_s[b][1][r]);
      // lazy reference update (identical in both groups)
      float m_use = m_run, alpha = 1.f;
      const bool raise = mx > m_run + kRescaleThreshold;
      if (raise) {
        m_use = mx;
        alpha = ex2_approx(m_run - mx);  // 0 on the first tile
      }
      const bool warp_rescale = __any_sync(0xffffffffu, raise && j > 0);
      if (warp_rescale) {
        // O must not be in flight: PV_{j-1} has to be complete
        if (!mbar_wait(&bars.pv_done, (j - 1) & 1, err, &abort_s)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          uint32_t v[16];
          tmem_ld16(tO + lane_off + c0 + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st16(tO + lane_off + c0 + c, v);
        }
        tmem_st_wait();
      }
      m_run = m_use;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; c += 32) {  // P as bf16 pairs: columns [32g, 32g+32) of the S buffer
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(fmaf(x[c + 2 * i], p.scale_log2, -m_use));
          const float p1 = ex2_approx(fmaf(x[c + 2 * i + 1], p.scale_log2, -m_use));
          ls[i & 3] += p0 + p1;
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          v[i] = *reinterpret_cast<uint32_t*>(&h2);
        }
        tmem_st16((b ? tS1 : tS0) + lane_off + 32 * g + c / 2, v);
      }
      l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[b]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && mbar_wait(&bars.o_full, 0, err, &abort_s)) {
      red_l[g][r] = l_run;
      tc_fence_after();
      float o[64];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t v[16];
        tmem_ld16(tO + lane_off + c0 + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[c + i] = __uint_as_float(v[i]);
      }
      tmem_ld_wait();
      mbar_arrive(&bars.red_l);
      mbar_wait(&bars.red_l, 0, err, &abort_s);
      const float l_tot = red_l[0][r] + red_l[1][r];
      if (qi < n) {
        const int64_t m = seq_begin + qi;
        const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) o[c] *= inv_l;
        const bool gs_ok = scale_ok(gs);
        const float kf = scale_factor(gs);
        uint32_t w[8];
        uint32_t sb[4];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          float R = 0.f;
          sb[blk] = gs_ok ? block_scale(fmaxf(amax8(o + 16 * blk), amax8(o + 16 * blk + 8)), kf, gs, R) : 0u;
          w[2 * blk] = gs_ok ? encode8(o + 16 * blk, R) : 0u;
          w[2 * blk + 1] = gs_ok ? encode8(o + 16 * blk + 8, R) : 0u;
        }
        uint4* dst = reinterpret_cast<uint4*>(p.codes + m * (static_cast<int64_t>(p.num_heads) * 64) + h * 64 + 32 * g);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        const int64_t kc = static_cast<int64_t>(h) * 8 + 4 * g;
        *reinterpret_cast<uint32_t*>(p.scales + sf_offset(m, kc, k_tiles_sf)) =
            sb[0] | (sb[1] << 8) | (sb[2] << 16) | (sb[3] << 24);
        if (g == 0 && p.lse != nullptr)
          p.lse[static_cast<int64_t>(h) * p.total + m] = l_tot > 0.f ? (m_run + log2f(l_tot)) * kLn2 : -INFINITY;
        if (!gs_ok && qi == 0 && g == 0) flag_error(err, MLA_DEVERR_SCALE);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// --------------------------------------------------------------- host side
// cuTensorMapEncodeTiled, fetched from the driver at run time (the library
// links only the CUDA runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [T, H, D] bf16 with element strides (st, sh, 1) as a 3-D map (D, H, T);
// box = 64 elements x 1 head x 128 tokens, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t D, int64_t H, int64_t T, int64_t st, int64_t sh) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(st * 2)};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream, int /*num_sms*/) {
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, kDqk, a.num_heads, a.total_tokens, a.q_st, a.q_sh) ||
      !make_map(&tk, a.k, kDqk, a.num_heads, a.total_tokens, a.k_st, a.k_sh) ||
      !make_map(&tv, a.v, kDv, a.num_heads, a.total_tokens, a.v_st, a.v_sh))
    return MLA_ERR_LAUNCH;
  Params p;
  p.cu = a.cu_seqlens;
  p.num_seqs = a.num_seqs;
  p.total = a.total_tokens;
  p.num_heads = a.num_heads;
  p.q_tiles = (a.max_seqlen + kBM - 1) / kBM;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.gs = a.gs;
  p.codes = a.out_codes;
  p.scales = a.out_scales;
  p.lse = a.lse;
  p.error_word = a.error_word;
  if (const int st = cuda_status(cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemAlloc)))) return st;
  dim3 grid(p.q_tiles, a.num_heads, a.num_seqs);
  if (grid.y > 65535u || grid.z > 65535u) return MLA_ERR_INVALID_ARG;
  prefill_tc_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(tq, tk, tv, p);
  return launch_status();
}

}  // namespace mla
