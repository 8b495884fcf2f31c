// NVFP4 x NVFP4 GEMM on tcgen05 block-scaled tensor cores: the output
// projection that consumes the fused prefill output as written.
//
// Source: "feat: MLA prefill NVFP4 fused output - #8" (vLLM fork), PR
// description: the prefill writes packed e2m1 codes and e4m3 block scales in
// the 128x4-swizzled layout that the NVFP4 GEMMs read directly, with no
// standalone quantisation pass.
//
//   C[m, n] = gs_a * gs_w * sum_k  e2m1(a[m,k]) s_a[m,k/16] * e2m1(w[n,k]) s_w[n,k/16]
//
// A [M, K] and W [N, K] are packed codes (two per byte, even element low)
// with swizzled scale buffers; C is bf16 [M, N] (row stride ldc).
//
// Tiles of 128 x 256 outputs, persistent CTAs (one per SM) walking the tiles
// in row-major order, so that the CTAs working at one time share a few rows
// of A and all of W through L2.  K runs in stages of 256 (128 code bytes per
// row: one 128-byte swizzle atom), four stages in flight:
//   warp 0        TMA producer: A and W code tiles (2-D tensor maps, 128-byte
//                 swizzle) and their scale tiles (1-D bulk copies: a 128-row
//                 x 4-block scale tile is one contiguous 512-byte block of the
//                 swizzled buffer, already in the order tcgen05.cp reads),
//   warp 1        MMA issuer: per stage, once its scale tiles are in TMEM,
//                 four tcgen05.mma kind::mxf4nvf4 (M 128, N 256, K 64, block
//                 scale 1x16 ue4m3) into the TMEM accumulator,
//   warps 2..5    epilogue: accumulator -> x gs_a gs_w -> bf16 -> C,
//   warps 6, 7    scale copies: per stage, the twelve tcgen05.cp of the
//                 scale tiles into TMEM (32x128b, replicated to the four
//                 lane quarters), split between the two warps, their
//                 completion releasing the stage to the MMA issuer.  The
//                 copies' issue rate, not the tensor pipe, set the pace when
//                 the MMA thread issued them itself (1.99 ms on 32768 x 7168
//                 x 16384 against 1.78 with one copy warp and 1.44 with two).
// TMEM: accumulator columns [0, 256), then per stage 16 columns of A scales
// and 32 of W scales.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "launch.h"
#include "nvfp4.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 256;
constexpr int kBKBytes = 128;            // K per stage: 256 fp4 codes
constexpr int kStages = 4;
constexpr int kCopyWarps = 2;  // 1: 1.78 ms, 2: 1.44, 3-4: 1.48, 6: 1.55 on 32768 x 7168 x 16384
constexpr int kThreads = 192 + 32 * kCopyWarps;
constexpr uint32_t kABytes = kBM * kBKBytes;      // 16 KB
constexpr uint32_t kBBytes = kBN * kBKBytes;      // 32 KB
constexpr uint32_t kSfTile = 512;                 // 128 rows x 4 blocks
constexpr uint32_t kSfaBytes = 4 * kSfTile;       // 4 k-tiles of 64
constexpr uint32_t kSfbBytes = 8 * kSfTile;       // 2 row tiles x 4 k-tiles
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr uint32_t kSmBytes = kStages * kStageBytes;
constexpr uint32_t kSmAlloc = kSmBytes + 1024;
static_assert(kSmAlloc + 256 <= 232448, "shared memory budget");

constexpr uint32_t kColD = 0;
__host__ __device__ constexpr uint32_t col_sfa(int s) { return 256u + 48u * s; }
__host__ __device__ constexpr uint32_t col_sfb(int s) { return 256u + 48u * s + 16u; }

// Instruction descriptor of kind::mxf4nvf4: e2m1 A and B (format 1), K-major,
// ue4m3 block scales (bit 23 = 0), scale-factor ids 0, N >> 3 in bits 17..22,
// M >> 4 in bits 24..28.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);

struct Params {
  const uint8_t* a_sf;
  const uint8_t* w_sf;
  int64_t M, N, K;
  int64_t a_sf_ktiles, w_sf_ktiles;  // 4-block scale tiles per 128-row tile
  const float* gs_a;
  const float* gs_w;
  __nv_bfloat16* c;
  int64_t ldc;
  int tiles_n;        // 256-column tiles
  uint32_t tn_magic;  // tiles_n's multiplier and shift for div_magic
  int tn_shift;
  uint32_t* error_word;
};

struct alignas(8) Barriers {
  uint64_t full[kStages], empty[kStages];
  uint64_t sf_full[kStages];  // the stage's scale tiles are in TMEM
  uint64_t acc_full, acc_empty;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Shared-memory descriptor of one 512-byte scale tile for tcgen05.cp
// 32x128b: 32 rows of 16 bytes, no swizzle, i.e. four 8-row core matrices
// 128 bytes apart.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 16;  // leading-dimension offset (one core matrix along K)
  d |= static_cast<uint64_t>(128u >> 4) << 32;  // stride-dimension offset: next 8 rows
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__device__ __forceinline__ void sf_copy(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(kIdesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w, Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  auto sA = [&](int s) { return s0 + s * kStageBytes; };
  auto sB = [&](int s) { return s0 + s * kStageBytes + kABytes; };
  auto sSfa = [&](int s) { return s0 + s * kStageBytes + kABytes + kBBytes; };
  auto sSfb = [&](int s) { return s0 + s * kStageBytes + kABytes + kBBytes + kSfaBytes; };

  const int64_t tiles_m = (p.M + kBM - 1) / kBM, tiles_n = p.tiles_n;
  const int64_t n_tiles = tiles_m * tiles_n;  // < 2^31 (checked at launch)
  const int nk = static_cast<int>(p.K / 256);
  uint32_t* err = p.error_word;

  if (threadIdx.x == 0) {
    abort_s = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
      mbar_init(&bars.sf_full[s], kCopyWarps);
    }
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.acc_empty, 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_a);
      prefetch_tmap(&tm_w);
      int it = 0;  // stage fills so far
      for (int64_t t = blockIdx.x; t < n_tiles && !abort_s; t += gridDim.x) {
        const int64_t mt = div_magic(static_cast<uint32_t>(t), p.tn_magic, p.tn_shift), ntile = t - mt * tiles_n;
        // the W scale rows of this tile: one or two 128-row tiles (N is a
        // multiple of 128; the second is absent on a half tile at the end)
        const int sfb_tiles = (ntile * kBN + 128 < p.N) ? 2 : 1;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&bars.empty[s], ((it / kStages) & 1) ^ 1, err, &abort_s)) break;
          mbar_expect_tx(&bars.full[s], kABytes + kBBytes + kSfaBytes + sfb_tiles * kSfaBytes);
          tma_load_2d(sA(s), &tm_a, kb * kBKBytes, static_cast<int>(mt * kBM), &bars.full[s]);
          tma_load_2d(sB(s), &tm_w, kb * kBKBytes, static_cast<int>(ntile * kBN), &bars.full[s]);
          // scale tiles (row tile r, k tiles 4 kb .. 4 kb + 3) are contiguous
          bulk_load(sSfa(s), p.a_sf + (mt * p.a_sf_ktiles + 4 * kb) * kSfTile, kSfaBytes, &bars.full[s]);
          for (int r = 0; r < sfb_tiles; ++r)
            bulk_load(sSfb(s) + r * kSfaBytes, p.w_sf + ((2 * ntile + r) * p.w_sf_ktiles + 4 * kb) * kSfTile,
                      kSfaBytes, &bars.full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int it = 0, tile_i = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++tile_i) {
        // the epilogue has read the previous tile's accumulator
        if (!mbar_wait(&bars.acc_empty, (tile_i & 1) ^ 1, err, &abort_s)) break;
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          // operands landed and the scale tiles copied into TMEM (warp 6)
          if (!mbar_wait(&bars.sf_full[s], (it / kStages) & 1, err, &abort_s)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = smem_desc_sw128(sA(s), 0, 1024), db = smem_desc_sw128(sB(s), 0, 1024);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // K 64 = 32 bytes a step along the swizzled row
            mma_fp4(tmem + kColD, da + 2 * j, db + 2 * j, tmem + col_sfa(s) + 4 * j, tmem + col_sfb(s) + 8 * j,
                    (kb > 0 || j > 0) ? 1u : 0u);
          mma_commit(&bars.empty[s]);
        }
        mma_commit(&bars.acc_full);
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------ scale copies
    // per stage, once its bytes have landed: scales into TMEM, k tile j of
    // A to columns sfa + 4 j; of W, row tiles 0 and 1 to columns sfb + 8 j
    // and sfb + 8 j + 4; the copies' completion releases the stage to the
    // MMA issuer.  A stage's columns are written again only after the
    // producer refilled it, which waits for the MMAs that read them.
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&bars.full[s], (it / kStages) & 1, err, &abort_s)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = warp - 6; c < 12; c += kCopyWarps) {
            const int j = c & 3, kind = c >> 2;  // 0: A, 1: W rows 0..127, 2: W rows 128..255
            const uint32_t col = kind == 0 ? col_sfa(s) + 4 * j : col_sfb(s) + 8 * j + 4 * (kind - 1);
            const uint32_t src = kind == 0 ? sSfa(s) + j * kSfTile : sSfb(s) + (kind - 1) * kSfaBytes + j * kSfTile;
            sf_copy(tmem + col, sf_desc(src));
          }
          mma_commit(&bars.sf_full[s]);
        }
      }
      if (it > 0) mbar_wait(&bars.sf_full[(it - 1) % kStages], ((it - 1) / kStages) & 1, err, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lane quarter this warp may access
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float alpha = *p.gs_a * *p.gs_w;
    int tile_i = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tile_i) {
      if (!mbar_wait(&bars.acc_full, tile_i & 1, err, &abort_s)) break;
      tc_fence_after();
      const int64_t mt = div_magic(static_cast<uint32_t>(t), p.tn_magic, p.tn_shift), ntile = t - mt * tiles_n;
      const int64_t row = mt * kBM + r;
      const int64_t n0 = ntile * kBN;
      __nv_bfloat16* crow = p.c + row * p.ldc + n0;
#pragma unroll 1
      for (int c = 0; c < kBN; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_off + kColD + c, v);
        tmem_ld_wait();
        if (row < p.M && n0 + c < p.N) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            __nv_bfloat162 h =
                __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * alpha, __uint_as_float(v[2 * i + 1]) * alpha);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
          }
          uint4* dst = reinterpret_cast<uint4*>(crow + c);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars.acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// cuTensorMapEncodeTiled from the driver at run time (the library links
// only the CUDA runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn gemm_encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(ptr);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// Packed codes [rows, K/2] bytes as a 2-D byte map; box = 128 bytes x
// box_rows rows, 128-byte swizzle (rows past the end read as zero).
bool make_code_map(CUtensorMap* m, const uint8_t* base, int64_t rows, int64_t K, uint32_t box_rows) {
  auto fn = gemm_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_gemm(const GemmArgs& a, cudaStream_t stream, int num_sms) {
  CUtensorMap tm_a, tm_w;
  if (!make_code_map(&tm_a, a.a_codes, a.M, a.K, kBM) || !make_code_map(&tm_w, a.w_codes, a.N, a.K, kBN)) {
    set_last_error("cuTensorMapEncodeTiled failed for the GEMM operands");
    return MLA_ERR_LAUNCH;
  }
  Params p;
  p.a_sf = a.a_scales;
  p.w_sf = a.w_scales;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.a_sf_ktiles = (a.K / 16 + 3) / 4;
  p.w_sf_ktiles = (a.K / 16 + 3) / 4;
  p.gs_a = a.gs_a;
  p.gs_w = a.gs_w;
  p.c = static_cast<__nv_bfloat16*>(a.out);
  p.ldc = a.ldc;
  p.error_word = a.error_word;
  const int64_t tiles = ((a.M + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN);
  if (tiles > (int64_t(1) << 31) - 1) return MLA_ERR_INVALID_ARG;
  p.tiles_n = static_cast<int>((a.N + kBN - 1) / kBN);
  magic_divisor(p.tiles_n, &p.tn_magic, &p.tn_shift);
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  if (const int st = smem_limit_once(reinterpret_cast<const void*>(nvfp4_gemm_kernel), static_cast<int>(kSmAlloc), 4))
    return st;
  nvfp4_gemm_kernel<<<grid, kThreads, kSmAlloc, stream>>>(tm_a, tm_w, p);
  return launch_status();
}

}  // namespace mla
