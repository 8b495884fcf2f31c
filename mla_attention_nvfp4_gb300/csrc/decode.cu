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
// tile holds c*s and k_pe, both exact in f16 (k_pe inside the f16 range),
// the query holds sigma*[q_lat, q_pe/gs] in f16 with sigma a per-head power
// of two keeping both parts inside the f16 range (q_lat then stays exact;
// q_pe/gs is rounded once, to 11 bits), the product is multiplied by
// softmax_scale*gs/sigma, and the output by gs.  All score MMAs are f16.
//
// Work unit = (sequence b, split, group of up to 128 heads), run by two
// independent CTAs.  Both compute the full 576-feature scores of every
// 64-key tile; CTA r accumulates only output features [256r, 256r+256).  The
// 128 x 512 fp32 output does not fit one SM's 512 TMEM columns next to the
// scores and the query, and exchanging partial scores between two SMs costs
// more than computing them twice, so the score product is duplicated and
// nothing crosses SMs.  The two CTAs are launched as a cluster of two: they
// read the same records, and a pair placed in one GPC finds the partner's
// records in the near L2 (without the cluster, a grid with CTAs that leave
// at once ran 13 us slower on 64 x 4096 keys, measured).
//
// Per CTA:
//   TMEM   O half [0,256), scores/P for two tiles [256,384), Q RoPE part and
//          latent features [0,192) [384,512) as MMA A operands.
//   SMEM   Q latent features [192,512) (f16, 128-byte swizzled, 80 KB), and
//          for two tiles: the "V part" (this CTA's 256 latent features, read
//          by both products) and the "T part" (the other 256 latent features
//          and the RoPE features, read by the score product only).
//   Each issuer runs  QK_T(j), QK_V(j), PV(j)  for its tiles; the softmax
//   of tile j overlaps the other issuer's tile j+1, and the V part of tile
//   j+2 may be written while QK_T(j+2) runs, so two buffers of each part
//   (one per tile parity) suffice.
//
// Warp roles (512 threads):
//   warps 0..3, 12..15  Q staging (two threads per head: warp w writes
//                TMEM lanes 32 (w % 4)..+32, warps 0..3 one half of each
//                query row, warps 12..15 the other), then the online
//                softmax, lazy O rescale and partial-output epilogue with
//                four threads per pair of heads: warp w takes TMEM lanes
//                32 (w % 4) + 16 [w >= 12] .. +16 through the 16-lane
//                shapes, thread t heads t/4 and t/4 + 8 of them and 16 of a
//                tile's 64 keys, so a head's threads share maxima and row
//                sums by shuffles (an earlier split over two warps had to
//                meet in shared memory behind an mbarrier every tile).
//   warps 4, 11  MMA issuers (one thread each) for even and odd tiles;
//                warp 4 owns the TMEM allocation.
//   warps 5..10  dequantisation: thread = (key, third of the record), 16-byte
//                loads straight from global memory as soon as the previous
//                tile is converted, e2m1 -> f16 conversion times the block
//                scale, stores into the swizzled operand tiles.
// With 128 SMs fetching this kernel's instructions at once, the size of the
// hot code counts: the MMA issue loops stay rolled, every wait shares one
// out-of-line polling loop, and each dequantising part has one copy of its
// conversion code (together ~25 % of the run time against unrolled forms).
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "nvfp4.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTok = 64;           // keys per tile (MMA N of the score product)
constexpr int kHeads = 128;        // heads per work unit (MMA M)
constexpr int kThreads = 384;    // NVFP4-query kernel: one softmax thread per head
constexpr int kThreadsTc = 512;  // exact kernel: two softmax threads per head
constexpr int kSoftWarp2 = 12;   // exact kernel: warps 12..15 take the second half of each tile's keys
constexpr int kMmaWarp = 4;    // MMA issuer for even tiles, TMEM owner
constexpr int kMmaWarp2 = 11;  // MMA issuer for odd tiles
constexpr int kDeqWarp0 = 5;
constexpr int kDeqWarps = 6;
constexpr uint32_t kChunk = kTok * 128;      // 64 keys x 64 features, f16
constexpr uint32_t kQChunk = kHeads * 128;   // 128 heads x 64 features, f16
constexpr uint32_t kVBytes = 4 * kChunk;     // V part: 4 latent chunks
constexpr uint32_t kTBytes = 5 * kChunk;     // T part: 4 latent chunks + RoPE
constexpr uint32_t kSmQ = 0;                 // Q latent chunks 3..7
constexpr uint32_t kSmV = kSmQ + 5 * kQChunk;
constexpr uint32_t kSmT = kSmV + 2 * kVBytes;
constexpr uint32_t kSmBytes = kSmT + 2 * kTBytes;
constexpr uint32_t kSmAlloc = kSmBytes + 1024;
static_assert(kSmAlloc + 512 <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t kTO = 0;                  // O half, 256 columns
__host__ __device__ constexpr uint32_t col_s(int buf) { return 256u + 64u * buf; }  // scores / P
constexpr uint32_t kTQRope = 384;            // sigma*q_pe/gs, f16 pairs, 32 columns
constexpr uint32_t kTQLat = 416;             // sigma*q_lat[0:192], f16 pairs, 96 columns

constexpr uint32_t kIdescQK = idesc_f16_f32(128, kTok, false, false);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 256, false, true);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The reference (running max, log2 units) is raised, and O rescaled, only
// when a tile's max exceeds it by more than kRescaleThreshold, and is then
// set kRefHeadroom above that max, so that the next raise needs the max to
// grow by both.  P = 2^(s - m) stays at most 2^15.5, inside f16 (max 65504),
// and sum P.V far inside fp32; right after a raise the largest P is 2^-4, so
// f16's subnormal range (below 2^-14) begins 10 log2 units under the max,
// where a P rounds to a multiple of 2^-24 against a row sum of at least
// 2^-4.  A rescale waits for the two previous P.V products; on the 64 x 4096
// workload (scores counted on the CPU) some softmax warp of a CTA rescales
// in ~8 % of tiles with these values, ~43 % with threshold 14 and no
// headroom.
constexpr float kRescaleThreshold = 15.5f;
constexpr float kRefHeadroom = 4.0f;

struct Params {
  const __nv_bfloat16* q;
  int batch, num_heads;
  const uint8_t* cache;
  int64_t num_slots;
  int record_bytes;
  const int32_t* page_table;
  int64_t pt_stride;
  int page_size;
  // page_size's multiplier and shift for div_magic
  uint32_t pg_magic;
  int pg_shift;
  const int32_t* seq_lens;
  const int32_t* topk;
  int topk_n;
  float softmax_scale;
  const float* gs;
  const float* gs_q;  // NVFP4-query mode: the query's global scale (null otherwise)
  float* part_o;    // [rows, heads, 512]: split partials
  float* part_lse;  // [rows, heads]
  int splits;       // uniform mode: key splits per sequence
  // planned mode (plan_items != null): CTA pair i runs item i of the plan
  const int32_t* plan_hdr;  // [0] items, [1] tiles per chunk
  const int2* plan_items;   // (sequence, chunk index)
  const int2* plan_seqs;    // (first partial row or -1, chunks) per sequence
  __nv_bfloat16* out;  // [batch, heads, 512]: written here directly when splits == 1
  float* lse;          // [batch, heads] or null (same)
  uint32_t* error_word;
};

// The kernel's waits: the first test inline, the polling loop (bounded as
// in sm100::mbar_wait) one out-of-line copy shared by every wait, which
// keeps the roles' hot code small.
__device__ __noinline__ bool bar_wait_poll(uint64_t* bar, uint32_t parity, uint32_t* error_word, volatile int* abort) {
  return mbar_wait(bar, parity, error_word, abort);
}
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, uint32_t* error_word, volatile int* abort) {
  return mbar_test(bar, parity) || bar_wait_poll(bar, parity, error_word, abort);
}

// Exchange between the two softmax threads of a head (exact kernel): one
// value per half and head row, behind an mbarrier that both halves arrive
// on: the query maxima of the staging pass (qx), each tile's maxima
// (mx_full, by tile parity), the row sums at the end (fin).  One slot per
// half serves all three; a value is overwritten only after the partner has
// read the previous one (the partner's P of the previous tile is in, or the
// item's last P.V has retired).
struct alignas(8) SoftX {
  uint64_t mx_full[2], fin, qx;
  float v[2][kHeads];
};
static_assert(kSmAlloc + sizeof(SoftX) + kHeads * sizeof(float) + 256 <= 232448, "shared memory budget of the exact kernel");

struct alignas(8) Barriers {
  uint64_t q_ready;
  uint64_t t_full[2], t_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_full;
  uint64_t sfa_ready;  // NVFP4-query mode: the query scales are in TMEM
};

// Key addressing in two halves so that the index load can be issued a tile
// ahead of its use: load_index() performs one unconditional, in-bounds load
// (the page-table entry or the top-k index of key position t, clamped into
// its row); key_slot() then turns that value into a slot id, or -1 for
// padding / positions past the sequence, and notes out-of-range ids.
__device__ __forceinline__ int32_t ldg_i32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// t / page_size for 0 <= t < 2^31
__device__ __forceinline__ int page_of(const Params& p, int t) {
  return static_cast<int>(div_magic(static_cast<uint32_t>(t), p.pg_magic, p.pg_shift));
}

// Key modes: kKeysAny decides paged or top-k from the arguments at run time;
// kKeysPaged and kKeysTopk fix it at compile time (the exact kernel is
// instantiated per mode, so each carries only its own addressing code), and
// kKeysPaged64 is paged with 64-token pages, a 64-key tile being one page
// (the page and the offset in it by shift and mask).
constexpr int kKeysAny = 0, kKeysPaged = 1, kKeysTopk = 2, kKeysPaged64 = 3;

template <int kMode = kKeysAny>
__device__ __forceinline__ bool topk_mode(const Params& p) {
  return kMode == kKeysTopk || (kMode == kKeysAny && p.topk != nullptr);
}

template <int kMode = kKeysAny>
__device__ __forceinline__ int32_t load_index(const Params& p, int b, int t) {
  if (topk_mode<kMode>(p)) {
    const int tc = min(max(t, 0), max(p.topk_n - 1, 0));
    return ldg_i32(p.topk + static_cast<int64_t>(b) * p.topk_n + tc);
  }
  const int pg = kMode == kKeysPaged64 ? max(t, 0) >> 6 : page_of(p, max(t, 0));
  const int pi = min(pg, static_cast<int>(p.pt_stride) - 1);
  return ldg_i32(p.page_table + static_cast<int64_t>(b) * p.pt_stride + pi);
}

template <int kMode = kKeysAny>
__device__ __forceinline__ int64_t key_slot(const Params& p, int32_t idx, int t, int n_keys, bool& bad) {
  if (t >= n_keys) return -1;
  int64_t slot;
  if (topk_mode<kMode>(p)) {
    if (idx < 0) return -1;  // padding entry
    slot = idx;
  } else {
    const int pg = kMode == kKeysPaged64 ? t >> 6 : page_of(p, t);
    if (pg >= p.pt_stride || idx < 0) {
      bad = true;
      return -1;
    }
    slot = kMode == kKeysPaged64 ? static_cast<int64_t>(idx) * 64 + (t & 63)
                                 : static_cast<int64_t>(idx) * p.page_size + (t - pg * p.page_size);
  }
  if (slot >= p.num_slots) {
    bad = true;
    return -1;
  }
  return slot;
}

// 16-byte read-only load issued where it is written (volatile): the raw
// record bytes of the next tile must be in flight while this tile converts,
// and an ordinary load may be scheduled next to its first use.
// Packed fp32 pair arithmetic (one instruction for two lanes of work) and a
// three-input max, to thin the softmax's instruction stream.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpk2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint4 ldg16(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

// bf16x2 -> f16x2; exact inside the f16 range (8 <= 11 significant bits),
// saturating to +-65504 outside it.  `amax` collects the magnitudes, so a
// value that saturated can be flagged.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_sat(uint32_t v, float& amax) {
  float lo, hi;
  bf16x2_to_f32(v, lo, hi);
  amax = max3(amax, fabsf(lo), fabsf(hi));
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t byte_of(const uint4& v, int i) {
  const uint32_t w = (i < 4) ? v.x : (i < 8) ? v.y : (i < 12) ? v.z : v.w;
  return (w >> (8 * (i & 3))) & 0xFFu;
}

// One 16-byte code segment (32 features, two 16-feature blocks with scale
// bytes s0, s1) -> four 16-byte units of c*s in f16, stored at feature units
// u0..u0+3 of a 128-byte-swizzled row (unit u of row `row` in chunk u/8).
__device__ __forceinline__ void dequant_segment(const uint4& c, uint32_t s0, uint32_t s1, uint32_t tile,
                                                int u0, int row) {
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
  const uint32_t f0 = e4m3x2_to_f16x2(s0 | (s0 << 8)), f1 = e4m3x2_to_f16x2(s1 | (s1 << 8));
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t h[4];
    e2m1x8_to_f16x8(words[w], h);
    const uint32_t f = (w < 2) ? f0 : f1;
    const int u = u0 + w;
    const uint32_t addr = tile + (u >> 3) * kChunk + row * 128 + (((u & 7) ^ (row & 7)) << 4);
    sts128(addr, make_uint4(hmul2_u32(h[0], f), hmul2_u32(h[1], f), hmul2_u32(h[2], f), hmul2_u32(h[3], f)));
  }
}

// ------------------------------------------------------------ dequantisation
// Thread = (key k of the tile, part Q): Q = 0 writes V units 0..23, Q = 1
// T units 0..15 and V units 24..31, Q = 2 T units 16..31 and the RoPE chunk
// (V = latent features [256 rank, +256), T = the other 256; a unit is 8
// features).  Each thread loads the raw bytes of its part with 16-byte loads
// straight from global memory into one register buffer, in two groups, each
// reloaded with the next tile's bytes as soon as this tile's conversion has
// read it: the loads land while the thread converts the rest and waits for
// the next tile's operand buffers (one buffer, and one copy of the conversion
// code, ran faster than two buffers a tile apart; a bulk L2 prefetch of each
// record, issued per key, made the kernel slower and was dropped).

template <int Q, int kRecord>
struct RawPart {
  static constexpr int kRope = (kRecord == 368) ? 4 : 8;  // RoPE segments
  static constexpr int kN = (Q == 0) ? 7 : (Q == 1) ? 8 : 5 + kRope;
  uint4 v[kN];
};

template <int Q, int kRecord>
__device__ __forceinline__ void load_part(RawPart<Q, kRecord>& r, const uint8_t* rec, int rank) {
  const int other = 1 - rank;
  if constexpr (Q == 0) {
#pragma unroll
    for (int i = 0; i < 6; ++i) r.v[i] = ldg16(rec + 128 * rank + 16 * i);
    r.v[6] = ldg16(rec + 256 + 16 * rank);
  } else if constexpr (Q == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) r.v[i] = ldg16(rec + 128 * other + 16 * i);
    r.v[4] = ldg16(rec + 256 + 16 * other);
#pragma unroll
    for (int i = 0; i < 2; ++i) r.v[5 + i] = ldg16(rec + 128 * rank + 96 + 16 * i);
    r.v[7] = ldg16(rec + 256 + 16 * rank);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) r.v[i] = ldg16(rec + 128 * other + 64 + 16 * i);
    r.v[4] = ldg16(rec + 256 + 16 * other);
#pragma unroll
    for (int i = 0; i < RawPart<Q, kRecord>::kRope; ++i) r.v[5 + i] = ldg16(rec + 288 + 16 * i);
  }
}

// Group g of part Q's raw bytes (g = 0: the registers the first conversion
// step reads, g = 1: the rest), from record `rec`, or zeros for rec == null.
template <int Q, int kRecord>
__device__ __forceinline__ void load_group(RawPart<Q, kRecord>& r, const uint8_t* rec, int rank, int g) {
  const int other = 1 - rank;
  const uint4 z = make_uint4(0, 0, 0, 0);
  if constexpr (Q == 0) {
    if (g == 0) {
#pragma unroll
      for (int i = 0; i < 3; ++i) r.v[i] = rec ? ldg16(rec + 128 * rank + 16 * i) : z;
    } else {
#pragma unroll
      for (int i = 3; i < 6; ++i) r.v[i] = rec ? ldg16(rec + 128 * rank + 16 * i) : z;
      r.v[6] = rec ? ldg16(rec + 256 + 16 * rank) : z;
    }
  } else if constexpr (Q == 1) {
    if (g == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) r.v[i] = rec ? ldg16(rec + 128 * other + 16 * i) : z;
      r.v[4] = rec ? ldg16(rec + 256 + 16 * other) : z;
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) r.v[5 + i] = rec ? ldg16(rec + 128 * rank + 96 + 16 * i) : z;
      r.v[7] = rec ? ldg16(rec + 256 + 16 * rank) : z;
    }
  } else {
    if (g == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) r.v[i] = rec ? ldg16(rec + 128 * other + 64 + 16 * i) : z;
      r.v[4] = rec ? ldg16(rec + 256 + 16 * other) : z;
    } else {
#pragma unroll
      for (int i = 0; i < RawPart<Q, kRecord>::kRope; ++i) r.v[5 + i] = rec ? ldg16(rec + 288 + 16 * i) : z;
    }
  }
}

struct DeqCtx {
  const Params& p;
  Barriers* bars;
  volatile int* abort_s;
  uint32_t sV, sT;
  int rank, b, tile0, nt, n_keys, k;
};

// Convert part Q of key k of tile j (raw bytes in r, or zeros for a padding
// key) into the tile's operand buffers.  False if a wait gave up.
template <int Q, int kRecord>
__device__ __forceinline__ bool convert_part(const DeqCtx& c, int j, RawPart<Q, kRecord>& r, float& rope_max,
                                             bool more, const uint8_t* nrec) {
  uint32_t* err = c.p.error_word;
  Barriers& bars = *c.bars;
  const int k = c.k;
  const uint32_t tV = c.sV + (j & 1) * kVBytes, tT = c.sT + (j & 1) * kTBytes;
  const uint32_t ph = ((j >> 1) & 1) ^ 1;  // phase in which the previous user released the buffer
  if constexpr (Q == 0) {
    if (!bar_wait(&bars.v_empty[j & 1], ph, err, c.abort_s)) return false;
#pragma unroll
    for (int i = 0; i < 3; ++i) dequant_segment(r.v[i], byte_of(r.v[6], 2 * i), byte_of(r.v[6], 2 * i + 1), tV, 4 * i, k);
    if (more) load_group<Q, kRecord>(r, nrec, c.rank, 0);
#pragma unroll
    for (int i = 3; i < 6; ++i) dequant_segment(r.v[i], byte_of(r.v[6], 2 * i), byte_of(r.v[6], 2 * i + 1), tV, 4 * i, k);
    if (more) load_group<Q, kRecord>(r, nrec, c.rank, 1);
    fence_async_smem();
    mbar_arrive(&bars.v_full[j & 1]);
  } else if constexpr (Q == 1) {
    if (!bar_wait(&bars.t_empty[j & 1], ph, err, c.abort_s)) return false;
#pragma unroll
    for (int i = 0; i < 4; ++i) dequant_segment(r.v[i], byte_of(r.v[4], 2 * i), byte_of(r.v[4], 2 * i + 1), tT, 4 * i, k);
    if (more) load_group<Q, kRecord>(r, nrec, c.rank, 0);
    fence_async_smem();
    mbar_arrive(&bars.t_full[j & 1]);
    if (!bar_wait(&bars.v_empty[j & 1], ph, err, c.abort_s)) return false;
#pragma unroll
    for (int i = 0; i < 2; ++i)
      dequant_segment(r.v[5 + i], byte_of(r.v[7], 12 + 2 * i), byte_of(r.v[7], 13 + 2 * i), tV, 24 + 4 * i, k);
    if (more) load_group<Q, kRecord>(r, nrec, c.rank, 1);
    fence_async_smem();
    mbar_arrive(&bars.v_full[j & 1]);
  } else {
    if (!bar_wait(&bars.t_empty[j & 1], ph, err, c.abort_s)) return false;
    const uint32_t rope_row = tT + 4 * kChunk + k * 128;
    {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dequant_segment(r.v[i], byte_of(r.v[4], 8 + 2 * i), byte_of(r.v[4], 9 + 2 * i), tT, 16 + 4 * i, k);
      if (more) load_group<Q, kRecord>(r, nrec, c.rank, 0);
      if constexpr (kRecord == 368) {  // e4m3 -> f16, exact
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 x = r.v[5 + i];
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 o = make_uint4(e4m3x2_to_f16x2(w[2 * h] & 0xFFFFu), e4m3x2_to_f16x2(w[2 * h] >> 16),
                                       e4m3x2_to_f16x2(w[2 * h + 1] & 0xFFFFu), e4m3x2_to_f16x2(w[2 * h + 1] >> 16));
            const int u = 2 * i + h;
            sts128(rope_row + ((u ^ (k & 7)) << 4), o);
          }
        }
      } else {  // bf16 -> f16
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = r.v[5 + u];
          sts128(rope_row + ((u ^ (k & 7)) << 4),
                 make_uint4(bf16x2_to_f16x2_sat(x.x, rope_max), bf16x2_to_f16x2_sat(x.y, rope_max),
                            bf16x2_to_f16x2_sat(x.z, rope_max), bf16x2_to_f16x2_sat(x.w, rope_max)));
        }
      }
      if (more) load_group<Q, kRecord>(r, nrec, c.rank, 1);
    }
    fence_async_smem();
    mbar_arrive(&bars.t_full[j & 1]);
  }
  return true;
}

// The dequantisation loop of one thread.  Returns whether an out-of-range
// page or slot id was met; flags a RoPE value beyond the f16 range.
template <int Q, int kRecord, int kMode>
__device__ bool dequant_role(const DeqCtx& c) {
  const Params& p = c.p;
  bool bad = false;
  float rope_max = 0.f;
  auto slot_of = [&](int j, int32_t idx) {
    return key_slot<kMode>(p, idx, (c.tile0 + j) * kTok + c.k, c.n_keys, bad);
  };
  auto index_of = [&](int j) { return load_index<kMode>(p, c.b, (c.tile0 + j) * kTok + c.k); };

  const int nt = c.nt;
  const int64_t s_cur = nt > 0 ? slot_of(0, index_of(0)) : -1;  // tile 0
  int64_t s_nxt = nt > 1 ? slot_of(1, index_of(1)) : -1;  // tile j + 1
  int32_t i_2 = nt > 2 ? index_of(2) : -1;                // index of tile j + 2
  RawPart<Q, kRecord> ra;
  // a padding key converts from zero bytes: codes and scale 0 give +0, the
  // bits of an empty operand row
  auto load_or_zero = [&](RawPart<Q, kRecord>& r, int64_t slot) {
    if (slot >= 0) {
      load_part(r, p.cache + slot * kRecord, c.rank);
    } else {
#pragma unroll
      for (int i = 0; i < RawPart<Q, kRecord>::kN; ++i) r.v[i] = make_uint4(0, 0, 0, 0);
    }
  };
  load_or_zero(ra, s_cur);
  // one buffer: tile j converts from `ra`, then tile j+1's bytes load into
  // it; the loads land while the thread waits for the next tile's buffers
#pragma unroll 1
  for (int j = 0; j < nt; ++j) {
    const int64_t s_2 = (j + 2 < nt) ? slot_of(j + 2, i_2) : -1;
    i_2 = (j + 3 < nt) ? index_of(j + 3) : -1;
    if constexpr (kMode == kKeysTopk) {
      // top-k keys are scattered records, each a DRAM access: this part's
      // bytes of tile j + 2 go to L2 while tile j converts (6 % on 32 x 2048
      // of 65,536 keys, measured; paged tiles do not need it)
      if (s_2 >= 0) {
        // first and last byte of the part's main span, both inside the record:
        // latent codes [128 r, +128) for parts 0 and 1, scales and RoPE
        // [256, kRecord - 16) for part 2
        constexpr int kSpan = (Q == 2) ? kRecord - 16 - 256 - 1 : 127;
        const uint8_t* rec = p.cache + s_2 * kRecord + (Q == 2 ? 256 : 128 * (Q == 0 ? c.rank : 1 - c.rank));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(rec));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + kSpan));
      }
    }
    // the next tile's bytes load into each register group as soon as this
    // tile's conversion has read it
    if (!convert_part<Q, kRecord>(c, j, ra, rope_max, j + 1 < nt, s_nxt >= 0 ? p.cache + s_nxt * kRecord : nullptr))
      break;
    s_nxt = s_2;
  }
  if (rope_max > 65504.f) flag_error(p.error_word, MLA_DEVERR_RANGE);
  return bad;
}

// The online softmax over an item's tiles (thread = head row; warps 0..3
// read their lane quarter of the scores): raw scores from TMEM, masking of
// padding keys, lazy max raise with an O rescale, probabilities as f16 into
// the scores' columns for P.V, running row sum.  The NVFP4-query kernel's
// (kSplit = 1; the exact kernel uses softmax_quad).
//
// kSplit = 2: two threads per head, thread `half` taking keys [32 half,
// 32 half + 32) of each tile and O columns [128 half, 128 half + 128) for
// the rescale; the halves exchange their tile maxima through `x` (so both
// take the same reference and the same rescale decisions) and keep
// separate row sums.  The exchange also orders the halves' score loads
// before the P stores that overwrite them.
template <int kSplit, int kMode>
__device__ __forceinline__ void softmax_tiles(const Params& p, Barriers& bars, volatile int& abort_s, uint32_t tmem,
                                              uint32_t lane_off, int b, int tile0, int nt, int n_keys,
                                              float score_scale, bool& ok, float& m_run, float& l_run, int half,
                                              SoftX* x_ch, int hr) {
  constexpr int kKeys = kTok / kSplit;  // keys of a tile per thread
  uint32_t* err = p.error_word;
  const int lane = threadIdx.x & 31;
  const int kb = half * kKeys;  // first key of this thread's part of a tile
  // per-tile validity: lane checks keys kb + lane (and kb + lane + 32)
  int32_t ia = load_index<kMode>(p, b, tile0 * kTok + kb + lane);
  int32_t ib = kSplit == 1 ? load_index<kMode>(p, b, tile0 * kTok + 32 + lane) : 0;
  for (int j = 0; j < nt; ++j) {
    const int pb = j & 1;
    const int key = (tile0 + j) * kTok + kb + lane;
    bool badv = false;
    const unsigned va = __ballot_sync(0xffffffffu, key_slot<kMode>(p, ia, key, n_keys, badv) >= 0);
    const unsigned vb = kSplit == 1 ? __ballot_sync(0xffffffffu, key_slot<kMode>(p, ib, key + 32, n_keys, badv) >= 0)
                                    : 0xffffffffu;
    if (j + 1 < nt) {
      ia = load_index<kMode>(p, b, key + kTok);
      if (kSplit == 1) ib = load_index<kMode>(p, b, key + kTok + 32);
    }
    if (!bar_wait(&bars.s_full[pb], (j >> 1) & 1, err, &abort_s)) {
      ok = false;
      break;
    }
    tc_fence_after();
    // raw scores: all loads in flight, one wait
    float x[kKeys];
    {
      uint32_t v[kKeys / 16][16];
#pragma unroll
      for (int c = 0; c < kKeys / 16; ++c) tmem_ld16(tmem + lane_off + col_s(pb) + kb + 16 * c, v[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kKeys; ++c) x[c] = __uint_as_float(v[c >> 4][c & 15]);
    }
    // max of the raw scores (score_scale > 0), padding keys at -inf; the
    // scale is applied inside the exponent below
    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if ((va & vb) != 0xffffffffu) {
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        const unsigned m = c < 32 ? va : vb;
        x[c] = ((m >> (c & 31)) & 1u) ? x[c] : -INFINITY;
      }
    }
#pragma unroll
    for (int c = 0; c < kKeys; c += 2) mq[(c >> 1) & 3] = max3(mq[(c >> 1) & 3], x[c], x[c + 1]);
    float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * score_scale;  // log2 units
    if constexpr (kSplit == 2) {
      // the partner has read this slot's previous value once its P of the
      // previous tile is in
      if (j > 0 && !bar_wait(&bars.p_full[(j - 1) & 1], ((j - 1) >> 1) & 1, err, &abort_s)) {
        ok = false;
        break;
      }
      x_ch->v[half][hr] = mx;
      tc_fence_before();
      mbar_arrive(&x_ch->mx_full[pb]);
      if (!bar_wait(&x_ch->mx_full[pb], (j >> 1) & 1, err, &abort_s)) {
        ok = false;
        break;
      }
      tc_fence_after();
      mx = fmaxf(mx, x_ch->v[half ^ 1][hr]);
    }
    float m_use = m_run, alpha = 1.f;
    const bool raise = mx > m_run + kRescaleThreshold;
    if (raise) {
      m_use = mx + kRefHeadroom;
      alpha = ex2_approx(m_run - m_use);
    }
    // an O rescale must follow every earlier P.V and precede PV(j).
    // PV(j-1) and PV(j-2) come from different issuers; each issuer's
    // earlier P.V products retire before its later ones.
    if (__any_sync(0xffffffffu, raise && j > 0)) {
      if (!bar_wait(&bars.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err, &abort_s) ||
          (j >= 2 && !bar_wait(&bars.pv_done[j & 1], ((j - 2) >> 1) & 1, err, &abort_s))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 4
      for (int c = 0; c < 256 / kSplit; c += 16) {
        uint32_t v[16];
        const uint32_t col = kTO + half * (256 / kSplit) + c;
        tmem_ld16(tmem + lane_off + col, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st16(tmem + lane_off + col, v);
      }
      tmem_st_wait();
    }
    m_run = m_use;
    const float m_ref = (m_use == -INFINITY) ? 0.f : m_use;  // no valid key so far
    // exponent arguments and row sums two at a time
    const uint64_t sc2 = pk2(score_scale, score_scale), nm2 = pk2(-m_ref, -m_ref);
    uint64_t ls2[4] = {0, 0, 0, 0};  // packed (+0, +0) partial sums
    uint32_t pv[kKeys / 2];
#pragma unroll
    for (int i = 0; i < kKeys / 2; ++i) {
      float a0, a1;
      unpk2(fma2(pk2(x[2 * i], x[2 * i + 1]), sc2, nm2), a0, a1);
      const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
      ls2[i & 3] = add2(ls2[i & 3], pk2(p0, p1));
      pv[i] = pack_f16(p0, p1);  // P <= 2^15.5 (lazy reference), f16 operand
    }
    float ls[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpk2(ls2[i], ls[2 * i], ls[2 * i + 1]);
    l_run = l_run * alpha + (((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7])));
    // P(j) over S(j): the buffer's previous P was read by PV(j-2), which
    // ran before QK(j) wrote S(j); key pair i of the tile in column i
#pragma unroll
    for (int c = 0; c < kKeys / 32; ++c) {
      uint32_t v0[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v0[i] = pv[16 * c + i];
      tmem_st16(tmem + lane_off + col_s(pb) + kb / 2 + 16 * c, v0);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars.p_full[pb]);
  }
}

// The partial output of an item (thread = head row): O half / l, scaled by
// gs, and the LSE, as the final bf16 output when the item is its sequence's
// only one, else as an fp32 partial row for the merge.  TMEM loads are
// warp-collective, so every lane loads; only stores depend on the head.
// kSplit = 2: thread `half` writes O columns [128 half, 128 half + 128) of
// this CTA's 256 with the row sum of both halves (exchanged through x).
template <int kSplit>
__device__ __forceinline__ void write_partial(const Params& p, uint32_t tmem, uint32_t lane_off, bool ok, int nt,
                                              float m_run, float l_run, float gs, int64_t row0, int b, int head,
                                              bool head_ok, bool direct, int rank, int half, SoftX* x_ch, int hr,
                                              volatile int* abort_s) {
  if constexpr (kSplit == 2) {
    if (nt > 0) {
      x_ch->v[half][hr] = l_run;
      mbar_arrive(&x_ch->fin);
      if (bar_wait(&x_ch->fin, 0, p.error_word, abort_s))
        l_run += x_ch->v[half ^ 1][hr];
      else
        ok = false;
    }
  }
  // partial output of this split: O half / l (scaled by gs), lse.  TMEM
  // loads are warp-collective, so every lane loads; only stores depend on
  // the head.
  const bool live = __all_sync(0xffffffffu, ok) && nt > 0;
  const bool have = live && l_run > 0.f;
  const float f = have ? gs / l_run : 0.f;
  const int64_t row = row0 + head;
  // For a sequence's only item the merge is the identity (weight
  // exp(0) = 1, sum 1): the final bf16 output and the LSE are written here
  // and no merge touches the sequence.
  constexpr int kCols = 256 / kSplit;
  float4* dst = reinterpret_cast<float4*>(p.part_o + row * 512 + 256 * rank + kCols * half);
  uint4* dst_bf = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * p.num_heads + head) * 512 + 256 * rank +
                                           kCols * half);
  if (live) tc_fence_after();
#pragma unroll 2
  for (int c = 0; c < kCols; c += 16) {
    uint32_t v[16];
    if (live) {
      tmem_ld16(tmem + lane_off + kTO + kCols * half + c, v);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0u;
    }
    if (head_ok) {
      if (direct) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * f, __uint_as_float(v[2 * i + 1]) * f);
          w[i] = *reinterpret_cast<uint32_t*>(&h2);
        }
        dst_bf[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
        dst_bf[c / 8 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[c / 4 + i] = make_float4(__uint_as_float(v[4 * i]) * f, __uint_as_float(v[4 * i + 1]) * f,
                                       __uint_as_float(v[4 * i + 2]) * f, __uint_as_float(v[4 * i + 3]) * f);
      }
    }
  }
  if (head_ok && rank == 0 && half == 0) {
    const float l = have ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    if (!direct)
      p.part_lse[row] = l;
    else if (p.lse != nullptr)
      p.lse[static_cast<int64_t>(b) * p.num_heads + head] = l;
  }
}

// The exact kernel's online softmax over an item's tiles, with four threads
// per pair of heads: the warp of TMEM subpartition q and group g (warps
// 0..3: g = 0, 12..15: g = 1) takes heads 32q + 16g .. +15, and its thread t
// heads 32q + 16g + t/4 and + 8, keys 8i + 2(t%4) and + 1 (i = 0..7) of each
// 64-key tile, the tcgen05.ld 16x256b layout.  A head's four threads are
// lanes of one warp: they share the tile maxima (and, at the end, the row
// sums) by shuffles, and each writes its keys' P pairs into the columns the
// 16x128b store gives it, which are its own (key pair k in column k).
// Otherwise as softmax_tiles: masking of padding keys, lazy reference raise
// with an O rescale, P as f16 for P.V, running row sums.
template <int kMode>
__device__ __forceinline__ void softmax_quad(const Params& p, Barriers& bars, volatile int& abort_s, uint32_t tmem,
                                             uint32_t lane_base, int b, int tile0, int nt, int n_keys,
                                             const float (&score_scale)[2], bool& ok, float (&m_run)[2],
                                             float (&l_run)[2]) {
  uint32_t* err = p.error_word;
  const int lane = threadIdx.x & 31, kq = 2 * (lane & 3);  // the thread's first key of each 8
  // per-tile validity: lane checks keys lane and 32 + lane
  int32_t ia = load_index<kMode>(p, b, tile0 * kTok + lane);
  int32_t ib = load_index<kMode>(p, b, tile0 * kTok + 32 + lane);
  for (int j = 0; j < nt; ++j) {
    const int pb = j & 1;
    const int key = (tile0 + j) * kTok + lane;
    bool badv = false;
    const unsigned va = __ballot_sync(0xffffffffu, key_slot<kMode>(p, ia, key, n_keys, badv) >= 0);
    const unsigned vb = __ballot_sync(0xffffffffu, key_slot<kMode>(p, ib, key + 32, n_keys, badv) >= 0);
    if (j + 1 < nt) {
      ia = load_index<kMode>(p, b, key + kTok);
      ib = load_index<kMode>(p, b, key + kTok + 32);
    }
    if (!bar_wait(&bars.s_full[pb], (j >> 1) & 1, err, &abort_s)) {
      ok = false;
      break;
    }
    tc_fence_after();
    // raw scores of both heads: x[h][2i + e] is key 8i + kq + e
    float x[2][16];
    {
      uint32_t v[32];
      tmem_ld_16x256b_x8(tmem + lane_base + col_s(pb), v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[0][2 * i] = __uint_as_float(v[4 * i]);
        x[0][2 * i + 1] = __uint_as_float(v[4 * i + 1]);
        x[1][2 * i] = __uint_as_float(v[4 * i + 2]);
        x[1][2 * i + 1] = __uint_as_float(v[4 * i + 3]);
      }
    }
    // padding keys at -inf; the maxima of the raw scores (score_scale > 0),
    // over the head's four threads; the scale is applied in the exponent
    if ((va & vb) != 0xffffffffu) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 8 * i + kq + e;
          if (!(((k < 32 ? va : vb) >> (k & 31)) & 1u)) {
            x[0][2 * i + e] = -INFINITY;
            x[1][2 * i + e] = -INFINITY;
          }
        }
    }
    float mx[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float m0 = max3(x[h][0], x[h][1], x[h][2]), m1 = max3(x[h][3], x[h][4], x[h][5]);
      m0 = max3(m0, x[h][6], x[h][7]);
      m1 = max3(m1, x[h][8], x[h][9]);
      m0 = max3(m0, x[h][10], x[h][11]);
      m1 = max3(m1, x[h][12], x[h][13]);
      float m = max3(m0, m1, fmaxf(x[h][14], x[h][15]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      mx[h] = m * score_scale[h];  // log2 units
    }
    float m_use[2], alpha[2];
    bool raise = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m_use[h] = m_run[h];
      alpha[h] = 1.f;
      if (mx[h] > m_run[h] + kRescaleThreshold) {
        m_use[h] = mx[h] + kRefHeadroom;
        alpha[h] = ex2_approx(m_run[h] - m_use[h]);
        raise = true;
      }
    }
    // an O rescale must follow every earlier P.V and precede PV(j).
    // PV(j-1) and PV(j-2) come from different issuers; each issuer's
    // earlier P.V products retire before its later ones.
    if (__any_sync(0xffffffffu, raise && j > 0)) {
      if (!bar_wait(&bars.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err, &abort_s) ||
          (j >= 2 && !bar_wait(&bars.pv_done[j & 1], ((j - 2) >> 1) & 1, err, &abort_s))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 256; c += 64) {
        uint32_t v[32];
        tmem_ld_16x256b_x8(tmem + lane_base + kTO + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha[(i >> 1) & 1]);
        tmem_st_16x256b_x8(tmem + lane_base + kTO + c, v);
      }
      tmem_st_wait();
    }
    // probabilities two at a time: x * score_scale - m_use, P <= 2^15.5
    // (lazy reference), f16 operand pairs; the row sums in packed halves
    uint32_t pv[16];  // pv[2i + h]: head h, key pair 8i + kq (column 4i + kq / 2)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m_run[h] = m_use[h];
      const float m_ref = (m_use[h] == -INFINITY) ? 0.f : m_use[h];  // no valid key so far
      const uint64_t sc2 = pk2(score_scale[h], score_scale[h]), nm2 = pk2(-m_ref, -m_ref);
      uint64_t ls2[2] = {0, 0};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float a0, a1;
        unpk2(fma2(pk2(x[h][2 * i], x[h][2 * i + 1]), sc2, nm2), a0, a1);
        const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
        ls2[i & 1] = add2(ls2[i & 1], pk2(p0, p1));
        pv[2 * i + h] = pack_f16(p0, p1);
      }
      float s0, s1, s2, s3;
      unpk2(ls2[0], s0, s1);
      unpk2(ls2[1], s2, s3);
      l_run[h] = l_run[h] * alpha[h] + ((s0 + s1) + (s2 + s3));
    }
    // P(j) over S(j): the warp's own lanes, read above; the buffer's
    // previous P was read by PV(j-2), which ran before QK(j) wrote S(j)
    tmem_st_16x128b_x8(tmem + lane_base + col_s(pb), pv);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars.p_full[pb]);
  }
}

// The output of an item for softmax_quad's heads (thread: heads `head0`
// and head0 + 8, O columns 8i + 2(t%4), +1 of each 64): O / l with the row
// sums of the head's four threads, scaled by gs, and the LSE, as the final
// bf16 output when the item is its sequence's only one, else as an fp32
// partial row for the merge.  TMEM loads are warp-collective, so every lane
// loads; only stores depend on the head.
__device__ __forceinline__ void write_partial_quad(const Params& p, uint32_t tmem, uint32_t lane_base, bool ok, int nt,
                                                   const float (&m_run)[2], float (&l_run)[2], float gs,
                                                   int64_t row0, int b, int head0, bool direct, int rank) {
  const int lane = threadIdx.x & 31, kq = 2 * (lane & 3);
  const bool live = __all_sync(0xffffffffu, ok) && nt > 0;
  float f[2];
  bool have[2], head_ok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_run[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l_run[h] = l;
    have[h] = live && l > 0.f;
    f[h] = have[h] ? gs / l : 0.f;
    head_ok[h] = head0 + 8 * h < p.num_heads;
  }
  if (live) tc_fence_after();
#pragma unroll 1
  for (int c = 0; c < 256; c += 64) {
    uint32_t v[32];
    if (live) {
      tmem_ld_16x256b_x8(tmem + lane_base + kTO + c, v);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!head_ok[h]) continue;
      const int head = head0 + 8 * h;
      if (direct) {
        __nv_bfloat16* dst = p.out + (static_cast<int64_t>(b) * p.num_heads + head) * 512 + 256 * rank + c + kq;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[4 * i + 2 * h]) * f[h],
                                                    __uint_as_float(v[4 * i + 2 * h + 1]) * f[h]);
          *reinterpret_cast<__nv_bfloat162*>(dst + 8 * i) = h2;
        }
      } else {
        float* dst = p.part_o + (row0 + head) * 512 + 256 * rank + c + kq;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float2*>(dst + 8 * i) =
              make_float2(__uint_as_float(v[4 * i + 2 * h]) * f[h], __uint_as_float(v[4 * i + 2 * h + 1]) * f[h]);
      }
    }
  }
  if (rank == 0 && (lane & 3) == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!head_ok[h]) continue;
      const int head = head0 + 8 * h;
      const float l = have[h] ? (m_run[h] + log2f(l_run[h])) * kLn2 : -INFINITY;
      if (!direct)
        p.part_lse[row0 + head] = l;
      else if (p.lse != nullptr)
        p.lse[static_cast<int64_t>(b) * p.num_heads + head] = l;
    }
  }
}

template <int kRecord, int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsTc, 1) decode_tc_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ SoftX xch;
  __shared__ float score_scale_s[kHeads];  // per head row: the softmax scale with its query's sigma
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x & 1;
  const int hg = blockIdx.z;
  // work item: (sequence b, key tiles [tile0, tile0 + nt)), where its
  // partial output goes (first row of its heads), and whether it is the
  // sequence's only item (then it writes out and lse itself)
  int b, tile0, per;
  int64_t row0;
  bool direct;
  if (p.plan_items != nullptr) {
    // launched as a programmatic dependent of the plan kernel: its tables
    // are read only once that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int item = blockIdx.x >> 1;
    if (item >= p.plan_hdr[0]) return;  // the plan has fewer items than the grid: the whole CTA leaves
    const int2 it = p.plan_items[item];
    if (it.x < 0 || it.x >= p.batch || it.y < 0) {  // not a plan of this batch: flag it, touch nothing
      if (threadIdx.x == 0) flag_error(p.error_word, MLA_DEVERR_BOUNDS);
      return;
    }
    const int2 sq = p.plan_seqs[it.x];
    b = it.x;
    per = p.plan_hdr[1];
    tile0 = it.y * per;
    direct = sq.x < 0;
    row0 = direct ? 0 : static_cast<int64_t>(sq.x + it.y) * p.num_heads;
  } else {
    const int split = blockIdx.x >> 1;
    b = blockIdx.y;
    const int n_keys_u = topk_mode<kMode>(p) ? p.topk_n : max(0, p.seq_lens[b]);
    per = ((n_keys_u + kTok - 1) / kTok + p.splits - 1) / p.splits;
    tile0 = split * per;
    direct = p.splits == 1;
    row0 = (static_cast<int64_t>(b) * p.splits + split) * p.num_heads;
  }
  const int n_keys = topk_mode<kMode>(p) ? p.topk_n : max(0, p.seq_lens[b]);
  const int n_tiles_all = n_keys / kTok + (n_keys % kTok != 0);
  const int nt = max(0, min(n_tiles_all, tile0 + per) - tile0);
  uint32_t* err = p.error_word;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + kSmQ), sV = smem_u32(smem + kSmV), sT = smem_u32(smem + kSmT);

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bars.q_ready, 256);  // both softmax halves stage part of Q
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.t_full[i], 128);
      mbar_init(&bars.t_empty[i], 1);
      mbar_init(&bars.v_full[i], 128);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 256);
      mbar_init(&xch.mx_full[i], 256);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.o_full, 2);
    mbar_init(&xch.fin, 256);
    mbar_init(&xch.qx, 256);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == kMmaWarp || warp == kMmaWarp2) {
    // ----------------------------------------------------------------- MMA
    // Two issuing threads: one thread issues tcgen05.mma at roughly one
    // instruction per 50 cycles, well below the tensor pipe's rate at N = 64,
    // so tiles alternate between two issuers.  Every buffer (scores, T, V)
    // is indexed by tile parity, so the issuer of parity p owns buffer p.
    const int par = (warp == kMmaWarp) ? 0 : 1;
    if (lane == 0 && nt > 0) {
      // Descriptors are formed once; a tile, chunk or K-step offset is added
      // to the start-address field (16-byte units, no carry: shared
      // addresses stay below 256 KB).
      const uint64_t dq = smem_desc_sw128(sQ, 0, 1024);
      const uint64_t dv = smem_desc_sw128(sV, 0, 1024);
      const uint64_t dt = smem_desc_sw128(sT, 0, 1024);
      const uint64_t dpv = smem_desc_sw128(sV, kChunk, 1024);
      bool ok = bar_wait(&bars.q_ready, 0, err, &abort_s);
      tc_fence_after();
      // latent chunk c of Q (TMEM for c < 3, shared memory otherwise) times
      // the K chunk at descriptor kd, into scores d.  The operand-form test
      // stays outside the K-steps: with it inside an unrolled K-step loop,
      // one K-step was observed to run with the previous step's A operand.
      // The issue loops stay rolled: with 128 SMs fetching this kernel's
      // instructions at once, unrolled issue code measured ~15 % slower.
      auto latent = [&](int c, uint64_t kd, uint32_t d) {
        if (c < 3) {
          const uint32_t a0 = tmem + kTQLat + 32 * c;
#pragma unroll 1
          for (int ks = 0; ks < 4; ++ks) mma_ts(d, a0 + 8 * ks, kd + 2 * ks, kIdescQK, 1u);
        } else {
          const uint64_t a0 = dq + static_cast<uint64_t>((c - 3) * (kQChunk / 16));
#pragma unroll 1
          for (int ks = 0; ks < 4; ++ks) mma_ss(d, a0 + 2 * ks, kd + 2 * ks, kIdescQK, 1u);
        }
      };
      auto issue_qk_t = [&](int j) -> bool {
        const int tb = j & 1;
        if (!bar_wait(&bars.t_full[tb], (j >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t d = tmem + col_s(tb);
        const uint64_t td = dt + tb * (kTBytes / 16);
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(d, tmem + kTQRope + 8 * kk, td + (4 * kChunk + 32 * kk) / 16, kIdescQK, kk > 0 ? 1u : 0u);
#pragma unroll 1
        for (int i = 0; i < 4; ++i) latent(4 * (1 - rank) + i, td + i * (kChunk / 16), d);
        mma_commit(&bars.t_empty[tb]);
        return true;
      };
      auto issue_qk_v = [&](int j) -> bool {
        const int vb = j & 1;
        if (!bar_wait(&bars.v_full[vb], (j >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t d = tmem + col_s(vb);
        const uint64_t vd = dv + vb * (kVBytes / 16);
#pragma unroll 1
        for (int i = 0; i < 4; ++i) latent(4 * rank + i, vd + i * (kChunk / 16), d);
        mma_commit(&bars.s_full[vb]);
        return true;
      };
      auto issue_pv = [&](int t) -> bool {
        const int pb = t & 1;
        if (!bar_wait(&bars.p_full[pb], (t >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint64_t vd = dpv + pb * (kVBytes / 16);
#pragma unroll 1
        for (int kk = 0; kk < kTok / 16; ++kk)
          mma_ts(tmem + kTO, tmem + col_s(pb) + 8 * kk, vd + (2048 * kk) / 16, kIdescPV, 1u);  // O starts at 0
        mma_commit(&bars.v_empty[pb]);
        mma_commit(&bars.pv_done[pb]);
        return true;
      };
      // per tile: the T part of the scores, the V part, then P.V once the
      // softmax has written P; the other issuer's tile fills the wait
      for (int j = par; ok && j < nt; j += 2) ok = issue_qk_t(j) && issue_qk_v(j) && issue_pv(j);
      mma_commit(&bars.o_full);
      bar_wait(&bars.o_full, 0, err, nullptr);  // both issuers' MMAs retired
    }
  } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // ---------------------------------------------------------- dequantise
    const int di = threadIdx.x - 32 * kDeqWarp0;
    const int k = di & 63, q = di >> 6;
    DeqCtx c{p, &bars, &abort_s, sV, sT, rank, b, tile0, nt, n_keys, k};
    bool bad;
    if (q == 0)
      bad = dequant_role<0, kRecord, kMode>(c);
    else if (q == 1)
      bad = dequant_role<1, kRecord, kMode>(c);
    else
      bad = dequant_role<2, kRecord, kMode>(c);
    if (bad && rank == 0 && q == 0) flag_error(err, MLA_DEVERR_BOUNDS);
  } else {
    // ------------------------------------------- softmax and epilogue
    // warps 0..3 (half 0) and 12..15 (half 1): two threads per head for the
    // query staging, warp w writing TMEM lanes 32 (w % 4) .. +32
    const int half = warp >= kSoftWarp2 ? 1 : 0;
    const int hr = (warp & 3) * 32 + lane;  // head row within the group
    const int head = hg * kHeads + hr;
    const bool head_ok = head < p.num_heads;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float gs = *p.gs;
    const bool gs_ok = scale_ok(gs);
    float score_scale = p.softmax_scale * gs * kLog2e;
    bool ok = true;
    if (nt > 0) {
      // Q -> f16 operands: TMEM [sigma*q_pe/gs, sigma*q_lat[0:192]], shared
      // memory sigma*q_lat[192:512] (swizzled rows).
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q + (static_cast<int64_t>(b) * p.num_heads + head) * 576);
      const float inv_gs = gs_ok ? 1.f / gs : 0.f;
      // Operand order of the 72 source units (8 bf16 each): positions 0..7
      // = q_pe (units 64..71), 8..31 = q_lat units 0..23 (TMEM, 4 columns a
      // unit), 32..71 = q_lat units 24..63 (shared memory chunks 0..4).
      // One pass in three batches of 24 loads converts with the given sigma
      // and returns max(|q_lat|, |q_pe/gs|).
      // Each half stages 36 of the units, in three batches of 12 loads.
      auto stage = [&](float sigma) -> float {
        float qmax = 0.f;
#pragma unroll 1
        for (int g = 0; g < 3; ++g) {
          const int ub = 36 * half + 12 * g;  // first unit position of the batch
          uint4 w[12];
#pragma unroll
          for (int i = 0; i < 12; ++i) {
            const int up = ub + i, u = up < 8 ? 64 + up : up - 8;
            w[i] = head_ok ? ldg16(qrow + 16 * u) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int i4 = 0; i4 < 12; i4 += 4) {
            uint32_t v[16];
#pragma unroll
            for (int i = i4; i < i4 + 4; ++i) {
              const int up = ub + i;
              const float f = up < 8 ? inv_gs : 1.f;
              const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
              for (int kx = 0; kx < 4; ++kx) {
                float lo, hi;
                bf16x2_to_f32(ws[kx], lo, hi);
                lo *= f;
                hi *= f;
                qmax = fmaxf(qmax, fmaxf(fabsf(lo), fabsf(hi)));
                v[4 * (i - i4) + kx] = pack_f16(lo * sigma, hi * sigma);
              }
            }
            const int up0 = ub + i4;
            if (up0 < 32) {
              tmem_st16(tmem + lane_off + kTQRope + 4 * up0, v);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int cu = up0 - 32 + i;
                sts128(sQ + (cu >> 3) * kQChunk + hr * 128 + (((cu & 7) ^ (hr & 7)) << 4),
                       make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
              }
            }
          }
        }
        return qmax;
      };
      // sigma = 2^-a with sigma*qmax < 2^16 (f16 max 65504); a = 0 unless a
      // query value reaches 2^15, in which case the row is staged again
      float qmax = stage(1.f);
      xch.v[half][hr] = qmax;  // the row's max over both halves' units
      mbar_arrive(&xch.qx);
      if (!bar_wait(&xch.qx, 0, err, &abort_s)) ok = false;
      qmax = fmaxf(qmax, xch.v[half ^ 1][hr]);
      const int qexp = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFFu) - 127;
      const int a_sh = max(0, min(qexp - 14, 100));
      if (__any_sync(0xffffffffu, a_sh > 0)) {
        tmem_st_wait();  // the first pass's TMEM stores land before the second's
        stage(__uint_as_float(static_cast<uint32_t>(127 - a_sh) << 23));
      }
      score_scale *= __uint_as_float(static_cast<uint32_t>(127 + a_sh) << 23);
      {  // O starts at zero: every P.V accumulates, whichever issuer runs first
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) tmem_st16(tmem + lane_off + kTO + 128 * half + c, z);
      }
      if (half == 0) score_scale_s[hr] = score_scale;
      fence_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.q_ready);
    }
    // the softmax and the output: four threads per pair of heads (the
    // 16-lane TMEM shapes), heads qh and qh + 8 of the group
    const int qh = (warp & 3) * 32 + 16 * half + (lane >> 2);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32 + 16 * half) << 16;
    float m_q[2] = {-INFINITY, -INFINITY}, l_q[2] = {0.f, 0.f};
    if (nt > 0) {
      // every head's scale is written before q_ready completes
      if (ok) ok = bar_wait(&bars.q_ready, 0, err, &abort_s);
      const float sc[2] = {score_scale_s[qh], score_scale_s[qh + 8]};
      if (ok) softmax_quad<kMode>(p, bars, abort_s, tmem, lane_base, b, tile0, nt, n_keys, sc, ok, m_q, l_q);
      if (ok) ok = bar_wait(&bars.o_full, 0, err, &abort_s);
    }
    write_partial_quad(p, tmem, lane_base, ok, nt, m_q, l_q, gs, row0, b, hg * kHeads + qh, direct, rank);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ================================================== NVFP4-query decode mode
// The absorbed query quantised to NVFP4 (16 features a block along the 576
// of a head, e4m3 scales, the query's global scale gs_q) in the staging
// pass, as the pages' caller-side query quantisation; the latent score
// product then runs on block-scaled fp4 tensor cores straight from the
// cache's codes and scales:
//   s_j = softmax_scale * gs_q * gs * ( sum_lat (c_q s_q)(c_k s_k)
//                                       + sum_rope (c_q s_q)(k_pe / gs) ),
// the first sum by eight kind::mxf4nvf4 MMAs (M 128 heads, N 64 keys, K 64)
// with the query scales and the keys' block scales in TMEM, the second by
// four f16 MMAs into the same accumulator: c_q s_q is exact in f16, k_pe / gs
// is rounded once to f16 (saturating, flagged MLA_DEVERR_RANGE).  P.V is the
// f16 product of the exact path.  Per key only this CTA's 256 output
// features are dequantised; the record's codes and scales go to shared
// memory as they are.
//
// Shared memory (1024-aligned parts): query codes 2 x 16 KB (128 heads x 256
// bytes, 128-byte swizzle), query scale tiles 4 KB; per tile parity: key
// codes 2 x 8 KB, RoPE f16 8 KB, key scale tiles 4 KB, V part 4 x 8 KB.
// TMEM: O [0,256), scores [256,384), query RoPE (f16) [384,416), query
// scales [416,448), key scales per parity [448,480) [480,512).
constexpr uint32_t kQ4Q = 0;
constexpr uint32_t kQ4Sfa = 32768;
constexpr uint32_t kQ4Buf0 = 36864;
constexpr uint32_t kQ4BufBytes = 61440;
constexpr uint32_t kQ4K = 0, kQ4Rope = 16384, kQ4Sfb = 24576, kQ4V = 28672;  // within a buffer
constexpr uint32_t kQ4SmBytes = kQ4Buf0 + 2 * kQ4BufBytes;
constexpr uint32_t kQ4SmAlloc = kQ4SmBytes + 1024;
static_assert(kQ4SmAlloc + 512 <= 232448, "shared memory budget");
constexpr uint32_t kQ4TRope = 384, kQ4TSfa = 416;
__host__ __device__ constexpr uint32_t q4_col_sfb(int buf) { return 448u + 32u * buf; }
constexpr uint32_t kIdescQ4 = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kTok >> 3) << 17) |
                              (static_cast<uint32_t>(kHeads >> 4) << 24);  // mxf4nvf4, e2m1 x e2m1, ue4m3 scales

// One 512-byte tile of 128 rows x 4 scale bytes, as tcgen05.cp 32x128b reads
// it: 32 rows of 16 bytes (byte (r % 32) * 16 + (r / 32) * 4 + block),
// four 8-row core matrices 128 bytes apart, no swizzle.
__device__ __forceinline__ uint64_t q4_sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__device__ __forceinline__ void q4_sf_copy(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void q4_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(kIdescQ4), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Raw record parts per key: 0 = all codes and scales (straight to the
// shared tiles), 1 = this CTA's 256 latent features and their scales
// (dequantised to the V part), 2 = the RoPE part (to f16, over gs).
template <int Q, int kRecord>
struct RawQ4 {
  static constexpr int kN = (Q == 0) ? 18 : (Q == 1) ? 9 : ((kRecord == 368) ? 4 : 8);
  uint4 v[kN];
};

template <int Q, int kRecord>
__device__ __forceinline__ void q4_load(RawQ4<Q, kRecord>& r, const uint8_t* rec, int rank) {
  if constexpr (Q == 0) {
#pragma unroll
    for (int i = 0; i < 18; ++i) r.v[i] = ldg16(rec + 16 * i);
  } else if constexpr (Q == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r.v[i] = ldg16(rec + 128 * rank + 16 * i);
    r.v[8] = ldg16(rec + 256 + 16 * rank);
  } else {
#pragma unroll
    for (int i = 0; i < RawQ4<Q, kRecord>::kN; ++i) r.v[i] = ldg16(rec + 288 + 16 * i);
  }
}

struct Q4Ctx {
  const Params& p;
  Barriers* bars;
  volatile int* abort_s;
  uint32_t sbuf;  // shared address of tile buffer 0
  int rank, b, tile0, nt, n_keys, k;
  float inv_gs;
};

// Write part Q of key k of tile j into the tile's buffers.  False if a wait
// gave up.
template <int Q, int kRecord>
__device__ __forceinline__ bool q4_convert(const Q4Ctx& c, int j, const RawQ4<Q, kRecord>& r, float& rope_max) {
  uint32_t* err = c.p.error_word;
  Barriers& bars = *c.bars;
  const int k = c.k;
  const uint32_t buf = c.sbuf + (j & 1) * kQ4BufBytes;
  const uint32_t ph = ((j >> 1) & 1) ^ 1;
  if constexpr (Q == 0) {
    if (!bar_wait(&bars.t_empty[j & 1], ph, err, c.abort_s)) return false;
#pragma unroll
    for (int u = 0; u < 16; ++u)  // codes: two 128-byte swizzled chunks
      sts128(buf + kQ4K + (u >> 3) * 8192 + k * 128 + (((u & 7) ^ (k & 7)) << 4), r.v[u]);
    const uint32_t w[8] = {r.v[16].x, r.v[16].y, r.v[16].z, r.v[16].w, r.v[17].x, r.v[17].y, r.v[17].z, r.v[17].w};
#pragma unroll
    for (int t = 0; t < 8; ++t)  // scales of blocks 4t..4t+3 into scale tile t
      sts32(buf + kQ4Sfb + 512 * t + (k & 31) * 16 + (k >> 5) * 4, w[t]);
    fence_async_smem();
    mbar_arrive(&bars.t_full[j & 1]);
  } else if constexpr (Q == 1) {
    if (!bar_wait(&bars.v_empty[j & 1], ph, err, c.abort_s)) return false;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      dequant_segment(r.v[i], byte_of(r.v[8], 2 * i), byte_of(r.v[8], 2 * i + 1), buf + kQ4V, 4 * i, k);
    fence_async_smem();
    mbar_arrive(&bars.v_full[j & 1]);
  } else {
    if (!bar_wait(&bars.t_empty[j & 1], ph, err, c.abort_s)) return false;
    const uint32_t row = buf + kQ4Rope + k * 128;
    auto put = [&](int u, const float (&f)[8]) {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = f[2 * i] * c.inv_gs, bb = f[2 * i + 1] * c.inv_gs;
        rope_max = max3(rope_max, fabsf(a), fabsf(bb));
        asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h[i]) : "f"(bb), "f"(a));
      }
      sts128(row + ((u ^ (k & 7)) << 4), make_uint4(h[0], h[1], h[2], h[3]));
    };
    if constexpr (kRecord == 368) {  // e4m3 -> f32 (exact) -> / gs -> f16
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t ws[4] = {r.v[i].x, r.v[i].y, r.v[i].z, r.v[i].w};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t two = ws[2 * hh + e];
            const uint32_t lo2 = e4m3x2_to_f16x2(two & 0xFFFFu), hi2 = e4m3x2_to_f16x2(two >> 16);
            const __half2 a = *reinterpret_cast<const __half2*>(&lo2), bq = *reinterpret_cast<const __half2*>(&hi2);
            f[4 * e] = __low2float(a);
            f[4 * e + 1] = __high2float(a);
            f[4 * e + 2] = __low2float(bq);
            f[4 * e + 3] = __high2float(bq);
          }
          put(2 * i + hh, f);
        }
      }
    } else {  // bf16 -> / gs -> f16
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t ws[4] = {r.v[u].x, r.v[u].y, r.v[u].z, r.v[u].w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) bf16x2_to_f32(ws[i], f[2 * i], f[2 * i + 1]);
        put(u, f);
      }
    }
    fence_async_smem();
    mbar_arrive(&bars.t_full[j & 1]);
  }
  return true;
}

template <int Q, int kRecord, int kMode>
__device__ bool q4_role(const Q4Ctx& c) {
  const Params& p = c.p;
  bool bad = false;
  float rope_max = 0.f;
  auto slot_of = [&](int j, int32_t idx) {
    return key_slot<kMode>(p, idx, (c.tile0 + j) * kTok + c.k, c.n_keys, bad);
  };
  auto index_of = [&](int j) { return load_index<kMode>(p, c.b, (c.tile0 + j) * kTok + c.k); };
  const int nt = c.nt;
  const int64_t s_cur = nt > 0 ? slot_of(0, index_of(0)) : -1;
  int64_t s_nxt = nt > 1 ? slot_of(1, index_of(1)) : -1;
  int32_t i_2 = nt > 2 ? index_of(2) : -1;
  RawQ4<Q, kRecord> ra;
  auto load_or_zero = [&](int64_t slot) {
    if (slot >= 0) {
      q4_load(ra, p.cache + slot * kRecord, c.rank);
    } else {
#pragma unroll
      for (int i = 0; i < RawQ4<Q, kRecord>::kN; ++i) ra.v[i] = make_uint4(0, 0, 0, 0);
    }
  };
  load_or_zero(s_cur);
#pragma unroll 1
  for (int j = 0; j < nt; ++j) {
    const int64_t s_2 = (j + 2 < nt) ? slot_of(j + 2, i_2) : -1;
    i_2 = (j + 3 < nt) ? index_of(j + 3) : -1;
    if (!q4_convert<Q, kRecord>(c, j, ra, rope_max)) break;
    if (j + 1 < nt) load_or_zero(s_nxt);
    s_nxt = s_2;
  }
  if (rope_max > 65504.f) flag_error(p.error_word, MLA_DEVERR_RANGE);
  return bad;
}

template <int kRecord, int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) decode_q4_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x & 1;
  const int hg = blockIdx.z;
  int b, tile0, per;
  int64_t row0;
  bool direct;
  if (p.plan_items != nullptr) {
    // launched as a programmatic dependent of the plan kernel: its tables
    // are read only once that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int item = blockIdx.x >> 1;
    if (item >= p.plan_hdr[0]) return;  // the plan has fewer items than the grid: the whole CTA leaves
    const int2 it = p.plan_items[item];
    if (it.x < 0 || it.x >= p.batch || it.y < 0) {  // not a plan of this batch: flag it, touch nothing
      if (threadIdx.x == 0) flag_error(p.error_word, MLA_DEVERR_BOUNDS);
      return;
    }
    const int2 sq = p.plan_seqs[it.x];
    b = it.x;
    per = p.plan_hdr[1];
    tile0 = it.y * per;
    direct = sq.x < 0;
    row0 = direct ? 0 : static_cast<int64_t>(sq.x + it.y) * p.num_heads;
  } else {
    const int split = blockIdx.x >> 1;
    b = blockIdx.y;
    const int n_keys_u = topk_mode<kMode>(p) ? p.topk_n : max(0, p.seq_lens[b]);
    per = ((n_keys_u + kTok - 1) / kTok + p.splits - 1) / p.splits;
    tile0 = split * per;
    direct = p.splits == 1;
    row0 = (static_cast<int64_t>(b) * p.splits + split) * p.num_heads;
  }
  const int n_keys = topk_mode<kMode>(p) ? p.topk_n : max(0, p.seq_lens[b]);
  const int n_tiles_all = n_keys / kTok + (n_keys % kTok != 0);
  const int nt = max(0, min(n_tiles_all, tile0 + per) - tile0);
  uint32_t* err = p.error_word;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + kQ4Q), sSfa = smem_u32(smem + kQ4Sfa), sBuf = smem_u32(smem + kQ4Buf0);

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bars.q_ready, 128);
    mbar_init(&bars.sfa_ready, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.t_full[i], 128);  // codes and scales (64 threads), RoPE (64)
      mbar_init(&bars.t_empty[i], 1);
      mbar_init(&bars.v_full[i], 64);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 128);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.o_full, 2);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == kMmaWarp || warp == kMmaWarp2) {
    // ----------------------------------------------------------------- MMA
    // issuer p runs the tiles of parity p: QK (scales of the tile into TMEM,
    // 8 block-scaled latent MMAs, 4 f16 RoPE MMAs), then P.V
    const int par = (warp == kMmaWarp) ? 0 : 1;
    if (lane == 0 && nt > 0) {
      const uint64_t dq = smem_desc_sw128(sQ, 0, 1024);
      const uint64_t dbuf = smem_desc_sw128(sBuf, 0, 1024);
      const uint64_t dbuf_mn = smem_desc_sw128(sBuf, kChunk, 1024);  // V read MN-major: 64-feature chunks 8 KB apart
      bool ok = bar_wait(&bars.q_ready, 0, err, &abort_s);
      tc_fence_after();
      if (ok && par == 0) {  // the query scales, for both issuers
#pragma unroll 1
        for (int t = 0; t < 8; ++t) q4_sf_copy(tmem + kQ4TSfa + 4 * t, q4_sf_desc(sSfa + 512 * t));
        mma_commit(&bars.sfa_ready);
      }
      ok = ok && bar_wait(&bars.sfa_ready, 0, err, &abort_s);
      tc_fence_after();
      auto issue_qk = [&](int j) -> bool {
        const int tb = j & 1;
        if (!bar_wait(&bars.t_full[tb], (j >> 1) & 1, err, &abort_s)) return false;
        tc_fence_after();
        const uint32_t bsh = sBuf + tb * kQ4BufBytes;
#pragma unroll 1
        for (int t = 0; t < 8; ++t) q4_sf_copy(tmem + q4_col_sfb(tb) + 4 * t, q4_sf_desc(bsh + kQ4Sfb + 512 * t));
        const uint32_t d = tmem + col_s(tb);
        const uint64_t dk = dbuf + (tb * kQ4BufBytes + kQ4K) / 16;
#pragma unroll 1
        for (int t = 0; t < 8; ++t)  // K 64 a step: chunk t / 4, 32 bytes along the swizzled row
          q4_mma(d, dq + (t >> 2) * (16384 / 16) + 2 * (t & 3), dk + (t >> 2) * (8192 / 16) + 2 * (t & 3),
                 tmem + kQ4TSfa + 4 * t, tmem + q4_col_sfb(tb) + 4 * t, t > 0 ? 1u : 0u);
        const uint64_t dr = dbuf + (tb * kQ4BufBytes + kQ4Rope) / 16;
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk) mma_ts(d, tmem + kQ4TRope + 8 * kk, dr + 2 * kk, kIdescQK, 1u);
        mma_commit(&bars.t_empty[tb]);
        mma_commit(&bars.s_full[tb]);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int pb = j & 1;
        if (!bar_wait(&bars.v_full[pb], (j >> 1) & 1, err, &abort_s) ||
            !bar_wait(&bars.p_full[pb], (j >> 1) & 1, err, &abort_s))
          return false;
        tc_fence_after();
        const uint64_t vd = dbuf_mn + (pb * kQ4BufBytes + kQ4V) / 16;
#pragma unroll 1
        for (int kk = 0; kk < kTok / 16; ++kk)
          mma_ts(tmem + kTO, tmem + col_s(pb) + 8 * kk, vd + (2048 * kk) / 16, kIdescPV, 1u);  // O starts at 0
        mma_commit(&bars.v_empty[pb]);
        mma_commit(&bars.pv_done[pb]);
        return true;
      };
      for (int j = par; ok && j < nt; j += 2) ok = issue_qk(j) && issue_pv(j);
      mma_commit(&bars.o_full);
      bar_wait(&bars.o_full, 0, err, nullptr);  // both issuers' MMAs retired
    }
  } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // ------------------------------------------------------- record parts
    const int di = threadIdx.x - 32 * kDeqWarp0;
    const int k = di & 63, q = di >> 6;
    const float gs = *p.gs;
    Q4Ctx c{p, &bars, &abort_s, sBuf, rank, b, tile0, nt, n_keys, k, scale_ok(gs) ? 1.f / gs : 0.f};
    bool bad;
    if (q == 0)
      bad = q4_role<0, kRecord, kMode>(c);
    else if (q == 1)
      bad = q4_role<1, kRecord, kMode>(c);
    else
      bad = q4_role<2, kRecord, kMode>(c);
    if (bad && rank == 0 && q == 0) flag_error(err, MLA_DEVERR_BOUNDS);
  } else {
    // ------------------------------ query quantisation, softmax, epilogue
    const int hr = warp * 32 + lane;
    const int head = hg * kHeads + hr;
    const bool head_ok = head < p.num_heads;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float gs = *p.gs, gs_q = *p.gs_q;
    const bool scales_ok = scale_ok(gs) && scale_ok(gs_q);
    const float score_scale = p.softmax_scale * gs_q * gs * kLog2e;
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    if (nt > 0) {
      // the query row to NVFP4 (correctly rounded, as the cache write):
      // latent codes to shared memory, their scales to the scale tiles, the
      // RoPE part's values c*s (exact in f16) to TMEM
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q + (static_cast<int64_t>(b) * p.num_heads + head) * 576);
      const float inv_gs_q = inv_scale(gs_q);
      uint32_t sf_word = 0, rope[16];
#pragma unroll 1
      for (int u = 0; u < 36; u += 2) {  // two blocks of 16 = one 16-byte unit of codes
        uint2 codes[2];
        uint32_t sbs[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int blk = u + h;
          const uint4 w0 = head_ok ? ldg16(qrow + 32 * blk) : make_uint4(0, 0, 0, 0);
          const uint4 w1 = head_ok ? ldg16(qrow + 32 * blk + 16) : make_uint4(0, 0, 0, 0);
          float x[16];
          const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) bf16x2_to_f32(ws[i], x[2 * i], x[2 * i + 1]);
          float R = 0.f, S = 0.f;
          bool bounded = true;
          sbs[h] = scales_ok ? block_scale_rn(fmaxf(amax8(x), amax8(x + 8)), inv_gs_q, gs_q, R, S, bounded) : 0u;
          codes[h] = scales_ok ? make_uint2(encode8_rn(x, R, S, bounded), encode8_rn(x + 8, R, S, bounded))
                               : make_uint2(0u, 0u);
        }
        if (u < 32) {
          const int cu = u >> 1;  // 16-byte unit of the 256-byte code row
          sts128(sQ + (cu >> 3) * 16384 + hr * 128 + (((cu & 7) ^ (hr & 7)) << 4),
                 make_uint4(codes[0].x, codes[0].y, codes[1].x, codes[1].y));
          sf_word |= (sbs[0] | (sbs[1] << 8)) << (16 * ((u >> 1) & 1));
          if ((u & 3) == 2) {  // blocks u-2 .. u+1 done: scale tile u / 4
            sts32(sSfa + 512 * (u >> 2) + (hr & 31) * 16 + (hr >> 5) * 4, sf_word);
            sf_word = 0;
          }
        } else {
          // RoPE values c * s (exact in f16), 8 f16 pairs a block: blocks u
          // and u + 1 fill 16 TMEM columns
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t f = e4m3x2_to_f16x2(sbs[h] | (sbs[h] << 8));
            uint32_t hh[4];
            e2m1x8_to_f16x8(codes[h].x, hh);
#pragma unroll
            for (int i = 0; i < 4; ++i) rope[8 * h + i] = hmul2_u32(hh[i], f);
            e2m1x8_to_f16x8(codes[h].y, hh);
#pragma unroll
            for (int i = 0; i < 4; ++i) rope[8 * h + 4 + i] = hmul2_u32(hh[i], f);
          }
          tmem_st16(tmem + lane_off + kQ4TRope + 8 * (u - 32), rope);
        }
      }
      {  // O starts at zero: every P.V accumulates, whichever issuer runs first
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll 1
        for (int cc = 0; cc < 256; cc += 16) tmem_st16(tmem + lane_off + kTO + cc, z);
      }
      fence_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.q_ready);
      if (!scales_ok && hr == 0 && rank == 0) flag_error(err, MLA_DEVERR_SCALE);
      softmax_tiles<1, kMode>(p, bars, abort_s, tmem, lane_off, b, tile0, nt, n_keys, score_scale, ok, m_run, l_run, 0,
                       nullptr, hr);
      if (ok) ok = bar_wait(&bars.o_full, 0, err, &abort_s);
    }
    write_partial<1>(p, tmem, lane_off, ok, nt, m_run, l_run, gs, row0, b, head, head_ok, direct, rank, 0, nullptr,
                     hr, &abort_s);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// Merge n partials of one (sequence, head), rows row0, row0 + stride, ...:
// LSE = ln sum exp(lse_i), out = sum exp(lse_i - LSE) o_i.  Thread t (of
// 128) handles features [4t, 4t + 4).
__device__ __forceinline__ void merge_rows(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                           int64_t row0, int64_t stride, int n, __nv_bfloat16* __restrict__ o,
                                           float* __restrict__ lse_out, int t) {
  float m = -INFINITY;
  for (int s = 0; s < n; ++s) m = fmaxf(m, part_lse[row0 + s * stride]);
  float tot = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (m != -INFINITY) {
    for (int s = 0; s < n; ++s) {
      const int64_t row = row0 + s * stride;
      const float l = part_lse[row];
      if (l == -INFINITY) continue;
      const float w = expf(l - m);
      tot += w;
      const float4 v = reinterpret_cast<const float4*>(part_o + row * 512)[t];
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(o + 4 * t) = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lse_out != nullptr && t == 0) *lse_out = (tot > 0.f) ? m + logf(tot) : -INFINITY;
}

// Uniform splits: one block per (batch, head), partial rows (b, split, h).
__global__ void __launch_bounds__(128) decode_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse,
                                                           int splits, int num_heads,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse) {
  const int b = blockIdx.x / num_heads, h = blockIdx.x % num_heads;
  const int64_t bh = static_cast<int64_t>(b) * num_heads + h;
  merge_rows(part_o, part_lse, static_cast<int64_t>(b) * splits * num_heads + h, num_heads, splits,
             out + bh * 512, lse != nullptr ? lse + bh : nullptr, threadIdx.x);
}

// Planned chunks: block (sequence b, group of kMergeHeads heads); a sequence
// with one chunk was written by the decode kernel and is skipped.
constexpr int kMergeHeads = 8;
__global__ void __launch_bounds__(256) decode_plan_merge_kernel(const float* __restrict__ part_o,
                                                                const float* __restrict__ part_lse,
                                                                const int2* __restrict__ seqs, int num_heads,
                                                                __nv_bfloat16* __restrict__ out,
                                                                float* __restrict__ lse) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as a dependent of the decode grid
  const int b = blockIdx.x;
  const int2 sq = seqs[b];
  if (sq.x < 0) return;
  for (int hh = threadIdx.x >> 7; hh < kMergeHeads; hh += 2) {
    const int h = blockIdx.y * kMergeHeads + hh;
    if (h >= num_heads) break;
    const int64_t bh = static_cast<int64_t>(b) * num_heads + h;
    merge_rows(part_o, part_lse, static_cast<int64_t>(sq.x) * num_heads + h, num_heads, sq.y, out + bh * 512,
               lse != nullptr ? lse + bh : nullptr, threadIdx.x & 127);
  }
}

// ------------------------------------------------------------------ plan
// Length-aware work list (num_splits <= 0).  Every sequence is cut into
// chunks of C key tiles (its last chunk shorter; an empty sequence is one
// empty chunk) and CTA pair i runs item i.  The list holds all full chunks
// first, then the shorter last chunks from longest to shortest (64 size
// buckets), so that the hardware, which starts CTAs in index order as SMs
// free up, schedules longest-first.  C is chosen among ceil(tmax / k),
// k = 1..32, by an estimate of the makespan over the resident CTA pairs P,
// with every item costing kItemOverhead tiles on top of its own:
//   max( ceil(full / P) * (C + o),  (tiles + o * items) / P + (mean last chunk + o) / 2 )
// (the full chunks' waves, or the average load plus half a typical last
// chunk), subject to the items and partial rows fitting the workspace.
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 64;
constexpr float kItemOverhead = 2.f;

// Key tiles of a sequence of n keys.
__host__ __device__ inline int plan_tiles_of(int n) {
  n = n > 0 ? n : 0;
  return n / kTok + (n % kTok != 0);
}

// Products and quotients rounded once on both sides, so that the device plan
// and its host form (decode_plan_one_chunk) rank the candidates alike.
__host__ __device__ inline float plan_mul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}

// The makespan estimate of chunk size C for a batch of `tot` tiles that C
// cuts into n items, `full` full chunks, `rows` partial rows (the chunks of
// sequences cut more than once) and `last` shorter last chunks (empty
// sequences included); infinity when the items or rows do not fit.
__host__ __device__ inline float plan_estimate(long long tot, long long n, long long full, long long rows,
                                               long long last, int C, int pairs, int max_items, int max_rows) {
  const float P = static_cast<float>(pairs > 1 ? pairs : 1), o = kItemOverhead;
  const float waves = plan_mul(ceilf(static_cast<float>(full) / P), static_cast<float>(C) + o);
  const float rem = static_cast<float>(tot - full * static_cast<long long>(C));
  const float spread = (static_cast<float>(tot) + plan_mul(o, static_cast<float>(n))) / P;
  const float tail = last > 0 ? plan_mul(0.5f, rem / static_cast<float>(last) + o) : 0.f;
  const float avg = spread + tail;
  const bool fits = n <= max_items && rows <= max_rows;
  return fits ? fmaxf(waves, avg) : INFINITY;
}

// The counts plan_estimate takes, of chunk size C over a sequence of t tiles.
struct PlanCounts {
  long long n = 0, full = 0, rows = 0, last = 0;
  __host__ __device__ void add(int t, int C) {
    const int f = t / C;
    const int chunks = f + (t % C != 0 ? 1 : 0);
    const int nb = chunks > 1 ? chunks : 1;  // an empty sequence is one empty chunk
    n += nb;
    full += f;
    rows += nb > 1 ? nb : 0;
    last += (t == 0 || t % C != 0) ? 1 : 0;
  }
};

struct PlanArgs {
  const int32_t* seq_lens;  // paged mode; null in top-k mode
  int topk_n;
  int batch, pairs, max_items, max_rows;
  int32_t* hdr;  // [0] items, [1] tiles per chunk
  int2* items;   // [max_items] (sequence, chunk)
  int2* seqs;    // [batch] (first partial row or -1, chunks)
};

__device__ __forceinline__ int plan_tiles(const PlanArgs& a, int b) {
  return plan_tiles_of(a.seq_lens != nullptr ? a.seq_lens[b] : a.topk_n);
}

// Tile counts of the first kPlanStaged sequences, read from global memory
// once per plan.
constexpr int kPlanStaged = 4096;
__device__ __forceinline__ int staged_tiles(const PlanArgs& a, const int* s_tiles, int b) {
  return b < kPlanStaged ? s_tiles[b] : plan_tiles(a, b);
}

// Bucket of a last chunk of r tiles (0 <= r < C): longer chunks first.
__device__ __forceinline__ int plan_bucket(int r, int C) {
  return kPlanBuckets - 1 - static_cast<int>(static_cast<long long>(r) * kPlanBuckets / C);
}

// Exclusive prefix sum over the 1024 threads of the block; *total gets the
// block's sum.  `sm` holds 32 ints.  Every thread must call it.
__device__ __forceinline__ int block_scan(int v, int* sm, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = sm[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sm[lane] = w;
  }
  __syncthreads();
  *total = sm[31];
  return x - v + (warp > 0 ? sm[warp - 1] : 0);
}

__global__ void __launch_bounds__(kPlanThreads, 1) decode_plan_kernel(PlanArgs a) {
  // the decode grid may be set up while the plan is built; it waits for
  // this grid's completion before reading the tables
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ int s_tiles[kPlanStaged];
  __shared__ long long s_tot[32];
  __shared__ int s_max[32], s_scan[32];
  __shared__ float s_est[32];
  __shared__ int s_hist[kPlanBuckets], s_fill[kPlanBuckets];
  __shared__ int s_chunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = a.batch;

  // total tiles and the longest sequence
  long long tot = 0;
  int tmax = 0;
  for (int b = threadIdx.x; b < B; b += kPlanThreads) {
    const int t = plan_tiles(a, b);
    if (b < kPlanStaged) s_tiles[b] = t;
    tot += t;
    tmax = max(tmax, t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
  }
  if (lane == 0) {
    s_tot[warp] = tot;
    s_max[warp] = tmax;
  }
  if (threadIdx.x < kPlanBuckets) {
    s_hist[threadIdx.x] = 0;
    s_fill[threadIdx.x] = 0;
  }
  __syncthreads();
  tot = 0;
  tmax = 0;
  for (int w = 0; w < 32; ++w) {
    tot += s_tot[w];
    tmax = max(tmax, s_max[w]);
  }

  // candidate C = ceil(tmax / (warp + 1)), evaluated by one warp each
  {
    const int C = max(1, (tmax + warp) / (warp + 1));
    PlanCounts c;
    for (int b = lane; b < B; b += 32) c.add(staged_tiles(a, s_tiles, b), C);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      c.n += __shfl_xor_sync(0xffffffffu, c.n, o);
      c.full += __shfl_xor_sync(0xffffffffu, c.full, o);
      c.rows += __shfl_xor_sync(0xffffffffu, c.rows, o);
      c.last += __shfl_xor_sync(0xffffffffu, c.last, o);
    }
    if (lane == 0) s_est[warp] = plan_estimate(tot, c.n, c.full, c.rows, c.last, C, a.pairs, a.max_items, a.max_rows);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // the first minimum (largest C); candidate 0 (one chunk per sequence)
    // always fits, since max_items >= batch and it needs no partial rows
    int best = 0;
    for (int w = 1; w < 32; ++w)
      if (s_est[w] < s_est[best]) best = w;
    s_chunk = max(1, (tmax + best) / (best + 1));
  }
  __syncthreads();
  const int C = s_chunk;

  // pass 1: per-sequence chunks and partial rows, full chunks in sequence
  // order, last-chunk size histogram
  int full_base = 0, row_base = 0;
  for (int b0 = 0; b0 < B; b0 += kPlanThreads) {
    const int b = b0 + threadIdx.x;
    int t = 0, nb = 0, f = 0;
    if (b < B) {
      t = staged_tiles(a, s_tiles, b);
      nb = max(1, t / C + (t % C != 0));
      f = t / C;
    }
    const int rows_b = nb > 1 ? nb : 0;
    int f_tot, r_tot;
    const int f_off = block_scan(f, s_scan, &f_tot);
    const int r_off = block_scan(rows_b, s_scan, &r_tot);
    if (b < B) {
      a.seqs[b] = make_int2(rows_b > 0 ? row_base + r_off : -1, nb);
      for (int c = 0; c < f; ++c) a.items[full_base + f_off + c] = make_int2(b, c);
      const int r = t - f * C;
      if (t == 0 || r > 0) atomicAdd(&s_hist[plan_bucket(r, C)], 1);
    }
    full_base += f_tot;
    row_base += r_tot;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the histogram (longest bucket first)
    int h0 = s_hist[lane], h1 = s_hist[32 + lane];
    int x0 = h0, x1 = h1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
      if (lane >= o) {
        x0 += y0;
        x1 += y1;
      }
    }
    const int sum0 = __shfl_sync(0xffffffffu, x0, 31);
    s_hist[lane] = x0 - h0;
    s_hist[32 + lane] = sum0 + x1 - h1;
    if (lane == 31) {
      a.hdr[0] = full_base + sum0 + x1;
      a.hdr[1] = C;
    }
  }
  __syncthreads();
  // pass 2: the last chunks, bucket by bucket after the full chunks
  for (int b = threadIdx.x; b < B; b += kPlanThreads) {
    const int t = staged_tiles(a, s_tiles, b);
    const int f = t / C, r = t - f * C;
    if (t == 0 || r > 0) {
      const int k = plan_bucket(r, C);
      a.items[full_base + s_hist[k] + atomicAdd(&s_fill[k], 1)] = make_int2(b, f);
    }
  }
}

}  // namespace

size_t decode_workspace_bytes(int batch, int num_heads, int num_splits) {
  const size_t rows = static_cast<size_t>(batch) * num_splits * num_heads;
  const size_t o_bytes = rows * 512 * sizeof(float);
  const size_t l_bytes = (rows * sizeof(float) + 255) / 256 * 256;
  return o_bytes + l_bytes;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

DecodePlanLayout decode_plan_layout(int batch, int num_heads, int num_sms, size_t bytes) {
  DecodePlanLayout l;
  l.pairs = num_sms / 2;
  // Items beyond one per sequence: one per resident CTA pair.  On the
  // log-uniform 1k..32k-token batch this balances as well as two per pair
  // (simulated makespan 239 against 240 tiles, lower bound 217), while each
  // slot the plan leaves unused is a CTA pair that still has to be launched
  // (~0.07 us each on GB300, measured).
  l.max_items = batch + l.pairs;
  l.items = 256;
  l.seqs = align256(l.items + static_cast<size_t>(l.max_items) * sizeof(int2));
  l.rows = align256(l.seqs + static_cast<size_t>(batch) * sizeof(int2));
  const size_t per_row = static_cast<size_t>(num_heads) * (512 + 1) * sizeof(float);  // o and lse per chunk
  const size_t slack = 512;                                                          // two 256-byte alignments
  size_t max_rows = static_cast<size_t>(l.max_items);
  if (bytes != 0) max_rows = bytes >= l.rows + slack ? (bytes - l.rows - slack) / per_row : 0;
  l.max_rows = static_cast<int>(max_rows < static_cast<size_t>(l.max_items) ? max_rows : l.max_items);
  l.lse = align256(l.rows + static_cast<size_t>(l.max_rows) * num_heads * 512 * sizeof(float));
  l.total = align256(l.lse + static_cast<size_t>(l.max_rows) * num_heads * sizeof(float));
  return l;
}

int decode_plan_one_chunk(const int32_t* lens, int batch, int num_heads, int num_sms, size_t bytes) {
  if (lens == nullptr || batch < 1 || num_heads < 1) return 0;
  const DecodePlanLayout l = decode_plan_layout(batch, num_heads, num_sms, bytes);
  long long tot = 0;
  int tmax = 0;
  for (int b = 0; b < batch; ++b) {
    const int t = plan_tiles_of(lens[b]);
    tot += t;
    tmax = t > tmax ? t : tmax;
  }
  // candidate 0 (C = tmax) against C = ceil(tmax / k), k = 2..32, exactly
  // as the device plan ranks them: the first minimum wins
  float est0 = 0.f;
  for (int w = 0; w < 32; ++w) {
    const int C = (tmax + w) / (w + 1) > 1 ? (tmax + w) / (w + 1) : 1;
    PlanCounts c;
    for (int b = 0; b < batch; ++b) c.add(plan_tiles_of(lens[b]), C);
    const float est = plan_estimate(tot, c.n, c.full, c.rows, c.last, C, l.pairs, l.max_items, l.max_rows);
    if (w == 0)
      est0 = est;
    else if (est < est0)
      return 0;
  }
  return 1;
}

int decode_default_splits(int batch, int num_heads, int num_sms) {
  const int groups = (num_heads + kHeads - 1) / kHeads;
  const int pairs = num_sms / 2;
  const int units = batch * groups;
  int s = pairs / (units > 0 ? units : 1);
  return s < 1 ? 1 : (s > 64 ? 64 : s);
}

// Launch with cudaLaunchKernelEx; `dependent` makes the grid a
// programmatic dependent of the previous kernel in the stream (it may start
// before that kernel completes and waits for it with griddepcontrol.wait).
static int launch_ex(const void* kern, dim3 grid, dim3 block, uint32_t smem, cudaStream_t stream, bool dependent,
                     void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  if (const int st = cuda_status(cudaLaunchKernelExC(&cfg, kern, args))) return st;
  return launch_status();
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream, int num_sms) {
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
  magic_divisor(a.page_size, &p.pg_magic, &p.pg_shift);
  p.seq_lens = a.seq_lens;
  p.topk = a.topk_indices;
  p.topk_n = a.topk;
  p.softmax_scale = a.softmax_scale;
  p.gs = a.gs;
  p.gs_q = a.gs_q;
  p.splits = a.num_splits;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.error_word = a.error_word;
  p.plan_hdr = nullptr;
  p.plan_items = nullptr;
  p.plan_seqs = nullptr;
  char* ws = static_cast<char*>(a.workspace);
  const unsigned groups = static_cast<unsigned>((a.num_heads + kHeads - 1) / kHeads);
  dim3 grid;
  DecodePlanLayout l{};
  if (a.planned) {
    l = decode_plan_layout(a.batch, a.num_heads, num_sms, a.workspace_bytes);
    p.plan_hdr = reinterpret_cast<int32_t*>(ws);
    p.plan_items = reinterpret_cast<int2*>(ws + l.items);
    p.plan_seqs = reinterpret_cast<int2*>(ws + l.seqs);
    p.part_o = reinterpret_cast<float*>(ws + l.rows);
    p.part_lse = reinterpret_cast<float*>(ws + l.lse);
    grid = dim3(2u * static_cast<unsigned>(l.max_items), 1u, groups);
    PlanArgs pa{a.seq_lens, a.topk, a.batch, l.pairs, l.max_items, l.max_rows,
                reinterpret_cast<int32_t*>(ws), reinterpret_cast<int2*>(ws + l.items),
                reinterpret_cast<int2*>(ws + l.seqs)};
    decode_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pa);
    if (const int st = launch_status()) return st;
  } else {
    const size_t rows = static_cast<size_t>(a.batch) * a.num_splits * a.num_heads;
    p.part_o = static_cast<float*>(a.workspace);
    p.part_lse = reinterpret_cast<float*>(ws + rows * 512 * sizeof(float));
    grid = dim3(2u * static_cast<unsigned>(a.num_splits), static_cast<unsigned>(a.batch), groups);
    if (grid.y > 65535u) return MLA_ERR_INVALID_ARG;
  }
  if (grid.z > 65535u) return MLA_ERR_INVALID_ARG;
  // planned: the decode grid is a programmatic dependent of the plan kernel
  // (set up while the plan is built, waiting for it before reading the
  // tables), and the merge of the decode
  const void* kern;
  uint32_t smem;
  int slot;
  if (a.gs_q != nullptr) {
    const bool r432 = a.record_bytes == 432;
    const bool topk = a.topk_indices != nullptr;
    kern = topk ? (r432 ? reinterpret_cast<const void*>(decode_q4_kernel<432, kKeysTopk>)
                        : reinterpret_cast<const void*>(decode_q4_kernel<368, kKeysTopk>))
                : (r432 ? reinterpret_cast<const void*>(decode_q4_kernel<432, kKeysPaged>)
                        : reinterpret_cast<const void*>(decode_q4_kernel<368, kKeysPaged>));
    smem = kQ4SmAlloc;
    slot = topk ? (r432 ? 10 : 11) : (r432 ? 5 : 6);
  } else {
    const bool r432 = a.record_bytes == 432, topk = a.topk_indices != nullptr;
    kern = topk ? (r432 ? reinterpret_cast<const void*>(decode_tc_kernel<432, kKeysTopk>)
                        : reinterpret_cast<const void*>(decode_tc_kernel<368, kKeysTopk>))
                : a.page_size == 64
                    ? (r432 ? reinterpret_cast<const void*>(decode_tc_kernel<432, kKeysPaged64>)
                            : reinterpret_cast<const void*>(decode_tc_kernel<368, kKeysPaged64>))
                    : (r432 ? reinterpret_cast<const void*>(decode_tc_kernel<432, kKeysPaged>)
                            : reinterpret_cast<const void*>(decode_tc_kernel<368, kKeysPaged>));
    smem = kSmAlloc;
    slot = topk ? (r432 ? 8 : 9) : a.page_size == 64 ? (r432 ? 12 : 13) : (r432 ? 1 : 2);
  }
  if (const int st = smem_limit_once(kern, static_cast<int>(smem), slot)) return st;
  {
    void* args[] = {&p};
    const int threads = a.gs_q != nullptr ? kThreads : kThreadsTc;
    if (const int st = launch_ex(kern, grid, dim3(threads), smem, stream, a.planned, args)) return st;
  }
  if (a.planned) {
    const float* po = p.part_o;
    const float* pl = p.part_lse;
    const int2* sq = p.plan_seqs;
    int heads = a.num_heads;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    float* lse = a.lse;
    void* args[] = {&po, &pl, &sq, &heads, &out, &lse};
    return launch_ex(reinterpret_cast<const void*>(decode_plan_merge_kernel),
                     dim3(static_cast<unsigned>(a.batch), (a.num_heads + kMergeHeads - 1) / kMergeHeads), dim3(256),
                     0, stream, true, args);
  }
  if (a.num_splits == 1) return MLA_OK;  // the decode kernel wrote out and lse
  decode_merge_kernel<<<a.batch * a.num_heads, 128, 0, stream>>>(
      p.part_o, p.part_lse, a.num_splits, a.num_heads, static_cast<__nv_bfloat16*>(a.out), a.lse);
  return launch_status();
}

}  // namespace mla
