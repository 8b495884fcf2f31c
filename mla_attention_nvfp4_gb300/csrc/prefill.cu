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
// Persistent: one CTA per SM takes work items (query tile of 128 rows of
// one sequence and head) from a launch-wide counter.  Items are numbered
// (sequence, head) major with the last query tile first, so the CTAs working
// at the same moment share the keys they read (L2 reuse) and each group's
// heaviest tile starts first.  The key blocks of one CTA's items form one
// stream, so the next item's first score product is issued before the
// current item's last P.V and the tensor pipe does not drain between items;
// a separate epilogue warpgroup quantises an item's output while the next
// item's first score products and softmax run.
// Warp roles (512 threads, four warpgroups):
//   warp 0       scheduler and TMA producer: takes items, hands their
//                indices to the other roles through a shared-memory ring,
//                loads K and V blocks of 128 keys into two-stage rings by
//                the CTA's global block count g (128-byte swizzled rows; the
//                K slot of block g is free once S of block g-2 completed,
//                the V slot once its P.V did)
//                and, per item, Q once the previous item's last score
//                products have read it; the next item is taken one item
//                ahead and its Q tile prefetched into L2.
//   warps 1, 3   MMA issuers, one thread each.  Issuer w takes the key
//                blocks j of each item with j mod 2 = w:
//                  S_g = Q K_g^T   M=128 N=128 K=192, A and B from smem
//                  O_w += P_g V_g  M=128 N=128 K=128, A (P) from TMEM,
//                                  B = V tile read MN-major
//                in the order S_j, P.V of j, S_{j+2}: in-order issue from
//                one thread keeps S_{j+2} behind the P.V that reads P_j in
//                the same TMEM buffer.  The split depends only on j, so an
//                item's arithmetic is the same whichever CTA runs it and the
//                output is identical from run to run.  A thread's barrier polls queue behind
//                its own MMAs, so one issuer per parity keeps the tensor pipe
//                fed from the other issuer while one waits.
//   warps 4..11  softmax: warpgroup w takes the same blocks as issuer w, one
//                thread per query row over all 128 keys, with its own
//                running max, row sum and partial O_w.  The two warpgroups
//                never exchange data inside an item.  A warpgroup signals
//                P_g ready only once V_g has landed, so the issuer waits on
//                one barrier before P.V.
//   warps 12..15 epilogue: thread = query row; merges the two partial
//                results by their row maxima and sums (the split-K merge of
//                online softmax), normalises, quantises to NVFP4 and stores.
// Registers are moved to the softmax warpgroups with setmaxnreg.
// TMEM columns: S/P of even and odd blocks [0,128) [128,256), partial O of
// even and odd blocks [256,384) [384,512).  P_g (bf16) overwrites the first
// 64 columns of its S buffer after the row is read.  A partial's reference
// max is only raised when a row's max grows by more than 8 (log2 units), so
// O_w is rarely rescaled; P stays <= 2^8, exact enough in bf16, and
// numerator and denominator share the same reference.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "launch.h"
#include "nvfp4.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 128, kDqk = 192, kDv = 128;
constexpr int kThreads = 512;
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
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 256 where the block's max is taken
constexpr float kSumLimit = 65536.0f;      // a block's P row sum formed against the reference: P <= 2^16
static_assert(kSmemAlloc <= 232448, "shared memory budget");

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);
// fake-quant mode: every operand is an exact f16 value code * scale
constexpr uint32_t kIdescS16 = idesc_f16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV16 = idesc_f16_f32(128, 128, false, true);
// P's global scale in fake-quant mode: amax/(6*448) with amax = 1 (P <= 1
// relative to its power-of-two reference)
constexpr float kGsP = 1.0f / 2688.0f;

struct Params {
  const int32_t* cu;
  int num_seqs;
  int64_t total;
  int num_heads;
  int q_tiles;          // query tiles of the longest sequence
  uint32_t num_items;   // q_tiles * num_seqs * num_heads
  // multipliers and shifts of q_tiles and num_heads for div_magic
  uint32_t qt_magic, h_magic;
  int qt_shift, h_shift;
  uint32_t* sched;      // [0] next item, [1] CTAs finished; zero between launches
  float scale_log2;
  const float* gs;
  uint8_t* codes;
  uint8_t* scales;
  float* lse;
  uint32_t* error_word;
  // partial mode (kPartial): the normalised fp32 output [total, H, 128]
  // (lse required), and, when cu_k is set, the key sequences of the key
  // tensors (total_k rows): queries of sequence s see every key of
  // [cu_k[s], cu_k[s+1]) (a context chunk), else the causal prefix of their
  // own sequence
  float* o_out;
  const int32_t* cu_k;
  int64_t total_k;
  // fake-quant mode (kQuant): global scales of the NVFP4 operands whose
  // code * scale values q, k, v hold, and 2:4 score sparsity on or off
  const float* gs_q;
  const float* gs_k;
  const float* gs_v;
  int sparse24;
};

// 2^d for an integer-valued d <= 0 (exact; 0 below the normal range).
__device__ __forceinline__ float exp2_int(float d) {
  return d < -126.f ? 0.f : __int_as_float((127 + static_cast<int>(d)) << 23);
}

constexpr int kRing = 4;  // item indices in flight from the producer to the other roles

struct alignas(8) Barriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2];  // K slots by global block parity
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2];  // by block parity = softmax warpgroup = MMA issuer
  uint64_t o_full;                // both issuers' P.V of an item retired
  uint64_t mma_done[2];           // every MMA of issuer 0 / 1 retired
  uint64_t o_empty[2], l_full[2];  // by item parity: epilogue -> MMA / softmax; softmax -> epilogue
  uint64_t item_full[kRing], item_empty[kRing];
};

// Register split (setmaxnreg), per thread: the launch gives 128 to each of
// the four warpgroups; producer/MMA and epilogue give some back to the two
// softmax warpgroups, which keep a whole score row in registers.
constexpr int kRegsCtl = 56, kRegsSoftmax = 176, kRegsEpi = 104;
static_assert(kRegsCtl + 2 * kRegsSoftmax + kRegsEpi <= 4 * 128, "register split exceeds the launch's registers");

struct Item {
  int h, seq_begin, n, row0, n_kv;
  int k_begin, n_k;  // key rows of the item's sequence (its own tokens unless a key table is given)
  bool valid;
};

__device__ __forceinline__ Item item_at(const Params& p, uint32_t idx, bool& bad) {
  const uint32_t group = div_magic(idx, p.qt_magic, p.qt_shift);
  const int qt = p.q_tiles - 1 - static_cast<int>(idx - group * static_cast<uint32_t>(p.q_tiles));
  const uint32_t seq_u = div_magic(group, p.h_magic, p.h_shift);
  const int seq = static_cast<int>(seq_u);
  Item it;
  it.h = static_cast<int>(group - seq_u * static_cast<uint32_t>(p.num_heads));
  it.seq_begin = p.cu[seq];
  const int seq_end = p.cu[seq + 1];
  it.n = seq_end - it.seq_begin;
  it.row0 = qt * kBM;
  if (it.seq_begin < 0 || seq_end > p.total || it.n < 0 || it.n > p.q_tiles * kBM) {
    bad = true;
    it.n = 0;
  }
  if (p.cu_k != nullptr) {
    it.k_begin = p.cu_k[seq];
    const int k_end = p.cu_k[seq + 1];
    it.n_k = k_end - it.k_begin;
    if (it.k_begin < 0 || k_end > p.total_k || it.n_k < 0) {
      bad = true;
      it.n_k = 0;
    }
    it.n_kv = (it.n_k + kBN - 1) / kBN;  // every key of the chunk
    it.valid = it.row0 < it.n && it.n_kv > 0;
  } else {
    it.k_begin = it.seq_begin;
    it.n_k = it.n;
    it.valid = it.row0 < it.n;
    it.n_kv = it.valid ? (min(it.n, it.row0 + kBM) - 1) / kBN + 1 : 0;  // causal: keys < row0 + 128
  }
  return it;
}

// Next valid item from the launch-wide counter, or -1 when none is left.
// The tiles of a group past its sequence's end come first in the group, so
// one invalid index moves the counter to the group's first valid tile.
__device__ int grab_item(const Params& p, bool& bad) {
  for (;;) {
    const uint32_t idx = atomicAdd(p.sched, 1u);
    if (idx >= p.num_items) return -1;
    const Item w = item_at(p, idx, bad);
    if (w.valid) return static_cast<int>(idx);
    const uint32_t group = idx / static_cast<uint32_t>(p.q_tiles);
    // a sequence with an empty key chunk has no item at all
    const uint32_t tiles = w.n_k > 0 || p.cu_k == nullptr ? static_cast<uint32_t>((w.n + kBM - 1) / kBM) : 0u;
    atomicMax(p.sched, group * static_cast<uint32_t>(p.q_tiles) + static_cast<uint32_t>(p.q_tiles) - tiles);
  }
}

// One copy per tile: the 4-D map (64 features, head, token, 64-feature chunk)
// lands as smem [chunk][token][64 features], the three (or two) 16 KB
// K-major 128-byte-swizzled chunks the MMAs read.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
// L2 prefetch of one box of the same map (no shared memory written).
__device__ __forceinline__ void tma_prefetch_4d(const void* tmap, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap), "r"(c0), "r"(c1),
               "r"(c2), "r"(c3) : "memory");
}

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

// A wait whose outcome is the same in every lane, so that the warp-wide
// tcgen05 loads and stores after it are reached by all lanes or by none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, abort));
}

template <bool kPartial, bool kQuant>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ int ring_s[kRing];     // item index, -1 = no more items
  __shared__ float l_s[2][2][kBM];  // [item parity][warpgroup][row] partial row sums
  __shared__ float m_s[2][2][kBM];  // matching reference maxima (log2 units)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t k_tiles_sf = (static_cast<int64_t>(p.num_heads) * 8 + 3) / 4;

  if constexpr (!kPartial) {
    // rows [total, roundup(total,128)) of the scale columns are zero
    const int64_t Mp = (p.total + 127) / 128 * 128;
    const int64_t pad = (Mp - p.total) * 8;
    for (int h = blockIdx.x; h < p.num_heads; h += gridDim.x)
      for (int64_t i = threadIdx.x; i < pad; i += kThreads)
        p.scales[sf_offset(p.total + i / 8, static_cast<int64_t>(h) * 8 + i % 8, k_tiles_sf)] = 0;
  } else if (p.cu_k != nullptr) {
    // queries whose key chunk is empty attend to nothing: O = 0, LSE = -inf
    for (int s = blockIdx.x; s < p.num_seqs; s += gridDim.x) {
      const int a = p.cu[s], e = p.cu[s + 1];
      if (p.cu_k[s + 1] - p.cu_k[s] != 0 || a < 0 || e > p.total || a > e) continue;
      for (int64_t i = threadIdx.x; i < static_cast<int64_t>(e - a) * p.num_heads * kDv; i += kThreads)
        p.o_out[static_cast<int64_t>(a) * p.num_heads * kDv + i] = 0.f;
      for (int64_t i = threadIdx.x; i < static_cast<int64_t>(e - a) * p.num_heads; i += kThreads)
        p.lse[(i / (e - a)) * p.total + a + i % (e - a)] = -INFINITY;
    }
  }
  const float gs = kPartial ? 0.f : *p.gs;  // the partial result is not quantised

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kSmemQ;
  uint8_t* sK = smem + kSmemK;
  uint8_t* sV = smem + kSmemV;

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 2);  // one arrival per MMA issuer
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], 128);
      mbar_init(&bars.mma_done[s], 1);
      mbar_init(&bars.o_empty[s], 128);
      mbar_init(&bars.l_full[s], 256);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&bars.item_full[s], 1);
      mbar_init(&bars.item_empty[s], 2 + 256 + 128);  // MMA issuers, softmax, epilogue
    }
    mbar_init(&bars.o_full, 2);  // one arrival per MMA issuer
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
  // TMEM columns: S of the even / odd key blocks, and the two partial O
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO[2] = {tmem + 256, tmem + 384};
  uint32_t* err = p.error_word;
  bool bad = false;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------ scheduler, K and Q
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int nq = 0, nk = 0, nv = 0;  // Q tiles, K and V blocks whose copies were issued
      int cur = grab_item(p, bad);
      for (int it = 0;; ++it) {
        // publish the item (or the end) to the other roles
        if (!mbar_wait(&bars.item_empty[it % kRing], ((it / kRing) & 1) ^ 1, err, &abort_s)) break;
        ring_s[it % kRing] = cur;
        mbar_arrive(&bars.item_full[it % kRing]);
        if (cur < 0) break;
        const Item w = item_at(p, static_cast<uint32_t>(cur), bad);
        // the next item is taken now so that its Q tile can be brought into L2
        const int nxt = grab_item(p, bad);
        if (nxt >= 0) {
          bool dummy = false;
          const Item w2 = item_at(p, static_cast<uint32_t>(nxt), dummy);
          tma_prefetch_4d(&tm_q, 0, w2.h, w2.seq_begin + w2.row0, 0);
        }
        bool ok = true;
        for (int j = 0; j < w.n_kv; ++j) {
          const int s = nk & 1;  // global block index
          const uint32_t ph = (nk >> 1) & 1;
          if (!(ok = mbar_wait(&bars.k_empty[s], ph ^ 1, err, &abort_s))) break;
          mbar_expect_tx(&bars.k_full[s], kKBytes);
          tma_load_4d(sK + s * kKBytes, &tm_k, 0, w.h, w.k_begin + j * kBN, 0, &bars.k_full[s]);
          ++nk;
          if (j == 0) {  // Q of this item, once the previous item's last score product has read it
            if (!(ok = mbar_wait(&bars.q_empty, (nq & 1) ^ 1, err, &abort_s))) break;
            mbar_expect_tx(&bars.q_full, kQBytes);
            tma_load_4d(sQ, &tm_q, 0, w.h, w.seq_begin + w.row0, 0, &bars.q_full);
            ++nq;
          }
          if (!(ok = mbar_wait(&bars.v_empty[s], ph ^ 1, err, &abort_s))) break;
          mbar_expect_tx(&bars.v_full[s], kVBytes);
          tma_load_4d(sV + s * kVBytes, &tm_v, 0, w.h, w.k_begin + j * kBN, 0, &bars.v_full[s]);
          ++nv;
        }
        if (!ok) break;
        cur = nxt;
      }
      // every copy issued has landed before the CTA can exit
      if (nq > 0) mbar_wait(&bars.q_full, (nq - 1) & 1, err, nullptr);
      for (int g = max(0, nk - 2); g < nk; ++g) mbar_wait(&bars.k_full[g & 1], (g >> 1) & 1, err, nullptr);
      for (int g = max(0, nv - 2); g < nv; ++g) mbar_wait(&bars.v_full[g & 1], (g >> 1) & 1, err, nullptr);
    } else if ((warp == 1 || warp == 3) && lane == 0) {
      // ------------------------------------------------------- MMA issuers
      // Issuer w (warp 1: w = 0, warp 3: w = 1) takes the key blocks j of
      // each item with j mod 2 = w, which use S/P buffer w and partial O_w,
      // and issues S_j then P.V of block j before S of block j+2: in-order
      // issue from one thread keeps S_{j+2} behind the P.V that reads P_j.
      // The split depends only on j, so an item's arithmetic is the same
      // whichever CTA runs it.  K/V slots follow the CTA's global block
      // count.  The two issuers' MMAs interleave on the tensor pipe.
      const int w = warp == 1 ? 0 : 1;
      // Descriptors are built once; a K-step only adds its byte offset >> 4
      // to the start-address field (addresses stay below 256 KB, no carry).
      const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 0, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 0, 1024);
      const uint64_t dk1 = smem_desc_sw128(smem_u32(sK) + kKBytes, 0, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), 16384, 1024);
      const uint64_t dv1 = smem_desc_sw128(smem_u32(sV) + kVBytes, 16384, 1024);
      const uint32_t sd = w ? tS[1] : tS[0];
      const uint32_t od = w ? tO[1] : tO[0];
      int gb = 0, cw = 0;  // global block counter; blocks of this issuer
      bool ok = true;
      for (int it = 0; ok; ++it) {
        if (!mbar_wait(&bars.item_full[it % kRing], (it / kRing) & 1, err, &abort_s)) break;
        const int idx = ring_s[it % kRing];
        mbar_arrive(&bars.item_empty[it % kRing]);
        if (idx < 0) break;
        bool dummy = false;
        const Item wi = item_at(p, static_cast<uint32_t>(idx), dummy);
        // this issuer's blocks of the item: j = w, w + 2, ...
        const int j0 = w;
        const int j_last = j0 < wi.n_kv ? j0 + ((wi.n_kv - 1 - j0) & ~1) : -1;
        for (int j = j0; j < wi.n_kv; j += 2, ++cw) {
          const uint32_t ph = cw & 1;
          const int g = gb + j;  // global block: K/V slot g mod 2
          const int s = g & 1;
          if ((j == j0 && !mbar_wait(&bars.q_full, it & 1, err, &abort_s)) ||
              !mbar_wait(&bars.k_full[s], (g >> 1) & 1, err, &abort_s)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // 12 K-steps: three 64-feature chunks of 16 KB, 32 bytes per step
          const uint64_t dk = s ? dk1 : dk0;
#pragma unroll 1
          for (int c = 0; c < kDqk / 64; ++c) {
            const uint64_t a = dq + c * (16384 >> 4), bdesc = dk + c * (16384 >> 4);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              mma_ss(sd, a + k4 * 2, bdesc + k4 * 2, kQuant ? kIdescS16 : kIdescS, (c | k4) != 0 ? 1u : 0u);
          }
          mma_commit(&bars.s_full[w]);
          mma_commit(&bars.k_empty[s]);
          if (j == j_last) mma_commit(&bars.q_empty);
          // P.V: the item's first one for this issuer overwrites O_w, which
          // the previous item's epilogue must have read; P_g implies V_g landed
          if ((j == j0 && it > 0 && !mbar_wait(&bars.o_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, err, &abort_s)) ||
              !mbar_wait(&bars.p_full[w], ph, err, &abort_s)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // 8 K-steps of 16 keys: P columns +8, V rows +2048 bytes
          const uint32_t first = j == j0 ? 1u : 0u;  // the item's first P.V overwrites O_w
          const uint64_t dv = s ? dv1 : dv0;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            const uint64_t bdesc = dv + h * ((4 * 2048) >> 4);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              mma_ts(od, sd + (4 * h + k4) * 8, bdesc + k4 * (2048 >> 4), kQuant ? kIdescPV16 : kIdescPV,
                     (first & (h == 0) & (k4 == 0)) ? 0u : 1u);
          }
          mma_commit(&bars.v_empty[s]);
          if (j == j_last) mma_commit(&bars.o_full);
        }
        if (!ok) break;
        if (j_last < 0) {
          // No block of this parity: nothing of this issuer reads Q or writes
          // O_w.  Its arrivals wait until the previous item's phases of
          // q_empty (implied by this item's Q having landed) and o_full
          // (implied by that item's epilogue being done) are complete, so
          // they cannot complete a phase that the other issuer still owes.
          if (!mbar_wait(&bars.q_full, it & 1, err, &abort_s)) break;
          mbar_arrive(&bars.q_empty);
          if (it > 0 && !mbar_wait(&bars.o_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, err, &abort_s)) break;
          mbar_arrive(&bars.o_full);
        }
        gb += wi.n_kv;
      }
      if (cw > 0) {
        mma_commit(&bars.mma_done[w]);
        mbar_wait(&bars.mma_done[w], 0, err, nullptr);  // every MMA of this issuer retired
      }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ softmax
    // Warpgroup wg takes the key blocks j of each item with j mod 2 = wg, one
    // thread per query row over all 128 keys of the block, with its own
    // running max, row sum and partial O; the epilogue merges the two
    // partial results.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t my_s = wg ? tS[1] : tS[0];
    const uint32_t my_o = wg ? tO[1] : tO[0];
    // fake-quant mode: the scores are products of code * scale values, so
    // the global scales of Q and K join the softmax scale
    const float sl2 = kQuant ? p.scale_log2 * *p.gs_q * *p.gs_k : p.scale_log2;
    const bool sparse = kQuant && p.sparse24 != 0;
    const float kf_p = scale_factor(kGsP);
    int gb = 0, cw = 0;  // global block counter; blocks of this warpgroup
    bool ok = true;
    for (int it = 0; ok; ++it) {
      if (!warp_wait(&bars.item_full[it % kRing], (it / kRing) & 1, err, &abort_s)) break;
      const int idx = ring_s[it % kRing];
      mbar_arrive(&bars.item_empty[it % kRing]);
      if (idx < 0) break;
      bool dummy = false;
      const Item w = item_at(p, static_cast<uint32_t>(idx), dummy);
      const int qi = w.row0 + r;  // query index within the sequence
      float m_run = -INFINITY, l_run = 0.f;
      bool any = false;  // this warpgroup had a block of this item
      for (int j = 0; j < w.n_kv; ++j, ++gb) {
        if ((j & 1) != wg) continue;
        if (!warp_wait(&bars.s_full[wg], cw & 1, err, &abort_s)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float x[128];
#pragma unroll
        for (int c = 0; c < 128; c += 64) {
          uint32_t v[64];
          tmem_ld64(my_s + lane_off + c, v);
#pragma unroll
          for (int i = 0; i < 64; ++i) x[c + i] = __uint_as_float(v[i]);
        }
        tmem_ld_wait();
        const int key0 = j * kBN;
        // the last visible key: the query itself (causal), or the chunk's last
        const int lim = (kPartial && p.cu_k != nullptr) ? w.n_k - 1 : qi;
        if (key0 + kBN - 1 > lim) {  // diagonal (or last) block: mask the keys beyond
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = (key0 + c <= lim) ? x[c] : -INFINITY;
        }
        // Exact mode, once the row has a reference max: P is first formed
        // against it without looking for the block's max; only a row whose
        // block sum then exceeds kSumLimit (or is not finite) takes the
        // block's max, raises its reference as below and forms P again.
        // Otherwise, and in fake-quant mode, the block's max comes first.
        bool fast = !kQuant && __all_sync(0xffffffffu, m_run != -INFINITY);
        float m_use = m_run, alpha = 1.f, l_blk = 0.f;
#pragma unroll 1
        for (int attempt = 0; attempt < 2; ++attempt) {
          if (!fast) {
            // max of the raw scores (scale_log2 > 0); the scale is applied
            // inside the exponent below
            float mq[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mq[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; c += 2) mq[(c >> 1) & 7] = max3(mq[(c >> 1) & 7], x[c], x[c + 1]);
            const float mx =
                fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])), fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7]))) *
                sl2;
            bool raise;
            if constexpr (kQuant) {
              // power-of-two reference: the running max rounded up (log2 units),
              // raised whenever it grows, so P <= 1 and O rescales exactly
              const float m_new = ceilf(mx);
              raise = m_new > m_run;
              if (raise) {
                m_use = m_new;
                alpha = m_run == -INFINITY ? 0.f : exp2_int(m_run - m_new);
              }
            } else {
              // lazy reference update
              raise = mx > m_run + kRescaleThreshold;
              if (raise) {
                m_use = mx;
                alpha = ex2_approx(m_run - mx);  // 0 on this warpgroup's first block
              }
            }
            // The partial O holds only this warpgroup's earlier blocks, whose
            // P.V retired before S of this block was committed.
            if (__any_sync(0xffffffffu, raise && any)) {
#pragma unroll
              for (int c = 0; c < 128; c += 16) {
                uint32_t v[16];
                tmem_ld16(my_o + lane_off + c, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                tmem_st16(my_o + lane_off + c, v);
              }
              tmem_st_wait();
            }
            m_run = m_use;
          }
          // exponent arguments two at a time: x * scale_log2 - m_use
          const uint64_t sc2 = pk2(sl2, sl2), nm2 = pk2(-m_use, -m_use);
          uint64_t ls2[4] = {0, 0, 0, 0};  // packed (+0, +0) partial row sums
#pragma unroll
          for (int c = 0; c < 128; c += 32) {  // P as 16-bit pairs: columns [0, 64) of the S buffer
            uint32_t v[16];
            if constexpr (kQuant) {
              // the row sum takes the unquantised P; the P.V operand is P
              // quantised to NVFP4 in blocks of 16 keys, as code * scale (f16)
#pragma unroll
              for (int blk = 0; blk < 2; ++blk) {
                float pb[16];
                if (sparse) {
                  // 2:4: of each group of 4 keys (aligned to the sequence's
                  // first key) keep the 2 largest scores, equal scores by lower
                  // key index; a key's rank counts the keys of its group that
                  // beat it.  A group's max is always kept, so the row max
                  // above is the max of the kept scores.
#pragma unroll
                  for (int g4 = c + 16 * blk; g4 < c + 16 * blk + 16; g4 += 4) {
                    const float a = x[g4], b = x[g4 + 1], cc = x[g4 + 2], d = x[g4 + 3];
                    const int ab = a >= b, ac = a >= cc, ad = a >= d, bc = b >= cc, bd = b >= d, cd = cc >= d;
                    const int ra = 3 - ab - ac - ad, rb = ab + 2 - bc - bd, rc = ac + bc + 1 - cd, rd = ad + bd + cd;
                    x[g4] = ra < 2 ? a : -INFINITY;
                    x[g4 + 1] = rb < 2 ? b : -INFINITY;
                    x[g4 + 2] = rc < 2 ? cc : -INFINITY;
                    x[g4 + 3] = rd < 2 ? d : -INFINITY;
                  }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  float a0, a1;
                  unpk2(fma2(pk2(x[c + 16 * blk + 2 * i], x[c + 16 * blk + 2 * i + 1]), sc2, nm2), a0, a1);
                  pb[2 * i] = ex2_approx(a0);
                  pb[2 * i + 1] = ex2_approx(a1);
                  ls2[i & 3] = add2(ls2[i & 3], pk2(pb[2 * i], pb[2 * i + 1]));
                }
                // amax of the block: P >= 0, so a plain three-input max
                float am = max3(pb[0], pb[1], pb[2]);
#pragma unroll
                for (int i = 3; i < 15; i += 2) am = max3(am, pb[i], pb[i + 1]);
                am = fmaxf(am, pb[15]);
                // block scale and 1/S in the reciprocal form, 1/S by the
                // approximate reciprocal: its decisions differ from the exact
                // quotient's only within a few float32 ulps of a midpoint
                const uint32_t sb = cvt_e4m3(__fmul_rn(am, kf_p));
                const float S = __fmul_rn(e4m3_to_f32(sb), kGsP);
                float R;
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(R) : "f"(S));
                if (!(S > 0.f)) R = 0.f;
                const uint32_t cw2[2] = {encode8(pb, R), encode8(pb + 8, R)};
                const uint32_t s2 = e4m3x2_to_f16x2_pair(sb | (sb << 8));
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const uint32_t byte = (cw2[i >> 2] >> (8 * (i & 3))) & 0xFFu;
                  uint32_t h2;
                  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h2) : "r"(byte));
                  const __half2 q2 = __hmul2(*reinterpret_cast<const __half2*>(&h2), *reinterpret_cast<const __half2*>(&s2));
                  v[8 * blk + i] = *reinterpret_cast<const uint32_t*>(&q2);
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float a0, a1;
                unpk2(fma2(pk2(x[c + 2 * i], x[c + 2 * i + 1]), sc2, nm2), a0, a1);
                const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                ls2[i & 3] = add2(ls2[i & 3], pk2(p0, p1));
                __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                v[i] = *reinterpret_cast<uint32_t*>(&h2);
              }
            }
            tmem_st16(my_s + lane_off + c / 2, v);
          }
          float ls[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) unpk2(ls2[i], ls[2 * i], ls[2 * i + 1]);
          l_blk = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
          if (!fast || !__any_sync(0xffffffffu, !(l_blk <= kSumLimit))) break;
          // P is formed again against the raised reference; its stores
          // replace these before P_g is signalled
          tmem_st_wait();
          fast = false;
        }
        l_run = l_run * alpha + l_blk;
        tmem_st_wait();
        tc_fence_before();
        if (!warp_wait(&bars.v_full[gb & 1], (gb >> 1) & 1, err, &abort_s)) {
          ok = false;
          break;
        }
        mbar_arrive(&bars.p_full[wg]);
        ++cw;
        any = true;
      }
      if (!ok) break;
      // partial row statistics for the epilogue; the slot of this item
      // parity is free once the epilogue of the item two before has read it
      if (!warp_wait(&bars.o_empty[it & 1], ((it >> 1) & 1) ^ 1, err, &abort_s)) break;
      l_s[it & 1][wg][r] = l_run;
      m_s[it & 1][wg][r] = m_run;
      mbar_arrive(&bars.l_full[it & 1]);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // thread = query row: merge the two partial results, normalise,
    // quantise to NVFP4 and store codes, scales and the LSE
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool gs_ok = scale_ok(gs);
    const float kf = scale_factor(gs);
    const float pv_scale = kQuant ? kGsP * *p.gs_v : 1.f;
    for (int it = 0;; ++it) {
      if (!warp_wait(&bars.item_full[it % kRing], (it / kRing) & 1, err, &abort_s)) break;
      const int idx = ring_s[it % kRing];
      mbar_arrive(&bars.item_empty[it % kRing]);
      if (idx < 0) break;
      bool dummy = false;
      const Item w = item_at(p, static_cast<uint32_t>(idx), dummy);
      const int o = it & 1;
      if (!warp_wait(&bars.o_full, it & 1, err, &abort_s) || !warp_wait(&bars.l_full[o], (it >> 1) & 1, err, &abort_s))
        break;
      tc_fence_after();
      const float l0 = l_s[o][0][r], l1 = l_s[o][1][r];
      const float m0 = m_s[o][0][r], m1 = m_s[o][1][r];
      const float m_row = fmaxf(m0, m1);
      // a partial with no block (l = 0) carries no weight, and its O is not read
      // (fake-quant mode: integer references, exact powers of two; the
      // global scales of P and V join the normalisation)
      const float a0 = l0 > 0.f ? (kQuant ? exp2_int(m0 - m_row) : ex2_approx(m0 - m_row)) : 0.f;
      const float a1 = l1 > 0.f ? (kQuant ? exp2_int(m1 - m_row) : ex2_approx(m1 - m_row)) : 0.f;
      const float l_tot = a0 * l0 + a1 * l1;
      const float inv_l = l_tot > 0.f ? pv_scale / l_tot : 0.f;
      const float c0 = a0 * inv_l, c1 = a1 * inv_l;
      const int qi = w.row0 + r;
      const int64_t m = w.seq_begin + qi;
      uint8_t* code_row = kPartial ? nullptr : p.codes + m * (static_cast<int64_t>(p.num_heads) * 64) + w.h * 64;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t sbits = 0;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int col = 64 * half + 32 * qq;
          float ov[32];
          uint32_t v0[16], v1[16], u0[16], u1[16];
          tmem_ld16(tO[0] + lane_off + col, v0);
          tmem_ld16(tO[0] + lane_off + col + 16, v1);
          tmem_ld16(tO[1] + lane_off + col, u0);
          tmem_ld16(tO[1] + lane_off + col + 16, u1);
          tmem_ld_wait();
          if (half == 1 && qq == 1) {
            // last read of O: the issuers may start the next item's PV
            // while this quarter is quantised and stored
            tc_fence_before();
            mbar_arrive(&bars.o_empty[o]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float y0 = c0 > 0.f ? c0 * __uint_as_float(v0[i]) : 0.f;
            float y1 = c0 > 0.f ? c0 * __uint_as_float(v1[i]) : 0.f;
            ov[i] = c1 > 0.f ? fmaf(c1, __uint_as_float(u0[i]), y0) : y0;
            ov[16 + i] = c1 > 0.f ? fmaf(c1, __uint_as_float(u1[i]), y1) : y1;
          }
          if constexpr (kPartial) {
            if (qi < w.n) {  // the normalised fp32 row, 32 features
              float4* dst = reinterpret_cast<float4*>(p.o_out + (m * p.num_heads + w.h) * kDv + col);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
            }
          } else if (qi < w.n) {
            uint32_t wd[4];
            uint32_t sb[2];
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              float R = 0.f;
              sb[blk] = gs_ok ? block_scale(fmaxf(amax8(ov + 16 * blk), amax8(ov + 16 * blk + 8)), kf, gs, R) : 0u;
              wd[2 * blk] = gs_ok ? encode8(ov + 16 * blk, R) : 0u;
              wd[2 * blk + 1] = gs_ok ? encode8(ov + 16 * blk + 8, R) : 0u;
            }
            *reinterpret_cast<uint4*>(code_row + col / 2) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            sbits |= (sb[0] | (sb[1] << 8)) << (16 * qq);
          }
        }
        if (!kPartial && qi < w.n) {
          const int64_t kc = static_cast<int64_t>(w.h) * 8 + 4 * half;
          *reinterpret_cast<uint32_t*>(p.scales + sf_offset(m, kc, k_tiles_sf)) = sbits;
        }
      }
      if (qi < w.n) {
        if (p.lse != nullptr)
          p.lse[static_cast<int64_t>(w.h) * p.total + m] = l_tot > 0.f ? (m_row + log2f(l_tot)) * kLn2 : -INFINITY;
        if (!kPartial && !gs_ok && qi == 0) flag_error(err, MLA_DEVERR_SCALE);
      }
    }
  }
  if (bad) flag_error(err, MLA_DEVERR_BOUNDS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // the last CTA to finish returns the counter to zero for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      __threadfence();
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
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

// [T, H, D] bf16 with element strides (st, sh, 1) as a 4-D map
// (64 features, H, T, D/64 chunks of 128 bytes); box = 64 features x 1 head x
// 128 tokens x all chunks, 128-byte swizzle: one copy per Q, K or V tile.
bool make_map(CUtensorMap* m, const void* base, int64_t D, int64_t H, int64_t T, int64_t st, int64_t sh) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(D / 64)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(st * 2), 128};
  cuuint32_t box[4] = {64, 1, 128, static_cast<cuuint32_t>(D / 64)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work counters: kSchedSlots pairs (next item, CTAs finished), each zero
// between launches.  Successive launches take successive slots, so launches
// that overlap on the device (other streams) use different counters unless
// kSchedSlots of them are in flight at once.
constexpr int kSchedSlots = 64;
__device__ uint32_t g_sched[kSchedSlots][2];

std::atomic<uint32_t> g_sched_next{0};

// A counter slot for the next launch.  The counters' address is looked up on
// every call: the lookup allocates nothing and follows the current context.
int sched_counter(uint32_t** out) {
  void* ptr = nullptr;
  if (const int st = cuda_status(cudaGetSymbolAddress(&ptr, g_sched))) return st;
  *out = static_cast<uint32_t*>(ptr) + 2 * (g_sched_next.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
  return MLA_OK;
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream, int num_sms) {
  const bool partial = a.o_out != nullptr;
  const int64_t total_k = a.cu_seqlens_k != nullptr ? a.total_k : a.total_tokens;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, kDqk, a.num_heads, a.total_tokens, a.q_st, a.q_sh) ||
      !make_map(&tk, a.k, kDqk, a.num_heads, total_k, a.k_st, a.k_sh) ||
      !make_map(&tv, a.v, kDv, a.num_heads, total_k, a.v_st, a.v_sh))
    return MLA_ERR_LAUNCH;
  Params p;
  p.cu = a.cu_seqlens;
  p.num_seqs = a.num_seqs;
  p.total = a.total_tokens;
  p.num_heads = a.num_heads;
  p.q_tiles = (a.max_seqlen + kBM - 1) / kBM;
  const int64_t items = static_cast<int64_t>(p.q_tiles) * a.num_seqs * a.num_heads;
  if (items > (int64_t(1) << 31) - 1) return MLA_ERR_INVALID_ARG;
  p.num_items = static_cast<uint32_t>(items);
  magic_divisor(p.q_tiles, &p.qt_magic, &p.qt_shift);
  magic_divisor(a.num_heads, &p.h_magic, &p.h_shift);
  if (const int st = sched_counter(&p.sched)) return st;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.gs = a.gs;
  p.codes = a.out_codes;
  p.scales = a.out_scales;
  p.lse = a.lse;
  p.error_word = a.error_word;
  p.o_out = a.o_out;
  p.cu_k = a.cu_seqlens_k;
  p.total_k = total_k;
  p.gs_q = a.gs_q;
  p.gs_k = a.gs_k;
  p.gs_v = a.gs_v;
  p.sparse24 = a.sparse24;
  const bool quant = a.gs_q != nullptr;
  if (quant && (partial || a.gs_k == nullptr || a.gs_v == nullptr)) return MLA_ERR_INVALID_ARG;
  const void* kern = partial ? reinterpret_cast<const void*>(prefill_tc_kernel<true, false>)
                     : quant ? reinterpret_cast<const void*>(prefill_tc_kernel<false, true>)
                             : reinterpret_cast<const void*>(prefill_tc_kernel<false, false>);
  if (const int st = smem_limit_once(kern, static_cast<int>(kSmemAlloc), partial ? 3 : quant ? 7 : 0)) return st;
  if (p.num_items == 0) return MLA_OK;
  // persistent: one CTA per SM
  const int grid = p.num_items < static_cast<uint32_t>(num_sms) ? static_cast<int>(p.num_items) : num_sms;
  if (partial)
    prefill_tc_kernel<true, false><<<grid, kThreads, kSmemAlloc, stream>>>(tq, tk, tv, p);
  else if (quant)
    prefill_tc_kernel<false, true><<<grid, kThreads, kSmemAlloc, stream>>>(tq, tk, tv, p);
  else
    prefill_tc_kernel<false, false><<<grid, kThreads, kSmemAlloc, stream>>>(tq, tk, tv, p);
  return launch_status();
}

}  // namespace mla
