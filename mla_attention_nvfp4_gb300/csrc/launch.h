// Internal launch interface between the C ABI (abi.cu) and the kernel files.
// Arguments are validated by the caller; these functions only launch.
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/mla_nvfp4.h"

namespace mla {

// Division by an invariant integer using multiplication (Granlund and
// Montgomery 1994): for a divisor d >= 1, shift = ceil(log2 d) and
// magic = floor(2^32 (2^shift - d) / d) + 1 give n / d as
// (umulhi(n, magic) + n) >> shift, exactly, for every n < 2^31.
inline void magic_divisor(int d, uint32_t* magic, int* shift) {
  d = d > 0 ? d : 1;
  int l = 0;
  while ((int64_t(1) << l) < d) ++l;
  *shift = l;
  *magic = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
}

// Record a CUDA failure for mla_nvfp4_last_error() and map it to a status.
int cuda_status(cudaError_t e);
// MLA_OK after a successful launch sequence, else the recorded failure.
int launch_status();
// Make mla_nvfp4_last_error() return `message` (which must outlive the
// calling thread's next library call) on this thread.
void set_last_error(const char* message);
// SM count of the current device, or -MLA_ERR_UNSUPPORTED_DEVICE when it
// is not sm_103.
int current_device_sms();
// Raise `kernel`'s dynamic shared memory limit to `bytes` on the current
// device, once per device and kernel slot (the attribute persists), so that
// launches inside a stream capture make no attribute calls.  `slot` names
// the kernel (0 .. 15).
int smem_limit_once(const void* kernel, int bytes, int slot);

int launch_cache_write(const void* kv_c, int64_t kv_stride, const void* k_pe, int64_t pe_stride,
                       const int64_t* slot_mapping, int64_t num_tokens, uint8_t* cache,
                       int64_t num_slots, int record_bytes, const float* gs,
                       uint32_t* error_word, cudaStream_t stream, int num_sms);

int launch_selftest_wait(uint32_t* error_word, int64_t limit_ns, unsigned long long* elapsed_ns,
                         cudaStream_t stream);
int launch_quantize_rows(const float* x, int64_t M, int64_t N, const float* gs, uint8_t* codes,
                         uint8_t* scales, uint32_t* error_word, cudaStream_t stream);

int launch_global_scale(const void* x, int64_t n, float* gs, cudaStream_t stream, int num_sms);

int launch_gather_latent(const uint8_t* cache, int64_t num_slots, int record_bytes, const float* gs,
                         const int64_t* slots, int64_t n, void* kv_c, void* k_pe, uint32_t* error_word,
                         cudaStream_t stream, int num_sms);
int launch_merge_fused_out(const float* o_parts, const float* lse_parts, int parts, int64_t T, int H,
                           const float* gs, uint8_t* codes, uint8_t* scales, float* lse, uint32_t* error_word,
                           cudaStream_t stream);

struct DecodeArgs {
  const void* q;
  int batch;
  int num_heads;
  const uint8_t* cache;
  int64_t num_slots;
  int record_bytes;
  const int32_t* page_table;
  int64_t page_table_stride;
  int page_size;
  const int32_t* seq_lens;
  const int32_t* topk_indices;
  int topk;
  float softmax_scale;
  const float* gs;
  const float* gs_q;  // non-null: NVFP4-query mode with this query global scale
  void* out;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  int num_splits;  // uniform mode: key splits per sequence
  bool planned;    // length-aware plan computed on the device (num_splits ignored)
  uint32_t* error_word;
};

// Decode workspace for uniform splits: partial rows (b, split, head).
size_t decode_workspace_bytes(int batch, int num_heads, int num_splits);
int decode_default_splits(int batch, int num_heads, int num_sms);

// Workspace of the planned decode: a 256-byte header, the item list, the
// per-sequence chunk table, then max_rows chunk rows of partial O (heads x
// 512 fp32 each) and their LSE.  `bytes` == 0 gives the full size (one row
// per possible item); otherwise max_rows is what fits in `bytes`.
struct DecodePlanLayout {
  int pairs, max_items, max_rows;
  size_t items, seqs, rows, lse, total;
};
DecodePlanLayout decode_plan_layout(int batch, int num_heads, int num_sms, size_t bytes);
// 1 when the planned decode of these (host) sequence lengths would keep one
// chunk per sequence, i.e. the one-split launch does the same work without
// the plan and merge kernels; 0 otherwise.  The same estimate as the device
// plan, on the host.
int decode_plan_one_chunk(const int32_t* lens, int batch, int num_heads, int num_sms, size_t bytes);
int launch_decode(const DecodeArgs& a, cudaStream_t stream, int num_sms);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const int32_t* cu_seqlens;
  int num_seqs;
  int64_t total_tokens;
  int max_seqlen;
  int num_heads;
  float softmax_scale;
  const float* gs;
  uint8_t* out_codes;
  uint8_t* out_scales;
  float* lse;
  uint32_t* error_word;
  // partial mode (o_out set): fp32 normalised output, no codes; a key table
  // (cu_seqlens_k over total_k key rows) makes every key of a sequence's
  // chunk visible instead of the causal prefix of its own tokens
  float* o_out = nullptr;
  const int32_t* cu_seqlens_k = nullptr;
  int64_t total_k = 0;
  // fake-quant mode (gs_q set): q, k, v hold the f16 code * scale values of
  // NVFP4 operands (launch_qdq_operands) with these global scales; P is
  // quantised to NVFP4 along the keys, optionally after 2:4 score sparsity
  const float* gs_q = nullptr;
  const float* gs_k = nullptr;
  const float* gs_v = nullptr;
  int sparse24 = 0;
};

int launch_prefill(const PrefillArgs& a, cudaStream_t stream, int num_sms);

// NVFP4 fake quantisation of the prefill operands (code * scale as f16).
struct QdqArgs {
  const void* q;
  const void* k;
  const void* v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const int32_t* cu_seqlens;
  int num_seqs;
  int64_t total;
  int max_seqlen;
  int num_heads;
  const float* gs_q;
  const float* gs_k;
  const float* gs_v;
  void* q_out;  // f16 [total, H, 192]
  void* k_out;  // f16 [total, H, 192]
  void* v_out;  // f16 [total, H, 128]
  uint32_t* error_word;
};
int launch_qdq_operands(const QdqArgs& a, cudaStream_t stream);

struct GemmArgs {
  const uint8_t* a_codes;
  const uint8_t* a_scales;
  int64_t M;
  const uint8_t* w_codes;
  const uint8_t* w_scales;
  int64_t N, K;
  const float* gs_a;
  const float* gs_w;
  void* out;
  int64_t ldc;
  uint32_t* error_word;
};

int launch_gemm(const GemmArgs& a, cudaStream_t stream, int num_sms);

}  // namespace mla
