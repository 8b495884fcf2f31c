// C ABI of the library: host-side argument checks, then one launch sequence
// on the caller's stream.  Nothing here allocates or keeps state beyond a
// per-device cache of the SM count and compute capability.
#include <cuda_runtime.h>

#include <atomic>

#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_info[kMaxDevices];  // 0 = unknown, else (cc << 16) | num_sms

// Current device's SM count, or a negative status when the device is not
// sm_103 (the only target the library is built for).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -MLA_ERR_UNSUPPORTED_DEVICE;
  int info = dev < kMaxDevices ? g_dev_info[dev].load(std::memory_order_relaxed) : 0;
  if (info == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return -MLA_ERR_UNSUPPORTED_DEVICE;
    info = ((major * 10 + minor) << 16) | (sms & 0xFFFF);
    if (dev < kMaxDevices) g_dev_info[dev].store(info, std::memory_order_relaxed);
  }
  if ((info >> 16) != 103) return -MLA_ERR_UNSUPPORTED_DEVICE;
  return info & 0xFFFF;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

thread_local const char* t_last_error = "";

}  // namespace

namespace mla {
int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  t_last_error = cudaGetErrorString(e);
  return MLA_ERR_LAUNCH;
}
int launch_status() { return cuda_status(cudaGetLastError()); }
void set_last_error(const char* message) { t_last_error = message; }
int current_device_sms() { return device_sms(); }
int smem_limit_once(const void* kernel, int bytes, int slot) {
  static std::atomic<uint64_t> done[16];  // bit d: set on device d
  int dev = 0;
  if (const int st = cuda_status(cudaGetDevice(&dev))) return st;
  if (slot < 0 || slot >= 16 || dev < 0 || dev >= 64) return MLA_ERR_LAUNCH;
  const uint64_t bit = uint64_t(1) << dev;
  if (done[slot].load(std::memory_order_acquire) & bit) return MLA_OK;
  if (const int st = cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)))
    return st;
  done[slot].fetch_or(bit, std::memory_order_acq_rel);
  return MLA_OK;
}
}  // namespace mla

extern "C" {

const char* mla_nvfp4_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null pointer, bad size or mode mix";
    case MLA_ERR_RECORD_BYTES: return "MLA_ERR_RECORD_BYTES: NVFP4 MLA cache record must be 368 or 432 bytes";
    case MLA_ERR_ALIGNMENT: return "MLA_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
    case MLA_ERR_UNSUPPORTED_DEVICE: return "MLA_ERR_UNSUPPORTED_DEVICE: current device is not sm_103 (GB300)";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: decode workspace missing or too small";
    case MLA_ERR_LAUNCH: return "MLA_ERR_LAUNCH: CUDA launch failed";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_nvfp4_abi_version(void) { return MLA_NVFP4_ABI_VERSION; }

const char* mla_nvfp4_last_error(void) { return t_last_error; }

int mla_nvfp4_global_scale(const void* x, int64_t n, float* gs, void* stream) {
  if (x == nullptr || gs == nullptr || n < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x)) return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  return mla::launch_global_scale(x, n, gs, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_cache_write(const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                          int64_t k_pe_stride, const int64_t* slot_mapping, int64_t num_tokens,
                          uint8_t* cache, int64_t num_slots, int record_bytes,
                          const float* global_scale, uint32_t* error_word, void* stream) {
  if (record_bytes != MLA_RECORD_BF16_ROPE && record_bytes != MLA_RECORD_FP8_ROPE)
    return MLA_ERR_RECORD_BYTES;
  if (num_tokens < 0 || num_slots < 0) return MLA_ERR_INVALID_ARG;
  if (num_tokens > 0 && (kv_c == nullptr || k_pe == nullptr || slot_mapping == nullptr ||
                         cache == nullptr || global_scale == nullptr))
    return MLA_ERR_INVALID_ARG;
  if (kv_c_stride < MLA_D_LATENT || k_pe_stride < MLA_D_ROPE) return MLA_ERR_INVALID_ARG;
  if (!aligned16(kv_c) || !aligned16(k_pe) || !aligned16(cache) || (kv_c_stride * 2) % 16 ||
      (k_pe_stride * 2) % 16)
    return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  return mla::launch_cache_write(kv_c, kv_c_stride, k_pe, k_pe_stride, slot_mapping, num_tokens,
                                 cache, num_slots, record_bytes, global_scale, error_word,
                                 static_cast<cudaStream_t>(stream), sms);
}

size_t mla_nvfp4_decode_workspace_size(int batch, int num_heads, int num_splits) {
  if (batch < 1 || num_heads < 1) return 0;
  if (num_splits == 1) return 0;
  if (num_splits <= 0) {
    const int sms = device_sms();
    return mla::decode_plan_layout(batch, num_heads, sms > 0 ? sms : 152, 0).total;
  }
  return mla::decode_workspace_bytes(batch, num_heads, num_splits);
}

int mla_nvfp4_decode_default_splits(int batch, int num_heads, int num_splits) {
  if (batch < 1 || num_heads < 1) return 0;
  if (num_splits > 0) return num_splits;
  const int sms = device_sms();
  return mla::decode_default_splits(batch, num_heads, sms > 0 ? sms : 152);
}

int mla_nvfp4_decode_plan_splits(const int32_t* seq_lens_host, int batch, int num_heads, size_t workspace_bytes) {
  if (seq_lens_host == nullptr || batch < 1 || num_heads < 1) return 0;
  const int sms = device_sms();
  if (sms <= 0) return 0;
  return mla::decode_plan_one_chunk(seq_lens_host, batch, num_heads, sms, workspace_bytes);
}

}  // extern "C"

namespace {

// The argument checks of mla_nvfp4_decode, run before anything is enqueued;
// on MLA_OK the launch arguments are in *a and the SM count in *sms.
int decode_prepare(const void* q, int batch, int num_heads, const uint8_t* cache, int64_t num_slots,
                   int record_bytes, const int32_t* page_table, int64_t page_table_stride,
                   int page_size, const int32_t* seq_lens, const int32_t* topk_indices, int topk,
                   float softmax_scale, const float* global_scale, void* out, float* lse,
                   void* workspace, size_t workspace_bytes, int num_splits, uint32_t* error_word,
                   mla::DecodeArgs* a, int* sms_out, const float* q_global_scale = nullptr) {
  if (record_bytes != MLA_RECORD_BF16_ROPE && record_bytes != MLA_RECORD_FP8_ROPE)
    return MLA_ERR_RECORD_BYTES;
  if (batch < 0 || num_heads < 1 || num_slots < 0) return MLA_ERR_INVALID_ARG;
  const bool paged = page_table != nullptr || seq_lens != nullptr;
  const bool sparse = topk_indices != nullptr;
  if (paged == sparse) return MLA_ERR_INVALID_ARG;  // exactly one mode
  if (paged && (page_table == nullptr || seq_lens == nullptr || page_size < 1 ||
                page_table_stride < 1))
    return MLA_ERR_INVALID_ARG;
  if (sparse && topk < 0) return MLA_ERR_INVALID_ARG;
  if (batch == 0) {
    *sms_out = 0;
    return MLA_OK;
  }
  if (q == nullptr || cache == nullptr || global_scale == nullptr || out == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !(softmax_scale < 3.0e38f)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(out)) return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  if (num_splits > 4096) return MLA_ERR_INVALID_ARG;
  // num_splits <= 0: in top-k mode every row has the same number of index
  // entries, so the split count follows from the sizes alone (enough splits
  // to fill the SMs); in paged mode, with a workspace, the length-aware
  // plan, and without one, one split per sequence.  One split needs no
  // workspace.
  if (num_splits <= 0 && sparse) num_splits = mla::decode_default_splits(batch, num_heads, sms);
  const bool planned = num_splits <= 0 && workspace != nullptr;
  if (num_splits <= 0 && !planned) num_splits = 1;
  if (planned || num_splits > 1) {
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLA_ERR_WORKSPACE;
    if (planned) {
      const mla::DecodePlanLayout l = mla::decode_plan_layout(batch, num_heads, sms, workspace_bytes);
      if (workspace_bytes < l.total) return MLA_ERR_WORKSPACE;
    } else if (workspace_bytes < mla::decode_workspace_bytes(batch, num_heads, num_splits)) {
      return MLA_ERR_WORKSPACE;
    }
  }
  *a = mla::DecodeArgs{q, batch, num_heads, cache, num_slots, record_bytes, page_table,
                       page_table_stride, page_size, seq_lens, topk_indices, sparse ? topk : 0,
                       softmax_scale, global_scale, q_global_scale, out, lse, workspace, workspace_bytes,
                       planned ? 0 : num_splits, planned, error_word};
  *sms_out = sms;
  return MLA_OK;
}

int copy_async(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t stream) {
  if (bytes == 0) return MLA_OK;
  return mla::cuda_status(cudaMemcpyAsync(dst, src, bytes, kind, stream));
}

}  // namespace

extern "C" {

int mla_nvfp4_decode(const void* q, int batch, int num_heads, const uint8_t* cache,
                     int64_t num_slots, int record_bytes, const int32_t* page_table,
                     int64_t page_table_stride, int page_size, const int32_t* seq_lens,
                     const int32_t* topk_indices, int topk, float softmax_scale,
                     const float* global_scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, int num_splits, uint32_t* error_word, void* stream) {
  mla::DecodeArgs a;
  int sms = 0;
  if (const int st = decode_prepare(q, batch, num_heads, cache, num_slots, record_bytes, page_table,
                                    page_table_stride, page_size, seq_lens, topk_indices, topk,
                                    softmax_scale, global_scale, out, lse, workspace,
                                    workspace_bytes, num_splits, error_word, &a, &sms))
    return st;
  if (batch == 0) return MLA_OK;
  return mla::launch_decode(a, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_decode_q4(const void* q, int batch, int num_heads, const uint8_t* cache,
                        int64_t num_slots, int record_bytes, const int32_t* page_table,
                        int64_t page_table_stride, int page_size, const int32_t* seq_lens,
                        const int32_t* topk_indices, int topk, float softmax_scale,
                        const float* global_scale, const float* q_global_scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, int num_splits, uint32_t* error_word,
                        void* stream) {
  if (batch > 0 && q_global_scale == nullptr) return MLA_ERR_INVALID_ARG;
  mla::DecodeArgs a;
  int sms = 0;
  if (const int st = decode_prepare(q, batch, num_heads, cache, num_slots, record_bytes, page_table,
                                    page_table_stride, page_size, seq_lens, topk_indices, topk,
                                    softmax_scale, global_scale, out, lse, workspace,
                                    workspace_bytes, num_splits, error_word, &a, &sms, q_global_scale))
    return st;
  if (batch == 0) return MLA_OK;
  return mla::launch_decode(a, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_decode_host(const void* q_host, void* q_dev, int batch, int num_heads,
                          const uint8_t* cache, int64_t num_slots, int record_bytes,
                          const int32_t* page_table_host, int32_t* page_table_dev,
                          int64_t page_table_stride, int page_size, const int32_t* seq_lens_host,
                          int32_t* seq_lens_dev, const int32_t* topk_host, int32_t* topk_dev,
                          int topk, float softmax_scale, const float* global_scale,
                          void* out_host, void* out_dev, float* lse_host, float* lse_dev,
                          void* workspace, size_t workspace_bytes, int num_splits,
                          uint32_t* error_word, void* stream) {
  // every host buffer comes with the device buffer that receives (or feeds) it
  if ((q_host == nullptr) != (q_dev == nullptr) || (out_host == nullptr) != (out_dev == nullptr) ||
      (page_table_host == nullptr) != (page_table_dev == nullptr) ||
      (seq_lens_host == nullptr) != (seq_lens_dev == nullptr) ||
      (topk_host == nullptr) != (topk_dev == nullptr) || (lse_host == nullptr) != (lse_dev == nullptr))
    return record_bytes != MLA_RECORD_BF16_ROPE && record_bytes != MLA_RECORD_FP8_ROPE
               ? MLA_ERR_RECORD_BYTES
               : MLA_ERR_INVALID_ARG;
  // the lengths are on the host: where the length-aware plan would keep one
  // chunk per sequence, launch that directly (no plan or merge kernel)
  if (num_splits <= 0 && seq_lens_host != nullptr && workspace != nullptr &&
      mla_nvfp4_decode_plan_splits(seq_lens_host, batch, num_heads, workspace_bytes) == 1)
    num_splits = 1;
  mla::DecodeArgs a;
  int sms = 0;
  if (const int st = decode_prepare(q_dev, batch, num_heads, cache, num_slots, record_bytes,
                                    page_table_dev, page_table_stride, page_size, seq_lens_dev,
                                    topk_dev, topk, softmax_scale, global_scale, out_dev, lse_dev,
                                    workspace, workspace_bytes, num_splits, error_word, &a, &sms))
    return st;
  if (batch == 0) return MLA_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t b = static_cast<size_t>(batch), h = static_cast<size_t>(num_heads);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  if (const int st = copy_async(q_dev, q_host, b * h * (MLA_D_LATENT + MLA_D_ROPE) * 2, h2d, s)) return st;
  if (page_table_dev != nullptr) {
    if (const int st = copy_async(page_table_dev, page_table_host,
                                  b * static_cast<size_t>(page_table_stride) * 4, h2d, s))
      return st;
    if (const int st = copy_async(seq_lens_dev, seq_lens_host, b * 4, h2d, s)) return st;
  } else {
    if (const int st = copy_async(topk_dev, topk_host, b * static_cast<size_t>(topk) * 4, h2d, s))
      return st;
  }
  if (const int st = mla::launch_decode(a, s, sms)) return st;
  if (const int st = copy_async(out_host, out_dev, b * h * MLA_D_LATENT * 2, d2h, s)) return st;
  if (lse_dev != nullptr)
    if (const int st = copy_async(lse_host, lse_dev, b * h * 4, d2h, s)) return st;
  return MLA_OK;
}

int mla_nvfp4_prefill_fused_out(const void* q, const void* k, const void* v,
                                int64_t q_stride_t, int64_t q_stride_h, int64_t k_stride_t,
                                int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                                const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                int max_seqlen, int num_heads, float softmax_scale,
                                const float* global_scale, uint8_t* out_codes,
                                uint8_t* out_scales, float* lse, uint32_t* error_word,
                                void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || num_heads < 1)
    return MLA_ERR_INVALID_ARG;
  if (total_tokens == 0 || num_seqs == 0) {
    if (total_tokens != 0) return MLA_ERR_INVALID_ARG;
    return MLA_OK;
  }
  if (max_seqlen < 1 || total_tokens > (int64_t(1) << 31) - 1) return MLA_ERR_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || cu_seqlens == nullptr ||
      global_scale == nullptr || out_codes == nullptr || out_scales == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !(softmax_scale < 3.0e38f)) return MLA_ERR_INVALID_ARG;
  if (q_stride_h < MLA_D_QK_PREFILL || k_stride_h < MLA_D_QK_PREFILL ||
      v_stride_h < MLA_D_V_PREFILL || q_stride_t < q_stride_h * (num_heads - 1) + MLA_D_QK_PREFILL ||
      k_stride_t < k_stride_h * (num_heads - 1) + MLA_D_QK_PREFILL ||
      v_stride_t < v_stride_h * (num_heads - 1) + MLA_D_V_PREFILL)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_codes) ||
      (reinterpret_cast<uintptr_t>(out_scales) & 3u) != 0 ||
      (q_stride_t * 2) % 16 || (q_stride_h * 2) % 16 || (k_stride_t * 2) % 16 ||
      (k_stride_h * 2) % 16 || (v_stride_t * 2) % 16 || (v_stride_h * 2) % 16)
    return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  mla::PrefillArgs a{q, k, v, q_stride_t, q_stride_h, k_stride_t, k_stride_h, v_stride_t,
                     v_stride_h, cu_seqlens, num_seqs, total_tokens, max_seqlen, num_heads,
                     softmax_scale, global_scale, out_codes, out_scales, lse, error_word};
  return mla::launch_prefill(a, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_scales, int64_t M, const uint8_t* w_codes,
                   const uint8_t* w_scales, int64_t N, int64_t K, const float* gs_a, const float* gs_w,
                   void* out, int64_t ldc, uint32_t* error_word, void* stream) {
  if (M < 0 || N < 0 || K < 0 || (N > 0 && N % 128 != 0) || (K > 0 && K % 256 != 0)) return MLA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MLA_OK;
  if (K == 0) return MLA_ERR_INVALID_ARG;
  if (a_codes == nullptr || a_scales == nullptr || w_codes == nullptr || w_scales == nullptr || gs_a == nullptr ||
      gs_w == nullptr || out == nullptr || ldc < N || M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) || !aligned16(w_scales) ||
      !aligned16(out) || (ldc * 2) % 16 != 0)
    return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  mla::GemmArgs a{a_codes, a_scales, M, w_codes, w_scales, N, K, gs_a, gs_w, out, ldc, error_word};
  return mla::launch_gemm(a, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_prefill_partial(const void* q, const void* k, const void* v, int64_t q_stride_t,
                              int64_t q_stride_h, int64_t k_stride_t, int64_t k_stride_h, int64_t v_stride_t,
                              int64_t v_stride_h, const int32_t* cu_seqlens, const int32_t* cu_seqlens_k,
                              int num_seqs, int64_t total_tokens, int64_t total_k, int max_seqlen,
                              int num_heads, float softmax_scale, float* out, float* lse,
                              uint32_t* error_word, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || num_heads < 1 || total_k < 0)
    return MLA_ERR_INVALID_ARG;
  if (total_tokens == 0 || num_seqs == 0) return total_tokens != 0 ? MLA_ERR_INVALID_ARG : MLA_OK;
  if (max_seqlen < 1 || total_tokens > (int64_t(1) << 31) - 1 || total_k > (int64_t(1) << 31) - 1)
    return MLA_ERR_INVALID_ARG;
  if (q == nullptr || cu_seqlens == nullptr || out == nullptr || lse == nullptr) return MLA_ERR_INVALID_ARG;
  const int64_t tk = cu_seqlens_k != nullptr ? total_k : total_tokens;
  if (tk > 0 && (k == nullptr || v == nullptr)) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !(softmax_scale < 3.0e38f)) return MLA_ERR_INVALID_ARG;
  if (q_stride_h < MLA_D_QK_PREFILL || k_stride_h < MLA_D_QK_PREFILL || v_stride_h < MLA_D_V_PREFILL ||
      q_stride_t < q_stride_h * (num_heads - 1) + MLA_D_QK_PREFILL ||
      k_stride_t < k_stride_h * (num_heads - 1) + MLA_D_QK_PREFILL ||
      v_stride_t < v_stride_h * (num_heads - 1) + MLA_D_V_PREFILL)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (q_stride_t * 2) % 16 ||
      (q_stride_h * 2) % 16 || (k_stride_t * 2) % 16 || (k_stride_h * 2) % 16 || (v_stride_t * 2) % 16 ||
      (v_stride_h * 2) % 16)
    return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  mla::PrefillArgs a{q, k, v, q_stride_t, q_stride_h, k_stride_t, k_stride_h, v_stride_t,
                     v_stride_h, cu_seqlens, num_seqs, total_tokens, max_seqlen, num_heads,
                     softmax_scale, nullptr, nullptr, nullptr, lse, error_word};
  a.o_out = out;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_k = total_k;
  if (cu_seqlens_k != nullptr && total_k == 0) {
    // every chunk empty (the kernel writes O = 0, LSE = -inf): the key maps
    // still need a valid base, and no key block is read
    a.k = q;
    a.v = q;
    a.k_st = q_stride_t;
    a.k_sh = q_stride_h;
    a.v_st = q_stride_t;
    a.v_sh = q_stride_h;
    a.total_k = 1;
  }
  return mla::launch_prefill(a, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_prefill_qdq(const void* q, const void* k, const void* v, int64_t q_stride_t, int64_t q_stride_h,
                          int64_t k_stride_t, int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                          const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int max_seqlen,
                          int num_heads, const float* gs_q, const float* gs_k, const float* gs_v, void* q_out,
                          void* k_out, void* v_out, uint32_t* error_word, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (total_tokens == 0 || num_seqs == 0) return total_tokens != 0 ? MLA_ERR_INVALID_ARG : MLA_OK;
  if (max_seqlen < 1 || total_tokens > (int64_t(1) << 31) - 1) return MLA_ERR_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || cu_seqlens == nullptr || gs_q == nullptr ||
      gs_k == nullptr || gs_v == nullptr || q_out == nullptr || k_out == nullptr || v_out == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (q_stride_h < MLA_D_QK_PREFILL || k_stride_h < MLA_D_QK_PREFILL || v_stride_h < MLA_D_V_PREFILL ||
      q_stride_t < q_stride_h * (num_heads - 1) + MLA_D_QK_PREFILL ||
      k_stride_t < k_stride_h * (num_heads - 1) + MLA_D_QK_PREFILL ||
      v_stride_t < v_stride_h * (num_heads - 1) + MLA_D_V_PREFILL)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || !aligned16(k_out) ||
      (reinterpret_cast<uintptr_t>(v) & 3u) != 0 || (reinterpret_cast<uintptr_t>(v_out) & 3u) != 0 ||
      (q_stride_t * 2) % 16 || (q_stride_h * 2) % 16 || (k_stride_t * 2) % 16 || (k_stride_h * 2) % 16 ||
      (v_stride_t * 2) % 4 || (v_stride_h * 2) % 4)
    return MLA_ERR_ALIGNMENT;
  mla::QdqArgs a{q, k, v, q_stride_t, q_stride_h, k_stride_t, k_stride_h, v_stride_t, v_stride_h, cu_seqlens,
                 num_seqs, total_tokens, max_seqlen, num_heads, gs_q, gs_k, gs_v, q_out, k_out, v_out, error_word};
  return mla::launch_qdq_operands(a, static_cast<cudaStream_t>(stream));
}

int mla_nvfp4_prefill_fakequant(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int num_seqs,
                                int64_t total_tokens, int max_seqlen, int num_heads, float softmax_scale,
                                const float* gs_q, const float* gs_k, const float* gs_v, int sparse24,
                                const float* global_scale, uint8_t* out_codes, uint8_t* out_scales, float* lse,
                                uint32_t* error_word, void* stream) {
  if (gs_q == nullptr || gs_k == nullptr || gs_v == nullptr || (sparse24 != 0 && sparse24 != 1))
    return MLA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (total_tokens == 0 || num_seqs == 0) return total_tokens != 0 ? MLA_ERR_INVALID_ARG : MLA_OK;
  if (max_seqlen < 1 || total_tokens > (int64_t(1) << 31) - 1) return MLA_ERR_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || cu_seqlens == nullptr || global_scale == nullptr ||
      out_codes == nullptr || out_scales == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !(softmax_scale < 3.0e38f)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out_codes) ||
      (reinterpret_cast<uintptr_t>(out_scales) & 3u) != 0)
    return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  const int64_t H = num_heads;
  mla::PrefillArgs a{q, k, v, H * MLA_D_QK_PREFILL, MLA_D_QK_PREFILL, H * MLA_D_QK_PREFILL, MLA_D_QK_PREFILL,
                     H * MLA_D_V_PREFILL, MLA_D_V_PREFILL, cu_seqlens, num_seqs, total_tokens, max_seqlen, num_heads,
                     softmax_scale, global_scale, out_codes, out_scales, lse, error_word};
  a.gs_q = gs_q;
  a.gs_k = gs_k;
  a.gs_v = gs_v;
  a.sparse24 = sparse24;
  return mla::launch_prefill(a, static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_merge_fused_out(const float* o_parts, const float* lse_parts, int num_parts, int64_t total_tokens,
                              int num_heads, const float* global_scale, uint8_t* out_codes, uint8_t* out_scales,
                              float* lse, uint32_t* error_word, void* stream) {
  if (num_parts < 1 || total_tokens < 0 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (total_tokens == 0) return MLA_OK;
  if (o_parts == nullptr || lse_parts == nullptr || global_scale == nullptr || out_codes == nullptr ||
      out_scales == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || (reinterpret_cast<uintptr_t>(out_codes) & 7u) != 0) return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  return mla::launch_merge_fused_out(o_parts, lse_parts, num_parts, total_tokens, num_heads, global_scale,
                                     out_codes, out_scales, lse, error_word, static_cast<cudaStream_t>(stream));
}

int mla_nvfp4_gather_latent(const uint8_t* cache, int64_t num_slots, int record_bytes, const float* global_scale,
                            const int64_t* slots, int64_t n, void* kv_c, void* k_pe, uint32_t* error_word,
                            void* stream) {
  if (record_bytes != MLA_RECORD_BF16_ROPE && record_bytes != MLA_RECORD_FP8_ROPE) return MLA_ERR_RECORD_BYTES;
  if (n < 0 || num_slots < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (cache == nullptr || global_scale == nullptr || slots == nullptr || kv_c == nullptr || k_pe == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(kv_c) || !aligned16(k_pe)) return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  return mla::launch_gather_latent(cache, num_slots, record_bytes, global_scale, slots, n, kv_c, k_pe, error_word,
                                   static_cast<cudaStream_t>(stream), sms);
}

int mla_nvfp4_quantize_rows(const float* x, int64_t M, int64_t N, const float* global_scale,
                            uint8_t* codes, uint8_t* scales, uint32_t* error_word, void* stream) {
  if (M < 0 || N < 0 || N % 16 != 0) return MLA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return MLA_OK;
  if (x == nullptr || global_scale == nullptr || codes == nullptr || scales == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u) != 0) return MLA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  return mla::launch_quantize_rows(x, M, N, global_scale, codes, scales, error_word,
                                   static_cast<cudaStream_t>(stream));
}

int mla_nvfp4_selftest_wait(uint32_t* error_word, int64_t limit_ns, unsigned long long* elapsed_ns,
                            void* stream) {
  if (error_word == nullptr || limit_ns < 1000 || limit_ns > 1000000000) return MLA_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms < 0) return -sms;
  return mla::launch_selftest_wait(error_word, limit_ns, elapsed_ns, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
