// mla_nvfp4_decode_noalloc: the absorbed decode with its split partials in a
// scratch array compiled into the library instead of a caller workspace.
//
// For callers that cannot pass device memory per call: a serving engine that
// has handed all free device memory to its KV-cache pool, a host program with
// no device allocator of its own, or a decode step that must not call
// cudaMalloc/cudaFree because they synchronise the device.  The call itself
// allocates nothing.  The scratch is one fixed array per device, so calls
// whose work overlaps on the device race; calls on one stream are ordered.
#include <cuda_runtime.h>

#include <cstdio>

#include "launch.h"

namespace {

constexpr size_t kScratchBytes = MLA_DECODE_STATIC_WORKSPACE_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch must stay a whole number of 256-byte units");

// One copy per device (module globals are per context).  Never cleared: the
// decode writes every partial row it merges.
__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

thread_local char t_message[512];

// Device address of the current device's scratch, looked up on every call
// (the lookup allocates nothing and follows the current context, so a reset
// device that loaded the module again gets the new address).
int scratch_address(void** ptr) {
  void* p = nullptr;
  if (const int st = mla::cuda_status(cudaGetSymbolAddress(&p, g_decode_scratch))) return st;
  if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 255u) != 0) return MLA_ERR_LAUNCH;
  *ptr = p;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_nvfp4_decode_noalloc(const void* q, int batch, int num_heads,
                                        const uint8_t* cache, int64_t num_slots, int record_bytes,
                                        const int32_t* page_table, int64_t page_table_stride,
                                        int page_size, const int32_t* seq_lens,
                                        const int32_t* topk_indices, int topk, float softmax_scale,
                                        const float* global_scale, void* out, float* lse,
                                        int num_splits, uint32_t* error_word, void* stream) {
  void* scratch = nullptr;
  if (batch >= 1 && num_heads >= 1) {
    const int sms = mla::current_device_sms();
    if (sms < 0) return -sms;
    if (num_splits > 1) {
      // uniform splits: batch x splits x heads partial rows must fit
      const long long rows = static_cast<long long>(batch) * num_splits * num_heads;
      if (rows > MLA_DECODE_STATIC_ROWS) {
        std::snprintf(t_message, sizeof t_message,
                      "mla_nvfp4_decode_noalloc: batch %d x splits %d x heads %d = %lld partial rows "
                      "exceed the built-in scratch of %d rows (%u bytes); pass fewer splits, 0 for the "
                      "length-aware plan, or use mla_nvfp4_decode with a caller workspace",
                      batch, num_splits, num_heads, rows, MLA_DECODE_STATIC_ROWS,
                      MLA_DECODE_STATIC_WORKSPACE_BYTES);
        mla::set_last_error(t_message);
        return MLA_ERR_WORKSPACE;
      }
    } else if (num_splits <= 0) {
      // the plan sizes its chunks to the scratch; its tables must fit
      const mla::DecodePlanLayout l = mla::decode_plan_layout(batch, num_heads, sms, kScratchBytes);
      if (l.total > kScratchBytes) {
        std::snprintf(t_message, sizeof t_message,
                      "mla_nvfp4_decode_noalloc: the work list of batch %d needs %zu bytes, more than the "
                      "built-in scratch of %u bytes; pass num_splits = 1 or use mla_nvfp4_decode",
                      batch, l.total, MLA_DECODE_STATIC_WORKSPACE_BYTES);
        mla::set_last_error(t_message);
        return MLA_ERR_WORKSPACE;
      }
    }
    if (num_splits != 1)
      if (const int st = scratch_address(&scratch)) return st;
  }
  return mla_nvfp4_decode(q, batch, num_heads, cache, num_slots, record_bytes, page_table,
                          page_table_stride, page_size, seq_lens, topk_indices, topk,
                          softmax_scale, global_scale, out, lse, scratch,
                          scratch != nullptr ? kScratchBytes : 0, num_splits, error_word, stream);
}
