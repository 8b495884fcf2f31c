/*
 * mla_nvfp4.h -- C ABI of the GB300 (sm_103a) MLA attention library with an
 * NVFP4 latent cache and NVFP4 fused prefill output.
 *
 * NVFP4 here: e2m1 codes packed two per byte (even element in the low
 * nibble), one e4m3 block scale per 16 elements along the contraction axis,
 * and an fp32 global scale gs in the dequantisation direction:
 *     x_hat = e2m1(code) * e4m3(scale) * gs,   gs = amax / (6 * 448).
 * Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
 * TRITON_MLA) - #2244", PR description, "Contract notes".
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers unless stated otherwise.  The caller
 *    owns every buffer (including decode workspace); the library allocates
 *    nothing and keeps no state between calls, except that
 *    mla_nvfp4_decode_noalloc uses a fixed scratch area compiled into the
 *    library (see there).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *    enqueued asynchronously; the return value covers host-side argument
 *    checks and the launch only.
 *  - `error_word` (nullable) is a device uint32 the kernels OR MLA_DEVERR_*
 *    bits into when they meet out-of-range indices (the access is skipped)
 *    or an invalid global scale.  The caller clears it; the library never
 *    does.
 *  - Return values are mla_status_t codes; nothing is launched when a check
 *    fails.  The library must run on an sm_103 device (GB300); any other
 *    device gives MLA_ERR_UNSUPPORTED_DEVICE before any launch.
 */
#ifndef MLA_NVFP4_H
#define MLA_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NVFP4_ABI_VERSION 2

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,        /* null pointer, bad size, bad mode mix    */
  MLA_ERR_RECORD_BYTES = 2,       /* record_bytes not 432 or 368             */
  MLA_ERR_ALIGNMENT = 3,          /* pointer or stride not 16-byte aligned   */
  MLA_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103            */
  MLA_ERR_WORKSPACE = 5,          /* decode workspace missing or too small   */
  MLA_ERR_LAUNCH = 6,             /* CUDA launch or attribute error          */
} mla_status_t;

/* Bits OR-ed into *error_word by the kernels. */
#define MLA_DEVERR_BOUNDS 0x1u  /* slot, page or index out of range: skipped */
#define MLA_DEVERR_TIMEOUT 0x2u /* a bounded pipeline wait gave up           */
#define MLA_DEVERR_SCALE 0x4u   /* global scale <= 0 or not finite           */
#define MLA_DEVERR_RANGE 0x8u   /* a value outside the kernel's operand range
                                   (decode: |k_pe| > 65504), saturated     */

/* Fixed MLA dimensions (DeepSeek-style absorbed MLA). */
#define MLA_D_LATENT 512   /* kv_c, the NVFP4 latent; also the decode V dim */
#define MLA_D_ROPE 64      /* k_pe                                          */
#define MLA_D_QK_DECODE 576
#define MLA_D_QK_PREFILL 192
#define MLA_D_V_PREFILL 128
#define MLA_RECORD_BF16_ROPE 432
#define MLA_RECORD_FP8_ROPE 368

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_nvfp4_status_string(int status);

/* MLA_NVFP4_ABI_VERSION of the loaded library. */
int mla_nvfp4_abi_version(void);

/* The CUDA runtime's message for the last failed launch or attribute call
 * behind an MLA_ERR_LAUNCH return on the calling host thread ("" if none). */
const char* mla_nvfp4_last_error(void);

/*
 * Global (outer) scale of a bf16 tensor: *gs = fp32(amax|x| / 2688).
 * Source: "#2244" PR description, "Contract notes" (amax/(6*448)); the
 * b12x "nvfp4 MLA KV cache + per-layer outer-scale ... - #33" description
 * restores this per-layer fp32 scale on read.
 *   x  : bf16 [n], 16-byte aligned.   n >= 1.
 *   gs : one fp32, overwritten (cleared and reduced on `stream`).
 */
int mla_nvfp4_global_scale(const void* x, int64_t n, float* gs, void* stream);

/*
 * Quantise-on-write of the MLA latent cache (one record per token).
 * Source: "#2244", second commit message (the latent is quantised once at
 * cache-write time and both attention products read those bytes); "#33",
 * review of api.py (432-byte record = bf16 RoPE, 368-byte = fp8 RoPE, any
 * other width is an error).
 *   kv_c         : bf16 [num_tokens, 512], row stride kv_c_stride elements.
 *   k_pe         : bf16 [num_tokens, 64], row stride k_pe_stride elements.
 *   slot_mapping : int64 [num_tokens]; -1 skips the token; a slot >= num_slots
 *                  is skipped and flagged MLA_DEVERR_BOUNDS.
 *   cache        : uint8 [num_slots, record_bytes], 16-byte aligned.
 *   record_bytes : 432 or 368.
 *   global_scale : device fp32 gs.
 * Record layout: [0,256) codes, [256,288) 32 e4m3 scales, then k_pe as 64
 * bf16 (432) or 64 e4m3 RNE-saturating (368), then 16 zero bytes.
 * kv_c, k_pe and both strides (in bytes) must be 16-byte aligned.
 */
int mla_nvfp4_cache_write(const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                          int64_t k_pe_stride, const int64_t* slot_mapping, int64_t num_tokens,
                          uint8_t* cache, int64_t num_slots, int record_bytes,
                          const float* global_scale, uint32_t* error_word, void* stream);

/*
 * Bytes of decode workspace mla_nvfp4_decode needs for (batch, num_heads,
 * num_splits) on the current device:
 *   num_splits <= 0 : paged mode's length-aware plan (see mla_nvfp4_decode):
 *                     a small header and work list plus room for the split
 *                     partials of batch + SMs/2 items, each num_heads x 2052
 *                     bytes (enough for top-k mode's default splits too);
 *   num_splits == 1 : 0 (one split per sequence needs no workspace);
 *   num_splits > 1  : batch * num_splits * num_heads * 2048 bytes of partial
 *                     outputs plus their LSE (256-byte rounded).
 * Never fails: returns 0 for invalid sizes.
 */
size_t mla_nvfp4_decode_workspace_size(int batch, int num_heads, int num_splits);

/*
 * The number of equal key splits mla_nvfp4_decode uses for (batch,
 * num_heads) on the current device: num_splits itself when > 0, else the
 * default that fills the SMs, which top-k calls and paged calls without a
 * workspace use (paged calls with a workspace and num_splits <= 0 are
 * planned from the lengths instead).  Returns 0 for invalid sizes.
 * Launches per call: one with one split, two (decode, merge) with more,
 * three (plan, decode, merge) when planned.
 */
int mla_nvfp4_decode_default_splits(int batch, int num_heads, int num_splits);

/*
 * The paged decode's length-aware plan, evaluated on the host for sequence
 * lengths the caller holds in host memory (seq_lens_host, int32 [batch]),
 * with the same makespan estimate as the device plan and the workspace that
 * would be passed (workspace_bytes, which bounds the partial rows).  Returns
 * 1 when that plan keeps one chunk per sequence: mla_nvfp4_decode with
 * num_splits = 1 then runs the same tiles in the same order, without the
 * plan and merge kernels and without a workspace (one launch instead of
 * three).  Returns 0 when the plan would cut sequences (pass num_splits = 0
 * and the workspace, so the device plans), and 0 for a NULL pointer,
 * batch < 1, num_heads < 1 or no usable device.  Costs O(32 * batch) host
 * work; enqueues nothing.  mla_nvfp4_decode_host applies it itself.
 * Source: "#2244", first commit message (split-K over the paged latent
 * cache, natural-log LSE merge): splitting a sequence is only needed to fill
 * the SMs.
 */
int mla_nvfp4_decode_plan_splits(const int32_t* seq_lens_host, int batch, int num_heads,
                                 size_t workspace_bytes);

/*
 * Absorbed MLA decode over the NVFP4 latent cache, split along the keys and
 * merged by natural-log LSE.
 * Source: "#2244", first commit message (split-K absorbed decode over the
 * paged latent cache, grouped query heads, natural-log LSE) and third commit
 * message (both products read the write-once latent; V is the latent);
 * "#33" (sparse top-k decode; bf16 Q staged unquantised, review of
 * kernel.py).
 *   q            : bf16 [batch, num_heads, 576] contiguous = [q_nope.W_UK (512),
 *                  q_pe (64)] per head, 16-byte aligned.
 *   cache        : uint8 [num_slots, record_bytes] written by
 *                  mla_nvfp4_cache_write with the same global_scale.
 *   Paged mode   : page_table int32 [batch, page_table_stride], seq_lens int32
 *                  [batch]; token t of sequence b is slot
 *                  page_table[b][t / page_size] * page_size + t % page_size.
 *                  topk_indices must be NULL.
 *   Top-k mode   : topk_indices int32 [batch, topk] of global slot ids, -1 =
 *                  padding; page_table and seq_lens must be NULL.
 *   out          : bf16 [batch, num_heads, 512].
 *   lse          : fp32 [batch, num_heads] natural-log LSE of the scaled
 *                  scores, or NULL.  A sequence with no keys gives out = 0 and
 *                  lse = -inf.
 *   num_splits   : > 0: every sequence's key tiles (64 keys each) are cut
 *                  into num_splits equal ranges, one CTA pair each, merged
 *                  by LSE.  <= 0 in top-k mode: as many equal splits as
 *                  fill the SMs (all rows have topk entries).  <= 0 in paged
 *                  mode with a workspace: length-aware plan, made on the
 *                  device from the lengths: every sequence is cut into
 *                  chunks of C tiles (C chosen per call from the tile
 *                  counts, the SM count and the workspace room), the CTA
 *                  pairs take the chunks longest first, and sequences with
 *                  one chunk are written directly.  <= 0 in paged mode
 *                  without a workspace (NULL): one split per sequence.
 *   workspace    : >= mla_nvfp4_decode_workspace_size(batch, num_heads,
 *                  num_splits) bytes, 256-byte aligned, contents ignored;
 *                  may be NULL for one split.  A planned call given less
 *                  than the full size uses fewer chunks (down to one per
 *                  sequence), as long as the work list itself fits.
 * scores = softmax_scale * q . [x_hat (512), k_pe (64)], out = softmax . x_hat.
 * k_pe values (432-byte records) enter the tensor cores as f16: a |k_pe|
 * above 65504 saturates there and is flagged MLA_DEVERR_RANGE.
 */
int mla_nvfp4_decode(const void* q, int batch, int num_heads, const uint8_t* cache,
                     int64_t num_slots, int record_bytes, const int32_t* page_table,
                     int64_t page_table_stride, int page_size, const int32_t* seq_lens,
                     const int32_t* topk_indices, int topk, float softmax_scale,
                     const float* global_scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, int num_splits, uint32_t* error_word, void* stream);

/*
 * mla_nvfp4_decode with the absorbed query quantised to NVFP4: the query's
 * 576 features per head in blocks of 16 (the contraction axis of Q K^T),
 * e4m3 block scales, global scale *q_global_scale (device fp32, e.g.
 * mla_nvfp4_global_scale of q), correctly rounded as the cache write does;
 * the scores are those of that quantised query:
 *   scores = softmax_scale * q_hat . [x_hat, k_pe],  out = softmax . x_hat.
 * Source: "#2244", first commit message (forward_mqa quantises the absorbed
 * query before the decode kernel) and PR description, "Contract notes"
 * (NVFP4 1x16 along the contraction axis).  The latent part of the score
 * product runs on block-scaled fp4 tensor cores straight from the cache's
 * codes and scales; the RoPE part in f16, with k_pe / gs rounded once to f16
 * (|k_pe / gs| above 65504 saturates and sets MLA_DEVERR_RANGE).  An invalid
 * q_global_scale gives zero scores' query and MLA_DEVERR_SCALE.  Other
 * arguments, the workspace, the splits and the result as mla_nvfp4_decode.
 */
int mla_nvfp4_decode_q4(const void* q, int batch, int num_heads, const uint8_t* cache,
                        int64_t num_slots, int record_bytes, const int32_t* page_table,
                        int64_t page_table_stride, int page_size, const int32_t* seq_lens,
                        const int32_t* topk_indices, int topk, float softmax_scale,
                        const float* global_scale, const float* q_global_scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, int num_splits, uint32_t* error_word,
                        void* stream);

/* Size of the library's built-in decode scratch: MLA_DECODE_STATIC_ROWS
 * partial rows (one head of one split each) and the bytes those rows take
 * (the value of mla_nvfp4_decode_workspace_size for that many rows). */
#define MLA_DECODE_STATIC_ROWS 16384
#define MLA_DECODE_STATIC_WORKSPACE_BYTES 33619968u /* 16384*2048 + 65536 */

/*
 * mla_nvfp4_decode without a caller workspace.  The pages describe no such
 * entry point; it exists for callers that cannot hand the library device
 * memory for each call: a serving engine that has given all free device
 * memory to its paged KV-cache pool at start-up, a host program in another
 * language with no device allocator of its own, or a decode step that must
 * not call cudaMalloc/cudaFree because those calls synchronise the device.
 * It takes the same arguments as mla_nvfp4_decode minus workspace and
 * workspace_bytes, and computes the same result with the same kernels.
 *
 *   Scratch      : the split partials and the work list live in a
 *                  file-scope __device__ array of
 *                  MLA_DECODE_STATIC_WORKSPACE_BYTES bytes (one copy per
 *                  device, 256-byte aligned).  The call allocates nothing:
 *                  no cudaMalloc, no cudaFree, no allocating library call.
 *                  Nothing in the scratch needs to start at zero: every
 *                  call writes the work list and each partial row before
 *                  they are read.
 *   Limit        : num_splits > 1: batch * num_splits * num_heads must not
 *                  exceed MLA_DECODE_STATIC_ROWS.  num_splits <= 0: the
 *                  plan cuts the sequences into no more chunks than the
 *                  scratch holds, and its work list (about 16 bytes per
 *                  sequence) must fit.  num_splits == 1 uses no scratch.
 *                  Calls beyond the limit return MLA_ERR_WORKSPACE without
 *                  launching, and mla_nvfp4_last_error() names the sizes.
 *   Scratch      : every call that uses the scratch looks up its device
 *                  address in the current context (cudaGetSymbolAddress,
 *                  which allocates nothing; the first call in a process may
 *                  load the library's device code, so make it before any
 *                  stream capture begins).  A reset device gets the address
 *                  of its new context.  A failed lookup returns
 *                  MLA_ERR_LAUNCH.
 *   Concurrency  : all calls on one device share the one scratch, so calls
 *                  whose work may overlap on the device (different
 *                  streams, or several host threads without ordering) race
 *                  and give wrong results.  Calls enqueued on one stream
 *                  run in order and are safe.
 */
int mla_nvfp4_decode_noalloc(const void* q, int batch, int num_heads, const uint8_t* cache,
                             int64_t num_slots, int record_bytes, const int32_t* page_table,
                             int64_t page_table_stride, int page_size, const int32_t* seq_lens,
                             const int32_t* topk_indices, int topk, float softmax_scale,
                             const float* global_scale, void* out, float* lse, int num_splits,
                             uint32_t* error_word, void* stream);

/*
 * mla_nvfp4_decode from and to host memory: the form a serving loop calls
 * once per step when the step's queries and page table are produced on the
 * host and its output is read there.  The pages describe no such entry
 * point; it keeps a step's host traffic inside one library call.  Enqueued
 * on `stream`, in order: one cudaMemcpyAsync per input from host memory
 * into the caller's device buffer for it (q; then page_table and seq_lens,
 * or topk), the decode of mla_nvfp4_decode on those device copies, and one
 * cudaMemcpyAsync per output back to host memory (out; then lse when both
 * lse pointers are given).
 *   *_host       : host memory with the shapes and types of the matching
 *                  mla_nvfp4_decode argument: q_host bf16 [batch, num_heads,
 *                  576]; page_table_host int32 [batch, page_table_stride]
 *                  (contiguous) and seq_lens_host int32 [batch], or
 *                  topk_host int32 [batch, topk]; out_host bf16 [batch,
 *                  num_heads, 512]; lse_host fp32 [batch, num_heads] or NULL.
 *                  Page-locked memory makes the copies asynchronous; with
 *                  pageable memory a copy may finish before the call returns.
 *   *_dev        : device buffers of the same sizes, owned by the caller,
 *                  that receive the inputs and hold the outputs before their
 *                  copy back (q_dev and out_dev 16-byte aligned).  Each host
 *                  pointer comes with its device pointer (both NULL or both
 *                  set).
 *   Other arguments and the result are those of mla_nvfp4_decode.  In paged
 *                  mode with num_splits <= 0 and a workspace, the lengths are
 *                  read on the host first (mla_nvfp4_decode_plan_splits): where
 *                  the plan would keep one chunk per sequence the call launches
 *                  the one-split decode instead of plan, decode and merge.
 *   Return       : argument checks run before anything is enqueued; a copy
 *                  that cannot be enqueued returns MLA_ERR_LAUNCH (see
 *                  mla_nvfp4_last_error).  The host buffers must stay
 *                  untouched until the stream has passed the call.
 */
int mla_nvfp4_decode_host(const void* q_host, void* q_dev, int batch, int num_heads,
                          const uint8_t* cache, int64_t num_slots, int record_bytes,
                          const int32_t* page_table_host, int32_t* page_table_dev,
                          int64_t page_table_stride, int page_size, const int32_t* seq_lens_host,
                          int32_t* seq_lens_dev, const int32_t* topk_host, int32_t* topk_dev,
                          int topk, float softmax_scale, const float* global_scale,
                          void* out_host, void* out_dev, float* lse_host, float* lse_dev,
                          void* workspace, size_t workspace_bytes, int num_splits,
                          uint32_t* error_word, void* stream);

/*
 * Causal varlen MLA prefill whose epilogue writes NVFP4 directly.
 * Source: "feat: MLA prefill NVFP4 fused output - #8" (PR description:
 * packed e2m1 output plus the global scale plus the 128x4-swizzled e4m3
 * block-scale buffer consumed by NVFP4 GEMMs, no standalone quantisation;
 * the call owns the whole scale buffer, which is why fusion needs a pure
 * prefill batch); "#2244", first commit (varlen, asymmetric 192/128 dims).
 *   q, k         : bf16 [total_tokens, num_heads, 192]; v: bf16 [total_tokens,
 *                  num_heads, 128]; element strides per token and per head
 *                  given, last dim contiguous; base and strides (in bytes)
 *                  16-byte aligned.
 *   cu_seqlens   : int32 [num_seqs + 1] on the device, cu_seqlens[0] = 0,
 *                  non-decreasing, cu_seqlens[num_seqs] = total_tokens;
 *                  max_seqlen (host) >= every sequence length.
 *   out_codes    : uint8 [total_tokens, num_heads * 64]: row m, byte
 *                  h*64 + d/2 holds features d, d+1 of head h.
 *   out_scales   : uint8 [roundup(T,128) * roundup(num_heads*8,4)]: e4m3 scale
 *                  of (row m, column k = h*8 + d/16) at
 *                  ((m/128)*(Kp/4) + k/4)*512 + (m%32)*16 + ((m%128)/32)*4 + k%4,
 *                  Kp = roundup(num_heads*8, 4); padding rows are zeroed.
 *   lse          : fp32 [num_heads, total_tokens] or NULL.
 * Query i of a sequence attends to keys 0..i of the same sequence; the
 * normalised fp32 output rows are quantised with blocks of 16 along d.
 *   Scheduling   : one CTA per SM takes work items from a device counter in
 *                  the library (64 counters, used in turn, each back at zero
 *                  when its launch ends).  Up to 64 calls may run at once on
 *                  one device (different streams).  Every call looks the
 *                  counters up (cudaGetSymbolAddress, which allocates
 *                  nothing); the first call in a process loads the module
 *                  and should come before any stream capture begins.
 *   Errors       : MLA_ERR_INVALID_ARG for bad sizes, strides or alignment
 *                  (nothing launched); device-side, MLA_DEVERR_BOUNDS in
 *                  *error_word when cu_seqlens is out of range or a sequence
 *                  is longer than max_seqlen, MLA_DEVERR_SCALE for a global
 *                  scale outside [2^-100, 2^100].
 */
int mla_nvfp4_prefill_fused_out(const void* q, const void* k, const void* v,
                                int64_t q_stride_t, int64_t q_stride_h, int64_t k_stride_t,
                                int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                                const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                int max_seqlen, int num_heads, float softmax_scale,
                                const float* global_scale, uint8_t* out_codes,
                                uint8_t* out_scales, float* lse, uint32_t* error_word,
                                void* stream);

/*
 * Chunked-context prefill over the quantised cache, in three calls.
 * Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
 * TRITON_MLA) - #2244", first commit message (the prefill's natural-log LSE
 * serves chunked-context merging; the chunked-context path projects context
 * keys and values from the latent) and second commit message (cached
 * context chunks are gathered from the quantised paged cache).  A prefill
 * of new tokens after a cached context: gather each context chunk's latent
 * (mla_nvfp4_gather_latent), project it to per-head keys and values (the
 * model's kv_b_proj; the caller's GEMM), attend the new queries to each
 * chunk and, causally, to the new tokens (mla_nvfp4_prefill_partial), then
 * merge the partial results and write the NVFP4 output
 * (mla_nvfp4_merge_fused_out).
 *
 * mla_nvfp4_gather_latent: cache records at slots[0..n) (int64; -1 gives
 * zeros, a slot >= num_slots zeros and MLA_DEVERR_BOUNDS) read back as
 *   kv_c : bf16 [n, 512], x_hat = e2m1 * e4m3 * gs rounded once to bf16
 *          (nearest, ties to even, from the exact product);
 *   k_pe : bf16 [n, 64], as stored (432-byte records) or the e4m3 value.
 */
int mla_nvfp4_gather_latent(const uint8_t* cache, int64_t num_slots, int record_bytes, const float* global_scale,
                            const int64_t* slots, int64_t n, void* kv_c, void* k_pe, uint32_t* error_word,
                            void* stream);

/*
 * mla_nvfp4_prefill_partial: the prefill's attention with an unquantised
 * result, for merging.  q bf16 [total_tokens, H, 192]; k bf16 [.., H, 192]
 * and v bf16 [.., H, 128] (strides as in mla_nvfp4_prefill_fused_out).
 *   cu_seqlens_k NULL : query i of sequence s attends causally to keys
 *                       0..i of its own tokens (k, v rows as q's).
 *   cu_seqlens_k set  : int32 [num_seqs + 1] over total_k rows of k and v;
 *                       the queries of sequence s attend to every key of
 *                       rows [cu_seqlens_k[s], cu_seqlens_k[s+1]) (a
 *                       context chunk); an empty chunk gives O = 0, LSE =
 *                       -inf.
 *   out  : fp32 [total_tokens, H, 128], the normalised output;
 *   lse  : fp32 [H, total_tokens], natural log (required).
 */
int mla_nvfp4_prefill_partial(const void* q, const void* k, const void* v, int64_t q_stride_t,
                              int64_t q_stride_h, int64_t k_stride_t, int64_t k_stride_h, int64_t v_stride_t,
                              int64_t v_stride_h, const int32_t* cu_seqlens, const int32_t* cu_seqlens_k,
                              int num_seqs, int64_t total_tokens, int64_t total_k, int max_seqlen,
                              int num_heads, float softmax_scale, float* out, float* lse,
                              uint32_t* error_word, void* stream);

/*
 * mla_nvfp4_merge_fused_out: num_parts partial results over the same
 * queries, o_parts fp32 [num_parts, T, H, 128] (each normalised) and
 * lse_parts fp32 [num_parts, H, T], merged by LSE (O = sum_i exp(lse_i -
 * LSE) O_i, LSE = ln sum_i exp(lse_i); all -inf gives O = 0) and written
 * as mla_nvfp4_prefill_fused_out writes its output: out_codes uint8
 * [T, H*64], out_scales 128x4-swizzled (padding zeroed), lse fp32 [H, T] or
 * NULL; the epilogue's quantiser with *global_scale.
 */
int mla_nvfp4_merge_fused_out(const float* o_parts, const float* lse_parts, int num_parts, int64_t total_tokens,
                              int num_heads, const float* global_scale, uint8_t* out_codes, uint8_t* out_scales,
                              float* lse, uint32_t* error_word, void* stream);

/*
 * Prefill with fake-quantised operands (an accuracy-study mode), in two
 * calls.  Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for
 * MLA (vLLM TRITON_MLA) - #2244", first commit message (mla_prefill: fused
 * Q/K/P/V fake quant, token-exact N:M score sparsity) and PR description
 * ("What does this PR do?": the projected Q/K/P/V operands quantised once,
 * optional 2:4 score sparsity on new-token attention; "Contract notes":
 * NVFP4 1x16 along the contraction axis, e4m3 block scale, amax/(6*448),
 * the softmax denominator unquantised).
 *
 * mla_nvfp4_prefill_qdq: each operand quantised to NVFP4 once along the axis
 * its product contracts, and written as the exact f16 value code * e4m3
 * scale (the global scale left out):
 *   q, k : bf16 [T, H, 192] (strides as in mla_nvfp4_prefill_fused_out), in
 *          blocks of 16 features of a (token, head) row, scales *gs_q / *gs_k;
 *   v    : bf16 [T, H, 128], in blocks of 16 tokens of a (head, feature)
 *          column counted from each sequence's first token (cu_seqlens), the
 *          last block of a sequence ragged, scale *gs_v;
 *   q_out, k_out : f16 [T, H, 192] contiguous;  v_out : f16 [T, H, 128].
 * The quotients are rounded exactly as the definition's float32 divisions.
 * Global scales are amax/(6*448) of each tensor (mla_nvfp4_global_scale).
 */
int mla_nvfp4_prefill_qdq(const void* q, const void* k, const void* v, int64_t q_stride_t, int64_t q_stride_h,
                          int64_t k_stride_t, int64_t k_stride_h, int64_t v_stride_t, int64_t v_stride_h,
                          const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int max_seqlen,
                          int num_heads, const float* gs_q, const float* gs_k, const float* gs_v, void* q_out,
                          void* k_out, void* v_out, uint32_t* error_word, void* stream);

/*
 * mla_nvfp4_prefill_fakequant: the causal varlen prefill of
 * mla_nvfp4_prefill_fused_out over the outputs of mla_nvfp4_prefill_qdq
 * (contiguous f16 q [T,H,192], k [T,H,192], v [T,H,128]) with their global
 * scales, and P quantised to NVFP4 in blocks of 16 keys (counted from the
 * sequence's first key) before P.V, relative to the power-of-two reference
 * 2^ceil(row max, log2 units) so that P <= 1 and gs_p = 1/2688; the row sum
 * takes the unquantised P.  sparse24 = 1: in each group of 4 keys (same
 * alignment) each query keeps its 2 largest scores (equal scores: the lower
 * key first) and drops the rest from numerator and denominator; keys hidden
 * by the causal mask count as dropped.  The output is written as by
 * mla_nvfp4_prefill_fused_out (codes, swizzled scales, optional LSE).
 */
int mla_nvfp4_prefill_fakequant(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int num_seqs,
                                int64_t total_tokens, int max_seqlen, int num_heads, float softmax_scale,
                                const float* gs_q, const float* gs_k, const float* gs_v, int sparse24,
                                const float* global_scale, uint8_t* out_codes, uint8_t* out_scales, float* lse,
                                uint32_t* error_word, void* stream);

/*
 * NVFP4 x NVFP4 GEMM on block-scaled tensor cores, reading the fused
 * prefill output as written (the attention output projection, o_proj):
 *     out[m, n] = gs_a * gs_w * sum_k a_hat[m, k] * w_hat[n, k]   (bf16)
 * with a_hat = e2m1(code) * e4m3(scale) per block of 16 along k.
 * Source: "feat: MLA prefill NVFP4 fused output - #8" (PR description: the
 * packed e2m1 output and its 128x4-swizzled e4m3 scales are what the NVFP4
 * GEMMs consume, with no standalone quantisation in between).
 *   a_codes      : uint8 [M, K/2] (e.g. out_codes of the prefill, K = heads*128).
 *   a_scales     : the 128x4-swizzled scale buffer of A's [M, K/16] scales
 *                  (layout as for out_scales of the prefill), padding readable.
 *   w_codes      : uint8 [N, K/2], the weight; w_scales likewise for [N, K/16].
 *   gs_a, gs_w   : device fp32 global scales of A and W.
 *   out          : bf16 [M, N] with row stride ldc >= N elements.
 * N must be a multiple of 128 and K of 256; all pointers and ldc*2
 * 16-byte aligned.  M == 0 or N == 0 is a no-op.
 */
int mla_nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_scales, int64_t M, const uint8_t* w_codes,
                   const uint8_t* w_scales, int64_t N, int64_t K, const float* gs_a, const float* gs_w,
                   void* out, int64_t ldc, uint32_t* error_word, void* stream);

/*
 * Self-test of the bounded waits (test hook; no counterpart on the pages).
 * Every wait of the library's pipelined kernels (decode, prefill) gives up
 * after a time limit, ORs MLA_DEVERR_TIMEOUT into the error word and raises
 * an abort flag that ends the CTA's other waits, so a stalled pipeline ends
 * its kernel with a status instead of holding the GPU.  This call launches
 * one CTA whose first wait, on a barrier nothing arrives on, runs out after
 * limit_ns, and whose second wait, with the kernels' full 2 s limit, must
 * then end through the abort flag.
 *   error_word   : device uint32, receives MLA_DEVERR_TIMEOUT.
 *   limit_ns     : the first wait's limit, 1 us .. 1 s.
 *   elapsed_ns   : device uint64 [2] or NULL: how long each wait ran.
 * Returns MLA_ERR_INVALID_ARG for a null error word or a limit out of range.
 */
int mla_nvfp4_selftest_wait(uint32_t* error_word, int64_t limit_ns, unsigned long long* elapsed_ns,
                            void* stream);

/*
 * The prefill epilogue's quantiser on its own (test hook): fp32 [M, N]
 * row-major, N a multiple of 16, into packed codes uint8 [M, N/2] and the
 * swizzled scale buffer of a [M, N/16] scale matrix (layout as for
 * out_scales above, padding zeroed).  Same device code as the epilogue.
 */
int mla_nvfp4_quantize_rows(const float* x, int64_t M, int64_t N, const float* global_scale,
                            uint8_t* codes, uint8_t* scales, uint32_t* error_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_NVFP4_H */
