"""CPU oracle for MLA attention over an NVFP4 latent cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library under
``mla_attention_nvfp4_gb300/csrc`` and imports nothing from the package.

The oracle is plain NumPy, written for a reader checking it against the
three pages it restates:

* "feat: MLA prefill NVFP4 fused output - #8" (vLLM fork): the prefill
  output written as packed e2m1 codes plus a 128x4-swizzled e4m3 block-scale
  buffer (PR description; review on the ``float4_e2m1fn_x2`` output view).
* "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
  TRITON_MLA) - #2244" (Model-Optimizer): NVFP4 = e2m1 codes, one e4m3 scale
  per 16 elements along the contraction axis, global scale amax/(6*448)
  ("Contract notes"); split-K absorbed decode over a paged latent cache with
  a natural-log LSE merge; the write-once latent consumed by both BMMs, with
  V = the latent (first and third commit messages).
* "nvfp4 MLA KV cache + per-layer outer-scale + fp8-RoPE KV-cell (sm120) -
  #33" (b12x): 432-byte (bf16 RoPE) and 368-byte (fp8 RoPE) records, the
  record size being the ABI (review of ``api.py``); bf16 Q (review of
  ``kernel.py``); the per-layer fp32 outer scale restored on read (PR
  description).

Floating point is float64, except the NVFP4 quantisation (scale byte and
codes), which evaluates its definition in IEEE float32 (divisions included)
and rounds the float32 quotients exactly onto the e4m3 / e2m1 grids.

Modules:
  nvfp4      e2m1 / e4m3 codecs, block quantisation, global scale.
  cache      the 432 / 368 byte cache record.
  attention  absorbed decode (paged and top-k), LSE merge, causal prefill.
  swizzle    the 128x4 scale-factor layout and the fused prefill output.
  gemm       the NVFP4 x NVFP4 product of packed codes and swizzled scales.
  fakequant  the causal prefill with NVFP4 fake-quantised Q, K, P, V and
             2:4 score sparsity.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, hand-worked examples, library routines (torch's
float8_e4m3fn cast, scaled_dot_product_attention in float64) or brute force.
The record byte order, the nibble order inside a byte, the fp8-RoPE cast and
the sign of a code that rounds to zero are readings of the pages (they fix
none of them), pinned only to those readings.
"""
