"""NVFP4 x NVFP4 GEMM on the fused prefill output (oracle; test
infrastructure only).

Source: "feat: MLA prefill NVFP4 fused output - #8" (vLLM fork), PR
description: the prefill writes its output as packed e2m1 codes plus e4m3
block scales in the 128x4-swizzled layout, which the NVFP4 GEMMs (the
attention output projection, o_proj) read directly, with no standalone
quantisation pass in between.

    C[m, n] = gs_a * gs_w * sum_k  a_hat[m, k] * w_hat[n, k]
    a_hat = e2m1(code) * e4m3(scale)   (blocks of 16 along k, as stored)

A is [M, K] (e.g. the prefill output, M tokens x K = heads * 128), W is the
weight [N, K]; both are packed codes [rows, K/2] with a swizzled scale
buffer for a [rows, K/16] scale matrix.  Computed in float64.
"""
from __future__ import annotations

import numpy as np

from . import swizzle


def nvfp4_gemm(a_codes, a_scales, w_codes, w_scales, M: int, N: int, K: int, gs_a, gs_w) -> np.ndarray:
    """float64 [M, N] = dequant(A) @ dequant(W)^T (global scales applied)."""
    a = swizzle.dequantize_rows(np.asarray(a_codes).reshape(M, K // 2), a_scales, M, K, gs_a)
    w = swizzle.dequantize_rows(np.asarray(w_codes).reshape(N, K // 2), w_scales, N, K, gs_w)
    return a @ w.T
