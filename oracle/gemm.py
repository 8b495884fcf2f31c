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

from . import nvfp4, swizzle


def nvfp4_gemm(a_codes, a_scales, w_codes, w_scales, M: int, N: int, K: int, gs_a, gs_w) -> np.ndarray:
    """float64 [M, N] = dequant(A) @ dequant(W)^T (global scales applied)."""
    a = swizzle.dequantize_rows(np.asarray(a_codes).reshape(M, K // 2), a_scales, M, K, gs_a)
    w = swizzle.dequantize_rows(np.asarray(w_codes).reshape(N, K // 2), w_scales, N, K, gs_w)
    return a @ w.T


def nvfp4_gemm_entries(a_codes, a_scales, w_codes, w_scales, K: int, gs_a, gs_w, rows, cols) -> np.ndarray:
    """nvfp4_gemm restricted to C[rows][:, cols] (sampling at full size):
    only the selected rows of A and W are dequantised (their scale bytes
    read from the swizzled buffers)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)

    def rows_hat(codes, sf_buf, idx, gs):
        kb = np.arange(K // 16)
        m, kk = np.meshgrid(idx, kb, indexing="ij")
        sf = np.asarray(sf_buf, dtype=np.uint8)[swizzle.sf_offset(m, kk, K // 16)]
        c = nvfp4.unpack_e2m1(np.asarray(codes)[idx].reshape(len(idx), K // 2))
        return nvfp4.dequantize_blocks(c, sf, gs)

    return rows_hat(a_codes, a_scales, rows, gs_a) @ rows_hat(w_codes, w_scales, cols, gs_w).T

