"""128x4-swizzled e4m3 scale-factor layout and the fused NVFP4 prefill output
(oracle; test infrastructure only).

Source: "feat: MLA prefill NVFP4 fused output - #8" (vLLM fork), PR
description: flash-attention writes the packed e2m1 output, and the e4m3
block scales in the 128x4-swizzled layout that the cutlass / flashinfer
NVFP4 GEMMs read, so no standalone quantisation pass runs; the 128-row
scale tiles are why fusion is limited to pure-prefill batches.  Review on
the output view: codes are ``float4_e2m1fn_x2``, shape [-1, H, v_head_dim/2].

The scale matrix is logically [M, K] with K = (row length) / 16.  It is
stored as tiles of 128 rows x 4 columns (512 bytes each), tiles ordered
row-major over (m // 128, k // 4) with Kp // 4 tiles per tile-row, where
Kp = K rounded up to a multiple of 4.  Inside a tile, the byte for (m, k)
sits at (m % 32) * 16 + ((m % 128) // 32) * 4 + k % 4.  Rows M..Mp-1 and
columns K..Kp-1 of the padded buffer (Mp = M rounded up to 128) are zero.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4

TILE_M = 128
TILE_K = 4
TILE_BYTES = 512


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def sf_buffer_bytes(M: int, K: int) -> int:
    return round_up(M, TILE_M) * round_up(K, TILE_K)


def sf_offset(m, k, K: int):
    """Byte offset of scale (m, k) in the swizzled buffer of a [M, K] matrix."""
    m = np.asarray(m, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    tiles_per_row = round_up(K, TILE_K) // TILE_K
    tile = (m // TILE_M) * tiles_per_row + (k // TILE_K)
    return tile * TILE_BYTES + (m % 32) * 16 + ((m % TILE_M) // 32) * 4 + (k % TILE_K)


def sf_unswizzle(off, K: int):
    """Inverse of sf_offset: byte offset -> (m, k)."""
    off = np.asarray(off, dtype=np.int64)
    tiles_per_row = round_up(K, TILE_K) // TILE_K
    tile, r = off // TILE_BYTES, off % TILE_BYTES
    tm, tk = tile // tiles_per_row, tile % tiles_per_row
    m_lo, rest = r // 16, r % 16
    m_mid, k_lo = rest // 4, rest % 4
    return tm * TILE_M + m_mid * 32 + m_lo, tk * TILE_K + k_lo


def swizzle_scales(sf) -> np.ndarray:
    """[M, K] scale bytes -> flat swizzled buffer (padding zero)."""
    sf = np.asarray(sf, dtype=np.uint8)
    M, K = sf.shape
    buf = np.zeros(sf_buffer_bytes(M, K), dtype=np.uint8)
    m, k = np.meshgrid(np.arange(M), np.arange(K), indexing="ij")
    buf[sf_offset(m, k, K)] = sf
    return buf


def unswizzle_scales(buf, M: int, K: int) -> np.ndarray:
    m, k = np.meshgrid(np.arange(M), np.arange(K), indexing="ij")
    return np.asarray(buf, dtype=np.uint8)[sf_offset(m, k, K)]


def quantize_rows(x, gs):
    """float32 [M, N] -> (packed codes [M, N/2] u8, swizzled scales u8).

    Blocks of 16 along each row, quantised as in ``nvfp4.quantize_blocks``.
    """
    x = np.asarray(x, dtype=np.float32)
    M, N = x.shape
    codes, sf = nvfp4.quantize_blocks(x, gs)
    return nvfp4.pack_e2m1(codes), swizzle_scales(sf.reshape(M, N // 16))


def dequantize_rows(packed, sf_buf, M: int, N: int, gs) -> np.ndarray:
    codes = nvfp4.unpack_e2m1(np.asarray(packed).reshape(M, N // 2))
    sf = unswizzle_scales(sf_buf, M, N // 16)
    return nvfp4.dequantize_blocks(codes, sf, gs)
