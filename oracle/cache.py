"""The per-token NVFP4 latent cache record (oracle; test infrastructure only).

Sources:
* "nvfp4 MLA KV cache + per-layer outer-scale + fp8-RoPE KV-cell (sm120) -
  #33", review of ``api.py``: the record is 432 bytes with a bf16 RoPE part
  or 368 bytes with an fp8 RoPE part, any other width is an error, and the
  record width is the authoritative ABI.  PR description: the fp8-RoPE cell
  and the per-layer fp32 outer scale restored on read.
* "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA ... - #2244",
  first and second commit messages: the latent is quantised once, when the
  cache is written, and both attention products read those bytes.

Byte layout (a reading: the pages give only the widths; the split follows
the widths 256 + 32 + 128 + 16 and 256 + 32 + 64 + 16):

    [0, 256)    512 e2m1 codes of kv_c, two per byte, even element low nibble
    [256, 288)  32 e4m3 block scales (block j covers kv_c[16j : 16j+16])
    [288, 416)  k_pe as 64 little-endian bf16              (432-byte record)
    [288, 352)  k_pe as 64 e4m3, RNE, saturating, scale 1  (368-byte record)
    rest        zero padding (16 bytes)

Only the latent carries the global (outer) scale; k_pe is stored unscaled.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4

D_LATENT = 512
D_ROPE = 64
RECORD_BF16_ROPE = 432
RECORD_FP8_ROPE = 368
CODES_OFF = 0
SCALES_OFF = 256
ROPE_OFF = 288


def check_record_bytes(record_bytes: int) -> bool:
    """432 = bf16 RoPE, 368 = fp8 RoPE; anything else is rejected."""
    if record_bytes not in (RECORD_BF16_ROPE, RECORD_FP8_ROPE):
        raise ValueError(f"NVFP4 MLA cache record must be 368 or 432 bytes, got {record_bytes}")
    return record_bytes == RECORD_FP8_ROPE


def bf16_bits(x_f32) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-representable."""
    u = np.asarray(x_f32, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "k_pe must hold bf16 values"
    return (u >> 16).astype(np.uint16)


def bf16_from_bits(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def encode_records(kv_c, k_pe, gs, record_bytes: int) -> np.ndarray:
    """kv_c [T,512], k_pe [T,64] (bf16 values held as float32) -> [T, record_bytes] u8."""
    fp8_rope = check_record_bytes(record_bytes)
    kv_c = np.asarray(kv_c, dtype=np.float32)
    k_pe = np.asarray(k_pe, dtype=np.float32)
    T = kv_c.shape[0]
    assert kv_c.shape == (T, D_LATENT) and k_pe.shape == (T, D_ROPE)
    codes, scales = nvfp4.quantize_blocks(kv_c, gs)
    rec = np.zeros((T, record_bytes), dtype=np.uint8)
    rec[:, CODES_OFF:SCALES_OFF] = nvfp4.pack_e2m1(codes)
    rec[:, SCALES_OFF:ROPE_OFF] = scales
    if fp8_rope:
        rec[:, ROPE_OFF:ROPE_OFF + D_ROPE] = nvfp4.e4m3_encode(k_pe.astype(np.float64))
    else:
        rope = bf16_bits(k_pe)
        rec[:, ROPE_OFF:ROPE_OFF + 2 * D_ROPE:2] = (rope & 0xFF).astype(np.uint8)
        rec[:, ROPE_OFF + 1:ROPE_OFF + 2 * D_ROPE:2] = (rope >> 8).astype(np.uint8)
    return rec


def write_cache(cache, kv_c, k_pe, slot_mapping, gs, record_bytes: int) -> np.ndarray:
    """Scatter encoded records into cache rows; slot -1 skips the token."""
    rec = encode_records(kv_c, k_pe, gs, record_bytes)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    cache[slots[keep]] = rec[keep]
    return cache


def decode_records(rec, gs, record_bytes: int):
    """[N, record_bytes] u8 -> (latent x_hat [N,512], rope [N,64]) in float64.

    x_hat = e2m1(code) * e4m3(scale) * gs; the rope part carries no scale.
    """
    fp8_rope = check_record_bytes(record_bytes)
    rec = np.asarray(rec, dtype=np.uint8)
    codes = nvfp4.unpack_e2m1(rec[:, CODES_OFF:SCALES_OFF])
    latent = nvfp4.dequantize_blocks(codes, rec[:, SCALES_OFF:ROPE_OFF], gs)
    if fp8_rope:
        rope = nvfp4.e4m3_decode(rec[:, ROPE_OFF:ROPE_OFF + D_ROPE])
    else:
        lo = rec[:, ROPE_OFF:ROPE_OFF + 2 * D_ROPE:2].astype(np.uint16)
        hi = rec[:, ROPE_OFF + 1:ROPE_OFF + 2 * D_ROPE:2].astype(np.uint16)
        rope = bf16_from_bits(lo | (hi << 8)).astype(np.float64)
    return latent, rope


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (8 significant bits,
    ties to even), returned as float32 (bf16 values are float32 values).
    Exact: the 8-bit mantissa is rounded from the float64 significand."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)  # numpy rint: half to even
    return r.astype(np.float32)


def gather_latent(cache, slots, gs, record_bytes: int):
    """The latent of cached tokens read back for a context chunk: records at
    `slots` dequantised (x_hat = e2m1 * e4m3 * gs, exactly) and rounded once
    to bf16; k_pe as stored (bf16, or the e4m3 value, exact in bf16).
    Source: "#2244", second commit message (cached-context prefill chunks
    gather from the quantised paged cache).  Returns (kv_c [n,512], k_pe
    [n,64]) as float32 holding bf16 values."""
    lat, rope = decode_records(np.asarray(cache)[np.asarray(slots, dtype=np.int64)], gs, record_bytes)
    return bf16_round(lat), bf16_round(rope)
