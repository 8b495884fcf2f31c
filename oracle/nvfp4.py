"""NVFP4 codecs and block quantisation (oracle; test infrastructure only).

Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
TRITON_MLA) - #2244", PR description, "Contract notes": NVFP4 is one e4m3
block scale per 16 elements along the contraction axis, with the global
scale amax/(6*448).  Codes are e2m1 with magnitudes {0, .5, 1, 1.5, 2, 3, 4,
6}; the block scale is e4m3(amax16 / 6 / global).

The definition is evaluated in IEEE float32 arithmetic, every operation
(divisions included) rounded to nearest even: for a block with maximum
magnitude amax16 and a float32 global scale gs,

    s_raw = f32( f32(amax16 / 6) / gs )
    sb    = e4m3 RNE-satfinite(s_raw)         (448 for anything above)
    S     = f32( e4m3(sb) * gs )
    code  = e2m1 RNE-satfinite( f32(x / S) )  (all codes 0 when S == 0)

Reading: the pages give the formula and float32 inputs but no precision or
evaluation order; float32, left to right, with true divisions is the plain
one.  The roundings onto the 8-bit and 4-bit grids are exact RNE of the
float32 quotient (computed here in float64, where they are exact).

A global scale outside [2^-100, 2^100] (or not finite) is invalid: codes
and scale bytes are then 0.

Saturation ("satfinite") clamps to the largest finite value, 448 for e4m3
and 6 for e2m1.  The sign of x is kept, so a negative value that rounds to
zero encodes as the e2m1 negative zero 0x8 (IEEE conversion semantics; the
pages do not say).
"""
from __future__ import annotations

import numpy as np

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
GLOBAL_SCALE_DIVISOR = 6.0 * 448.0  # 2688
BLOCK = 16


# ----------------------------------------------------------------------------
# e2m1
# ----------------------------------------------------------------------------
def e2m1_decode(codes) -> np.ndarray:
    """4-bit code -> value: bit 3 is the sign, bits 0..2 index the magnitudes."""
    c = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e2m1_encode(x) -> np.ndarray:
    """Round to nearest e2m1 magnitude, ties to the even code, saturate at 6.

    Between adjacent magnitudes k and k+1 the midpoint goes to whichever of
    the two codes is even.  Counting the midpoints strictly below |x| gives
    the round-to-nearest code; a value exactly on the midpoint after an odd
    code k moves up to the even code k+1.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    mids = (E2M1_MAGNITUDES[:-1] + E2M1_MAGNITUDES[1:]) * 0.5  # 7 midpoints
    code = np.zeros(a.shape, dtype=np.int64)
    for k, m in enumerate(mids):
        code += (a > m)
        if k % 2 == 1:
            code += (a == m)
    sign = np.signbit(x).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


# ----------------------------------------------------------------------------
# e4m3 (the OCP "e4m3fn" format: bias 7, no infinities, 0x7F/0xFF are NaN)
# ----------------------------------------------------------------------------
def e4m3_decode(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.int64)
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where((b >> 7) & 1, -mag, mag)


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto the e4m3 grid, saturating at +-448.

    For |x| in binade [2^E, 2^(E+1)) the spacing is 2^(E-3); below the
    smallest normal 2^-6 the spacing stays 2^-9 (subnormals).  With
    E = max(floor(log2|x|), -6) and n = rint(|x| / 2^(E-3)) the code is
    (E + 7) * 8 + n - 8: for subnormals (E = -6) this is n itself, and n = 16
    rolls over into the next binade on its own.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # log2 of an exact power of two is exact; guard the other side anyway
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    e = np.where(a > 0, np.maximum(e, -6.0), -6.0)
    n = np.rint(a / np.exp2(e - 3.0))  # numpy rint: half to even
    code = (e + 7.0) * 8.0 + n - 8.0
    code = np.minimum(code, 126.0)  # 0x7E = 448, satfinite
    sign = np.signbit(x).astype(np.int64)
    return (code.astype(np.int64) | (sign << 7)).astype(np.uint8)


# ----------------------------------------------------------------------------
# block quantisation
# ----------------------------------------------------------------------------
def global_scale(amax) -> np.float32:
    """gs = amax / (6 * 448), one float32 rounding ("Contract notes")."""
    return np.float32(np.float32(amax) / np.float32(GLOBAL_SCALE_DIVISOR))


GS_MIN, GS_MAX = 2.0 ** -100, 2.0 ** 100


def scale_valid(gs) -> bool:
    g = float(np.float32(gs))
    return GS_MIN <= g <= GS_MAX


def choose_scale(amax, gs) -> np.ndarray:
    """Scale byte sb = e4m3 RNE-satfinite of f32(f32(amax / 6) / gs)."""
    a = np.asarray(amax, dtype=np.float32)
    with np.errstate(over="ignore"):
        s_raw = (a / np.float32(6.0)).astype(np.float32) / np.float32(gs)  # IEEE float32 divisions
    s_raw = np.minimum(s_raw.astype(np.float64), 1e4)  # anything above 464 saturates to 448
    return e4m3_encode(s_raw)


def encode_with_scale(x, sb, gs) -> np.ndarray:
    """Codes of float32 blocks x [..., nb, 16] given their scale bytes sb
    [..., nb]: code = e2m1 RNE-satfinite of f32(x / S), S = f32(e4m3(sb) *
    gs), sign of x kept; all 16 codes 0 when S == 0."""
    x = np.asarray(x, dtype=np.float32)
    S = (e4m3_decode(sb).astype(np.float32) * np.float32(gs)).astype(np.float32)
    ok = S > 0
    with np.errstate(over="ignore"):
        q = (x / np.where(ok, S, np.float32(1.0))[..., None]).astype(np.float32)  # IEEE float32 division
    codes = e2m1_encode(q.astype(np.float64))
    return np.where(ok[..., None], codes, np.uint8(0)).astype(np.uint8)


def quantize_blocks(x, gs):
    """Quantise rows of 16 float32 values with the NVFP4 definition.

    x: float32 array [..., 16*nb] (row length a multiple of 16).
    gs: float32 global scale (dequantisation direction: x ~ code*scale*gs).
    Returns (codes uint8 [..., 16*nb], scale bytes uint8 [..., nb]).
    """
    x = np.asarray(x, dtype=np.float32)
    gs = np.float32(gs)
    assert x.shape[-1] % BLOCK == 0
    blocks = x.reshape(x.shape[:-1] + (x.shape[-1] // BLOCK, BLOCK))
    if not scale_valid(gs):
        return np.zeros(x.shape, dtype=np.uint8), np.zeros(blocks.shape[:-1], dtype=np.uint8)
    amax = np.max(np.abs(blocks), axis=-1)  # exact in float32
    sb = choose_scale(amax, gs)
    codes = encode_with_scale(blocks, sb, gs)
    return codes.reshape(x.shape), sb


def dequantize_blocks(codes, scale_bytes, gs) -> np.ndarray:
    """x_hat = e2m1(code) * e4m3(scale) * gs, in float64."""
    codes = np.asarray(codes)
    vals = e2m1_decode(codes)
    nb = codes.shape[-1] // BLOCK
    vals = vals.reshape(codes.shape[:-1] + (nb, BLOCK))
    s = e4m3_decode(scale_bytes)[..., None]
    return (vals * s * np.float64(np.float32(gs))).reshape(codes.shape)


def pack_e2m1(codes) -> np.ndarray:
    """Two codes per byte, even element in the low nibble (the little-endian
    ``torch.float4_e2m1fn_x2`` convention of the vLLM output view)."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out

