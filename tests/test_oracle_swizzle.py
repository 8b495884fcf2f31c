"""Pins for the 128x4 scale-factor swizzle and the fused prefill output
layout (CPU only)."""
import numpy as np
import pytest

from oracle import nvfp4, swizzle


def test_known_offsets():
    K = 8  # 2 tiles per tile-row
    cases = {(0, 0): 0, (0, 1): 1, (0, 3): 3, (1, 0): 16, (31, 0): 496, (32, 0): 4,
             (64, 0): 8, (96, 3): 15, (127, 3): 511, (0, 4): 512, (128, 0): 1024,
             (129, 5): 1024 + 512 + 16 + 1}
    for (m, k), off in cases.items():
        assert swizzle.sf_offset(m, k, K) == off, (m, k)


@pytest.mark.parametrize("M,K", [(256, 8), (200, 12), (128, 4), (1, 1), (130, 9)])
def test_bijection_and_inverse(M, K):
    Mp, Kp = swizzle.round_up(M, 128), swizzle.round_up(K, 4)
    m, k = np.meshgrid(np.arange(Mp), np.arange(Kp), indexing="ij")
    off = swizzle.sf_offset(m, k, K)
    assert np.array_equal(np.sort(off.ravel()), np.arange(Mp * Kp))
    m2, k2 = swizzle.sf_unswizzle(np.arange(Mp * Kp), K)
    assert np.array_equal(swizzle.sf_offset(m2, k2, K), np.arange(Mp * Kp))


def test_bijection_full_prefill_output():
    # 32768 rows x 128 heads * 8 scale columns (no padding at this size)
    M, K = 32768, 1024
    off = np.arange(M * K)
    m, k = swizzle.sf_unswizzle(off, K)
    assert m.min() == 0 and m.max() == M - 1 and k.max() == K - 1
    assert np.array_equal(swizzle.sf_offset(m, k, K), off)
    counts = np.bincount(m * K + k, minlength=M * K)
    assert np.all(counts == 1)


def test_padding_is_zero_and_round_trip():
    rng = np.random.default_rng(20)
    M, N = 130, 3 * 16
    x = rng.standard_normal((M, N)).astype(np.float32)
    gs = nvfp4.global_scale(np.abs(x).max())
    packed, buf = swizzle.quantize_rows(x, gs)
    assert packed.shape == (M, N // 2)
    assert buf.size == 256 * 4
    sf = swizzle.unswizzle_scales(buf, M, N // 16)
    codes, sb = nvfp4.quantize_blocks(x, gs)
    assert np.array_equal(sf, sb)
    mask = np.ones(buf.size, dtype=bool)
    mm, kk = np.meshgrid(np.arange(M), np.arange(N // 16), indexing="ij")
    mask[swizzle.sf_offset(mm, kk, N // 16)] = False
    assert np.all(buf[mask] == 0)
    xh = swizzle.dequantize_rows(packed, buf, M, N, gs)
    assert np.array_equal(xh, nvfp4.dequantize_blocks(codes, sb, gs))
