"""Pins for the oracle's NVFP4 codecs (CPU only).

Each test ties oracle.nvfp4 to something other than itself: hand-worked
blocks (tests/golden/nvfp4_blocks.txt), torch's independent float8_e4m3fn
cast, exhaustive enumeration, or closed forms.
"""
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        gs, xs, sb, codes = [p.strip() for p in line.split("|")]
        rows.append((np.float32(gs), np.array(xs.split(), dtype=np.float32), int(sb, 16),
                     [int(c, 16) for c in codes.split()]))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"sb{r[2]:02x}")
def test_hand_worked_blocks(row):
    gs, x, sb, codes = row
    got_codes, got_sb = nvfp4.quantize_blocks(x[None, :], gs)
    assert int(got_sb[0, 0]) == sb
    assert got_codes[0].tolist() == codes


def test_e2m1_decode_table():
    # magnitudes of the e2m1 format: 2 exponent bits (bias 1), 1 mantissa bit
    for c in range(16):
        e, m, s = (c >> 1) & 3, c & 1, c >> 3
        mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert nvfp4.e2m1_decode(c) == (-mag if s else mag)


def test_e2m1_encode_is_nearest_with_even_ties():
    # brute force: every value is mapped to a nearest grid point; exact ties
    # go to the even code; values beyond 6 saturate.
    grid = nvfp4.E2M1_MAGNITUDES
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-8, 8, 20000), (grid[:-1] + grid[1:]) / 2,
                         -(grid[:-1] + grid[1:]) / 2, grid, -grid, [7.0, 1e9, -1e9]])
    codes = nvfp4.e2m1_encode(xs)
    vals = nvfp4.e2m1_decode(codes)
    for x, c, v in zip(xs, codes, vals):
        a = min(abs(x), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        assert abs(abs(v) - a) == d.min()
        if len(best) == 2:
            assert (c & 7) == best[best % 2 == 0][0]
        assert bool(c & 8) == bool(np.signbit(x))


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = nvfp4.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_in_range():
    # torch's float32 -> float8_e4m3fn cast rounds to nearest even; it gives
    # NaN above 448 instead of saturating, so compare within range only.
    rng = np.random.default_rng(1)
    grid = nvfp4.e4m3_decode(np.arange(127))
    mids = (grid[:-1] + grid[1:]) / 2
    xs = np.concatenate([
        rng.uniform(0, 448, 50000), np.exp2(rng.uniform(-14, 8.8, 50000)), mids, grid,
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1000))]).astype(np.float32)
    xs = np.concatenate([xs, -xs])
    xs = xs[np.abs(xs) <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = nvfp4.e4m3_encode(xs.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    assert nvfp4.e4m3_encode(np.array([448.0, 463.9, 464.0, 500.0, 1e30])).tolist() == [0x7E] * 5
    assert nvfp4.e4m3_encode(np.array([-1e30])).tolist() == [0xFE]
    # smallest subnormal 2^-9; half of it ties to even (zero)
    assert nvfp4.e4m3_encode(np.array([2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -10])).tolist() == [1, 0, 1]


def test_global_scale():
    assert nvfp4.global_scale(2688.0) == np.float32(1.0)
    assert nvfp4.global_scale(6.0 * 448.0 * 0.25) == np.float32(0.25)


def test_scale_never_saturates_under_global_scale():
    # with gs = amax/(6*448), amax16/6/gs <= 448 up to float32 rounding, and
    # the largest element of the block reconstructs within one e2m1 step.
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((4096, 64)) * np.exp(rng.uniform(-3, 3, (4096, 1)))).astype(np.float32)
    gs = nvfp4.global_scale(np.abs(x).max())
    codes, sb = nvfp4.quantize_blocks(x, gs)
    assert sb.max() <= 0x7E
    xh = nvfp4.dequantize_blocks(codes, sb, gs).reshape(x.shape)
    # per-element error bound: half the widest e2m1 gap (1.0 at [4, 6]) of S,
    # plus the e4m3 scale rounding (2^-4 relative) times 6
    S = (nvfp4.e4m3_decode(sb) * np.float64(gs)).repeat(16, axis=1)
    blk_amax = np.abs(x.reshape(4096, 4, 16)).max(-1).repeat(16, axis=1)
    ok = np.abs(xh - x) <= np.maximum(1.0 * S, blk_amax * 2 ** -3) + 1e-30
    assert ok.all()


def test_pack_nibble_order():
    # even element in the low nibble: codes [1, 2] -> 0x21
    assert nvfp4.pack_e2m1(np.array([1, 2], dtype=np.uint8)).tolist() == [0x21]
    c = np.random.default_rng(3).integers(0, 16, 64).astype(np.uint8)
    assert np.array_equal(nvfp4.unpack_e2m1(nvfp4.pack_e2m1(c)), c)


def test_lossless_on_grid():
    # values already of the form code * e4m3 * gs with gs a power of two and
    # each block's amax = 6 * scale * gs are reproduced exactly.
    rng = np.random.default_rng(4)
    gs = np.float32(2.0 ** -4)
    sbytes = rng.integers(0x08, 0x70, (256, 4))
    scale = nvfp4.e4m3_decode(sbytes)
    codes = rng.integers(0, 16, (256, 4, 16))
    codes[..., 0] = 7  # magnitude 6 in every block
    x = (nvfp4.e2m1_decode(codes) * scale[..., None] * np.float64(gs)).astype(np.float32)
    got_c, got_s = nvfp4.quantize_blocks(x.reshape(256, 64), gs)
    assert np.array_equal(got_s, sbytes)
    xh = nvfp4.dequantize_blocks(got_c, got_s, gs)
    assert np.array_equal(xh, x.reshape(256, 64).astype(np.float64))
