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


def _nearest_even_argmin(d):
    """Row-wise index of the smallest distance; of two equal smallest
    distances the even index (round half to even on the code)."""
    dmin = d.min(axis=-1, keepdims=True)
    hit = d == dmin
    lo = np.argmax(hit, axis=-1)
    hi = d.shape[-1] - 1 - np.argmax(hit[..., ::-1], axis=-1)
    return np.where(lo % 2 == 0, lo, hi)


def _brute_force_quantize(x, gs):
    """The float32 quotients from torch's float32 division, then the nearest
    e4m3 scale and the nearest e2m1 magnitude by exhaustive search over the
    grid (ties to the even code).  Distances are exact in float64: a float32
    quotient and a grid value (at most 4 significant bits) differ by a value
    float64 holds."""
    g32 = torch.tensor(np.float32(gs))
    blocks = torch.from_numpy(np.asarray(x, dtype=np.float32).reshape(-1, 16))
    amax = blocks.abs().amax(dim=1)
    s32 = ((amax / 6.0) / g32).double().clamp(max=1e4).numpy()
    grid = nvfp4.e4m3_decode(np.arange(0x7F))
    sb = _nearest_even_argmin(np.abs(s32[:, None] - grid[None, :]))
    S32 = (torch.from_numpy(grid[sb]).float() * g32).float()
    ok = (S32 > 0).numpy()
    q32 = (blocks / torch.where(S32 > 0, S32, torch.ones_like(S32))[:, None]).double().abs().numpy()
    mags = nvfp4.E2M1_MAGNITUDES
    mag = _nearest_even_argmin(np.abs(q32[..., None] - mags[None, None, :]))
    codes = np.where(ok[:, None], mag | (np.signbit(blocks.numpy()).astype(np.int64) << 3), 0)
    return codes.astype(np.uint8).reshape(np.shape(x)), sb.astype(np.uint8)


def _tie_blocks(rng, n, gs):
    """Blocks whose float32 quotients sit exactly on a rounding midpoint.  gs
    has at most 16 significant bits, so 6*gs*midpoint (scale ties, whose
    quotient (amax/6)/gs is then the midpoint exactly) and
    e2m1-midpoint*e4m3*gs (code ties, with S = e4m3*gs exact) are float32
    values."""
    grid = nvfp4.e4m3_decode(np.arange(0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    out = np.zeros((2 * n, 16), dtype=np.float32)
    # scale ties: amax exactly 6*gs*midpoint, the rest of the block below it
    k = rng.integers(0, len(mids), n)
    amax = 6.0 * float(gs) * mids[k]
    out[:n] = (rng.uniform(-1, 1, (n, 16)) * amax[:, None]).astype(np.float32)
    out[np.arange(n), rng.integers(0, 16, n)] = (amax * rng.choice([-1, 1], n)).astype(np.float32)
    # code ties: amax = 6*S reproduces the scale byte, the other elements are
    # +-(e2m1 midpoint)*S
    sb = rng.integers(1, 0x7F, n)
    S = grid[sb] * float(gs)
    e_mids = (nvfp4.E2M1_MAGNITUDES[:-1] + nvfp4.E2M1_MAGNITUDES[1:]) / 2
    vals = e_mids[rng.integers(0, 7, (n, 16))] * rng.choice([-1, 1], (n, 16)) * S[:, None]
    vals[:, 0] = 6.0 * S
    out[n:] = vals.astype(np.float32)
    assert np.array_equal(out[n:].astype(np.float64), vals)  # the ties are exact
    return out


def _f32_16bit(v) -> np.float32:
    """v as float32 with its mantissa cut to 16 significant bits."""
    u = np.array([v], dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFFF80)
    return u.view(np.float32)[0]


@pytest.mark.parametrize("gs", [1.0, 0.37, 2.0 ** -20, 4.5e-3])
def test_quantize_blocks_against_brute_force(gs):
    # >= 10^5 random blocks at magnitudes spanning the e4m3 range (subnormal
    # scales, saturation, zero blocks) plus exact scale and code ties
    rng = np.random.default_rng(20)
    g = np.float32(gs)
    n = 100_000
    mag = np.exp2(rng.uniform(-14, 14, (n, 1))) * float(g) * 6
    x = (rng.standard_normal((n, 16)) * mag).astype(np.float32)
    x[:50] = 0.0
    x[50:100] = (rng.standard_normal((50, 16)) * 1e4 * 6 * 448 * float(g)).astype(np.float32)  # saturating
    g_tie = _f32_16bit(gs)
    ties = _tie_blocks(rng, 5000, g_tie)
    for xs, gg in ((x, g), (ties, g_tie)):
        codes, sb = nvfp4.quantize_blocks(xs, gg)
        bc, bsb = _brute_force_quantize(xs, gg)
        assert np.array_equal(sb.reshape(-1), bsb)
        assert np.array_equal(codes.reshape(-1, 16), bc.reshape(-1, 16))
    # the code-tie blocks really sit on ties: every tied element took an even
    # magnitude code (0.25 -> 0, 0.75 -> 2, 1.25 -> 2, 1.75 -> 4, 2.5 -> 4,
    # 3.5 -> 6, 5 -> 6)
    codes, _ = nvfp4.quantize_blocks(ties[5000:], g_tie)
    assert np.all((codes[:, 1:] & 7) % 2 == 0)
    assert np.all((codes[:, 0] & 7) == 7)


def test_quantize_blocks_exact_definition_spot_values():
    # amax/6/gs exactly halfway between e4m3 0x30 (0.5) and 0x31 (0.5625):
    # the tie goes to the even code 0x30; a hair above goes up
    gs = np.float32(1.0)
    half = (0.5 + 0.5625) / 2 * 6  # 3.1875, exact in float32
    x = np.zeros((2, 16), dtype=np.float32)
    x[0, 0] = half
    x[1, 0] = np.nextafter(np.float32(half), np.float32(10))
    _, sb = nvfp4.quantize_blocks(x, gs)
    assert sb[:, 0].tolist() == [0x30, 0x31]
    # with S = 0.5 (sb 0x30, gs 1): x/S = 0.75 is a tie between codes 1 and 2
    # (0.5, 1.0) and goes to 2; 1.25 between 2 and 3 goes to 2
    y = np.array([[3.0, 0.375, 0.625, -0.375] + [0.0] * 12], dtype=np.float32)
    codes, sb = nvfp4.quantize_blocks(y, gs)
    assert sb[0, 0] == 0x30
    assert codes[0, :4].tolist() == [0x7, 0x2, 0x2, 0xA]


def _reciprocal_form(x, gs):
    """A float32 model of a kernel that evaluates the quotients as products
    with reciprocals: k = 1/(6 gs), s_raw = amax16 * k, r = 1/S, q = x * r
    (each an IEEE float32 operation), then the same roundings."""
    x = np.asarray(x, dtype=np.float32).reshape(-1, 16)
    g = np.float32(gs)
    k = np.float32(np.float32(1) / np.float32(np.float32(6) * g))
    s_raw = (np.abs(x).max(1) * k).astype(np.float32)
    sb = nvfp4.e4m3_encode(s_raw.astype(np.float64))
    S = (nvfp4.e4m3_decode(sb).astype(np.float32) * g).astype(np.float32)
    r = (np.float32(1) / np.where(S > 0, S, np.float32(1))).astype(np.float32)
    q = (x * r[:, None]).astype(np.float32)
    codes = np.where((S > 0)[:, None], nvfp4.e2m1_encode(q.astype(np.float64)), 0).astype(np.uint8)
    return codes, sb


def test_tie_flip_rule_accepts_float32_kernels_and_rejects_errors():
    # Tie blocks with a gs whose reciprocals are inexact: the float32
    # reciprocal form rounds some exact ties the other way; the comparison
    # rule accepts exactly those (counted) and rejects a planted wrong code.
    from tests.helpers import quant_flips
    rng = np.random.default_rng(30)
    g = _f32_16bit(0.37)
    x = np.concatenate([_tie_blocks(rng, 2000, g),
                        (rng.standard_normal((20000, 16)) * 3).astype(np.float32)]).reshape(-1, 64)
    codes, sb = _reciprocal_form(x, g)
    flips, n = quant_flips(x, g, codes.reshape(x.shape), sb.reshape(x.shape[0], 4), "reciprocal model", budget=1.0)
    assert 0 < flips < n  # some exact ties do round the other way
    # a code one magnitude step off on a random (non-tie) element is rejected
    bad = codes.copy().reshape(x.shape)
    row, col = 3000, 5  # rows >= 1000 hold the random blocks
    m = bad[row, col] & 7
    bad[row, col] = (bad[row, col] & 8) | (m + 1 if m < 7 else 6)
    with pytest.raises(AssertionError):
        quant_flips(x, g, bad, sb.reshape(x.shape[0], 4), "planted error", budget=1.0)


def _fma32(a, b, c):
    """float32 fma: a * b + c exactly, rounded once to float32.  The product
    is exact in float64; the sum is carried as float64 plus its exact error
    (two-sum), which decides a float32 rounding that float64 left halfway."""
    a, b, c = (np.asarray(v, dtype=np.float32).astype(np.float64) for v in (a, b, c))
    p = a * b
    s_ = p + c
    bb = s_ - p
    err = (p - (s_ - bb)) + (c - bb)
    r = s_.astype(np.float32)
    lo = np.nextafter(r, np.float32(-np.inf))
    hi = np.nextafter(r, np.float32(np.inf))
    down = (s_ == (r.astype(np.float64) + lo.astype(np.float64)) / 2) & (err < 0)
    up = (s_ == (r.astype(np.float64) + hi.astype(np.float64)) / 2) & (err > 0)
    return np.where(down, lo, np.where(up, hi, r)).astype(np.float32)


def _div_rn_model(a, b, y):
    """The kernels' correctly rounded division: q0 = a * y, then
    q0 + (a - q0 * b) * y, both corrections as float32 fmas."""
    a = np.asarray(a, dtype=np.float32)
    q0 = (a * y).astype(np.float32)
    return _fma32(_fma32(-q0, b, a), y, q0)


def _cache_write_model(x, gs):
    """A float32 model of the cache write's quantiser: every division from a
    correctly rounded reciprocal plus two fmas."""
    x = np.asarray(x, dtype=np.float32).reshape(-1, 16)
    g = np.float32(gs)
    amax = np.abs(x).max(1)
    q6 = _div_rn_model(amax, np.float32(6), np.float32(1) / np.float32(6))
    s_raw = _div_rn_model(q6, g, np.float32(1) / g)
    sb = nvfp4.e4m3_encode(np.minimum(s_raw.astype(np.float64), 1e4))
    S = (nvfp4.e4m3_decode(sb).astype(np.float32) * g).astype(np.float32)
    R = (np.float32(1) / np.where(S > 0, S, np.float32(1))).astype(np.float32)
    q = _div_rn_model(x, S[:, None], R[:, None])
    codes = np.where((S > 0)[:, None], nvfp4.e2m1_encode(q.astype(np.float64)), 0)
    return codes.astype(np.uint8), sb.astype(np.uint8)


@pytest.mark.parametrize("gs", [0.37, 1.0, 4.5e-3])
def test_correctly_rounded_division_reproduces_the_definition(gs):
    # bf16 latents with the global scale of their own amax (whose thresholds
    # sit within 2^-24 of bf16 values at a rate of ~1e-3), exact tie blocks
    # and random floats: the fma-corrected reciprocal gives the definition's
    # float32 quotients exactly, the plain reciprocal does not
    rng = np.random.default_rng(40)
    bf = torch.from_numpy(rng.standard_normal(400_000).astype(np.float32)).to(torch.bfloat16).float().numpy()
    g_bf = nvfp4.global_scale(np.abs(bf).max())
    g_tie = _f32_16bit(gs)
    cases = [(bf.reshape(-1, 16), g_bf), (_tie_blocks(rng, 5000, g_tie), g_tie),
             ((rng.standard_normal((50_000, 16)) * np.exp2(rng.uniform(-10, 10, (50_000, 1)))).astype(np.float32),
              np.float32(gs))]
    for x, g in cases:
        codes, sb = nvfp4.quantize_blocks(x, g)
        mc, msb = _cache_write_model(x, g)
        assert np.array_equal(msb, sb.reshape(-1))
        assert np.array_equal(mc, codes.reshape(-1, 16))
