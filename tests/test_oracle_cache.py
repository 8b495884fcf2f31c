"""Pins for the oracle's cache record (CPU only): hand-built records with
known bytes at known offsets, and the record-width rule."""
import numpy as np
import pytest

from oracle import cache, nvfp4


def test_record_widths_rejected():
    for bad in (0, 416, 431, 433, 367, 512):
        with pytest.raises(ValueError):
            cache.check_record_bytes(bad)
    assert cache.check_record_bytes(432) is False
    assert cache.check_record_bytes(368) is True


def _hand_token():
    kv = np.zeros((1, 512), dtype=np.float32)
    kv[0, 0], kv[0, 1] = 6.0, 0.5      # block 0: amax 6 -> scale 1.0 (0x38); codes 7, 1
    kv[0, 16] = -3.0                   # block 1: amax 3 -> scale 0.5 (0x30); code -6 -> 0xF
    kv[0, 511] = 1.5                   # block 31: amax 1.5 -> 0.25 (0x28); code 6 -> 7 (high nibble)
    pe = np.zeros((1, 64), dtype=np.float32)
    pe[0, 0], pe[0, 63] = 1.0, -2.0
    return kv, pe


@pytest.mark.parametrize("rb", [432, 368])
def test_hand_built_record(rb):
    kv, pe = _hand_token()
    rec = cache.encode_records(kv, pe, np.float32(1.0), rb)[0]
    assert rec.shape == (rb,)
    assert rec[0] == 0x17            # codes 7 (low) and 1 (high)
    assert rec[8] == 0x0F            # element 16 -> byte 8 low nibble
    assert rec[255] == 0x70          # element 511 -> byte 255 high nibble
    assert rec[256] == 0x38 and rec[257] == 0x30 and rec[256 + 31] == 0x28
    assert np.all(rec[258:256 + 31] == 0)
    if rb == 432:
        assert rec[288] == 0x80 and rec[289] == 0x3F          # bf16 1.0 = 0x3F80, little endian
        assert rec[288 + 126] == 0x00 and rec[288 + 127] == 0xC0  # bf16 -2.0 = 0xC000
        assert np.all(rec[416:432] == 0)
    else:
        assert rec[288] == 0x38 and rec[288 + 63] == 0xC0      # e4m3 1.0, -2.0
        assert np.all(rec[352:368] == 0)


@pytest.mark.parametrize("rb", [432, 368])
def test_round_trip_random(rb):
    rng = np.random.default_rng(5)
    kv = rng.standard_normal((64, 512)).astype(np.float32)
    kv = (kv.view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16 values
    pe = (rng.standard_normal((64, 64)).astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    gs = nvfp4.global_scale(np.abs(kv).max())
    rec = cache.encode_records(kv, pe, gs, rb)
    lat, rope = cache.decode_records(rec, gs, rb)
    codes, sb = nvfp4.quantize_blocks(kv, gs)
    assert np.array_equal(lat, nvfp4.dequantize_blocks(codes, sb, gs))
    if rb == 432:
        assert np.array_equal(rope, pe.astype(np.float64))
    else:
        assert np.array_equal(rope, nvfp4.e4m3_decode(nvfp4.e4m3_encode(pe.astype(np.float64))))
    # relative L2 reconstruction error of NVFP4 on Gaussian data is a few percent
    err = np.linalg.norm(lat - kv) / np.linalg.norm(kv)
    assert 0.02 < err < 0.15


def test_write_cache_skips_negative_slots():
    kv, pe = _hand_token()
    kv2 = np.concatenate([kv, kv * 2])
    pe2 = np.concatenate([pe, pe])
    c = np.full((4, 432), 0xAB, dtype=np.uint8)
    cache.write_cache(c, kv2, pe2, np.array([2, -1]), np.float32(1.0), 432)
    assert np.all(c[[0, 1, 3]] == 0xAB)
    assert c[2, 0] == 0x17


def test_bf16_round_is_nearest_even():
    # against a search over the two bf16 neighbours of each value, with
    # exact ties (the midpoint of two bf16 values) going to the even one
    import torch
    from oracle import cache as oc
    rng = np.random.default_rng(70)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))
    lo = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    cand = []
    b = lo.view(torch.int16).numpy().astype(np.int32)
    for d in (-1, 0, 1):
        cand.append(torch.from_numpy((b + d).astype(np.int16)).view(torch.bfloat16).double().numpy())
    cand = np.stack(cand, 1)
    dist = np.abs(cand - x[:, None])
    best = cand[np.arange(len(x)), dist.argmin(1)]
    got = oc.bf16_round(x).astype(np.float64)
    assert np.array_equal(got, best)
    mids = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7)])
    assert oc.bf16_round(mids).tolist() == [1.0, 1.0 + 4 * 2.0 ** -8, -2.0]
