"""GPU parity of the elementwise NVFP4 kernels against the oracle: the
quantise-rows hook (the prefill epilogue's quantiser), the cache write and
the global scale.  The oracle takes the exact NVFP4 decisions; the kernels
evaluate the quotients in float32, so a code or scale byte may differ only
where the exact quotient lies within that float32 error of a rounding
midpoint, and such flips are counted against a budget of 1e-4 of the codes
(tests.helpers.quant_flips).  Everything else (RoPE bytes, padding, skipped
slots, the global scale) is bit-exact."""
import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import nvfp4, swizzle
from tests.helpers import f32, oracle_gs, quant_flips, record_flips

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def _edge_matrix(M, N, seed):
    """Gaussian rows at many magnitudes plus hand-placed edge blocks: exact
    e2m1 ties, negatives that round to zero, saturating values, zero and
    subnormal-scale blocks."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((M, N)) * np.exp(rng.uniform(-8, 8, (M, 1)))).astype(np.float32)
    if M >= 4 and N >= 32:
        x[0, :16] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, 6, 0.1, -0.6, 2.9, 4.4, -5.5, 0, 6]
        x[1, :16] = 0.0
        x[1, 16:32] = -1e-30
        x[2, :16] = np.float32(1e-38) * np.arange(16)
        x[3, :16] = [-0.01, 3000, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, -3000]
    return x


@pytest.mark.parametrize("M,N,gs", [(1, 16, 1.0), (130, 48, 1.0), (256, 1024, 0.37), (300, 8192, 0.002)])
def test_quantize_rows_matches_definition(M, N, gs):
    x = _edge_matrix(M, N, seed=M + N)
    g = np.float32(gs)
    xt = torch.from_numpy(x).to(DEV)
    gst = torch.tensor([g], dtype=torch.float32, device=DEV)
    codes, sf = mla.mla_nvfp4_quantize_rows(xt, gst)
    torch.cuda.synchronize()
    codes, sf = codes.cpu().numpy(), sf.cpu().numpy()
    assert sf.size == swizzle.sf_buffer_bytes(M, N // 16)
    quant_flips(x, g, nvfp4.unpack_e2m1(codes), swizzle.unswizzle_scales(sf, M, N // 16),
                f"quantize_rows {M}x{N} gs={gs}")
    # padding rows and columns of the swizzled buffer are zero
    pad = np.ones(sf.size, dtype=bool)
    m, k = np.meshgrid(np.arange(M), np.arange(N // 16), indexing="ij")
    pad[swizzle.sf_offset(m, k, N // 16)] = False
    assert np.all(sf[pad] == 0)


def test_quantize_rows_scale_guard():
    x = torch.ones((128, 16), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes, sf = mla.mla_nvfp4_quantize_rows(x, torch.tensor([0.0], device=DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & mla.DEVERR_SCALE
    assert int(codes.abs().sum()) == 0 and int(sf.sum()) == 0


@pytest.mark.parametrize("rb", [432, 368])
def test_cache_write_tiny(rb):
    w = workloads.decode_tiny(record_bytes=rb)
    gs = oracle_gs(w.kv_c)
    cache = torch.zeros((w.num_slots, rb), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache, gst, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    c = cache.cpu().numpy()
    slots = w.slot_mapping.numpy()
    record_flips(c[slots], f32(w.kv_c), f32(w.k_pe), gs, rb, f"cache write tiny {rb}")
    untouched = np.ones(w.num_slots, dtype=bool)
    untouched[slots] = False
    assert np.all(c[untouched] == 0)


@pytest.mark.parametrize("rb", [432, 368])
def test_cache_write_ragged_skip_and_bounds(rb):
    # 37 tokens (not a multiple of the 8 tokens per block), strided rows,
    # skipped (-1) and out-of-range slots, k_pe with exact e4m3 ties
    rng = np.random.default_rng(7)
    T, S = 37, 50
    kv_full = torch.from_numpy(rng.standard_normal((T, 520)).astype(np.float32)).to(torch.bfloat16)
    kv = kv_full[:, :512]
    pe = torch.from_numpy(rng.standard_normal((T, 64)).astype(np.float32) * 30).to(torch.bfloat16)
    pe[0, :8] = torch.tensor([0.0, -0.0, 1.0625, 1.1875, -600.0, 500.0, 2 ** -10, -(2 ** -10)])
    slots = torch.from_numpy(rng.permutation(S)[:T].astype(np.int64))
    slots[3] = -1
    slots[5] = S + 10  # out of range: skipped and flagged
    gs = oracle_gs(kv)
    cache = torch.full((S, rb), 0xEE, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(kv.to(DEV), pe.to(DEV), slots.to(DEV), cache,
                              torch.tensor([gs], device=DEV), err)
    torch.cuda.synchronize()
    assert int(err.item()) == mla.DEVERR_BOUNDS
    c = cache.cpu().numpy()
    keep = slots.numpy().copy()
    keep[5] = -1
    written = keep >= 0
    record_flips(c[keep[written]], f32(kv)[written], f32(pe)[written], gs, rb, f"cache write ragged {rb}")
    untouched = np.ones(S, dtype=bool)
    untouched[keep[written]] = False
    assert np.all(c[untouched] == 0xEE)  # skipped and out-of-range tokens wrote nothing


def test_global_scale_exact():
    rng = np.random.default_rng(8)
    x = torch.from_numpy(rng.standard_normal(1000003).astype(np.float32) * 3).to(torch.bfloat16)
    x[123457] = -77.5
    gs = mla.mla_nvfp4_global_scale(x.to(DEV))
    torch.cuda.synchronize()
    assert gs.item() == float(oracle_gs(x))
    assert gs.item() == float(np.float32(77.5) / np.float32(2688))


@pytest.mark.parametrize("rb", [432, 368])
def test_cache_write_many_tokens_per_warp(rb):
    # 50,003 tokens: the grid is one wave of resident blocks, so every warp
    # loops over about ten tokens (two per iteration, ragged last iteration);
    # records land in a permuted slot order
    rng = np.random.default_rng(11)
    T = 50_003
    kv = torch.from_numpy(rng.standard_normal((T, 512)).astype(np.float32)).to(torch.bfloat16)
    pe = torch.from_numpy(rng.standard_normal((T, 64)).astype(np.float32)).to(torch.bfloat16)
    slots = torch.from_numpy(rng.permutation(T).astype(np.int64))
    gs = oracle_gs(kv)
    cache = torch.zeros((T, rb), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(kv.to(DEV), pe.to(DEV), slots.to(DEV), cache, torch.tensor([gs], device=DEV), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    c = cache.cpu().numpy()
    record_flips(c[slots.numpy()], f32(kv), f32(pe), gs, rb, f"cache write 50003 tokens {rb}")
