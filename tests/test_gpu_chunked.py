"""GPU parity of the chunked-context prefill (new tokens after a cached
context) against the float64 oracle: the cache read-back of a context chunk
(bit-exact), the partial attention over a chunk and over the new tokens'
causal prefix (unquantised fp32 output and LSE), and the LSE merge written
as the fused NVFP4 output, end to end after the kernels' own cache write."""
import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import attention, cache as ocache, nvfp4, swizzle
from tests.helpers import (MEAN_REL, P_ROUNDING, assert_lse_close, check_fused_blocks, check_fused_output, f32,
                           oracle_cache, oracle_gs, quant_flips)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"
# flip rate of the fused output (see the prefill tests: set by the attention
# error, not by the quantiser)
FUSED_FLIP_RATE = 2e-2


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _assert_partial_close(got, ref, o_abs, what):
    """Unquantised prefill output: the bf16 rounding of P bounds the error
    by P_ROUNDING * softmax @ |v| (fp32 accumulation adds ~1e-6 relative)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    excess = err - P_ROUNDING * o_abs - 1e-6 * np.abs(ref)
    mean_rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
    print(f"[partial] {what}: raw max-abs {err.max():.3e}, beyond the P rounding {excess.max():.3e}, "
          f"mean rel {mean_rel:.3e}")
    assert excess.max() <= 1e-5 and mean_rel <= MEAN_REL, what


@pytest.mark.parametrize("record_bytes", [432, 368])
def test_gather_latent_bit_exact(record_bytes):
    w = workloads.decode_tiny(seed=3, heads=4, seq_lens=(200, 77), record_bytes=record_bytes)
    gs = oracle_gs(w.kv_c)
    cache = oracle_cache(w, gs)
    g = torch.Generator().manual_seed(5)
    slots = torch.randint(0, w.num_slots, (1000,), generator=g, dtype=torch.int64)
    slots[::97] = -1
    err = _err()
    kv, pe = mla.mla_nvfp4_gather_latent(torch.from_numpy(cache).to(DEV), torch.tensor([gs], device=DEV),
                                         slots.to(DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    s = slots.numpy()
    lat, rope = ocache.gather_latent(cache, np.where(s < 0, 0, s), gs, record_bytes)
    lat[s < 0] = 0
    rope[s < 0] = 0
    assert np.array_equal(f32(kv), lat)
    assert np.array_equal(f32(pe), rope)


def test_gather_latent_out_of_range_flags():
    w = workloads.decode_tiny(seed=4, heads=4, seq_lens=(64,))
    gs = oracle_gs(w.kv_c)
    cache = torch.from_numpy(oracle_cache(w, gs)).to(DEV)
    slots = torch.tensor([0, w.num_slots, 5], dtype=torch.int64, device=DEV)
    err = _err()
    kv, pe = mla.mla_nvfp4_gather_latent(cache, torch.tensor([gs], device=DEV), slots, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & mla.DEVERR_BOUNDS
    assert not kv[1].any() and not pe[1].any()
    lat, _ = ocache.gather_latent(cache.cpu().numpy(), [0, 5], gs, 432)
    assert np.array_equal(f32(kv[[0, 2]]), lat)


def _partial(q, k, v, cu, max_len, scale, cu_k=None):
    err = _err()
    o, lse = mla.mla_nvfp4_prefill_partial(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), max_len, scale,
                                           cu_seqlens_k=None if cu_k is None else cu_k.to(DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o, lse


@pytest.mark.parametrize("lens,ctx,heads", [((1, 37, 200), (300, 0, 129), 4), ((129,), (1,), 2),
                                            ((300, 5, 64), (1000, 2500, 0), 8)])
def test_partial_context_chunk(lens, ctx, heads):
    w = workloads.prefill_context(lens, ctx, heads=heads, seed=sum(lens) + sum(ctx))
    o, lse = _partial(w.q, w.k_ctx, w.v_ctx, w.cu_seqlens, w.max_seqlen, w.softmax_scale, cu_k=w.cu_ctx)
    args = (f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(), f32(w.k_ctx), f32(w.v_ctx), w.cu_ctx.numpy(),
            w.softmax_scale)
    o_ref, l_ref = attention.attend_all(*args)
    o_abs, _ = attention.attend_all(*args[:5], np.abs(f32(w.v_ctx)), *args[6:])
    _assert_partial_close(f32(o), o_ref, o_abs, f"context chunk {lens}/{ctx}")
    assert_lse_close(f32(lse), l_ref, f"context chunk {lens}/{ctx}")


@pytest.mark.parametrize("lens,heads", [((1, 37, 128, 200), 4), ((1000, 0, 300), 8)])
def test_partial_causal(lens, heads):
    w = workloads.prefill("small", seq_lens=lens, heads=heads, seed=sum(lens) + 1)
    o, lse = _partial(w.q, w.k, w.v, w.cu_seqlens, w.max_seqlen, w.softmax_scale)
    o_ref, l_ref, o_abs = attention.prefill(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(), w.softmax_scale,
                                            with_abs=True)
    _assert_partial_close(f32(o), o_ref, o_abs, f"causal {lens}")
    assert_lse_close(f32(lse), l_ref, f"causal {lens}")


def test_partial_every_chunk_empty():
    w = workloads.prefill_context((40, 7), (0, 0), heads=2, seed=9)
    o, lse = _partial(w.q, w.k, w.v, w.cu_seqlens, w.max_seqlen, w.softmax_scale,
                      cu_k=torch.zeros(3, dtype=torch.int32))
    assert not o.any() and bool(torch.isneginf(lse).all())


@pytest.mark.parametrize("parts", [1, 3])
def test_merge_fused_out(parts):
    T, H = 300, 4
    g = torch.Generator().manual_seed(parts)
    o_parts = torch.randn((parts, T, H, 128), generator=g)
    lse_parts = torch.randn((parts, H, T), generator=g) * 3
    lse_parts[0, :, :7] = float("-inf")  # a part that saw no key
    gs = np.float32(2.0 / 2688)
    err = _err()
    codes, sf = mla.mla_nvfp4_merge_fused_out(o_parts.to(DEV), lse_parts.to(DEV), torch.tensor([gs], device=DEV),
                                              error_word=err)
    lse_out = torch.empty((H, T), device=DEV)
    mla.mla_nvfp4_merge_fused_out(o_parts.to(DEV), lse_parts.to(DEV), torch.tensor([gs], device=DEV),
                                  lse=lse_out, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    op, lp = o_parts.numpy().astype(np.float64), lse_parts.numpy().astype(np.float64)
    o_m, l_m = np.zeros((T, H, 128)), np.zeros((H, T))
    for t in range(T):
        o_m[t], l_m[:, t] = attention.lse_merge(op[:, t], lp[:, :, t])
    assert_lse_close(f32(lse_out), l_m, "merged lse", tol=1e-5)
    # the merge in fp32 moves each value by ~1e-6 relative: compare the
    # quantisation of the merged fp32 values through the fused-output rule
    # with a tiny error in place of the attention error
    o2 = o_m.reshape(T, H * 128)
    counts = check_fused_output(codes.cpu().numpy(), sf.cpu().numpy(), o2,
                                np.abs(o2) * (4e-6 / P_ROUNDING), gs, f"merge P={parts}")
    assert counts["rate"] <= 1e-3, counts


@pytest.mark.parametrize("record_bytes", [432, 368])
def test_chunked_prefill_end_to_end(record_bytes):
    """Cache write (kernel) -> gather of each sequence's context (kernel) ->
    per-head projection of the gathered latent (the model's kv_b_proj, here
    a float64 matmul rounded to bf16 on the host, the same input for both
    sides) -> partial attention over the chunk and over the new tokens
    (kernel) -> LSE merge into the fused NVFP4 output (kernel), against the
    oracle's single-softmax prefill_with_context over the same keys."""
    H, lens, ctx = 4, (33, 150, 1), (500, 64, 0)
    g = torch.Generator().manual_seed(record_bytes)
    Tc = sum(ctx)
    kv_c = (torch.randn((Tc, 512), generator=g)).to(torch.bfloat16)
    k_pe = (torch.randn((Tc, 64), generator=g)).to(torch.bfloat16)
    perm = torch.randperm(4 * Tc, generator=g)[:Tc].to(torch.int64)  # scattered slots
    num_slots = 4 * Tc
    gs = oracle_gs(kv_c)
    gst = torch.tensor([gs], device=DEV)
    cache = torch.zeros((num_slots, record_bytes), dtype=torch.uint8, device=DEV)
    err = _err()
    mla.mla_nvfp4_cache_write(kv_c.to(DEV), k_pe.to(DEV), perm.to(DEV), cache, gst, error_word=err)
    kv, pe = mla.mla_nvfp4_gather_latent(cache, gst, perm.to(DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lat_ref, rope_ref = ocache.gather_latent(cache.cpu().numpy(), perm.numpy(), gs, record_bytes)
    assert np.array_equal(f32(kv), lat_ref) and np.array_equal(f32(pe), rope_ref)
    # the projection (caller's GEMM): k_nope and v per head from the latent
    w_kv = torch.randn((512, H * 256), generator=g, dtype=torch.float64) / 512 ** 0.5
    kvp = (lat_ref.astype(np.float64) @ w_kv.numpy()).reshape(Tc, H, 256)
    k_ctx = np.concatenate([kvp[..., :128], np.broadcast_to(rope_ref[:, None, :], (Tc, H, 64))], axis=2)
    k_ctx = torch.from_numpy(ocache.bf16_round(k_ctx)).to(torch.bfloat16)
    v_ctx = torch.from_numpy(ocache.bf16_round(kvp[..., 128:])).to(torch.bfloat16)
    w = workloads.prefill("new", seq_lens=lens, heads=H, seed=11)
    cu_ctx = torch.tensor(np.concatenate([[0], np.cumsum(ctx)]), dtype=torch.int32)
    o1, l1 = _partial(w.q, k_ctx, v_ctx, w.cu_seqlens, w.max_seqlen, w.softmax_scale, cu_k=cu_ctx)
    o2, l2 = _partial(w.q, w.k, w.v, w.cu_seqlens, w.max_seqlen, w.softmax_scale)
    o_ref, l_ref, o_abs = attention.prefill_with_context(
        f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(), f32(k_ctx), f32(v_ctx), cu_ctx.numpy(),
        w.softmax_scale, with_abs=True)
    T = w.total_tokens
    o_ref2 = o_ref.reshape(T, H * 128)
    gso = nvfp4.global_scale(np.abs(o_ref).max())
    lse = torch.empty((H, T), device=DEV)
    codes, sf = mla.mla_nvfp4_merge_fused_out(torch.stack([o1, o2]), torch.stack([l1, l2]),
                                              torch.tensor([gso], device=DEV), lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_lse_close(f32(lse), l_ref, "chunked prefill lse")
    counts = check_fused_output(codes.cpu().numpy(), sf.cpu().numpy(), o_ref2, o_abs.reshape(T, H * 128), gso,
                                f"chunked prefill {record_bytes}")
    assert counts["rate"] <= FUSED_FLIP_RATE, counts
    deq = swizzle.dequantize_rows(codes.cpu().numpy(), sf.cpu().numpy(), T, H * 128, gso)
    ref_deq = swizzle.dequantize_rows(*swizzle.quantize_rows(o_ref2.astype(np.float32), gso), T, H * 128, gso)
    rel = np.abs(deq - ref_deq).sum() / np.abs(ref_deq).sum()
    assert rel <= 5e-3, rel


def test_chunked_full_size_sampled():
    """The benchmark's chunked-context shape: 8 x 4096 new tokens after 8 x
    4096 context tokens per sequence, 128 heads, in its launch order
    (partial over the context, partial causal, merge); sampled rows of two
    sequences and two heads against the oracle's single-softmax prefill."""
    w = workloads.prefill_context((4096,) * 8, (4096,) * 8, heads=128, seed=3, device=DEV)
    err = _err()
    o1, l1 = mla.mla_nvfp4_prefill_partial(w.q, w.k_ctx, w.v_ctx, w.cu_seqlens, w.max_seqlen, w.softmax_scale,
                                           cu_seqlens_k=w.cu_ctx, error_word=err)
    o2, l2 = mla.mla_nvfp4_prefill_partial(w.q, w.k, w.v, w.cu_seqlens, w.max_seqlen, w.softmax_scale,
                                           error_word=err)
    gs_out = nvfp4.global_scale(max(float(w.v.abs().max()), float(w.v_ctx.abs().max())))
    lse = torch.empty((w.heads, w.total_tokens), device=DEV)
    codes, sf = mla.mla_nvfp4_merge_fused_out(torch.stack([o1, o2]), torch.stack([l1, l2]),
                                              torch.tensor([gs_out], device=DEV), lse=lse, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    del o1, o2
    H = w.heads
    cu, cc = w.cu_seqlens.cpu().numpy(), w.cu_ctx.cpu().numpy()
    rng = np.random.default_rng(23)
    rows = sorted({a + r for a in (0, 3 * 4096, 6 * 4096)
                   for r in (0, 1, 127, 128, 4095, *rng.integers(2, 4095, 11).tolist())})
    sf_np, lse_np = sf.cpu().numpy(), f32(lse)
    # the flip rate is a rate over many codes: taken over all sampled rows
    # of both heads (each flip is checked to lie at a rounding boundary)
    total = {"scale_flips": 0, "code_flips": 0, "zero_sign": 0, "codes": 0}
    for h in (0, 100):
        sl = slice(h, h + 1)
        o_ref, l_ref, o_abs = attention.prefill_with_context_rows(
            f32(w.q[:, sl]), f32(w.k[:, sl]), f32(w.v[:, sl]), cu, f32(w.k_ctx[:, sl]), f32(w.v_ctx[:, sl]), cc,
            w.softmax_scale, rows, 0, with_abs=True)
        c_rows = codes[rows][:, h * 64:(h + 1) * 64].cpu().numpy()
        m, kk = np.meshgrid(np.array(rows), np.arange(h * 8, h * 8 + 8), indexing="ij")
        counts = check_fused_blocks(c_rows, sf_np[swizzle.sf_offset(m, kk, H * 8)], o_ref, o_abs, gs_out,
                                    f"chunked 8x4096+4096 head {h} sampled rows")
        for key in total:
            total[key] += counts[key]
        assert_lse_close(lse_np[h, rows], l_ref, f"chunked lse head {h}")
    rate = (17 * total["scale_flips"] + total["code_flips"] + total["zero_sign"]) / total["codes"]
    print(f"[fused] chunked 8x4096+4096, both heads: {total} -> mismatch rate {rate:.2e}")
    assert rate <= FUSED_FLIP_RATE, total
