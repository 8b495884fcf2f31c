"""Pins for the oracle's decode, LSE merge and prefill (CPU only).

The oracle is tied to torch's scaled_dot_product_attention in float64 on
inputs where NVFP4 quantisation is lossless, to closed forms, and to
invariances that a wrong index, sign or operand would break.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention, cache, nvfp4

SCALE = 1.0 / math.sqrt(192.0)


def _on_grid_latent(rng, T, gs):
    """bf16-representable latent rows that NVFP4 reproduces exactly."""
    sb = rng.integers(0x20, 0x48, (T, 32))
    codes = rng.integers(0, 16, (T, 32, 16))
    codes[..., 3] = 7 | (rng.integers(0, 2, (T, 32)) << 3)  # |.| = 6 in every block
    x = nvfp4.e2m1_decode(codes) * nvfp4.e4m3_decode(sb)[..., None] * float(gs)
    return x.reshape(T, 512).astype(np.float32)


def _bf16(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _sdpa(q, k, v, scale, causal=False):
    return F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                          torch.from_numpy(v), scale=scale,
                                          is_causal=causal).numpy()


@pytest.mark.parametrize("rb", [432, 368])
def test_decode_lossless_matches_sdpa(rb):
    rng = np.random.default_rng(10)
    B, H, P = 2, 4, 64
    lens = [64, 100]
    gs = np.float32(2.0 ** -3)
    n_pages = 4
    perm = np.array([3, 0, 2, 1])
    table = np.array([[perm[0], 0], [perm[1], perm[2]]])
    slots = attention.decode_slots_paged(table, lens, P)
    kv = _on_grid_latent(rng, sum(lens), gs)
    pe = _bf16(rng, (sum(lens), 64))
    if rb == 368:  # fp8 rope must be on the e4m3 grid to be lossless
        pe = nvfp4.e4m3_decode(nvfp4.e4m3_encode(pe.astype(np.float64))).astype(np.float32)
    c = np.zeros((n_pages * P, rb), dtype=np.uint8)
    cache.write_cache(c, kv, pe, np.concatenate(slots), gs, rb)
    q = _bf16(rng, (B, H, 576)).astype(np.float64)
    out, lse = attention.decode(q, c, rb, gs, SCALE, slots)
    pos = 0
    for b, L in enumerate(lens):
        k = np.concatenate([kv[pos:pos + L], pe[pos:pos + L]], axis=1).astype(np.float64)
        v = kv[pos:pos + L].astype(np.float64)
        ref = _sdpa(q[b][:, None, :], np.broadcast_to(k, (H, L, 576)).copy(),
                    np.broadcast_to(v, (H, L, 512)).copy(), SCALE)[:, 0]
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)
        s = SCALE * q[b] @ k.T
        np.testing.assert_allclose(lse[b], np.log(np.exp(s).sum(1)), rtol=1e-13)
        pos += L


def test_lse_is_natural_log():
    q = np.zeros((1, 576))
    k = np.zeros((5, 576))
    v = np.arange(5 * 512, dtype=np.float64).reshape(5, 512)
    o, lse = attention.attend(q, k, v, 1.0)
    assert lse[0] == pytest.approx(math.log(5.0), abs=1e-15)
    np.testing.assert_allclose(o[0], v.mean(0))


def test_split_merge_invariance():
    rng = np.random.default_rng(11)
    H, N = 8, 300
    q = rng.standard_normal((H, 576))
    k = rng.standard_normal((N, 576))
    v = rng.standard_normal((N, 512))
    o_full, l_full = attention.attend(q, k, v, SCALE)
    for cuts in ([0, 100, 300], [0, 1, 64, 65, 299, 300], [0, 150, 150, 300]):
        parts = [attention.attend(q, k[a:b], v[a:b], SCALE) for a, b in zip(cuts[:-1], cuts[1:])]
        o, l = attention.lse_merge([p[0] for p in parts], [p[1] for p in parts])
        np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, l_full, rtol=1e-14)


def test_merge_all_empty():
    o, l = attention.lse_merge(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_paged_addressing_matches_contiguous():
    rng = np.random.default_rng(12)
    lens = [130, 64, 1]
    P = 64
    pages = [(L + P - 1) // P for L in lens]
    n_pages = sum(pages)
    perm = rng.permutation(n_pages)
    table = np.zeros((3, max(pages)), dtype=np.int64)
    pos = 0
    for b, n in enumerate(pages):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    slots = attention.decode_slots_paged(table, lens, P)
    # token t of sequence b must sit in page table[b][t//64] at row t%64
    assert slots[0][129] == table[0, 2] * 64 + 1
    assert slots[2][0] == table[2, 0] * 64
    allslots = np.concatenate(slots)
    assert len(np.unique(allslots)) == len(allslots)
    gs = np.float32(0.01)
    kv = _bf16(rng, (sum(lens), 512))
    pe = _bf16(rng, (sum(lens), 64))
    c = np.zeros((n_pages * P, 432), dtype=np.uint8)
    cache.write_cache(c, kv, pe, allslots, gs, 432)
    q = _bf16(rng, (3, 2, 576))
    out, _ = attention.decode(q, c, 432, gs, SCALE, slots)
    rec = cache.encode_records(kv, pe, gs, 432)
    pos = 0
    for b, L in enumerate(lens):
        lat, rope = cache.decode_records(rec[pos:pos + L], gs, 432)
        o, _ = attention.attend(q[b], np.concatenate([lat, rope], 1), lat, SCALE)
        np.testing.assert_allclose(out[b], o, atol=1e-13)
        pos += L


def test_topk_padding_and_order():
    rng = np.random.default_rng(13)
    gs = np.float32(0.005)
    kv = _bf16(rng, (50, 512))
    pe = _bf16(rng, (50, 64))
    c = np.zeros((50, 432), dtype=np.uint8)
    cache.write_cache(c, kv, pe, np.arange(50), gs, 432)
    q = _bf16(rng, (3, 4, 576))
    idx = np.array([[5, 7, 9, -1], [9, 5, 7, -1], [-1, -1, -1, -1]])
    out, lse = attention.decode(q, c, 432, gs, SCALE, attention.decode_slots_topk(idx))
    q1 = q.copy()
    q1[1] = q[0]
    out1, _ = attention.decode(q1, c, 432, gs, SCALE, attention.decode_slots_topk(idx))
    np.testing.assert_allclose(out1[1], out[0], atol=1e-14)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


def test_decode_brute_force_vs_unquantised():
    # tiny case: quantised attention stays within the NVFP4 error of exact
    # attention on the unquantised latent
    rng = np.random.default_rng(14)
    L, H = 8, 2
    kv = _bf16(rng, (L, 512))
    pe = _bf16(rng, (L, 64))
    gs = nvfp4.global_scale(np.abs(kv).max())
    c = np.zeros((L, 432), dtype=np.uint8)
    cache.write_cache(c, kv, pe, np.arange(L), gs, 432)
    q = _bf16(rng, (1, H, 576))
    out, _ = attention.decode(q, c, 432, gs, SCALE, [np.arange(L)])
    k = np.concatenate([kv, pe], 1).astype(np.float64)
    s = SCALE * q[0].astype(np.float64) @ k.T
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    exact = p @ kv.astype(np.float64)
    rel = np.linalg.norm(out[0] - exact) / np.linalg.norm(exact)
    assert rel < 0.2
    # and the quantised output is not the exact one (quantisation is live)
    assert rel > 1e-3


def test_prefill_matches_causal_sdpa():
    rng = np.random.default_rng(15)
    lens = [1, 37, 128, 5]
    H = 3
    T = sum(lens)
    q, k = _bf16(rng, (T, H, 192)), _bf16(rng, (T, H, 192))
    v = _bf16(rng, (T, H, 128))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, lse = attention.prefill(q, k, v, cu, SCALE)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        ref = _sdpa(q[a:e].transpose(1, 0, 2).astype(np.float64),
                    k[a:e].transpose(1, 0, 2).astype(np.float64),
                    v[a:e].transpose(1, 0, 2).astype(np.float64), SCALE, causal=True)
        np.testing.assert_allclose(o[a:e].transpose(1, 0, 2), ref, atol=1e-12)
    # first row of each sequence attends to itself only: o = v, lse = s_00
    for s in range(len(lens)):
        a = cu[s]
        np.testing.assert_allclose(o[a], v[a], atol=1e-15)
        np.testing.assert_allclose(lse[:, a], SCALE * np.einsum("hd,hd->h", q[a].astype(np.float64),
                                                                k[a].astype(np.float64)), rtol=1e-13)
    rows = [0, 1, 37, 100, T - 1]
    orow, lrow = attention.prefill_rows(q, k, v, cu, SCALE, rows, head=2)
    np.testing.assert_allclose(orow, o[rows, 2], atol=1e-14)
    np.testing.assert_allclose(lrow, lse[2, rows], rtol=1e-14)
    # the sampled |v| bound: >= |o| elementwise, and equal to the full
    # oracle's; for the first row of a sequence it is |v| of that row
    o_f, _, oabs_f = attention.prefill(q, k, v, cu, SCALE, heads=[2], with_abs=True)
    orow2, _, oabs_rows = attention.prefill_rows(q, k, v, cu, SCALE, rows, head=2, with_abs=True)
    np.testing.assert_allclose(orow2, orow, atol=0)
    np.testing.assert_allclose(oabs_rows, oabs_f[rows, 2], atol=1e-14)
    assert np.all(oabs_rows >= np.abs(orow2) - 1e-14)
    np.testing.assert_allclose(oabs_rows[0], np.abs(v[0, 2].astype(np.float64)), atol=1e-15)


def test_absorption_identity():
    # q_nope . (W_UK c) == (q_nope W_UK) . c: the 512-d latent query is exact
    rng = np.random.default_rng(16)
    W = rng.standard_normal((128, 512))
    qn = rng.standard_normal(128)
    c = rng.standard_normal(512)
    assert np.isclose(qn @ (W @ c), (qn @ W) @ c, rtol=1e-12)


def test_bf16_rounding_allowance_matches_bf16():
    # the decode tolerance allows half a bf16 ulp for the output rounding:
    # rounding to bf16 must never exceed it, and must reach it at ties
    import torch
    from tests.helpers import bf16_half_ulp
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [1.0 + 2.0 ** -8, 77.25, -300.5]])
    r = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()
    d = np.abs(r - x)
    assert np.all(d <= bf16_half_ulp(x) * (1 + 1e-12))
    assert np.isclose(d[-3], bf16_half_ulp(x[-3]))  # exact tie at 1 + 2^-8


def test_decode_with_abs_bounds_output():
    # softmax @ |v| bounds |softmax @ v| elementwise
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 6))
    k = rng.standard_normal((9, 6))
    v = rng.standard_normal((9, 3))
    o, _ = attention.attend(q, k, v, 0.5)
    oa, _ = attention.attend(q, k, np.abs(v), 0.5)
    assert np.all(oa >= np.abs(o) - 1e-15)
    assert np.any(oa > np.abs(o) + 1e-3)  # mixed signs: strictly larger somewhere


def test_query_quantisation_is_the_block_quantiser_and_lossless_on_grid():
    # a query already on the NVFP4 grid (gs_q a power of two, a magnitude-6
    # code in every block) is unchanged, so decode_q4 equals decode; and a
    # generic query moves by at most half an e2m1 step of its block scale
    from oracle import attention, cache as ocache, nvfp4
    rng = np.random.default_rng(60)
    B, H = 2, 4
    gs_q = np.float32(2.0 ** -5)
    sb = rng.integers(0x20, 0x58, (B * H, 36))
    codes = rng.integers(0, 16, (B * H, 36, 16))
    codes[..., 3] = 7
    q_grid = (nvfp4.e2m1_decode(codes) * nvfp4.e4m3_decode(sb)[..., None] * float(gs_q)).reshape(B, H, 576)
    assert np.array_equal(attention.quantize_query(q_grid.astype(np.float32), gs_q), q_grid)
    kv = rng.standard_normal((100, 512)).astype(np.float32)
    pe = rng.standard_normal((100, 64)).astype(np.float32)
    gs = nvfp4.global_scale(np.abs(kv).max())
    cache = ocache.encode_records(kv, pe.astype(np.float32), gs, 368)
    slots = [np.arange(0, 60), np.arange(60, 100)]
    o1, l1 = attention.decode_q4(q_grid.astype(np.float32), cache, 368, gs, 0.07, slots, gs_q)
    o2, l2 = attention.decode(q_grid, cache, 368, gs, 0.07, slots)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    q = rng.standard_normal((B, H, 576)).astype(np.float32)
    g = nvfp4.global_scale(np.abs(q).max())
    qh = attention.quantize_query(q, g)
    blocks = q.reshape(-1, 36, 16)
    S = (np.abs(blocks).max(-1) / 6.0)[..., None]
    assert np.all(np.abs(qh.reshape(-1, 36, 16) - blocks) <= S * (1.0 + 2.0 ** -3) + 1e-12)


def test_context_prefill_is_the_merge_of_its_parts():
    # attention over [context chunk; causal new keys] in one softmax equals
    # the LSE merge of the chunk's all-keys attention and the causal
    # attention of the new keys, and reduces to the causal prefill when the
    # chunk is empty
    from oracle import attention
    rng = np.random.default_rng(71)
    H, lens, ctx = 2, (5, 1, 9), (7, 0, 3)
    T, Tc = sum(lens), sum(ctx)
    q, k = rng.standard_normal((T, H, 192)), rng.standard_normal((T, H, 192))
    v = rng.standard_normal((T, H, 128))
    kc, vc = rng.standard_normal((Tc, H, 192)), rng.standard_normal((Tc, H, 128))
    cu = np.concatenate([[0], np.cumsum(lens)])
    cc = np.concatenate([[0], np.cumsum(ctx)])
    o, lse = attention.prefill_with_context(q, k, v, cu, kc, vc, cc, 0.07)
    o1, l1 = attention.attend_all(q, k, v, cu, kc, vc, cc, 0.07)
    o2, l2 = attention.prefill(q, k, v, cu, 0.07)
    for h in range(H):
        om, lm = attention.lse_merge(np.stack([o1[:, h], o2[:, h]]), np.stack([l1[h], l2[h]]))
        assert np.allclose(om, o[:, h], atol=1e-12) and np.allclose(lm, lse[h], atol=1e-12)
    z = np.zeros((0, H, 192))
    o0, l0 = attention.prefill_with_context(q, k, v, cu, z, np.zeros((0, H, 128)), np.zeros(4, dtype=int), 0.07)
    assert np.allclose(o0, o2, atol=1e-12) and np.allclose(l0, l2, atol=1e-12)


def test_context_rows_match_the_full_oracle():
    rng = np.random.default_rng(9)
    H, lens, ctx = 2, (5, 9), (7, 0)
    T, Tc = sum(lens), sum(ctx)
    q, k = rng.standard_normal((T, H, 192)), rng.standard_normal((T, H, 192))
    v = rng.standard_normal((T, H, 128))
    kc, vc = rng.standard_normal((Tc, H, 192)), rng.standard_normal((Tc, H, 128))
    cu, cc = np.array([0, 5, 14]), np.array([0, 7, 7])
    o, lse, o_abs = attention.prefill_with_context(q, k, v, cu, kc, vc, cc, 0.07, with_abs=True)
    rows = [0, 4, 5, 13]
    ro, rl, ra = attention.prefill_with_context_rows(q, k, v, cu, kc, vc, cc, 0.07, rows, 1, with_abs=True)
    assert np.allclose(ro, o[rows, 1], rtol=1e-12) and np.allclose(rl, lse[1, rows], rtol=1e-12)
    assert np.allclose(ra, o_abs[rows, 1], rtol=1e-12)
