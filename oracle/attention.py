"""Absorbed MLA decode, LSE merge and causal prefill (oracle; test
infrastructure only).  Plain float64 softmax attention, no blocking.

Sources:
* "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
  TRITON_MLA) - #2244", first commit message: split-K absorbed decode over
  the paged latent cache with grouped query heads; natural-log LSE for
  merging chunks; varlen prefill with asymmetric 192/128 head dims.  Third
  commit message: the decode reads the write-once latent for both products,
  V being the latent itself.
* "nvfp4 MLA KV cache + per-layer outer-scale + fp8-RoPE KV-cell (sm120) -
  #33": sparse (top-k indexed) decode; bf16 Q staged unquantised (review of
  ``kernel.py``).

Decode (absorbed "MQA" form): q = [q_nope . W_UK (512), q_pe (64)] per head,
K_j = [x_hat_j (512), rope_j (64)], V_j = x_hat_j,
s_j = scale * q . K_j, o = sum_j softmax(s)_j V_j,
lse = max(s) + ln(sum exp(s - max(s))).
"""
from __future__ import annotations

import numpy as np

from . import cache as cache_mod, nvfp4

D_QK_DECODE = 576
D_V_DECODE = 512


def attend(q, k, v, scale):
    """q [H, D], k [N, D], v [N, Dv] (float64) -> (o [H, Dv], lse [H]).

    N == 0 gives o = 0 and lse = -inf (nothing to attend to).
    """
    q = np.asarray(q, dtype=np.float64)
    H = q.shape[0]
    if k.shape[0] == 0:
        return np.zeros((H, v.shape[1])), np.full(H, -np.inf)
    s = scale * (q @ k.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e / l) @ v
    lse = (m + np.log(l))[:, 0]
    return o, lse


def lse_merge(os, lses):
    """Merge partial attention results over disjoint key sets.

    LSE = ln sum_i exp(lse_i); O = sum_i exp(lse_i - LSE) O_i.  Partials
    with lse = -inf (empty) carry no weight; all-empty gives O = 0.
    """
    lses = np.asarray(lses, dtype=np.float64)  # [P, H]
    os = np.asarray(os, dtype=np.float64)  # [P, H, D]
    m = np.max(lses, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    o = np.einsum("ph,phd->hd", w, os) / np.where(finite, tot, 1.0)[:, None]
    return o, lse


def decode_slots_paged(page_table, seq_lens, page_size: int):
    """Slot ids per sequence: slot = page_table[b][t // P] * P + t % P."""
    out = []
    for b, L in enumerate(np.asarray(seq_lens)):
        t = np.arange(int(L))
        out.append(np.asarray(page_table)[b, t // page_size].astype(np.int64) * page_size + t % page_size)
    return out


def decode_slots_topk(topk_indices):
    """Slot ids per sequence from global top-k slot ids; -1 entries are padding."""
    out = []
    for row in np.asarray(topk_indices):
        out.append(row[row >= 0].astype(np.int64))
    return out


def decode(q, cache, record_bytes, gs, softmax_scale, slots_per_seq, with_abs=False):
    """q [B,H,576] (bf16 values), cache [num_slots, record_bytes] u8.

    Returns (out [B,H,512], lse [B,H]) in float64; with ``with_abs`` also
    softmax(s) @ |x_hat|, the scale of any rounding of the probabilities.
    """
    q = np.asarray(q, dtype=np.float64)
    B, H, D = q.shape
    assert D == D_QK_DECODE
    out = np.zeros((B, H, D_V_DECODE))
    out_abs = np.zeros((B, H, D_V_DECODE)) if with_abs else None
    lse = np.zeros((B, H))
    for b in range(B):
        slots = slots_per_seq[b]
        lat, rope = cache_mod.decode_records(cache[slots], gs, record_bytes)
        k = np.concatenate([lat, rope], axis=1)
        out[b], lse[b] = attend(q[b], k, lat, softmax_scale)
        if with_abs:
            out_abs[b], _ = attend(q[b], k, np.abs(lat), softmax_scale)
    return (out, lse, out_abs) if with_abs else (out, lse)


def quantize_query(q, gs_q):
    """The absorbed query quantised to NVFP4 and read back (the caller-side
    query quantisation of the absorbed decode): blocks of 16 along the 576
    features of each head (the contraction axis of Q K^T), e4m3 block scales,
    the float32 global scale gs_q of the whole query tensor.

    Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
    TRITON_MLA) - #2244", first commit message (forward_mqa runs the
    absorbed-Q quantise-dequantise before the decode kernel) and PR
    description, "Contract notes" (NVFP4 is 1x16 along the contraction axis,
    E4M3 block scale, amax/(6*448)).  Reading: the RoPE features are part of
    the contraction and quantised with the rest (36 blocks per head); gs_q is
    amax|q| / 2688 over the tensor.
    Returns q_hat [B, H, 576] in float64."""
    q = np.asarray(q, dtype=np.float32)
    B, H, D = q.shape
    codes, sb = nvfp4.quantize_blocks(q.reshape(B * H, D), gs_q)
    return nvfp4.dequantize_blocks(codes, sb, gs_q).reshape(B, H, D)


def decode_q4(q, cache, record_bytes, gs, softmax_scale, slots_per_seq, gs_q, with_abs=False):
    """decode() of the NVFP4-quantised query quantize_query(q, gs_q)."""
    return decode(quantize_query(q, gs_q), cache, record_bytes, gs, softmax_scale, slots_per_seq, with_abs)


def prefill(q, k, v, cu_seqlens, softmax_scale, heads=None, with_abs=False):
    """Causal varlen prefill.

    q, k [T,H,Dqk], v [T,H,Dv] (bf16 values); cu_seqlens [S+1].  Query i of a
    sequence sees keys 0..i of the same sequence.  ``heads`` restricts the
    computation to a subset of heads (the others are left zero).
    Returns (o [T,H,Dv], lse [H,T]) in float64; with ``with_abs`` also
    softmax(s) @ |v|, the scale of any rounding of the probabilities.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, H, _ = q.shape
    Dv = v.shape[2]
    heads = range(H) if heads is None else heads
    o = np.zeros((T, H, Dv))
    o_abs = np.zeros((T, H, Dv)) if with_abs else None
    lse = np.full((H, T), -np.inf)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        n = e - a
        if n == 0:
            continue
        mask = np.tril(np.ones((n, n), dtype=bool))
        for h in heads:
            sc = softmax_scale * (q[a:e, h] @ k[a:e, h].T)
            sc = np.where(mask, sc, -np.inf)
            m = sc.max(axis=1, keepdims=True)
            p = np.exp(sc - m)
            l = p.sum(axis=1, keepdims=True)
            o[a:e, h] = (p / l) @ v[a:e, h]
            if with_abs:
                o_abs[a:e, h] = (p / l) @ np.abs(v[a:e, h])
            lse[h, a:e] = (m + np.log(l))[:, 0]
    return (o, lse, o_abs) if with_abs else (o, lse)


def prefill_with_context(q, k, v, cu_seqlens, k_ctx, v_ctx, cu_ctx, softmax_scale, with_abs=False):
    """Prefill of new tokens after a cached context (chunked-context
    prefill): query i of sequence s attends to every context key of s
    (k_ctx / v_ctx rows cu_ctx[s]..cu_ctx[s+1]) and to the new keys 0..i of
    s, in one softmax.

    Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
    TRITON_MLA) - #2244", first commit message (the prefill's natural-log
    LSE serves chunked-context merging; forward_mha keeps the chunked-context
    path, whose context keys and values are projected from the latent
    gathered out of the paged cache) and second commit message (cached
    context chunks are gathered from the quantised paged cache).
    q, k [T,H,192], v [T,H,128] (new tokens); k_ctx [Tc,H,192], v_ctx
    [Tc,H,128].  Returns (o [T,H,128], lse [H,T]) in float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    kc = np.asarray(k_ctx, dtype=np.float64)
    vc = np.asarray(v_ctx, dtype=np.float64)
    T, H, _ = q.shape
    o = np.zeros((T, H, v.shape[2]))
    o_abs = np.zeros((T, H, v.shape[2])) if with_abs else None
    lse = np.full((H, T), -np.inf)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = np.asarray(cu_ctx, dtype=np.int64)
    for s_ in range(len(cu) - 1):
        a, e = int(cu[s_]), int(cu[s_ + 1])
        ca, ce = int(cc[s_]), int(cc[s_ + 1])
        for i in range(a, e):
            for h in range(H):
                keys = np.concatenate([kc[ca:ce, h], k[a:i + 1, h]])
                vals = np.concatenate([vc[ca:ce, h], v[a:i + 1, h]])
                oi, li = attend(q[i:i + 1, h], keys, vals, softmax_scale)
                o[i, h], lse[h, i] = oi[0], li[0]
                if with_abs:
                    o_abs[i, h] = attend(q[i:i + 1, h], keys, np.abs(vals), softmax_scale)[0][0]
    return (o, lse, o_abs) if with_abs else (o, lse)


def attend_all(q, k, v, cu_seqlens, k_ctx, v_ctx, cu_ctx, softmax_scale):
    """Each query of sequence s over all keys of its context chunk only (no
    mask): the partial result a context chunk contributes.  Returns (o
    [T,H,Dv], lse [H,T]); a sequence with an empty chunk gives o = 0, lse =
    -inf."""
    q = np.asarray(q, dtype=np.float64)
    T, H, _ = q.shape
    o = np.zeros((T, H, np.asarray(v_ctx).shape[2]))
    lse = np.full((H, T), -np.inf)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = np.asarray(cu_ctx, dtype=np.int64)
    for s_ in range(len(cu) - 1):
        a, e = int(cu[s_]), int(cu[s_ + 1])
        ca, ce = int(cc[s_]), int(cc[s_ + 1])
        for h in range(H):
            oo, ll = attend(q[a:e, h], np.asarray(k_ctx, np.float64)[ca:ce, h],
                            np.asarray(v_ctx, np.float64)[ca:ce, h], softmax_scale)
            o[a:e, h], lse[h, a:e] = oo, ll
    return o, lse


def prefill_rows(q, k, v, cu_seqlens, softmax_scale, rows, head, with_abs=False):
    """Causal prefill for selected global query rows of one head (sampling).
    With ``with_abs`` also softmax(s) @ |v| for those rows."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    o = np.zeros((len(rows), v.shape[2]))
    o_abs = np.zeros((len(rows), v.shape[2]))
    lse = np.zeros(len(rows))
    for i, r in enumerate(rows):
        s = int(np.searchsorted(cu, r, side="right") - 1)
        a = int(cu[s])
        kk = k[a:r + 1, head]
        o_i, l_i = attend(q[r:r + 1, head], kk, v[a:r + 1, head], softmax_scale)
        o[i], lse[i] = o_i[0], l_i[0]
        if with_abs:
            o_abs[i] = attend(q[r:r + 1, head], kk, np.abs(v[a:r + 1, head]), softmax_scale)[0][0]
    return (o, lse, o_abs) if with_abs else (o, lse)


def prefill_with_context_rows(q, k, v, cu_seqlens, k_ctx, v_ctx, cu_ctx, softmax_scale, rows, head, with_abs=False):
    """prefill_with_context for selected global query rows of one head
    (sampling at full size).  Returns (o [len(rows), Dv], lse [len(rows)])
    and with ``with_abs`` also softmax @ |v|."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = np.asarray(cu_ctx, dtype=np.int64)
    Dv = np.asarray(v).shape[2]
    o = np.zeros((len(rows), Dv))
    o_abs = np.zeros((len(rows), Dv))
    lse = np.zeros(len(rows))
    for i, r in enumerate(rows):
        s_ = int(np.searchsorted(cu, r, side="right") - 1)
        a, ca, ce = int(cu[s_]), int(cc[s_]), int(cc[s_ + 1])
        keys = np.concatenate([np.asarray(k_ctx[ca:ce, head], np.float64), np.asarray(k[a:r + 1, head], np.float64)])
        vals = np.concatenate([np.asarray(v_ctx[ca:ce, head], np.float64), np.asarray(v[a:r + 1, head], np.float64)])
        qr = np.asarray(q[r:r + 1, head], np.float64)
        oo, ll = attend(qr, keys, vals, softmax_scale)
        o[i], lse[i] = oo[0], ll[0]
        if with_abs:
            o_abs[i] = attend(qr, keys, np.abs(vals), softmax_scale)[0][0]
    return (o, lse, o_abs) if with_abs else (o, lse)

