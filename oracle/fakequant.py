"""Fake-quantised causal prefill: NVFP4 Q/K/P/V and 2:4 score sparsity.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Add NVFP4/FP8 Q/K/P/V + 2:4 attention quantization for MLA (vLLM
TRITON_MLA) - #2244": the first commit message (mla_prefill: varlen prefill
with asymmetric head dims, fused Q/K/P/V fake quant, token-exact N:M score
sparsity, natural-log LSE) and the PR description ("What does this PR do?":
the prefill quantises the projected Q/K/P/V operands once, with optional
token-exact N:M (2:4) score sparsity on new-token attention; "Contract
notes": NVFP4 is 1x16 along the contraction axis with an e4m3 block scale
and amax/(6*448) as the global scale, the softmax denominator stays
unquantised, P is quantised after the row sum).

Each operand is quantised once along the axis its product contracts:

  Q, K   blocks of 16 along the 192 features of a (token, head) row
         (Q K^T contracts the features), global scales gs_q, gs_k;
  V      blocks of 16 tokens of one (head, feature) column, counted from
         the sequence's first token, the last block of a sequence ragged
         (P V contracts the keys), global scale gs_v;
  P      blocks of 16 keys of one query row, counted from the sequence's
         first key, global scale gs_p = amax/(6*448) with amax = 1.

Readings (the pages fix the block rule and the global-scale rule, not the
rest):
  * The global scales of Q, K and V are amax/(6*448) over each whole tensor
    (per-tensor, as for the cache's latent); the caller passes them.
  * P is quantised relative to a reference that is a power of two, namely
    the row's max score rounded up in log2 units: p_j = 2^(x_j - M),
    x_j = s_j log2(e), M = ceil(max_j x_j), so every p_j <= 1 and the amax
    of P is taken as 1 (gs_p = f32(1/2688)).  NVFP4 quantisation commutes
    with scaling by a power of two as long as the block scales stay normal
    e4m3 values, so any running reference that differs from M by a power
    of two (a one-pass kernel's) quantises P the same way.
  * p is rounded to float32 (the softmax's precision) before it is
    quantised; the row sum l = sum_j p_j is taken from the unquantised p.
  * 2:4 sparsity: for each query row, each group of 4 consecutive keys
    counted from the sequence's first key keeps its 2 largest scores (equal
    scores: the lower key index first) and drops the others from the
    softmax (numerator and denominator); keys hidden by the causal mask
    count as -inf, so a group cut by the diagonal keeps its visible keys up
    to 2.
  * O = (P_hat V_hat) / l and LSE = ln l + M ln 2, natural log.
"""
from __future__ import annotations

import math

import numpy as np

from . import nvfp4

P_GLOBAL_SCALE = nvfp4.global_scale(1.0)
LOG2E = 1.0 / math.log(2.0)


def qdq(x, gs) -> np.ndarray:
    """NVFP4 quantise-dequantise along the last axis (a multiple of 16):
    x_hat = e2m1 * e4m3 * gs in float64, from float32 x."""
    codes, sb = nvfp4.quantize_blocks(np.asarray(x, dtype=np.float32), gs)
    return nvfp4.dequantize_blocks(codes, sb, gs)


def qdq_padded(x, gs) -> np.ndarray:
    """qdq along the last axis of any length: the last block is completed
    with zeros (which leave its amax unchanged) and the padding dropped."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    pad = (-n) % nvfp4.BLOCK
    if pad:
        x = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,), dtype=np.float32)], axis=-1)
    return qdq(x, gs)[..., :n]


def qdq_tokens(v, cu_seqlens, gs) -> np.ndarray:
    """V [T, H, D] quantised along the tokens: per sequence, blocks of 16
    tokens of each (head, feature) column from the sequence's first token."""
    v = np.asarray(v, dtype=np.float32)
    out = np.zeros(v.shape)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        if e > a:
            cols = np.moveaxis(v[a:e], 0, -1)  # [H, D, n]
            out[a:e] = np.moveaxis(qdq_padded(cols, gs), -1, 0)
    return out


def select_2of4(s) -> np.ndarray:
    """2:4 sparsity of a score matrix [rows, keys] (-inf = hidden): in each
    group of 4 consecutive keys from key 0, keep the 2 largest per row
    (ties: lower key index first); the rest become -inf."""
    s = np.asarray(s, dtype=np.float64)
    out = np.full(s.shape, -np.inf)
    for g in range(0, s.shape[1], 4):
        grp = s[:, g:g + 4]
        # stable sort on -value: equal values keep their index order
        order = np.argsort(-grp, axis=1, kind="stable")[:, :2]
        rows = np.arange(s.shape[0])[:, None]
        out[rows, g + order] = grp[rows, order]
    return out


def softmax_fq(s, v_hat):
    """The softmax and P V of one head of one sequence, from its kept scores
    s [n, n_k] (-inf = dropped or hidden) and V_hat [n_k, Dv]: p = 2^(x - M)
    in float32 (x = s log2 e, M = ceil(max x) per row), l = sum p, P_hat =
    NVFP4(p) in blocks of 16 keys with gs_p, O = P_hat V_hat / l, LSE =
    ln l + M ln 2.  Returns (o, lse, p, p_hat, l)."""
    x = np.asarray(s, dtype=np.float64) * LOG2E
    M = np.ceil(x.max(axis=1, keepdims=True))
    p = np.exp2(x - M).astype(np.float32)  # dropped and hidden keys: exactly 0
    l = p.astype(np.float64).sum(axis=1, keepdims=True)
    p_hat = qdq_padded(p, P_GLOBAL_SCALE)
    o = (p_hat @ np.asarray(v_hat, dtype=np.float64)) / l
    lse = (M[:, 0] + np.log2(l[:, 0])) / LOG2E
    return o, lse, p, p_hat, l


def prefill_fakequant(q, k, v, cu_seqlens, softmax_scale, gs_q, gs_k, gs_v, sparse24=False, with_abs=False,
                      tie_rel=None):
    """Causal varlen prefill with NVFP4 fake-quantised Q, K, P, V and
    optional 2:4 score sparsity (module docstring for the readings).

    q, k [T, H, 192], v [T, H, 128] (bf16 values); cu_seqlens [S+1];
    gs_q, gs_k, gs_v float32 global scales.
    Returns (o [T, H, 128], lse [H, T]) in float64; with ``with_abs`` also
    (P_hat |V_hat|) / l.  With ``tie_rel`` also a per-element allowance
    [T, H, 128] for the decisions a kernel computing in float32 may take
    differently: every P element whose quotient p/S (or whose block's
    amax/6/gs_p) lies within tie_rel (relative) of a rounding midpoint may
    move by one grid step of its block (at most amax16/3, or 1/8 of amax16
    for the scale), and every 2:4 group whose 2nd and 3rd largest scores lie
    within tie_rel * (1 + |s|) of each other may swap them; the allowance is
    the sum of those moves times |v_hat| (plus |o| for a swap, which also
    moves l), over l."""
    q_hat = qdq(q, gs_q)
    k_hat = qdq(k, gs_k)
    v_hat = qdq_tokens(v, cu_seqlens, gs_v)
    T, H, _ = q_hat.shape
    Dv = v_hat.shape[2]
    o = np.zeros((T, H, Dv))
    o_abs = np.zeros((T, H, Dv)) if with_abs else None
    allow = np.zeros((T, H, Dv)) if tie_rel is not None else None
    lse = np.full((H, T), -np.inf)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    mids_c = (nvfp4.E2M1_MAGNITUDES[:-1] + nvfp4.E2M1_MAGNITUDES[1:]) / 2
    grid_s = nvfp4.e4m3_decode(np.arange(0x7F))
    mids_s = (grid_s[:-1] + grid_s[1:]) / 2
    for sq in range(len(cu) - 1):
        a, e = int(cu[sq]), int(cu[sq + 1])
        n = e - a
        if n == 0:
            continue
        mask = np.tril(np.ones((n, n), dtype=bool))
        for h in range(H):
            s = softmax_scale * (q_hat[a:e, h] @ k_hat[a:e, h].T)
            s = np.where(mask, s, -np.inf)
            s_dense = s
            if sparse24:
                s = select_2of4(s)
            vv = v_hat[a:e, h]
            o[a:e, h], lse[h, a:e], p, p_hat, l = softmax_fq(s, vv)
            if with_abs:
                o_abs[a:e, h] = (p_hat @ np.abs(vv)) / l
            if tie_rel is not None:
                allow[a:e, h] = _allowance(p, s_dense if sparse24 else None, s, vv, o[a:e, h], l, tie_rel,
                                           mids_c, mids_s)
    if tie_rel is not None:
        return o, lse, o_abs, allow
    return (o, lse, o_abs) if with_abs else (o, lse)


def _allowance(p, s_dense, s_kept, vv, o, l, rel, mids_c, mids_s):
    """Per-row allowance of prefill_fakequant (its docstring)."""
    n = p.shape[1]
    pad = (-n) % nvfp4.BLOCK
    pb = np.concatenate([p.astype(np.float64), np.zeros((p.shape[0], pad))], axis=1)
    pb = pb.reshape(p.shape[0], -1, nvfp4.BLOCK)
    amax = pb.max(axis=-1)
    g = float(P_GLOBAL_SCALE)
    sraw = amax / 6.0 / g
    near_s = np.min(np.abs(sraw[..., None] - mids_s), axis=-1) <= rel * sraw
    sb = nvfp4.choose_scale(amax.astype(np.float32), P_GLOBAL_SCALE)
    S = nvfp4.e4m3_decode(sb) * g
    qv = np.where(S[..., None] > 0, pb / np.where(S > 0, S, 1.0)[..., None], 0.0)
    near_c = np.min(np.abs(qv[..., None] - mids_c), axis=-1) <= rel * np.maximum(qv, 1e-30)
    move = np.where(near_c, 2.0 * S[..., None], 0.0)  # one e2m1 step is at most 2 S
    move = np.maximum(move, np.where(near_s, amax / 8.0 + 2.0 * S, 0.0)[..., None])
    move = move.reshape(p.shape[0], -1)[:, :n]
    allow = move @ np.abs(vv)
    if s_dense is not None:
        # 2:4 groups whose 2nd and 3rd scores nearly tie: both keys may swap
        x = np.exp(s_dense - np.max(np.where(np.isfinite(s_kept), s_kept, -np.inf), axis=1, keepdims=True))
        for g0 in range(0, n, 4):
            grp = s_dense[:, g0:g0 + 4]
            if grp.shape[1] < 3:
                continue
            srt = -np.sort(-grp, axis=1)
            fin = np.isfinite(srt[:, 2])
            gap = np.abs(srt[:, 1] - np.where(fin, srt[:, 2], 0.0))  # (hidden 3rd key: no tie)
            near = fin & (gap <= rel * (1.0 + np.abs(srt[:, 1])))
            if near.any():
                w = x[:, g0:g0 + 4] * near[:, None]
                allow += 2.0 * (w @ np.abs(vv[g0:g0 + 4]) + w.sum(axis=1, keepdims=True) * np.abs(o))
    return allow / l


def prefill_fakequant_seq_rows(q_seq, k_seq, v_seq, softmax_scale, gs_q, gs_k, gs_v, rows, sparse24=False,
                               tie_rel=None):
    """prefill_fakequant for selected rows of one sequence and head (sampling
    at full size): q_seq, k_seq [n, 192], v_seq [n, 128] are the head's
    values over the whole sequence; rows are indices within it.  Returns
    (o [len(rows), 128], lse [len(rows)], o_abs, allowance) as
    prefill_fakequant does for those rows."""
    q_hat = qdq(q_seq, gs_q)
    k_hat = qdq(k_seq, gs_k)
    n = np.asarray(v_seq).shape[0]
    v_hat = qdq_tokens(np.asarray(v_seq)[:, None, :], [0, n], gs_v)[:, 0, :]
    mids_c = (nvfp4.E2M1_MAGNITUDES[:-1] + nvfp4.E2M1_MAGNITUDES[1:]) / 2
    grid_s = nvfp4.e4m3_decode(np.arange(0x7F))
    mids_s = (grid_s[:-1] + grid_s[1:]) / 2
    Dv = v_hat.shape[1]
    o = np.zeros((len(rows), Dv))
    o_abs = np.zeros((len(rows), Dv))
    allow = np.zeros((len(rows), Dv))
    lse = np.zeros(len(rows))
    for i, r in enumerate(rows):
        s = softmax_scale * (q_hat[r:r + 1] @ k_hat[:r + 1].T)
        s_kept = select_2of4(s) if sparse24 else s
        vv = v_hat[:r + 1]
        oo, ll, p, p_hat, l = softmax_fq(s_kept, vv)
        o[i], lse[i] = oo[0], ll[0]
        o_abs[i] = ((p_hat @ np.abs(vv)) / l)[0]
        if tie_rel is not None:
            allow[i] = _allowance(p, s if sparse24 else None, s_kept, vv, oo, l, tie_rel, mids_c, mids_s)[0]
    return o, lse, o_abs, allow

