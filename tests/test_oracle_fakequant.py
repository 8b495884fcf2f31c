"""Pins for the oracle's fake-quantised prefill (CPU only): the operand
quantisers against brute force and hand-worked blocks, the 2:4 selection
against exhaustive enumeration, the P quantisation and softmax against
hand-computed rows, and whole-prefill properties that a wrong axis, index or
reference would break."""
import itertools
import math

import numpy as np
import pytest

from oracle import attention, fakequant, nvfp4
from tests.test_oracle_nvfp4 import _brute_force_quantize

RNG = np.random.default_rng(2244)


def _bf16(shape, scale=1.0):
    x = (RNG.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _brute_qdq(x, gs):
    codes, sb = _brute_force_quantize(x, gs)
    return nvfp4.dequantize_blocks(codes.reshape(-1, 16), sb.reshape(-1, 1), gs).reshape(np.shape(x))


def test_qdq_is_identity_on_grid():
    # a block whose max is 6 * e4m3 * gs: the scale and every code are exact
    gs = np.float32(0.01)
    sb = 0x38  # 1.0
    codes = RNG.integers(0, 16, (50, 16))
    codes[:, 5] = 7  # |x| = 6 in every block
    x = (nvfp4.e2m1_decode(codes) * nvfp4.e4m3_decode(sb) * float(gs)).astype(np.float32)
    assert np.array_equal(fakequant.qdq(x, gs), x.astype(np.float64))


def test_qdq_matches_brute_force():
    gs = nvfp4.global_scale(3.0)
    x = _bf16((400, 64))
    assert np.array_equal(fakequant.qdq(x, gs), _brute_qdq(x, gs))


@pytest.mark.parametrize("n", [1, 5, 16, 21, 40])
def test_qdq_tokens_blocks_follow_the_sequence(n):
    """V blocks are 16 tokens of one (head, feature) column from each
    sequence's first token; the last block is ragged."""
    H, D = 2, 128
    lens = [n, 3, n + 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    v = _bf16((cu[-1], H, D))
    gs = nvfp4.global_scale(np.abs(v).max())
    got = fakequant.qdq_tokens(v, cu, gs)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        for b0 in range(a, e, 16):
            b1 = min(b0 + 16, e)
            blk = np.zeros((16, H, D), dtype=np.float32)
            blk[:b1 - b0] = v[b0:b1]
            cols = blk.transpose(1, 2, 0).reshape(-1, 16)  # one block per (h, d)
            want = _brute_qdq(cols, gs).reshape(H, D, 16).transpose(2, 0, 1)[:b1 - b0]
            assert np.array_equal(got[b0:b1], want)


def test_qdq_tokens_single_token_block_closed_form():
    # a block of one token: amax = |v|, code 6 unless the scale rounds far
    v = np.array([[[0.3]], [[-1.7]], [[2.2]]], dtype=np.float32)  # 3 sequences of 1 token
    gs = np.float32(0.01)
    got = fakequant.qdq_tokens(v, [0, 1, 2, 3], gs)
    for i in range(3):
        x = float(v[i, 0, 0])
        s_raw = float(np.float32(np.float32(abs(x) / np.float32(6)) / gs))
        S = float(nvfp4.e4m3_decode(nvfp4.e4m3_encode(s_raw))) * float(gs)
        mag = nvfp4.E2M1_MAGNITUDES[np.argmin(np.abs(nvfp4.E2M1_MAGNITUDES - abs(x) / S))]
        assert got[i, 0, 0] == math.copysign(mag * S, x)


def test_select_2of4_exhaustive():
    vals = [-np.inf, -1.0, 0.0, 0.5, 2.0]
    for row in itertools.product(vals, repeat=4):
        got = fakequant.select_2of4(np.array([row]))[0]
        # brute force: rank by (value desc, index asc)
        order = sorted(range(4), key=lambda i: (-row[i], i))
        want = np.full(4, -np.inf)
        for i in order[:2]:
            want[i] = row[i]
        assert np.array_equal(got, want), row


def test_select_2of4_groups_start_at_key_zero_and_tail():
    s = np.array([[5.0, 4, 3, 2, 1, 0, -1]])  # groups [0,4) and [4,7)
    got = fakequant.select_2of4(s)[0]
    assert np.array_equal(np.isfinite(got), [True, True, False, False, True, True, False])


def test_softmax_fq_hand_worked_row():
    """Scores 0, -ln 2, -2 ln 2, ln(2/3): p = 1, 1/2, 1/4, 2/3 (M = 0); one
    block, amax 1 -> scale byte e4m3(448) (the largest), S = 448 gs_p = 1/6
    (up to gs_p's float32 rounding); p/S = 6, 3, 1.5, 4 are grid values, so
    P_hat = p exactly up to S's rounding; l = 29/12 from the unquantised p."""
    s = np.array([[0.0, -math.log(2), -2 * math.log(2), math.log(2 / 3)]])
    v = np.array([[1.0, 0], [0, 1.0], [2.0, 2.0], [-1.0, 3.0]])
    o, lse, p, p_hat, l = fakequant.softmax_fq(s, v)
    S = 448.0 * float(fakequant.P_GLOBAL_SCALE)
    assert np.allclose(p_hat[0], np.array([6, 3, 1.5, 4]) * S, rtol=0, atol=1e-15)
    assert l[0, 0] == pytest.approx(1 + 0.5 + 0.25 + 2 / 3, rel=1e-7)
    want = (np.array([6, 3, 1.5, 4]) * S) @ v / (29 / 12)
    assert np.allclose(o[0], want, rtol=1e-7)
    assert lse[0] == pytest.approx(math.log(29 / 12), abs=1e-7)


def test_softmax_fq_reference_is_a_power_of_two():
    """Adding c to every score of a row shifts the reference M by ceil; as
    long as c is a multiple of ln 2, P_hat scales by 2^(c/ln 2 - dM) exactly
    and O does not change; LSE moves by c."""
    s = RNG.standard_normal((5, 37)) * 3
    v = RNG.standard_normal((37, 8))
    o0, l0, *_ = fakequant.softmax_fq(s, v)
    for c in (math.log(2) * 3, -math.log(2) * 5):
        o1, l1, *_ = fakequant.softmax_fq(s + c, v)
        assert np.allclose(o1, o0, rtol=1e-12, atol=1e-12)
        assert np.allclose(l1, l0 + c, atol=1e-12)


def test_softmax_fq_single_key_closed_form():
    """One visible key: p = 2^(x - ceil x) in (1/2, 1]; the block's amax is p,
    its code 6 (p/S = 6 up to the scale's e4m3 rounding of at most 1/16), so
    O = v * 6 S / p and LSE = s."""
    for sv in (-3.3, 0.0, 0.2, 7.9):
        s = np.array([[sv]])
        v = np.array([[1.5, -2.0]])
        o, lse, p, p_hat, l = fakequant.softmax_fq(s, v)
        x = sv / math.log(2)
        pv = float(np.float32(2.0 ** (x - math.ceil(x))))
        g = fakequant.P_GLOBAL_SCALE
        s_raw = float(np.float32(np.float32(pv / np.float32(6)) / g))
        S = float(nvfp4.e4m3_decode(nvfp4.e4m3_encode(s_raw))) * float(g)
        assert p_hat[0, 0] == 6 * S
        assert np.allclose(o[0], v[0] * 6 * S / pv, rtol=1e-12)
        assert lse[0] == pytest.approx(sv, abs=1e-6)


def _case(lens, H=2, seed=0):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q, k = _bf16((T, H, 192)), _bf16((T, H, 192))
    v = _bf16((T, H, 128))
    cu = np.concatenate([[0], np.cumsum(lens)])
    g = [nvfp4.global_scale(np.abs(t).max()) for t in (q, k, v)]
    return q, k, v, cu, g


def test_prefill_fakequant_first_row_and_lse():
    """Row 0 of each sequence sees one key: O = v_hat[0] * 6 S / p, and its
    LSE is the quantised score itself."""
    q, k, v, cu, g = _case([7, 20])
    scale = 1 / math.sqrt(192)
    o, lse = fakequant.prefill_fakequant(q, k, v, cu, scale, *g)
    q_hat, k_hat = fakequant.qdq(q, g[0]), fakequant.qdq(k, g[1])
    v_hat = fakequant.qdq_tokens(v, cu, g[2])
    for a in cu[:-1]:
        for h in range(2):
            s0 = scale * float(q_hat[a, h] @ k_hat[a, h])
            assert lse[h, a] == pytest.approx(s0, abs=1e-7)  # l from p in float32
            x = s0 / math.log(2)
            pv = float(np.float32(2.0 ** (x - math.ceil(x))))
            gp = fakequant.P_GLOBAL_SCALE
            S = float(nvfp4.e4m3_decode(nvfp4.e4m3_encode(float(np.float32(np.float32(pv / np.float32(6)) / gp))))) * float(gp)
            assert np.allclose(o[a, h], v_hat[a, h] * 6 * S / pv, rtol=1e-12)


def test_prefill_fakequant_close_to_exact_prefill():
    """NVFP4 noise only: within ~20% (L1) of the unquantised prefill, and
    the LSE within the quantisation of the scores."""
    q, k, v, cu, g = _case([40, 70], seed=3)
    scale = 1 / math.sqrt(192)
    o, lse = fakequant.prefill_fakequant(q, k, v, cu, scale, *g)
    o_ref, l_ref = attention.prefill(q, k, v, cu, scale)
    rel = np.abs(o - o_ref).sum() / np.abs(o_ref).sum()
    assert 0.01 < rel < 0.2, rel
    assert np.abs(lse - l_ref).max() < 0.5


def test_prefill_fakequant_sparse_short_sequences_are_dense():
    """With at most 2 keys visible to every row, 2:4 keeps everything."""
    q, k, v, cu, g = _case([1, 2, 2], seed=4)
    scale = 0.1
    a = fakequant.prefill_fakequant(q, k, v, cu, scale, *g)
    b = fakequant.prefill_fakequant(q, k, v, cu, scale, *g, sparse24=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_prefill_fakequant_sparse_keeps_two_of_each_group():
    """The sparse LSE of a row is the log-sum over the top-2 keys of each
    group of its visible keys (scores from the quantised operands),
    evaluated here directly."""
    q, k, v, cu, g = _case([13], seed=5)
    scale = 1 / math.sqrt(192)
    _, lse = fakequant.prefill_fakequant(q, k, v, cu, scale, *g, sparse24=True)
    q_hat, k_hat = fakequant.qdq(q, g[0]), fakequant.qdq(k, g[1])
    for h in range(2):
        for i in range(13):
            sc = [scale * float(q_hat[i, h] @ k_hat[j, h]) for j in range(i + 1)]
            kept = []
            for g0 in range(0, i + 1, 4):
                kept += sorted(sc[g0:g0 + 4], reverse=True)[:2]
            want = math.log(sum(math.exp(t) for t in kept))
            assert lse[h, i] == pytest.approx(want, abs=1e-6)


def test_allowance_is_zero_without_near_ties_and_covers_a_planted_flip():
    q, k, v, cu, g = _case([50], seed=6)
    scale = 1 / math.sqrt(192)
    o, lse, o_abs, allow = fakequant.prefill_fakequant(q, k, v, cu, scale, *g, with_abs=True, tie_rel=1e-12)
    assert np.all(allow >= 0)
    o2, _, _, allow2 = fakequant.prefill_fakequant(q, k, v, cu, scale, *g, with_abs=True, tie_rel=2e-2)
    assert np.array_equal(o, o2)
    assert (allow2 > 0).any() and (allow2 >= allow).all()


def test_seq_rows_match_the_full_oracle():
    """The sampling form (one sequence and head, selected rows) gives the
    full oracle's rows, dense and 2:4, with the same allowances."""
    q, k, v, cu, g = _case([37], H=1, seed=8)
    scale = 1 / math.sqrt(192)
    rows = [0, 1, 15, 16, 17, 36]
    for sparse in (False, True):
        o, lse, o_abs, allow = fakequant.prefill_fakequant(q, k, v, cu, scale, *g, sparse24=sparse, with_abs=True,
                                                           tie_rel=1e-3)
        ro, rl, ra, rw = fakequant.prefill_fakequant_seq_rows(q[:, 0], k[:, 0], v[:, 0], scale, *g, rows,
                                                              sparse24=sparse, tie_rel=1e-3)
        assert np.allclose(ro, o[rows, 0], rtol=1e-12, atol=1e-15)
        assert np.allclose(rl, lse[0, rows], rtol=1e-12)
        assert np.allclose(ra, o_abs[rows, 0], rtol=1e-12, atol=1e-15)
        assert np.allclose(rw, allow[rows, 0], rtol=1e-12, atol=1e-15)
