"""GPU parity of the fake-quantised prefill (NVFP4 Q/K/P/V, optional 2:4
score sparsity) against the float64 oracle.  The operand quantisation is
bit-exact; the attention is compared element by element with an allowance
for the P-quantisation and 2:4 decisions whose exact quotient lies within
the kernel's float32 error of a rounding midpoint (or a score tie), which
the oracle derives per element."""
import math

import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import fakequant, nvfp4, swizzle
from tests.helpers import P_ROUNDING, assert_lse_close, check_fused_blocks, check_fused_output, f32

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"
# Relative error of the kernel's P before quantisation: the fp32 score sum
# (~1e-6 of sum |q_i k_i|, i.e. ~1e-5 in log2 units at these magnitudes)
# and ex2.approx; decisions within this of a midpoint may go either way.
TIE_REL = 5e-5
# The rest of the kernel's error relative to softmax @ |v|: fp32
# accumulation and the row sum of approximate exponentials.
ACCUM_REL = 3e-5


def _gs(x):
    return nvfp4.global_scale(np.abs(f32(x)).max())


def test_qdq_bit_exact():
    w = workloads.prefill("qdq", seq_lens=(1, 37, 16, 200, 0, 33), heads=3, seed=5)
    # q and k as strided views of a wider buffer
    big = torch.zeros((w.total_tokens, 3, 256), dtype=torch.bfloat16)
    big[..., :192] = w.q
    q = big.to(DEV)[..., :192]
    gs = [_gs(t) for t in (w.q, w.k, w.v)]
    gst = [torch.tensor([g], device=DEV) for g in gs]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    qc, kc, vc = mla.mla_nvfp4_prefill_qdq(q, w.k.to(DEV), w.v.to(DEV), w.cu_seqlens.to(DEV), w.max_seqlen, *gst,
                                           error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    cu = w.cu_seqlens.numpy()
    want_q = fakequant.qdq(f32(w.q), gs[0])
    want_k = fakequant.qdq(f32(w.k), gs[1])
    want_v = fakequant.qdq_tokens(f32(w.v), cu, gs[2])
    for got, want, g, name in ((qc, want_q, gs[0], "q"), (kc, want_k, gs[1], "k"), (vc, want_v, gs[2], "v")):
        got64 = got.cpu().double().numpy() * float(g)
        assert np.array_equal(got64, want), f"{name}: {int((got64 != want).sum())} values differ"


def _run(w, sparse, gs_out):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes, sf, lse = mla.mla_nvfp4_prefill_quantized(
        w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.cu_seqlens.to(DEV), w.max_seqlen, w.softmax_scale,
        torch.tensor([gs_out], device=DEV), sparse24=sparse, return_lse=True, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return codes.cpu().numpy(), sf.cpu().numpy(), f32(lse)


@pytest.mark.parametrize("sparse", [False, True])
@pytest.mark.parametrize("lens,heads", [((1, 37, 128, 200), 4), ((129, 0, 2), 2), ((300, 5, 64), 3), ((2000,), 2)])
def test_fakequant_prefill(lens, heads, sparse):
    w = workloads.prefill("fq", seq_lens=lens, heads=heads, seed=sum(lens) + heads)
    gs = [_gs(t) for t in (w.q, w.k, w.v)]
    o, lse, o_abs, allow = fakequant.prefill_fakequant(
        f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(), w.softmax_scale, *gs, sparse24=sparse, with_abs=True,
        tie_rel=TIE_REL)
    T = w.total_tokens
    gs_out = nvfp4.global_scale(np.abs(o).max())
    codes, sf, lse_g = _run(w, sparse, gs_out)
    assert_lse_close(lse_g, lse, f"fake-quant lse {lens}", tol=2e-4)
    o2 = o.reshape(T, heads * 128)
    err = allow + ACCUM_REL * o_abs
    print(f"[fakequant] {lens} H{heads} sparse={sparse}: elements with a decision allowance "
          f"{int((allow > 0).sum())} of {allow.size}")
    counts = check_fused_output(codes, sf, o2, (err / P_ROUNDING).reshape(T, heads * 128), gs_out,
                                f"fake-quant {lens} sparse={sparse}")
    assert counts["rate"] <= 2e-3, counts
    deq = swizzle.dequantize_rows(codes, sf, T, heads * 128, gs_out)
    ref = swizzle.dequantize_rows(*swizzle.quantize_rows(o2.astype(np.float32), gs_out), T, heads * 128, gs_out)
    rel = np.abs(deq - ref).sum() / np.abs(ref).sum()
    assert rel <= 1e-3, rel


def test_fakequant_sparse_differs_from_dense():
    """The 2:4 switch is live: sequences longer than 2 keys change."""
    w = workloads.prefill("fq", seq_lens=(64,), heads=2, seed=1)
    a = _run(w, False, np.float32(1e-3))
    b = _run(w, True, np.float32(1e-3))
    assert not np.array_equal(a[2], b[2])
    assert np.array_equal(a[2][:, :2], b[2][:, :2])  # rows 0 and 1 see at most 2 keys


@pytest.mark.parametrize("sparse", [False, True])
def test_fakequant_full_size_sampled(sparse):
    """8 sequences x 4096 tokens x 128 heads (the benchmark's fake-quant
    legs): sampled rows of two sequences and two heads against the oracle,
    one sequence-head at a time."""
    w = workloads.prefill_8x4096(device=DEV)
    gs = [nvfp4.global_scale(float(t.abs().max())) for t in (w.q, w.k, w.v)]
    gs_out = nvfp4.global_scale(float(w.v.abs().max()))
    codes, sf, lse = _run(w, sparse, gs_out)
    H = w.heads
    rng = np.random.default_rng(17)
    # rates over all sampled rows: magnitude decisions (a differing scale
    # byte counting 17) and, separately, the sign of a code that is zero on
    # both sides (a value within its error of zero; each checked so)
    total = {"scale_flips": 0, "code_flips": 0, "zero_sign": 0, "codes": 0}
    for s in (0, 5):
        a = 4096 * s
        local = sorted({0, 1, 127, 128, 2047, 4095, *rng.integers(2, 4095, 3).tolist()})
        rows = [a + r for r in local]
        for h in (0, 77):
            o, l_ref, o_abs, allow = fakequant.prefill_fakequant_seq_rows(
                f32(w.q[a:a + 4096, h]), f32(w.k[a:a + 4096, h]), f32(w.v[a:a + 4096, h]), w.softmax_scale, *gs,
                local, sparse24=sparse, tie_rel=TIE_REL)
            c_rows = codes[rows][:, h * 64:(h + 1) * 64]
            m, kk = np.meshgrid(np.array(rows), np.arange(h * 8, h * 8 + 8), indexing="ij")
            sf_rows = sf[swizzle.sf_offset(m, kk, H * 8)]
            err = allow + ACCUM_REL * o_abs
            counts = check_fused_blocks(c_rows, sf_rows, o, err / P_ROUNDING, gs_out,
                                        f"fake-quant 8x4096 seq {s} head {h} sparse={sparse}")
            for key in total:
                total[key] += counts[key]
            assert_lse_close(lse[h, rows], l_ref, f"fake-quant lse seq {s} head {h}", tol=2e-4)
    flips = (17 * total["scale_flips"] + total["code_flips"]) / total["codes"]
    signs = total["zero_sign"] / total["codes"]
    print(f"[fakequant] 8x4096 sparse={sparse}: {total} -> magnitude flips {flips:.2e}, zero signs {signs:.2e}")
    assert flips <= 2e-3 and signs <= 1e-2, total
