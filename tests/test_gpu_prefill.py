"""GPU parity of the causal varlen prefill with fused NVFP4 output against
the float64 oracle.  The kernel quantises its own fp32 output, so codes and
scale bytes may differ from the oracle's quantisation of the exact output
only where the exact value sits within the attention error of a rounding
boundary; dequantised outputs meet the attention tolerance."""
import math

import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import attention, swizzle
from tests.helpers import assert_lse_close, check_fused_output, f32, oracle_gs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def _run(w, gs):
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes, sf, lse = mla.mla_nvfp4_prefill_fused_out(
        w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.cu_seqlens.to(DEV), w.max_seqlen, w.softmax_scale,
        gst, return_lse=True, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return codes.cpu().numpy(), sf.cpu().numpy(), f32(lse)


@pytest.mark.parametrize("lens,heads", [((1, 37, 128, 200), 4), ((129,), 2), ((64, 64, 1), 3)])
def test_prefill_small(lens, heads):
    w = workloads.prefill("small", seq_lens=lens, heads=heads, seed=sum(lens))
    gs = oracle_gs(w.v)
    codes, sf, lse = _run(w, gs)
    o_ref, l_ref, o_abs = attention.prefill(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(),
                                             w.softmax_scale, with_abs=True)
    T = w.total_tokens
    o2 = o_ref.reshape(T, heads * 128)
    n_sf, n_codes = check_fused_output(codes, sf, o2, o_abs.reshape(T, heads * 128), gs)
    deq = swizzle.dequantize_rows(codes, sf, T, heads * 128, gs)
    ref_deq = swizzle.dequantize_rows(*swizzle.quantize_rows(o2.astype(np.float32), gs), T, heads * 128, gs)
    # codes agree up to boundary flips (checked above), so the dequantised
    # outputs agree in mean relative L1; a flipped code moves one e2m1 step
    rel = np.abs(deq - ref_deq).sum() / np.abs(ref_deq).sum()
    assert rel <= 5e-3, rel
    assert_lse_close(lse, l_ref, "prefill lse")
    # padding rows of the scale buffer are zero
    Mp = (T + 127) // 128 * 128
    m, k = np.meshgrid(np.arange(T, Mp), np.arange(heads * 8), indexing="ij")
    assert np.all(sf[swizzle.sf_offset(m, k, heads * 8)] == 0)
