"""GPU parity of the NVFP4-query decode (block-scaled fp4 scores) against the
float64 oracle's decode of the NVFP4-quantised query (decode_q4), with the
decode tolerances (max-abs 2e-2 beyond the output and P roundings, mean
relative 5e-3; LSE ln(1 + 5e-3)).  The query scale is computed by the oracle
from the query (amax / 2688)."""
import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import attention, nvfp4
from tests.helpers import assert_attention_close, assert_lse_close, f32, oracle_cache, oracle_gs, oracle_slots

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def _run(w, num_splits=0):
    gs = oracle_gs(w.kv_c)
    gs_q = oracle_gs(w.q)
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache, gst, err)
    kw = dict(page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV)) if w.paged else \
        dict(topk_indices=w.topk_indices.to(DEV))
    out, lse = mla.mla_nvfp4_decode_q4(w.q.to(DEV), cache, gst, w.softmax_scale, torch.tensor([gs_q], device=DEV),
                                       num_splits=num_splits, error_word=err, return_lse=True, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, l_ref, o_abs = attention.decode_q4(f32(w.q), oracle_cache(w, gs), w.record_bytes, gs, w.softmax_scale,
                                              oracle_slots(w), gs_q, with_abs=True)
    return f32(out), f32(lse), o_ref, l_ref, o_abs


@pytest.mark.parametrize("rb", [432, 368])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_q4_tiny(rb, splits):
    w = workloads.decode_tiny(record_bytes=rb)
    out, lse, o_ref, l_ref, o_abs = _run(w, splits)
    assert_attention_close(out, o_ref, f"decode q4 tiny rb={rb} splits={splits}", o_abs)
    assert_lse_close(lse, l_ref, "decode q4 tiny lse")


@pytest.mark.parametrize("rb", [432, 368])
def test_decode_q4_many_tiles_and_shapes(rb):
    lens = (1000, 129, 2049, 64, 1, 0, 65)
    w = workloads.decode_paged("q4", len(lens), 128, lens, rb, perm_pages=True, outlier_frac=0.01,
                               outlier_mult=20.0, seed=61)
    out, lse, o_ref, l_ref, o_abs = _run(w)
    assert_attention_close(out, o_ref, f"decode q4 many tiles rb={rb}", o_abs)
    assert_lse_close(lse, l_ref, "decode q4 many tiles lse")


def test_decode_q4_heads_and_topk():
    w = workloads.decode_paged("q4h", 3, 20, (300, 77, 5), 432, perm_pages=True, seed=62)
    out, lse, o_ref, l_ref, o_abs = _run(w)
    assert_attention_close(out, o_ref, "decode q4 20 heads", o_abs)
    w = workloads.decode_topk(batch=3, heads=64, context=4096, topk=300, max_pad=8, seed=63)
    out, lse, o_ref, l_ref, o_abs = _run(w)
    assert_attention_close(out, o_ref, "decode q4 top-k", o_abs)
    assert_lse_close(lse, l_ref, "decode q4 top-k lse")


def test_decode_q4_full_dsv3_sampled():
    # the 64 x 4096 x 128-head batch in the benchmark's configuration
    # (planned split); three sequences against the oracle
    w = workloads.decode_dsv3(device=DEV)
    gs = nvfp4.global_scale(float(w.kv_c.abs().max()))
    gs_q = nvfp4.global_scale(float(w.q.abs().max()))
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, gst, err)
    out, lse = mla.mla_nvfp4_decode_q4(w.q, cache, gst, w.softmax_scale, torch.tensor([gs_q], device=DEV),
                                       page_table=w.page_table, seq_lens=w.seq_lens, error_word=err,
                                       return_lse=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    from oracle import cache as ocache
    for b in (0, 41, 63):
        tok = torch.arange(4096 * b, 4096 * (b + 1), device=DEV)
        rec = ocache.encode_records(f32(w.kv_c[tok]), f32(w.k_pe[tok]), gs, 432)
        lat, rope = ocache.decode_records(rec, gs, 432)
        k = np.concatenate([lat, rope], 1)
        qh = attention.quantize_query(f32(w.q[b:b + 1]), gs_q)[0]
        o_ref, l_ref = attention.attend(qh, k, lat, w.softmax_scale)
        o_abs, _ = attention.attend(qh, k, np.abs(lat), w.softmax_scale)
        assert_attention_close(f32(out[b]), o_ref, f"decode q4 dsv3 seq {b}", o_abs)
        assert_lse_close(f32(lse[b]), l_ref, f"decode q4 dsv3 seq {b} lse")
