"""GPU parity of the absorbed NVFP4 decode against the float64 oracle
(max-abs 2e-2, mean relative L1 5e-3 on the bf16 output; LSE within 2e-3)."""
import math

import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import attention
from tests.helpers import assert_attention_close, assert_lse_close, f32, oracle_cache, oracle_gs, oracle_slots

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def run_gpu(w, gs, num_splits=0):
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache, gst, err)
    kw = dict(page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV)) if w.paged else \
        dict(topk_indices=w.topk_indices.to(DEV))
    out, lse = mla.mla_nvfp4_decode(w.q.to(DEV), cache, gst, w.softmax_scale, num_splits=num_splits,
                                    error_word=err, return_lse=True, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return f32(out), f32(lse)


def run_oracle(w, gs):
    """(out, lse, softmax @ |v|) of the float64 oracle."""
    c = oracle_cache(w, gs)
    return attention.decode(f32(w.q), c, w.record_bytes, gs, w.softmax_scale, oracle_slots(w), with_abs=True)


@pytest.mark.parametrize("rb", [432, 368])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_tiny(rb, splits):
    w = workloads.decode_tiny(record_bytes=rb)
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, splits)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(out, o_ref, f"decode tiny rb={rb} splits={splits}", o_abs)
    assert_lse_close(lse, l_ref, "decode tiny lse")


@pytest.mark.parametrize("heads,lens", [(128, (1, 63, 64, 65, 100)), (64, (200, 7)), (20, (129,))])
def test_decode_shapes(heads, lens):
    w = workloads.decode_paged("sweep", len(lens), heads, lens, 432, perm_pages=True, seed=3)
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(out, o_ref, f"decode heads={heads} lens={lens}", o_abs)
    assert_lse_close(lse, l_ref, "decode lse")


@pytest.mark.parametrize("splits", [0, 1])  # 1: output written by the decode kernel itself
def test_decode_topk_small(splits):
    w = workloads.decode_topk(batch=3, heads=32, context=4096, topk=300, max_pad=8, seed=5)
    w.topk_indices[2, :] = -1  # a row with nothing to attend to
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, splits)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))
    assert_attention_close(out, o_ref, "decode top-k small", o_abs)
    assert_lse_close(lse, l_ref, "decode top-k lse")


@pytest.mark.parametrize("rb", [432, 368])
@pytest.mark.parametrize("splits", [1, 2, 7])
def test_decode_many_tiles_per_split(rb, splits):
    # several 64-key tiles per CTA: exercises both operand buffers, the score
    # product split around P.V, and the lazy rescale across tiles (outliers)
    lens = (1000, 129, 2049, 64)
    w = workloads.decode_paged("tiles", len(lens), 128, lens, rb, perm_pages=True, outlier_frac=0.01,
                               outlier_mult=20.0, seed=7)
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, splits)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(out, o_ref, f"decode many tiles rb={rb} splits={splits}", o_abs)
    assert_lse_close(lse, l_ref, "decode many tiles lse")


@pytest.mark.parametrize("case", ["small_latent", "large_query"])
def test_decode_query_range_scaling(case):
    # q_pe/gs or q itself beyond the f16 range: the query is staged with a
    # per-head power-of-two scale, undone in the score scale
    w = workloads.decode_paged("range", 2, 64, (300, 77), 432, perm_pages=True, seed=9)
    if case == "small_latent":
        w.kv_c = (w.kv_c.float() * 1e-3).to(torch.bfloat16)  # gs ~ 2e-6: q_pe/gs ~ 1e6
    else:
        w.q = (w.q.float() * 3e4).to(torch.bfloat16)
        w.softmax_scale = w.softmax_scale / 3e4
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, 1)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(out, o_ref, f"decode query range {case}", o_abs)
    assert_lse_close(lse, l_ref, f"decode query range {case} lse")


@pytest.mark.parametrize("mode,rb,with_lse", [("paged", 432, True), ("topk", 432, True), ("paged", 368, False)])
def test_decode_host_buffers_match_device_call(mode, rb, with_lse):
    # the host-buffer entry runs the same kernels on device copies of the
    # inputs: its output (and LSE) equal the device call's bit for bit
    if mode == "paged":
        w = workloads.decode_paged("host", 3, 128, (700, 64, 1500), rb, perm_pages=True, seed=12)
    else:
        w = workloads.decode_topk(batch=3, heads=64, context=4096, topk=300, max_pad=8, seed=13)
    gs = oracle_gs(w.kv_c)
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache, gst, err)
    if w.paged:
        kw = dict(page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV))
        hw = dict(page_table_host=w.page_table.contiguous().pin_memory(),
                  page_table_dev=torch.empty_like(w.page_table, device=DEV),
                  seq_lens_host=w.seq_lens.pin_memory(), seq_lens_dev=torch.empty_like(w.seq_lens, device=DEV))
    else:
        kw = dict(topk_indices=w.topk_indices.to(DEV))
        hw = dict(topk_host=w.topk_indices.contiguous().pin_memory(),
                  topk_dev=torch.empty_like(w.topk_indices, device=DEV))
    out_d, lse_d = mla.mla_nvfp4_decode(w.q.to(DEV), cache, gst, w.softmax_scale, error_word=err,
                                        return_lse=True, **kw)
    B, H, _ = w.q.shape
    q_host = w.q.contiguous().pin_memory()
    out_host = torch.empty((B, H, 512), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((B, H), dtype=torch.float32).pin_memory() if with_lse else None
    lse_dev = torch.empty((B, H), dtype=torch.float32, device=DEV) if with_lse else None
    mla.mla_nvfp4_decode_host(q_host, torch.empty_like(q_host, device=DEV), cache, gst, w.softmax_scale,
                              out_host, torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV),
                              lse_host=lse_host, lse_dev=lse_dev, error_word=err, **hw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_host, out_d.cpu())
    if with_lse:
        assert torch.equal(lse_host, lse_d.cpu())
