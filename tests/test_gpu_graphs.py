"""CUDA-graph capture and concurrent streams: the launch paths make no
attribute or allocation calls once a device has been used, so a prefill or
decode captured in a graph replays to the same bytes as a direct call, and
prefill calls running at the same time on two streams use different work
counters."""
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from tests.helpers import oracle_gs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def _prefill_buffers(w):
    T, H = w.total_tokens, w.heads
    return dict(out_codes=torch.empty((T, H * 64), dtype=torch.uint8, device=DEV),
                out_scales=torch.empty(mla.prefill_scale_bytes(T, H), dtype=torch.uint8, device=DEV),
                lse=torch.empty((H, T), dtype=torch.float32, device=DEV),
                error_word=torch.zeros(1, dtype=torch.int32, device=DEV))


def _prefill(w, gst, bufs):
    return mla.mla_nvfp4_prefill_fused_out(w.q, w.k, w.v, w.cu_seqlens, w.max_seqlen, w.softmax_scale, gst,
                                           return_lse=True, **bufs)


def _on_device(w):
    w.q, w.k, w.v, w.cu_seqlens = w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.cu_seqlens.to(DEV)
    return w


def test_prefill_graph_replay():
    w = _on_device(workloads.prefill("graph", seq_lens=(300, 1000, 37), heads=4, seed=31))
    gst = torch.tensor([oracle_gs(w.v.cpu())], device=DEV)
    direct = _prefill_buffers(w)
    ref = [t.clone() for t in _prefill(w, gst, direct)]
    bufs = _prefill_buffers(w)
    _prefill(w, gst, bufs)  # first use on this device happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _prefill(w, gst, bufs)
    for _ in range(3):
        for t in (bufs["out_codes"], bufs["out_scales"], bufs["lse"]):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(bufs["out_codes"], ref[0])
        assert torch.equal(bufs["out_scales"], ref[1])
        assert torch.equal(bufs["lse"], ref[2])
    assert int(bufs["error_word"].item()) == 0


def test_prefill_two_streams():
    wa = _on_device(workloads.prefill("sa", seq_lens=(2000, 300), heads=8, seed=32))
    wb = _on_device(workloads.prefill("sb", seq_lens=(129, 1500, 700), heads=8, seed=33))
    ga = torch.tensor([oracle_gs(wa.v.cpu())], device=DEV)
    gb = torch.tensor([oracle_gs(wb.v.cpu())], device=DEV)
    ref_a = [t.clone() for t in _prefill(wa, ga, _prefill_buffers(wa))]
    ref_b = [t.clone() for t in _prefill(wb, gb, _prefill_buffers(wb))]
    torch.cuda.synchronize()
    ba, bb = _prefill_buffers(wa), _prefill_buffers(wb)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    for _ in range(4):  # several rounds, so the two streams' launches overlap
        with torch.cuda.stream(s1):
            out_a = _prefill(wa, ga, ba)
        with torch.cuda.stream(s2):
            out_b = _prefill(wb, gb, bb)
    torch.cuda.synchronize()
    for got, ref in zip(out_a, ref_a):
        assert torch.equal(got, ref)
    for got, ref in zip(out_b, ref_b):
        assert torch.equal(got, ref)
    assert int(ba["error_word"].item()) == 0 and int(bb["error_word"].item()) == 0


@pytest.mark.parametrize("splits", [0, 1, 2])  # 0: planned (three kernels in the graph)
def test_decode_graph_replay(splits):
    w = workloads.decode_paged("graph", 3, 128, (700, 65, 1500), 432, perm_pages=True, seed=34)
    gs = torch.tensor([oracle_gs(w.kv_c)], device=DEV)
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache, gs)
    q, pt, sl = w.q.to(DEV), w.page_table.to(DEV), w.seq_lens.to(DEV)
    need = mla.mla_nvfp4_decode_workspace_size(3, 128, splits)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV) if need > 0 else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run(out, lse):
        mla.mla_nvfp4_decode(q, cache, gs, w.softmax_scale, page_table=pt, seq_lens=sl, out=out, lse=lse,
                             workspace=ws, num_splits=splits, error_word=err)

    ref_o = torch.empty((3, 128, 512), dtype=torch.bfloat16, device=DEV)
    ref_l = torch.empty((3, 128), dtype=torch.float32, device=DEV)
    run(ref_o, ref_l)
    out = torch.empty_like(ref_o)
    lse = torch.empty_like(ref_l)
    run(out, lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(out, lse)
    for _ in range(3):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert int(err.item()) == 0
