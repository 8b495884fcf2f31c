"""Decode parity at the full workload sizes, in the launch configuration the
benchmark times (default split count): sampled sequences against the float64
oracle, computed one sequence at a time, and the sampled tokens' cache
records against the oracle's encoder (RoPE and padding bit-exact, codes and
scales up to counted rounding-tie flips)."""
import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import attention, cache as ocache, nvfp4
from tests.helpers import assert_attention_close, assert_lse_close, f32, record_flips

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def _run(w):
    amax = float(w.kv_c.abs().max())  # exact: a maximum of bf16 magnitudes
    gs = nvfp4.global_scale(amax)
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, gst, err)
    kw = dict(page_table=w.page_table, seq_lens=w.seq_lens) if w.paged else dict(topk_indices=w.topk_indices)
    out, lse = mla.mla_nvfp4_decode(w.q, cache, gst, w.softmax_scale, error_word=err, return_lse=True, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse, cache, gs


def _tokens_of(w, b):
    """Written-token indices of sequence b, in key order."""
    if w.paged:
        lens = w.seq_lens.to("cpu", torch.int64)
        off = int(lens[:b].sum())
        return torch.arange(off, off + int(lens[b]))
    valid = (w.topk_indices >= 0).sum(1).to("cpu", torch.int64)
    off = int(valid[:b].sum())
    return torch.arange(off, off + int(valid[b]))


def _check(w, samples):
    out, lse, cache, gs = _run(w)
    for b in samples:
        tok = _tokens_of(w, b).to(DEV)
        rec = ocache.encode_records(f32(w.kv_c[tok]), f32(w.k_pe[tok]), gs, w.record_bytes)
        got = cache[w.slot_mapping[tok]].cpu().numpy()
        record_flips(got, f32(w.kv_c[tok]), f32(w.k_pe[tok]), gs, w.record_bytes, f"{w.name} seq {b} records")
        lat, rope = ocache.decode_records(rec, gs, w.record_bytes)
        k = np.concatenate([lat, rope], 1)
        o_ref, l_ref = attention.attend(f32(w.q[b]), k, lat, w.softmax_scale)
        o_abs, _ = attention.attend(f32(w.q[b]), k, np.abs(lat), w.softmax_scale)
        assert_attention_close(f32(out[b]), o_ref, f"{w.name} seq {b}", o_abs)
        assert_lse_close(f32(lse[b]), l_ref, f"{w.name} seq {b} lse")


def test_decode_dsv3_full_sampled():
    w = workloads.decode_dsv3(device=DEV)
    _check(w, [0, 37, 63])


def test_decode_mixed_full_sampled():
    w = workloads.decode_mixed(device=DEV)
    lens = w.seq_lens.cpu()
    _check(w, sorted({0, int(lens.argmax()), int(lens.argmin())}))


def test_decode_topk_full_sampled():
    w = workloads.decode_topk(device=DEV)
    _check(w, [0, 17, 31])
