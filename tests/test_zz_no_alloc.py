"""The decode entry point without a caller workspace (built-in scratch).

Two calls in a row through the C ABI, on different workloads, must give the
bytes of mla_nvfp4_decode (caller workspace of the scratch's size, so both
make the same plan) at the same split setting; a later call must not change
the device's free memory; a call larger than the scratch must be refused
with a message; one-split calls need no scratch, whatever their size.  This file is collected last so it
also runs after every other GPU test in the same process, and it sets up its
own inputs so it passes alone in a fresh process."""
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from tests.helpers import oracle_gs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"
MLA_ERR_WORKSPACE = 5
STATIC_ROWS = 16384


def _prepare(w):
    gs = oracle_gs(w.kv_c)
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    gst = torch.tensor([gs], device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache, gst, err)
    kw = dict(page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV)) if w.paged else \
        dict(topk_indices=w.topk_indices.to(DEV))
    return dict(q=w.q.to(DEV), cache=cache, gst=gst, err=err, scale=w.softmax_scale, kw=kw)


def _outputs(p):
    B, H, _ = p["q"].shape
    return (torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV),
            torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV))


def _noalloc(p, splits):
    out, lse = _outputs(p)
    mla.mla_nvfp4_decode_noalloc(p["q"], p["cache"], p["gst"], p["scale"], out, lse=lse,
                                 num_splits=splits, error_word=p["err"], **p["kw"])
    return out, lse


STATIC_BYTES = 33619968


def _with_workspace(p, splits):
    ws = torch.empty(STATIC_BYTES, dtype=torch.uint8, device=DEV) if splits != 1 else None
    return mla.mla_nvfp4_decode(p["q"], p["cache"], p["gst"], p["scale"], num_splits=splits,
                                error_word=p["err"], return_lse=True, workspace=ws, **p["kw"])


def _same(got, ref, what):
    (o, l), (o_ref, l_ref) = got, ref
    assert torch.equal(o, o_ref), f"{what}: output differs from mla_nvfp4_decode"
    assert torch.equal(l, l_ref), f"{what}: lse differs from mla_nvfp4_decode"


CASES = [
    # (workload, num_splits)
    (lambda: workloads.decode_paged("noalloc_a", 3, 128, (700, 65, 0), 432, perm_pages=True, seed=11), 0),
    (lambda: workloads.decode_topk(batch=2, heads=64, context=4096, topk=500, max_pad=8, seed=12), 5),
]


def test_two_calls_in_a_row_match_decode():
    preps = [(_prepare(make()), splits) for make, splits in CASES]
    torch.cuda.synchronize()
    # the two no-alloc calls back to back on one stream, then the references
    got = [_noalloc(p, s) for p, s in preps]
    ref = [_with_workspace(p, s) for p, s in preps]
    torch.cuda.synchronize()
    for i, ((p, s), g, r) in enumerate(zip(preps, got, ref)):
        assert int(p["err"].item()) == 0
        _same(g, r, f"no-alloc decode call {i} (splits={s})")


def test_later_call_allocates_nothing():
    p = _prepare(CASES[0][0]())
    _noalloc(p, 0)  # the first call on the device may do the set-up
    torch.cuda.synchronize()
    out, lse = _outputs(p)
    free0 = torch.cuda.mem_get_info()[0]
    torch_bytes0 = torch.cuda.memory_allocated()
    mla.mla_nvfp4_decode_noalloc(p["q"], p["cache"], p["gst"], p["scale"], out, lse=lse,
                                 error_word=p["err"], **p["kw"])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == torch_bytes0
    _same((out, lse), _with_workspace(p, 0), "no-alloc decode, later call")


def test_oversize_call_refused():
    w = workloads.decode_paged("noalloc_big", 2, 128, (64, 64), 432, perm_pages=True, seed=13)
    p = _prepare(w)
    out, lse = _outputs(p)
    splits = STATIC_ROWS // (2 * 128) + 1  # one split more than the scratch holds
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_nvfp4_decode_noalloc(p["q"], p["cache"], p["gst"], p["scale"], out, lse=lse,
                                     num_splits=splits, error_word=p["err"], **p["kw"])
    assert ei.value.status == MLA_ERR_WORKSPACE
    assert str(STATIC_ROWS) in str(ei.value) and "rows" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()  # nothing was launched
    # the largest call that fits is accepted
    mla.mla_nvfp4_decode_noalloc(p["q"], p["cache"], p["gst"], p["scale"], out, lse=lse,
                                 num_splits=splits - 1, error_word=p["err"], **p["kw"])
    ref = _with_workspace(p, splits - 1)
    torch.cuda.synchronize()
    _same((out, lse), ref, "no-alloc decode at the scratch limit")


def test_one_split_beyond_scratch_rows():
    # one split writes out directly and uses no scratch: batch x heads above
    # the scratch's row count is accepted
    lens = (3,) * 130
    p = _prepare(workloads.decode_paged("noalloc_rows", len(lens), 128, lens, 432, perm_pages=True, seed=14))
    got = _noalloc(p, 1)
    ref = _with_workspace(p, 1)
    torch.cuda.synchronize()
    assert int(p["err"].item()) == 0
    _same(got, ref, "no-alloc decode, one split, 16640 rows")
