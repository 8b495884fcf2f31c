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
    kw = dict(page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV), page_size=w.page_size) if w.paged \
        else dict(topk_indices=w.topk_indices.to(DEV))
    out, lse = mla.mla_nvfp4_decode(w.q.to(DEV), cache, gst, w.softmax_scale, num_splits=num_splits,
                                    error_word=err, return_lse=True, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return f32(out), f32(lse)


@pytest.mark.parametrize("page_size", [1, 16, 48, 100, 64])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_page_sizes(page_size, splits):
    # a key's page and offset within it are taken with the page size's
    # multiplier and shift: page sizes that are and are not powers of two,
    # sequences over several pages ending mid-page, permuted pages
    w = workloads.decode_paged("pages", 4, 32, (1, 257, 700, 1000), 432, perm_pages=True, seed=page_size,
                               page_size=page_size)
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, splits)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(out, o_ref, f"decode page size {page_size} splits={splits}", o_abs)
    assert_lse_close(lse, l_ref, f"decode page size {page_size} lse")


def run_oracle(w, gs):
    """(out, lse, softmax @ |v|) of the float64 oracle."""
    c = oracle_cache(w, gs)
    return attention.decode(f32(w.q), c, w.record_bytes, gs, w.softmax_scale, oracle_slots(w), with_abs=True)


@pytest.mark.parametrize("growth", [0.5, 2.0])
@pytest.mark.parametrize("splits", [0, 1])
def test_decode_growing_scores(growth, splits):
    # the latent of key tile j scaled by 1 + growth * j: a head's scores grow
    # from tile to tile by more than the lazy rescale's threshold, so its
    # reference is raised (with headroom) and O rescaled many times per
    # sequence, against both issuers' earlier P.V products
    lens = (1000, 700)
    w = workloads.decode_paged("growing", len(lens), 128, lens, 432, perm_pages=True, seed=int(4 * growth))
    tile = torch.cat([torch.arange(L) // 64 for L in lens]).float()
    w.kv_c = (w.kv_c.float() * (1.0 + growth * tile)[:, None]).to(torch.bfloat16)
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, splits)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(out, o_ref, f"decode growing scores x{growth} splits={splits}", o_abs)
    assert_lse_close(lse, l_ref, f"decode growing scores x{growth} lse")


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


@pytest.mark.parametrize("rb", [432, 368])
@pytest.mark.parametrize("splits", [0, 1])  # 1: output written by the decode kernel itself
def test_decode_topk_small(splits, rb):
    w = workloads.decode_topk(batch=3, heads=32, context=4096, topk=300, max_pad=8, seed=5, record_bytes=rb)
    w.topk_indices[2, :] = -1  # a row with nothing to attend to
    gs = oracle_gs(w.kv_c)
    out, lse = run_gpu(w, gs, splits)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))
    assert_attention_close(out, o_ref, f"decode top-k small rb={rb}", o_abs)
    assert_lse_close(lse, l_ref, f"decode top-k lse rb={rb}")


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


def _decode(w, gs, cache, err, **kw):
    pk = dict(page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV)) if w.paged else \
        dict(topk_indices=w.topk_indices.to(DEV))
    return mla.mla_nvfp4_decode(w.q.to(DEV), cache, torch.tensor([gs], device=DEV), w.softmax_scale,
                                error_word=err, return_lse=True, **pk, **kw)


def _written_cache(w, gs):
    cache = torch.zeros((w.num_slots, w.record_bytes), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache,
                              torch.tensor([gs], device=DEV), err)
    return cache, err


@pytest.mark.parametrize("rb", [432, 368])
def test_decode_planned_mixed_lengths(rb):
    # the length-aware plan (num_splits = 0 with a workspace): empty
    # sequences, one-key sequences, tile edges and long sequences in one
    # batch, so that the plan cuts some sequences into several chunks (merged)
    # and leaves others whole (written directly)
    lens = (0, 1, 64, 65, 4000, 130, 0, 2500, 3, 1999, 64 * 37, 700)
    w = workloads.decode_paged("planned", len(lens), 128, lens, rb, perm_pages=True, outlier_frac=0.01,
                               outlier_mult=20.0, seed=31)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    out, lse = _decode(w, gs, cache, err, num_splits=0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    out, lse = f32(out), f32(lse)
    assert np.all(out[[0, 6]] == 0) and np.all(np.isneginf(lse[[0, 6]]))
    assert_attention_close(out, o_ref, f"decode planned rb={rb}", o_abs)
    assert_lse_close(lse, l_ref, "decode planned lse")


def test_decode_planned_workspace_room():
    # a planned call given only room for its work list (no partial rows) cuts
    # no sequence: one chunk each, written directly, the same bytes as one
    # uniform split; given the full workspace it may split and still agrees
    lens = (3000, 10, 5000, 64)
    w = workloads.decode_paged("room", len(lens), 64, lens, 432, perm_pages=True, seed=32)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    # 64 KB: the header, the item list (batch + one per SM pair) and the chunk
    # table fit, one chunk row (64 heads x 2052 bytes) does not
    tables_only = torch.empty(65536, dtype=torch.uint8, device=DEV)
    o_small, l_small = _decode(w, gs, cache, err, num_splits=0, workspace=tables_only)
    o_one, l_one = _decode(w, gs, cache, err, num_splits=1)  # no workspace at all
    o_full, l_full = _decode(w, gs, cache, err, num_splits=0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o_small, o_one) and torch.equal(l_small, l_one)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(f32(o_full), o_ref, "decode planned, full workspace", o_abs)
    assert_lse_close(f32(l_full), l_ref, "decode planned lse, full workspace")


def test_decode_uniform_splits_need_their_workspace():
    w = workloads.decode_paged("ws", 2, 16, (300, 77), 432, perm_pages=True, seed=33)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    short = torch.empty(mla.mla_nvfp4_decode_workspace_size(2, 16, 3) - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(mla.MLAError) as ei:
        _decode(w, gs, cache, err, num_splits=3, workspace=short)
    assert ei.value.status == 5  # MLA_ERR_WORKSPACE


def test_decode_one_split_many_rows_without_workspace():
    # one split, batch x heads above the no-allocation scratch's row count:
    # no workspace is needed or checked
    lens = (5,) * 130
    w = workloads.decode_paged("rows", len(lens), 128, lens, 432, perm_pages=True, seed=34)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    out, lse = _decode(w, gs, cache, err, num_splits=1)
    torch.cuda.synchronize()
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(f32(out), o_ref, "decode 130 x 128 heads, one split", o_abs)
    assert_lse_close(f32(lse), l_ref, "decode 130 x 128 heads lse")


@pytest.mark.parametrize("peak,flagged", [(6.0e4, False), (7.0e4, True)])
def test_decode_rope_range(peak, flagged):
    # bf16 k_pe enters the tensor cores as f16: inside the f16 range it is
    # exact (the result matches the oracle); beyond it saturates and the
    # call flags MLA_DEVERR_RANGE
    w = workloads.decode_paged("rope", 2, 32, (100, 70), 432, perm_pages=True, seed=35)
    w.k_pe[7, 3] = peak
    w.k_pe[120, 0] = -peak
    w.q[:, :, 512:] *= 1e-4  # keeps the scores of those keys moderate
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    out, lse = _decode(w, gs, cache, err, num_splits=1)
    torch.cuda.synchronize()
    assert bool(int(err.item()) & mla.DEVERR_RANGE) == flagged
    if not flagged:
        o_ref, l_ref, o_abs = run_oracle(w, gs)
        assert_attention_close(f32(out), o_ref, "decode rope near the f16 limit", o_abs)
        assert_lse_close(f32(lse), l_ref, "decode rope near the f16 limit lse")
    else:
        assert torch.isfinite(out.float()).all()


def _plan_choice(tiles, pairs, max_items, max_rows, overhead=2.0):
    """The chunk size the plan documents: among C = ceil(tmax / k), k = 1..32,
    the first minimum of max(ceil(full / P) * (C + o), (tiles + o * items) /
    P + (mean last chunk + o) / 2) over the candidates whose items and
    partial rows fit."""
    tmax, tot = max(tiles), sum(tiles)
    best, best_est = None, math.inf
    for k in range(1, 33):
        C = max(1, -(-tmax // k))
        nb = [max(1, -(-t // C)) for t in tiles]
        n, full = sum(nb), sum(t // C for t in tiles)
        rows = sum(x for x in nb if x > 1)
        last = sum(1 for t in tiles if t == 0 or t % C)
        waves = math.ceil(full / pairs) * (C + overhead)
        avg = (tot + overhead * n) / pairs + (0.5 * ((tot - full * C) / last + overhead) if last else 0.0)
        est = max(waves, avg) if (n <= max_items and rows <= max_rows) else math.inf
        if est < best_est * (1 - 1e-6):  # float32 on the device: a near tie keeps the larger C
            best, best_est = C, est
    return best


def _random_lens(seed, batch, max_len):
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(0, max_len, batch))


@pytest.mark.parametrize("lens", [(4096,) * 64, (0, 1, 64, 65, 4000, 130, 0, 2500, 3, 1999, 2368, 700),
                                  (32768, 1024, 1500, 20000, 5000, 8000, 1100),
                                  _random_lens(51, 90, 3000), _random_lens(52, 40, 9000)])
def test_decode_plan_covers_every_chunk_once(lens):
    w = workloads.decode_paged("plan", len(lens), 16, lens, 432, perm_pages=True, seed=36)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    B = len(lens)
    ws = torch.zeros(mla.mla_nvfp4_decode_workspace_size(B, 16, 0), dtype=torch.uint8, device=DEV)
    _decode(w, gs, cache, err, num_splits=0, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    raw = ws.cpu().numpy()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs, max_items = sms // 2, B + sms // 2
    n_items, C = (int(x) for x in raw[:8].view(np.int32))
    items = raw[256:256 + 8 * n_items].view(np.int32).reshape(-1, 2)
    seq_off = (256 + 8 * max_items + 255) // 256 * 256
    seqs = raw[seq_off:seq_off + 8 * B].view(np.int32).reshape(-1, 2)
    tiles = [-(-L // 64) for L in lens]
    assert C == _plan_choice(tiles, pairs, max_items, max_items)
    # the host form of the plan makes the same choice between one chunk per
    # sequence and cut sequences
    one = mla.mla_nvfp4_decode_plan_splits(torch.tensor(lens, dtype=torch.int32), 16, ws.numel())
    assert one == (1 if C >= max(1, max(tiles)) else 0)
    nb = [max(1, -(-t // C)) for t in tiles]
    # every (sequence, chunk) exactly once
    assert sorted(map(tuple, items.tolist())) == sorted((b, c) for b in range(B) for c in range(nb[b]))
    # the chunk table: one-chunk sequences are direct, the others own
    # consecutive, disjoint partial rows
    assert seqs[:, 1].tolist() == nb
    rows = [(int(seqs[b, 0]), nb[b]) for b in range(B) if nb[b] > 1]
    assert all(seqs[b, 0] == -1 for b in range(B) if nb[b] == 1)
    used = sorted(r for base, n in rows for r in range(base, base + n))
    assert used == list(range(len(used)))
    # longest first: full chunks, then the last chunks by non-increasing
    # size bucket (64 buckets over [0, C))
    size = [min(C, tiles[b] - c * C) for b, c in items.tolist()]
    n_full = sum(t // C for t in tiles)
    assert all(s_ == C for s_ in size[:n_full])
    buckets = [63 - s_ * 64 // C for s_ in size[n_full:]]
    assert buckets == sorted(buckets)


@pytest.mark.parametrize("lens,one", [((640,) * 48, 1), ((700, 64, 1500), 0), ((0,) * 49 + (64,), 1)])
def test_decode_host_plans_from_host_lengths(lens, one):
    # mla_nvfp4_decode_host reads the lengths on the host: where the plan
    # keeps one chunk per sequence it launches the one-split decode (the plan
    # kernel never writes the workspace), otherwise the device plans; either
    # way the output is the planned device call's, bit for bit
    B, H = len(lens), 16
    w = workloads.decode_paged("hostplan", B, H, lens, 432, perm_pages=True, seed=44)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = [-(-L // 64) for L in lens]
    ws_bytes = mla.mla_nvfp4_decode_workspace_size(B, H, 0)
    assert (_plan_choice(tiles, sms // 2, B + sms // 2, B + sms // 2) == max(1, max(tiles))) == bool(one)
    assert mla.mla_nvfp4_decode_plan_splits(w.seq_lens, H, ws_bytes) == one
    out_d, lse_d = _decode(w, gs, cache, err, num_splits=0,
                           workspace=torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV))
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device=DEV)
    q_host = w.q.contiguous().pin_memory()
    out_host = torch.empty((B, H, 512), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((B, H), dtype=torch.float32).pin_memory()
    mla.mla_nvfp4_decode_host(q_host, torch.empty_like(q_host, device=DEV), cache, torch.tensor([gs], device=DEV),
                              w.softmax_scale, out_host, torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV),
                              page_table_host=w.page_table.contiguous().pin_memory(),
                              page_table_dev=torch.empty_like(w.page_table, device=DEV),
                              seq_lens_host=w.seq_lens.pin_memory(),
                              seq_lens_dev=torch.empty_like(w.seq_lens, device=DEV),
                              lse_host=lse_host, lse_dev=torch.empty((B, H), dtype=torch.float32, device=DEV),
                              workspace=ws, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    header_untouched = bool((ws[:8] == 0xFF).all())
    assert header_untouched == bool(one)
    assert torch.equal(out_host, out_d.cpu()) and torch.equal(lse_host, lse_d.cpu())


@pytest.mark.parametrize("batch,heads,max_len,seed", [(300, 16, 600, 41), (40, 160, 3000, 42)])
def test_decode_planned_many_items_per_cta(batch, heads, max_len, seed):
    # more work items than resident CTA pairs (several waves, items taken
    # longest first), and more than 128 heads (two head groups per item)
    rng = np.random.default_rng(seed)
    lens = tuple(int(x) for x in rng.integers(0, max_len, batch))
    w = workloads.decode_paged("items", batch, heads, lens, 432, perm_pages=True, seed=seed)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    out, lse = _decode(w, gs, cache, err, num_splits=0)
    again, lse2 = _decode(w, gs, cache, err, num_splits=0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the schedule differs from call to call; the bytes do not
    assert torch.equal(out, again) and torch.equal(lse, lse2)
    o_ref, l_ref, o_abs = run_oracle(w, gs)
    assert_attention_close(f32(out), o_ref, f"decode planned B{batch} H{heads}", o_abs)
    assert_lse_close(f32(lse), l_ref, f"decode planned B{batch} H{heads} lse")


def test_decode_planned_is_stream_ordered():
    # the planned decode is three kernels (plan, decode, merge); work queued
    # after the call on the same stream sees the finished output and LSE
    w = workloads.decode_paged("order", 16, 128, (4096,) * 15 + (9000,), 432, perm_pages=True, seed=43)
    gs = oracle_gs(w.kv_c)
    cache, err = _written_cache(w, gs)
    torch.cuda.synchronize()
    out = torch.full((16, 128, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((16, 128), float("nan"), dtype=torch.float32, device=DEV)
    mla.mla_nvfp4_decode(w.q.to(DEV), cache, torch.tensor([gs], device=DEV), w.softmax_scale,
                         page_table=w.page_table.to(DEV), seq_lens=w.seq_lens.to(DEV), out=out, lse=lse,
                         num_splits=0, error_word=err)
    out_copy, lse_copy = out.clone(), lse.clone()  # same stream, no synchronisation in between
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not torch.isnan(out_copy.float()).any() and not torch.isnan(lse_copy).any()
    assert torch.equal(out_copy, out) and torch.equal(lse_copy, lse)
