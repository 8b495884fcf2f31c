"""Seeded synthetic inputs for the MLA NVFP4 kernels.

This module only draws random tensors and index structures (shapes, value
distributions, page tables, top-k index sets, sequence-length mixes).  It
holds none of the method's arithmetic: no quantisation, no attention, no
scale computation.  The tests feed its output to both the CUDA library and
the float64 oracle; the benchmark feeds it to the library.

Named workloads (all seeded, default seed 0):

  decode_tiny      batch 2, 16 heads, sequence lengths 64 and 100, pages in
                   order, 432-byte records, everything ~N(0,1).
  decode_dsv3      batch 64, 128 heads, every sequence 4096 tokens, a random
                   permutation of 4096 pages of 64 tokens, 432-byte records,
                   latent ~N(0,1) with 1% of elements multiplied by 20.
  decode_mixed     batch 128, 128 heads, lengths floor(exp(U(ln 1024,
                   ln 32768))), permuted pages, 368-byte (fp8 RoPE) records.
  decode_topk      batch 32, 128 heads, 65536-token context per sequence in
                   432-byte records; each query picks 2048 distinct positions
                   uniformly without replacement, the last r in [1, 8] of them
                   replaced by -1; the global slot of (b, t) is b * 65536 + t.
  prefill_8x4096   8 sequences x 4096 tokens, 128 heads, q/k head dim 192,
                   v head dim 128, all ~N(0,1) bf16.
  prefill_context  new tokens after a cached context: per sequence a chunk
                   of context keys / values (k_ctx [Tc, H, 192], v_ctx
                   [Tc, H, 128], ~N(0,1) bf16, rows cu_ctx[s]..cu_ctx[s+1])
                   besides the new tokens' q / k / v.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

PAGE = 64
D_LATENT = 512
D_ROPE = 64
D_QK = 576
D_V = 512


@dataclass
class DecodeWorkload:
    name: str
    batch: int
    heads: int
    record_bytes: int
    q: torch.Tensor  # [B, H, 576] bf16
    kv_c: torch.Tensor  # [T, 512] bf16, one row per written token
    k_pe: torch.Tensor  # [T, 64] bf16
    slot_mapping: torch.Tensor  # [T] int64
    num_slots: int
    seq_lens: Optional[torch.Tensor] = None  # [B] int32 (paged mode)
    page_table: Optional[torch.Tensor] = None  # [B, max_pages] int32 (paged mode)
    topk_indices: Optional[torch.Tensor] = None  # [B, topk] int32 (top-k mode)
    softmax_scale: float = 1.0 / math.sqrt(192.0)
    page_size: int = PAGE  # tokens per page (paged mode)
    meta: dict = field(default_factory=dict)

    @property
    def paged(self) -> bool:
        return self.page_table is not None

    def tokens_attended(self) -> int:
        if self.paged:
            return int(self.seq_lens.to(torch.int64).sum())
        return int((self.topk_indices >= 0).sum())


@dataclass
class PrefillWorkload:
    name: str
    heads: int
    q: torch.Tensor  # [T, H, 192] bf16
    k: torch.Tensor  # [T, H, 192] bf16
    v: torch.Tensor  # [T, H, 128] bf16
    cu_seqlens: torch.Tensor  # [S+1] int32
    max_seqlen: int
    softmax_scale: float = 1.0 / math.sqrt(192.0)
    k_ctx: Optional[torch.Tensor] = None  # [Tc, H, 192] bf16 (context chunk keys)
    v_ctx: Optional[torch.Tensor] = None  # [Tc, H, 128] bf16
    cu_ctx: Optional[torch.Tensor] = None  # [S+1] int32

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def _paged_layout(seq_lens, perm_pages: bool, g, device, page=PAGE):
    """Page table and slot mapping for sequences laid out page by page."""
    pages_per_seq = [(int(L) + page - 1) // page for L in seq_lens]
    n_pages = sum(pages_per_seq)
    if perm_pages:
        ids = torch.randperm(n_pages, generator=g, device=device).to("cpu")
    else:
        ids = torch.arange(n_pages)
    max_pages = max(pages_per_seq)
    table = torch.zeros((len(seq_lens), max_pages), dtype=torch.int32)
    slots = []
    pos = 0
    for b, (L, npg) in enumerate(zip(seq_lens, pages_per_seq)):
        table[b, :npg] = ids[pos:pos + npg].to(torch.int32)
        pos += npg
        t = torch.arange(int(L))
        slots.append(table[b, t // page].to(torch.int64) * page + t % page)
    return table, torch.cat(slots), n_pages * page


def decode_paged(name, batch, heads, seq_lens, record_bytes, perm_pages, outlier_frac=0.0,
                 outlier_mult=1.0, seed=0, device="cpu", page_size=PAGE) -> DecodeWorkload:
    g = _gen(seed, device)
    seq_lens = [int(x) for x in seq_lens]
    table, slots, num_slots = _paged_layout(seq_lens, perm_pages, g, device, page_size)
    T = int(sum(seq_lens))
    q = _randn_bf16((batch, heads, D_QK), g, device)
    kv = torch.randn((T, D_LATENT), generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        mask = torch.rand((T, D_LATENT), generator=g, device=device) < outlier_frac
        kv = torch.where(mask, kv * outlier_mult, kv)
    kv_c = kv.to(torch.bfloat16)
    k_pe = _randn_bf16((T, D_ROPE), g, device)
    return DecodeWorkload(
        name=name, batch=batch, heads=heads, record_bytes=record_bytes, q=q, kv_c=kv_c,
        k_pe=k_pe, slot_mapping=slots.to(device), num_slots=num_slots,
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
        page_table=table.to(device), page_size=page_size)


def decode_tiny(seed=0, device="cpu", heads=16, seq_lens=(64, 100), record_bytes=432) -> DecodeWorkload:
    return decode_paged("decode_tiny", len(seq_lens), heads, seq_lens, record_bytes,
                        perm_pages=False, seed=seed, device=device)


def decode_dsv3(seed=0, device="cpu", batch=64, heads=128, seq_len=4096) -> DecodeWorkload:
    return decode_paged("decode_dsv3", batch, heads, [seq_len] * batch, 432, perm_pages=True,
                        outlier_frac=0.01, outlier_mult=20.0, seed=seed, device=device)


def mixed_lengths(batch, lo, hi, g, device) -> list:
    u = torch.rand(batch, generator=g, device=device, dtype=torch.float64).to("cpu")
    return [int(math.floor(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
            for x in u]


def decode_mixed(seed=0, device="cpu", batch=128, heads=128, lo=1024, hi=32768) -> DecodeWorkload:
    g = _gen(seed + 1000, device)
    lens = mixed_lengths(batch, lo, hi, g, device)
    w = decode_paged("decode_mixed", batch, heads, lens, 368, perm_pages=True, seed=seed,
                     device=device)
    return w


def decode_topk(seed=0, device="cpu", batch=32, heads=128, context=65536, topk=2048,
                max_pad=8, record_bytes=432) -> DecodeWorkload:
    g = _gen(seed, device)
    idx = torch.empty((batch, topk), dtype=torch.int64)
    for b in range(batch):
        t = torch.randperm(context, generator=g, device=device)[:topk].to("cpu")
        idx[b] = b * context + t
    pads = torch.randint(1, max_pad + 1, (batch,), generator=g, device=device).to("cpu")
    for b in range(batch):
        idx[b, topk - int(pads[b]):] = -1
    ref = idx[idx >= 0]  # referenced slots; only these rows are written
    T = int(ref.numel())
    q = _randn_bf16((batch, heads, D_QK), g, device)
    kv_c = _randn_bf16((T, D_LATENT), g, device)
    k_pe = _randn_bf16((T, D_ROPE), g, device)
    return DecodeWorkload(
        name="decode_topk", batch=batch, heads=heads, record_bytes=record_bytes, q=q, kv_c=kv_c,
        k_pe=k_pe, slot_mapping=ref.to(device), num_slots=batch * context,
        topk_indices=idx.to(torch.int32).to(device), meta={"context": context, "topk": topk})


def prefill(name="prefill_8x4096", seq_lens=(4096,) * 8, heads=128, d_qk=192, d_v=128, seed=0,
            device="cpu") -> PrefillWorkload:
    g = _gen(seed, device)
    T = int(sum(seq_lens))
    q = _randn_bf16((T, heads, d_qk), g, device)
    k = _randn_bf16((T, heads, d_qk), g, device)
    v = _randn_bf16((T, heads, d_v), g, device)
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int32), 0)
    return PrefillWorkload(name=name, heads=heads, q=q, k=k, v=v, cu_seqlens=cu.to(device),
                           max_seqlen=int(max(seq_lens)))


def prefill_8x4096(seed=0, device="cpu") -> PrefillWorkload:
    return prefill(seed=seed, device=device)


def prefill_context(seq_lens, ctx_lens, heads=16, seed=0, device="cpu") -> PrefillWorkload:
    w = prefill("prefill_context", seq_lens=seq_lens, heads=heads, seed=seed, device=device)
    g = _gen(seed + 7, device)
    Tc = int(sum(ctx_lens))
    w.k_ctx = _randn_bf16((Tc, heads, 192), g, device)
    w.v_ctx = _randn_bf16((Tc, heads, 128), g, device)
    cc = torch.zeros(len(ctx_lens) + 1, dtype=torch.int32)
    cc[1:] = torch.cumsum(torch.tensor(ctx_lens, dtype=torch.int32), 0)
    w.cu_ctx = cc.to(device)
    return w
