"""Shared test helpers: running the oracle on workload tensors and the
comparison rules (tolerances from the method's stated acceptance bar)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention, cache as ocache, nvfp4, swizzle

# Dequantised attention outputs: max-abs error and mean relative (L1) error
# against the float64 oracle.
MAX_ABS = 2e-2
MEAN_REL = 5e-3
# Rounding-tie budget: mismatching codes (a mismatching scale byte counts as
# 17: itself and its block's 16 codes) per code compared.
TIE_BUDGET = 1e-4
# The kernels evaluate the NVFP4 quotients in float32 as products with
# reciprocals (1/(6 gs), then amax16 times it; 1/S, then x times it): three
# roundings of 2^-24 relative each, so their pre-rounding value lies within
# 3 * 2^-24 < 2^-22 (relative) of the exact quotient, and a decision can
# differ from the exact one only where the exact quotient lies that close to
# a grid midpoint.
NEAR_TIE = 2.0 ** -22


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def oracle_gs(x: torch.Tensor) -> np.float32:
    return nvfp4.global_scale(np.abs(f32(x)).max())


def oracle_cache(w, gs) -> np.ndarray:
    c = np.zeros((w.num_slots, w.record_bytes), dtype=np.uint8)
    ocache.write_cache(c, f32(w.kv_c), f32(w.k_pe), w.slot_mapping.cpu().numpy(), gs, w.record_bytes)
    return c


def oracle_slots(w):
    if w.paged:
        return attention.decode_slots_paged(w.page_table.cpu().numpy(), w.seq_lens.cpu().numpy(), w.page_size)
    return attention.decode_slots_topk(w.topk_indices.cpu().numpy())


def bf16_half_ulp(x) -> np.ndarray:
    """Half a bf16 unit in the last place at |x|: the largest change that
    rounding x to bf16 (8 significant bits) can make."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8)


# Decode rounds the probabilities to f16 for the tensor-core P.V product
# (11 significant bits): each output element may move by up to 2^-11 times
# sum_j p_j |v_j| / sum_j p_j, plus ~1e-7 relative from fp32 accumulation.
P16_ROUNDING = 2.0 ** -11


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str, o_abs=None):
    """Decode outputs (bf16) against the float64 oracle.  The max-abs bar
    applies to the error beyond the two roundings the output and the tensor
    cores force: half a bf16 ulp at the element's magnitude (the output type;
    at |o| ~ 80, reached with x20 latent outliers, that alone is 0.25) and,
    when o_abs = softmax @ |v| is given, the f16 probability rounding
    P16_ROUNDING * o_abs.  The mean relative L1 error is taken as is."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    excess = err - np.maximum(bf16_half_ulp(ref), bf16_half_ulp(got))
    if o_abs is not None:
        excess = excess - P16_ROUNDING * np.asarray(o_abs, dtype=np.float64)
    max_abs = float(excess.max()) if err.size else 0.0
    raw = float(err.max()) if err.size else 0.0
    allowance = float((err - excess).max()) if err.size else 0.0
    denom = float(np.abs(ref).sum())
    mean_rel = float(err.sum() / denom) if denom > 0 else float(err.sum())
    print(f"[attention] {what}: raw max-abs {raw:.3e}, largest rounding allowance {allowance:.3e}, "
          f"max-abs beyond it {max_abs:.3e} (bar {MAX_ABS}), mean rel {mean_rel:.3e} (bar {MEAN_REL})")
    assert max_abs <= MAX_ABS and mean_rel <= MEAN_REL, \
        f"{what}: max_abs beyond output rounding={max_abs:.3e} (<= {MAX_ABS}), " \
        f"mean_rel={mean_rel:.3e} (<= {MEAN_REL})"
    return max_abs, mean_rel


# LSE: the partition function to within the mean relative error bar of the
# outputs, ln(1 + 5e-3).
LSE_TOL = float(np.log1p(MEAN_REL))


def assert_lse_close(got, ref, what: str, tol=LSE_TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf), f"{what}: -inf pattern differs"
    d = np.abs(got[~inf] - ref[~inf])
    assert d.size == 0 or d.max() <= tol, f"{what}: lse max diff {d.max():.3e}"


def code_boundary_distance(q: np.ndarray) -> np.ndarray:
    """Distance of |q| (value / block scale) to the nearest e2m1 rounding
    midpoint, in code units."""
    mids = (nvfp4.E2M1_MAGNITUDES[:-1] + nvfp4.E2M1_MAGNITUDES[1:]) / 2
    return np.min(np.abs(np.abs(q)[..., None] - mids), axis=-1)


# Bound on the kernel's output error from rounding the probabilities to bf16
# for the tensor-core P.V product: |dO| <= 2^-9 * sum_j p_j |v_j| / sum_j p_j
# per element (fp32 accumulation adds ~1e-6 relative); 2^-8 leaves a 2x margin.
P_ROUNDING = 2.0 ** -8


def check_fused_output(codes_gpu, scales_gpu, o_ref, o_abs, gs, what="fused output"):
    """End-to-end NVFP4 output check where the kernel quantises its own fp32
    attention output.  Each output element may differ from the exact one by
    err = P_ROUNDING * o_abs (+1e-6 relative).  A scale byte may differ from
    the oracle's quantisation of the exact output only where the block's raw
    scale lies within the error of an e4m3 rounding midpoint, and a code only
    where value/scale lies within err/scale of an e2m1 midpoint (or its
    block's scale differs); a code of magnitude 0 may differ in its sign bit
    only (a value within err of zero).  Returns the counts (check_fused_blocks)."""
    M, N = o_ref.shape
    return check_fused_blocks(codes_gpu, swizzle.unswizzle_scales(scales_gpu, M, N // 16), o_ref, o_abs, gs,
                              what)


def check_fused_blocks(codes_gpu, sf_gpu, o_ref, o_abs, gs, what="fused output"):
    """check_fused_output with the kernel's scale bytes already in row-major
    [M, N/16] order (used for sampled rows of a large output).  Returns a
    dict: scale bytes that differ, codes that differ in a block whose scale
    agrees (magnitude flips at a boundary), codes that differ only in the
    sign of a zero, and the number of codes compared; prints it."""
    M, N = o_ref.shape
    K = N // 16
    x = o_ref.astype(np.float32)
    err = (P_ROUNDING * np.asarray(o_abs, dtype=np.float64) + 1e-6 * np.abs(o_ref)).reshape(M, N) + 1e-30
    codes_ref, sb_ref = nvfp4.quantize_blocks(x, gs)
    sf_gpu = np.asarray(sf_gpu).reshape(M, K)
    codes_g = nvfp4.unpack_e2m1(codes_gpu.reshape(M, N // 2))
    sb_ref = sb_ref.reshape(M, K)
    # scales
    amax = np.abs(x.reshape(M, K, 16)).max(-1).astype(np.float64)
    d_amax = err.reshape(M, K, 16).max(-1)
    s_raw = amax / 6.0 / float(gs)
    ds = d_amax / 6.0 / float(gs)
    grid = nvfp4.e4m3_decode(np.arange(127))
    mids = (grid[:-1] + grid[1:]) / 2
    near_s = np.min(np.abs(s_raw[..., None] - mids), axis=-1) <= ds
    bad_s = (sf_gpu != sb_ref)
    assert not np.any(bad_s & ~near_s), f"{what}: {int((bad_s & ~near_s).sum())} scale bytes differ away from a tie"
    # codes (only in blocks whose scale agrees)
    S = (nvfp4.e4m3_decode(sb_ref) * float(gs)).repeat(16, axis=1)
    safe = np.where(S > 0, S, 1.0)
    q = np.where(S > 0, x.astype(np.float64) / safe, 0)
    near_c = code_boundary_distance(q) <= err / safe
    same_scale = (~bad_s).repeat(16, axis=1)
    diff = (codes_g != codes_ref) & same_scale
    # a zero magnitude on both sides may differ in its sign bit, only for a
    # value within its error of zero
    zero_sign = diff & ((codes_g & 7) == 0) & ((codes_ref & 7) == 0)
    assert np.all(np.abs(x[zero_sign]) <= err[zero_sign]), f"{what}: sign of a zero code differs away from zero"
    flips = diff & ~zero_sign
    bad = flips & ~near_c
    assert not np.any(bad), f"{what}: {int(bad.sum())} codes differ away from a rounding boundary"
    counts = {"scale_flips": int(bad_s.sum()), "code_flips": int(flips.sum()), "zero_sign": int(zero_sign.sum()),
              "codes": int(codes_g.size)}
    rate = (17 * counts["scale_flips"] + counts["code_flips"] + counts["zero_sign"]) / max(1, counts["codes"])
    print(f"[fused] {what}: {counts} -> mismatch rate {rate:.2e}")
    counts["rate"] = rate
    return counts


def _near_midpoint(v, mids, rel):
    """|v - nearest midpoint| <= rel * v (v >= 0, float64)."""
    return np.min(np.abs(v[..., None] - mids), axis=-1) <= rel * v


def quant_flips(x, gs, codes_gpu, sb_gpu, what: str, budget: float = TIE_BUDGET):
    """The kernel's NVFP4 quantisation of float32 x ([..., 16*nb]; unpacked
    codes [..., 16*nb], scale bytes [..., nb]) against the oracle's exact
    definition.  A scale byte may differ only by one code and only where
    amax16/6/gs lies within NEAR_TIE of an e4m3 midpoint; a code only by one
    magnitude step, with the same sign, where x/S lies within NEAR_TIE of an
    e2m1 midpoint (codes of a block whose scale differs are compared with the
    definition under the kernel's scale).  Asserts all of that and that the
    mismatches (a scale byte counting 17) are at most `budget` of the codes;
    returns (mismatches, codes compared) and prints them."""
    x = np.asarray(x, dtype=np.float32)
    nb = x.shape[-1] // 16
    blocks = x.reshape(-1, nb, 16)
    codes_gpu = np.asarray(codes_gpu, dtype=np.uint8).reshape(blocks.shape)
    sb_gpu = np.asarray(sb_gpu, dtype=np.uint8).reshape(blocks.shape[:-1])
    codes_ref, sb_ref = nvfp4.quantize_blocks(blocks.reshape(-1, nb * 16), gs)
    codes_ref = codes_ref.reshape(blocks.shape)
    sb_ref = sb_ref.reshape(sb_gpu.shape)
    g = float(np.float32(gs))
    bad_s = sb_gpu != sb_ref
    if bad_s.any():
        amax = np.abs(blocks).max(-1).astype(np.float64)[bad_s]
        grid = nvfp4.e4m3_decode(np.arange(0x7F))
        near = _near_midpoint(amax / 6.0 / g, (grid[:-1] + grid[1:]) / 2, NEAR_TIE)
        step = np.abs(sb_gpu[bad_s].astype(int) - sb_ref[bad_s].astype(int)) == 1
        assert np.all(near & step), f"{what}: {int((~(near & step)).sum())} scale bytes differ away from a tie"
        # the differing blocks' codes follow the definition under the kernel's scale
        codes_ref[bad_s] = nvfp4.encode_with_scale(blocks[bad_s], sb_gpu[bad_s], gs)
    diff = codes_gpu != codes_ref
    if diff.any():
        S = (nvfp4.e4m3_decode(sb_gpu) * g)[..., None] * np.ones(16)
        q = np.abs(blocks.astype(np.float64))[diff] / S[diff]
        mids = (nvfp4.E2M1_MAGNITUDES[:-1] + nvfp4.E2M1_MAGNITUDES[1:]) / 2
        cg, cr = codes_gpu[diff].astype(int), codes_ref[diff].astype(int)
        ok = _near_midpoint(q, mids, NEAR_TIE) & ((cg >> 3) == (cr >> 3)) & (np.abs((cg & 7) - (cr & 7)) == 1)
        assert np.all(ok), f"{what}: {int((~ok).sum())} codes differ away from a tie"
    n_codes = codes_gpu.size
    flips = 17 * int(bad_s.sum()) + int((diff & ~bad_s[..., None]).sum())
    print(f"[quant] {what}: {flips} tie flips in {n_codes} codes (budget {budget:g} = {budget * n_codes:.1f})")
    assert flips <= budget * n_codes, f"{what}: {flips} tie flips exceed {budget:g} of {n_codes} codes"
    return flips, n_codes


def record_flips(rec_gpu, kv_c, k_pe, gs, record_bytes: int, what: str):
    """Cache records from the kernel against the oracle's encoder: the RoPE
    part and the padding bit-exact, the codes and scales up to counted tie
    flips (quant_flips).  kv_c / k_pe: the tokens' bf16 values as float32."""
    rec_gpu = np.asarray(rec_gpu, dtype=np.uint8)
    ref = ocache.encode_records(kv_c, k_pe, gs, record_bytes)
    assert np.array_equal(rec_gpu[:, ocache.ROPE_OFF:], ref[:, ocache.ROPE_OFF:]), f"{what}: RoPE part or padding differs"
    codes = nvfp4.unpack_e2m1(rec_gpu[:, ocache.CODES_OFF:ocache.SCALES_OFF])
    return quant_flips(kv_c, gs, codes, rec_gpu[:, ocache.SCALES_OFF:ocache.ROPE_OFF], what)
