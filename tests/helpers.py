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
# Rounding-tie budget for codes where both sides do not see the same input.
TIE_BUDGET = 1e-4


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
        return attention.decode_slots_paged(w.page_table.cpu().numpy(), w.seq_lens.cpu().numpy(), 64)
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
    denom = float(np.abs(ref).sum())
    mean_rel = float(err.sum() / denom) if denom > 0 else float(err.sum())
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


def check_fused_output(codes_gpu, scales_gpu, o_ref, o_abs, gs):
    """End-to-end NVFP4 output check where the kernel quantises its own fp32
    attention output.  Each output element may differ from the exact one by
    err = P_ROUNDING * o_abs (+1e-6 relative).  A scale byte may differ from
    the oracle's quantisation of the exact output only where the block's raw
    scale lies within the error of an e4m3 rounding midpoint, and a code only
    where value/scale lies within err/scale of an e2m1 midpoint (or its
    block's scale differs).  Returns (scale mismatches, code mismatches)."""
    M, N = o_ref.shape
    return check_fused_blocks(codes_gpu, swizzle.unswizzle_scales(scales_gpu, M, N // 16), o_ref, o_abs, gs)


def check_fused_blocks(codes_gpu, sf_gpu, o_ref, o_abs, gs):
    """check_fused_output with the kernel's scale bytes already in row-major
    [M, N/16] order (used for sampled rows of a large output)."""
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
    assert not np.any(bad_s & ~near_s), f"{int((bad_s & ~near_s).sum())} scale bytes differ away from a tie"
    # codes (only in blocks whose scale agrees)
    S = (nvfp4.e4m3_decode(sb_ref) * float(gs)).repeat(16, axis=1)
    safe = np.where(S > 0, S, 1.0)
    q = np.where(S > 0, x.astype(np.float64) / safe, 0)
    near_c = code_boundary_distance(q) <= err / safe
    same_scale = (~bad_s).repeat(16, axis=1)
    diff = (codes_g != codes_ref)
    # the sign of a value that rounds to zero may differ
    zero_both = ((codes_g & 7) == 0) & ((codes_ref & 7) == 0)
    diff &= ~zero_both
    bad = diff & same_scale & ~near_c
    assert not np.any(bad), f"{int(bad.sum())} codes differ away from a rounding boundary"
    return int(bad_s.sum()), int((diff & same_scale).sum())
