"""GPU parity of the NVFP4 x NVFP4 GEMM against the float64 oracle.

Both sides get the same packed codes and swizzled scale bytes (random, so no
quantiser is involved).  Every product of two e2m1 codes and two e4m3 scales
is exact in float32; the kernel sums K of them in float32 (error at most
K * 2^-24 of the sum of magnitudes, bound used with a factor 2), scales by
gs_a * gs_w and rounds to bf16 (half a bf16 ulp)."""
import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from oracle import attention, gemm, nvfp4, swizzle
from tests.helpers import bf16_half_ulp, f32

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def _random_nvfp4(rng, rows, K, sb_lo=0x28, sb_hi=0x48, pad=0):
    """Random packed codes and a swizzled scale buffer (scales in [sb_lo,
    sb_hi)); the buffer's padding holds `pad` (a byte) or random bytes (-1)."""
    codes = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    sf = rng.integers(sb_lo, sb_hi, (rows, K // 16)).astype(np.uint8)
    buf = swizzle.swizzle_scales(sf)
    if pad != 0:
        mask = np.ones(buf.size, dtype=bool)
        m, k = np.meshgrid(np.arange(rows), np.arange(K // 16), indexing="ij")
        mask[swizzle.sf_offset(m, k, K // 16)] = False
        buf[mask] = rng.integers(0, 256, int(mask.sum()), dtype=np.uint8) if pad < 0 else pad
    return codes, buf


def _abs_product(ac, asf, wc, wsf, M, N, K, gs_a, gs_w):
    """sum_k |a_hat||w_hat| (gs applied), for the accumulation bound."""
    a = np.abs(swizzle.dequantize_rows(ac, asf, M, K, gs_a))
    w = np.abs(swizzle.dequantize_rows(wc, wsf, N, K, gs_w))
    return a @ w.T


def _check(got, ref, absprod, K, what):
    bound = bf16_half_ulp(ref) + 2.0 * K * 2.0 ** -24 * absprod + 1e-30
    err = np.abs(got - ref)
    worst = float((err / bound).max())
    rel = float(err.sum() / np.abs(ref).sum())
    print(f"[gemm] {what}: max err / bound {worst:.3f}, mean rel {rel:.2e}")
    assert worst <= 1.0, f"{what}: error {worst:.3f} x the bound"


@pytest.mark.parametrize("M,N,K,pad", [(128, 256, 256, 0), (200, 384, 512, -1), (1, 128, 1024, 0),
                                       (300, 512, 4096, -1)])
def test_gemm_matches_oracle(M, N, K, pad):
    rng = np.random.default_rng(M + N + K)
    ac, asf = _random_nvfp4(rng, M, K, pad=pad)
    wc, wsf = _random_nvfp4(rng, N, K, pad=pad)
    gs_a, gs_w = np.float32(0.37), np.float32(1.0 / 3000)
    ref = gemm.nvfp4_gemm(ac, asf, wc, wsf, M, N, K, gs_a, gs_w)
    t = lambda x: torch.from_numpy(x).to(DEV)
    out = mla.mla_nvfp4_gemm(t(ac), t(asf), t(wc), t(wsf), torch.tensor([gs_a], device=DEV),
                             torch.tensor([gs_w], device=DEV))
    torch.cuda.synchronize()
    _check(f32(out), ref, _abs_product(ac, asf, wc, wsf, M, N, K, gs_a, gs_w), K, f"{M}x{N}x{K}")


def test_gemm_rejects_bad_shapes():
    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8, device=DEV)
    g = torch.ones(1, device=DEV)
    with pytest.raises(mla.MLAError):  # N not a multiple of 128
        mla.mla_nvfp4_gemm(u8(4, 128), u8(4096), u8(100, 128), u8(4096), g, g)
    with pytest.raises(mla.MLAError):  # K (= 2 x 64 code bytes) not a multiple of 256
        mla.mla_nvfp4_gemm(u8(4, 64), u8(4096), u8(128, 64), u8(4096), g, g)


def test_prefill_output_into_gemm():
    # the prefill's fused output is the GEMM's A as written: codes [T, H*64]
    # and the swizzled scale buffer; against the oracle chain (exact
    # attention -> the oracle's quantisation -> the oracle's GEMM), whose
    # codes differ from the kernel's at ~1e-2 boundary flips (the attention
    # error), hence the relative bound
    w = workloads.prefill("gemm_in", seq_lens=(300, 77), heads=2, seed=50)
    gs = nvfp4.global_scale(float(w.v.abs().max()))
    gst = torch.tensor([gs], device=DEV)
    codes, sf = mla.mla_nvfp4_prefill_fused_out(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.cu_seqlens.to(DEV),
                                                w.max_seqlen, w.softmax_scale, gst)
    T, K, N = w.total_tokens, 2 * 128, 384
    rng = np.random.default_rng(51)
    wc, wsf = _random_nvfp4(rng, N, K)
    gs_w = np.float32(1.0 / 1000)
    out = mla.mla_nvfp4_gemm(codes, sf, torch.from_numpy(wc).to(DEV), torch.from_numpy(wsf).to(DEV), gst,
                             torch.tensor([gs_w], device=DEV))
    torch.cuda.synchronize()
    o, _ = attention.prefill(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(), w.softmax_scale)
    oc, osf = swizzle.quantize_rows(o.reshape(T, K).astype(np.float32), gs)
    ref = gemm.nvfp4_gemm(oc, osf, wc, wsf, T, N, K, gs, gs_w)
    rel = float(np.abs(f32(out) - ref).sum() / np.abs(ref).sum())
    print(f"[gemm] prefill output -> gemm: mean rel {rel:.2e}")
    assert rel <= 2e-2


def test_gemm_full_size_sampled():
    """The benchmark's GEMM: the fused output of the 8 x 4096 x 128 prefill
    ([32768, 16384] codes + swizzled scales, as written) times a random
    NVFP4 weight [7168, 16384] drawn as the benchmark draws it; 64 x 64
    sampled outputs against the oracle."""
    w = workloads.prefill_8x4096(device=DEV)
    gsp = nvfp4.global_scale(float(w.v.abs().max()))
    gst = torch.tensor([gsp], device=DEV)
    codes, sf = mla.mla_nvfp4_prefill_fused_out(w.q, w.k, w.v, w.cu_seqlens, w.max_seqlen, w.softmax_scale, gst)
    n_out, k_in = 7168, w.heads * 128
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    wc = torch.randint(0, 256, (n_out, k_in // 2), dtype=torch.uint8, device=DEV, generator=g)
    wsf = torch.randint(0x28, 0x48, (n_out * k_in // 16,), dtype=torch.uint8, device=DEV, generator=g)
    gs_w = np.float32(1.0 / 4096)
    out = mla.mla_nvfp4_gemm(codes, sf, wc, wsf, gst, torch.tensor([gs_w], device=DEV))
    torch.cuda.synchronize()
    rng = np.random.default_rng(29)
    rows = np.unique(np.concatenate([[0, 127, 128, 32767], rng.integers(0, 32768, 60)]))
    cols = np.unique(np.concatenate([[0, 255, 256, 7167], rng.integers(0, 7168, 60)]))
    ac, asf = codes.cpu().numpy(), sf.cpu().numpy()
    wc_np, wsf_np = wc.cpu().numpy(), wsf.cpu().numpy()
    ref = gemm.nvfp4_gemm_entries(ac, asf, wc_np, wsf_np, k_in, gsp, gs_w, rows, cols)

    def rows_abs(c, buf, idx, gs):
        m, kk = np.meshgrid(idx, np.arange(k_in // 16), indexing="ij")
        sfb = buf[swizzle.sf_offset(m, kk, k_in // 16)]
        return np.abs(nvfp4.dequantize_blocks(nvfp4.unpack_e2m1(c[idx]), sfb, gs))

    absprod = rows_abs(ac, asf, rows, gsp) @ rows_abs(wc_np, wsf_np, cols, gs_w).T
    _check(f32(out[rows][:, cols]), ref, absprod, k_in, "32768x7168x16384 sampled")
