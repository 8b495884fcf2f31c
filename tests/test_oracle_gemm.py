"""Pins for the oracle's NVFP4 GEMM (CPU only): a triple loop over values
decoded by table lookup (e2m1) and torch's float8_e4m3fn view (scales), the
lossless case where both operands lie on the NVFP4 grid, and ragged sizes
whose scale buffers carry padding."""
import numpy as np
import pytest
import torch

from oracle import gemm, nvfp4, swizzle

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _decode_loop(codes, sf_buf, rows, K, gs):
    """Values of a packed NVFP4 matrix, element by element: the nibble of
    byte k/2 (low nibble for even k), its e4m3 scale read at the 128x4
    offset of (row, k/16) through torch's float8 view."""
    Kp = (K // 16 + 3) // 4 * 4
    sf = torch.from_numpy(np.asarray(sf_buf, dtype=np.uint8).copy()).view(torch.float8_e4m3fn).double().numpy()
    out = np.zeros((rows, K))
    for r in range(rows):
        for k in range(K):
            byte = int(codes[r, k // 2])
            c = byte & 0xF if k % 2 == 0 else byte >> 4
            v = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
            kb = k // 16
            off = ((r // 128) * (Kp // 4) + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
            out[r, k] = v * sf[off] * float(np.float32(gs))
    return out


@pytest.mark.parametrize("M,N,K", [(3, 5, 32), (130, 7, 48), (2, 129, 80)])
def test_gemm_against_triple_loop(M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K)
    a = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, (M, 1)))).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32)
    gs_a, gs_w = nvfp4.global_scale(np.abs(a).max()), nvfp4.global_scale(np.abs(w).max())
    ac, asf = swizzle.quantize_rows(a, gs_a)
    wc, wsf = swizzle.quantize_rows(w, gs_w)
    got = gemm.nvfp4_gemm(ac, asf, wc, wsf, M, N, K, gs_a, gs_w)
    A = _decode_loop(ac, asf, M, K, gs_a)
    W = _decode_loop(wc, wsf, N, K, gs_w)
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += A[m, k] * W[n, k]
            ref[m, n] = s
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gemm_lossless_on_grid():
    # operands already of the form code * e4m3 * gs (gs a power of two, each
    # block holding a code of magnitude 6): quantisation is the identity, so
    # the GEMM equals the float64 product of the original values
    rng = np.random.default_rng(5)
    M, N, K = 64, 48, 128
    gs = np.float32(2.0 ** -3)

    def on_grid(rows):
        sb = rng.integers(0x20, 0x50, (rows, K // 16))
        codes = rng.integers(0, 16, (rows, K // 16, 16))
        codes[..., 0] = 7
        x = nvfp4.e2m1_decode(codes) * nvfp4.e4m3_decode(sb)[..., None] * float(gs)
        return x.reshape(rows, K).astype(np.float32)

    a, w = on_grid(M), on_grid(N)
    ac, asf = swizzle.quantize_rows(a, gs)
    wc, wsf = swizzle.quantize_rows(w, gs)
    got = gemm.nvfp4_gemm(ac, asf, wc, wsf, M, N, K, gs, gs)
    assert np.array_equal(got, a.astype(np.float64) @ w.astype(np.float64).T)


def test_gemm_entries_match_the_full_product():
    rng = np.random.default_rng(5)
    M, N, K = 300, 256, 512
    ac = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    wc = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    asf = swizzle.swizzle_scales(rng.integers(0x28, 0x48, (M, K // 16)).astype(np.uint8))
    wsf = swizzle.swizzle_scales(rng.integers(0x28, 0x48, (N, K // 16)).astype(np.uint8))
    full = gemm.nvfp4_gemm(ac, asf, wc, wsf, M, N, K, np.float32(0.5), np.float32(0.25))
    rows, cols = [0, 7, 128, 299], [1, 130, 255]
    sub = gemm.nvfp4_gemm_entries(ac, asf, wc, wsf, K, np.float32(0.5), np.float32(0.25), rows, cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])
