"""MLA attention with an NVFP4 latent cache and NVFP4 fused prefill output,
for one GB300 (sm_103a).

This package is a thin ctypes binding over libmla_nvfp4.so (C ABI declared
in include/mla_nvfp4.h).  The Python functions carry the same names as the C
entry points and only marshal arguments: every step of the computation runs
in the library's CUDA kernels.  PyTorch supplies device memory and the
current stream.  There is no CPU fallback: if the library is missing or the
device is not sm_103, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "load_library", "MLAError", "mla_nvfp4_global_scale", "mla_nvfp4_cache_write",
    "mla_nvfp4_decode_workspace_size", "mla_nvfp4_decode_default_splits", "mla_nvfp4_decode_plan_splits",
    "decode_launches",
    "mla_nvfp4_decode", "mla_nvfp4_decode_q4", "mla_nvfp4_prefill_fused_out",
    "mla_nvfp4_quantize_rows", "mla_nvfp4_gemm", "mla_nvfp4_gather_latent", "mla_nvfp4_prefill_partial",
    "mla_nvfp4_merge_fused_out", "mla_nvfp4_prefill_qdq", "mla_nvfp4_prefill_fakequant",
    "mla_nvfp4_prefill_quantized", "abi_symbols", "RECORD_BF16_ROPE", "RECORD_FP8_ROPE",
    "LAUNCHES_PER_CALL",
]

RECORD_BF16_ROPE = 432
RECORD_FP8_ROPE = 368
DEVERR_BOUNDS, DEVERR_TIMEOUT, DEVERR_SCALE, DEVERR_RANGE = 0x1, 0x2, 0x4, 0x8

# Kernels each entry point launches (for launch accounting in the benchmark);
# decode launches one kernel with one key split, two (plus the merge) with
# uniform splits and three (plan, decode, merge) when planned, see
# decode_launches().
LAUNCHES_PER_CALL = {"cache_write": 1, "decode": 3, "prefill": 1, "global_scale": 2, "gemm": 1,
                     "gather_latent": 1, "prefill_partial": 1, "merge_fused_out": 1, "prefill_qdq": 2,
                     "prefill_fakequant": 1}
# What bounds each hot kernel as built: "hbm", "tensor" (tcgen05 MMA) or
# "alu" (CUDA-core arithmetic).
KERNEL_BOUND = {"cache_write": "hbm", "decode": "tensor", "prefill": "tensor", "gemm": "tensor"}
# Operand type of each kernel's tensor-core products (fp32 accumulation):
# the decode multiplies f16 operands (the dequantised latent c*s is exact in
# f16), the prefill bf16 inputs as given.
OPERAND_DTYPE = {"decode": "f16", "prefill": "bf16", "gemm": "nvfp4"}


def kernel_kind(name: str) -> str:
    return KERNEL_BOUND[name]


def operand_dtype(name: str) -> str:
    return OPERAND_DTYPE[name]

_LIB = None

_c_i64, _c_int, _c_vp, _c_f = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
_SIGS = {
    "mla_nvfp4_status_string": (ctypes.c_char_p, [_c_int]),
    "mla_nvfp4_abi_version": (_c_int, []),
    "mla_nvfp4_last_error": (ctypes.c_char_p, []),
    "mla_nvfp4_global_scale": (_c_int, [_c_vp, _c_i64, _c_vp, _c_vp]),
    "mla_nvfp4_cache_write": (_c_int, [_c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_i64,
                                       _c_int, _c_vp, _c_vp, _c_vp]),
    "mla_nvfp4_decode_workspace_size": (ctypes.c_size_t, [_c_int, _c_int, _c_int]),
    "mla_nvfp4_decode_default_splits": (_c_int, [_c_int, _c_int, _c_int]),
    "mla_nvfp4_decode_plan_splits": (_c_int, [_c_vp, _c_int, _c_int, ctypes.c_size_t]),
    "mla_nvfp4_decode": (_c_int, [_c_vp, _c_int, _c_int, _c_vp, _c_i64, _c_int, _c_vp, _c_i64, _c_int,
                                  _c_vp, _c_vp, _c_int, _c_f, _c_vp, _c_vp, _c_vp, _c_vp,
                                  ctypes.c_size_t, _c_int, _c_vp, _c_vp]),
    "mla_nvfp4_decode_q4": (_c_int, [_c_vp, _c_int, _c_int, _c_vp, _c_i64, _c_int, _c_vp, _c_i64, _c_int,
                                     _c_vp, _c_vp, _c_int, _c_f, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                     ctypes.c_size_t, _c_int, _c_vp, _c_vp]),
    "mla_nvfp4_decode_noalloc": (_c_int, [_c_vp, _c_int, _c_int, _c_vp, _c_i64, _c_int, _c_vp, _c_i64,
                                          _c_int, _c_vp, _c_vp, _c_int, _c_f, _c_vp, _c_vp, _c_vp,
                                          _c_int, _c_vp, _c_vp]),
    "mla_nvfp4_decode_host": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp, _c_i64, _c_int, _c_vp, _c_vp,
                                       _c_i64, _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_f, _c_vp,
                                       _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_int, _c_vp,
                                       _c_vp]),
    "mla_nvfp4_prefill_fused_out": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64,
                                             _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_int, _c_int,
                                             _c_f, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_nvfp4_quantize_rows": (_c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_nvfp4_gather_latent": (_c_int, [_c_vp, _c_i64, _c_int, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_nvfp4_prefill_partial": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64,
                                           _c_vp, _c_vp, _c_int, _c_i64, _c_i64, _c_int, _c_int, _c_f, _c_vp,
                                           _c_vp, _c_vp, _c_vp]),
    "mla_nvfp4_merge_fused_out": (_c_int, [_c_vp, _c_vp, _c_int, _c_i64, _c_int, _c_vp, _c_vp, _c_vp, _c_vp,
                                           _c_vp, _c_vp]),
    "mla_nvfp4_prefill_qdq": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp,
                                       _c_int, _c_i64, _c_int, _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                       _c_vp, _c_vp]),
    "mla_nvfp4_prefill_fakequant": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_i64, _c_int, _c_int, _c_f,
                                             _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_nvfp4_gemm": (_c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64,
                                _c_vp, _c_vp]),
    "mla_nvfp4_selftest_wait": (_c_int, [_c_vp, _c_i64, _c_vp, _c_vp]),
}


def abi_symbols():
    """Entry points the header declares (and the library must export)."""
    return list(_SIGS)


class MLAError(RuntimeError):
    def __init__(self, fn, status, detail=None):
        self.status = status
        if detail is not None:
            detail = ": " + detail
        else:
            detail = ""
            if status == 6:  # MLA_ERR_LAUNCH: add the CUDA runtime's message
                detail = ": " + load_library().mla_nvfp4_last_error().decode()
        super().__init__(f"{fn}: {status_string(status)} (status {status}){detail}")


def load_library(path: str | None = None, build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libmla_nvfp4.so."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    lib_path = path or _build.LIB
    if path is None and build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(lib_path):
        raise RuntimeError(f"libmla_nvfp4.so not found at {lib_path}; run the package build")
    lib = ctypes.CDLL(lib_path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load_library().mla_nvfp4_status_string(status).decode()


def _check(fn, status):
    if status != 0:
        raise MLAError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, name, dtype, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def mla_nvfp4_global_scale(x: torch.Tensor, gs: torch.Tensor | None = None) -> torch.Tensor:
    """gs = amax|x| / (6 * 448) as a device fp32 scalar tensor (shape [1])."""
    _need(x, "x", torch.bfloat16)
    if gs is None:
        gs = torch.empty(1, dtype=torch.float32, device=x.device)
    _need(gs, "gs", torch.float32, x.device)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    with torch.cuda.device(x.device):
        _check("mla_nvfp4_global_scale",
               load_library().mla_nvfp4_global_scale(_ptr(x), x.numel(), _ptr(gs), _stream(x)))
    return gs


def mla_nvfp4_cache_write(kv_c, k_pe, slot_mapping, cache, global_scale, error_word=None):
    """Quantise kv_c [T,512] / k_pe [T,64] (bf16) into cache [num_slots, 432|368] (uint8)."""
    dev = cache.device
    _need(kv_c, "kv_c", torch.bfloat16, dev)
    _need(k_pe, "k_pe", torch.bfloat16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    _need(cache, "cache", torch.uint8, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    if cache.dim() != 2 or kv_c.dim() != 2 or k_pe.dim() != 2:
        raise ValueError("kv_c, k_pe and cache must be 2-D")
    if kv_c.stride(1) != 1 or k_pe.stride(1) != 1 or not cache.is_contiguous() or not slot_mapping.is_contiguous():
        raise ValueError("last dimensions must be contiguous")
    T = kv_c.shape[0]
    if k_pe.shape[0] != T or slot_mapping.numel() != T or kv_c.shape[1] != 512 or k_pe.shape[1] != 64:
        raise ValueError("shape mismatch")
    with torch.cuda.device(dev):
        _check("mla_nvfp4_cache_write", load_library().mla_nvfp4_cache_write(
            _ptr(kv_c), kv_c.stride(0), _ptr(k_pe), k_pe.stride(0), _ptr(slot_mapping), T,
            _ptr(cache), cache.shape[0], cache.shape[1], _ptr(global_scale), _ptr(error_word),
            _stream(cache)))


def mla_nvfp4_decode_workspace_size(batch: int, num_heads: int, num_splits: int = 0) -> int:
    return int(load_library().mla_nvfp4_decode_workspace_size(batch, num_heads, num_splits))


def mla_nvfp4_decode_default_splits(batch: int, num_heads: int, num_splits: int = 0) -> int:
    """Equal key splits a decode of (batch, num_heads) uses: num_splits when
    > 0, else the library default on the current device (top-k calls, and
    paged calls without a workspace; paged calls with one are planned)."""
    return int(load_library().mla_nvfp4_decode_default_splits(batch, num_heads, num_splits))


def mla_nvfp4_decode_plan_splits(seq_lens_host, num_heads: int, workspace_bytes: int = 0) -> int:
    """The device plan's choice, made on the host from lengths held there
    (int32 CPU tensor or array [batch]): 1 when it would keep one chunk per
    sequence (call mla_nvfp4_decode with num_splits=1: one launch, no
    workspace), 0 when it would cut sequences (num_splits=0 with a
    workspace of workspace_bytes)."""
    lens = torch.as_tensor(seq_lens_host, device="cpu").to(torch.int32).contiguous()
    if lens.dim() != 1:
        raise ValueError("seq_lens_host must be one-dimensional")
    return int(load_library().mla_nvfp4_decode_plan_splits(lens.data_ptr(), int(lens.shape[0]), num_heads,
                                                           int(workspace_bytes)))


def decode_launches(batch: int, num_heads: int, num_splits: int = 0, *, paged: bool = True,
                    workspace: bool = True) -> int:
    """Kernels one mla_nvfp4_decode call launches: plan, decode and merge
    when planned (paged, num_splits <= 0, a workspace); otherwise the decode,
    plus the merge with more than one split."""
    if paged and num_splits <= 0 and workspace:
        return 3
    return 1 if mla_nvfp4_decode_default_splits(batch, num_heads, num_splits) == 1 else 2


def mla_nvfp4_decode_q4(q, cache, global_scale, softmax_scale, q_global_scale, **kw):
    """mla_nvfp4_decode with the query quantised to NVFP4 (global scale
    q_global_scale, a device fp32 [1]) and block-scaled fp4 scores."""
    return mla_nvfp4_decode(q, cache, global_scale, softmax_scale, _q_global_scale=q_global_scale, **kw)


def mla_nvfp4_decode(q, cache, global_scale, softmax_scale, *, page_table=None, seq_lens=None,
                     page_size=64, topk_indices=None, out=None, lse=None, workspace=None,
                     num_splits=0, error_word=None, return_lse=False, _q_global_scale=None):
    """Absorbed MLA decode.  q [B,H,576] bf16 -> out [B,H,512] bf16 (and lse [B,H] fp32)."""
    dev = q.device
    _need(q, "q", torch.bfloat16)
    _need(cache, "cache", torch.uint8, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(page_table, "page_table", torch.int32, dev)
    _need(seq_lens, "seq_lens", torch.int32, dev)
    _need(topk_indices, "topk_indices", torch.int32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    if q.dim() != 3 or q.shape[2] != 576 or not q.is_contiguous():
        raise ValueError("q must be contiguous [B, H, 576]")
    B, H, _ = q.shape
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    if return_lse and lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    _need(lse, "lse", torch.float32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        need = int(lib.mla_nvfp4_decode_workspace_size(B, H, num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, dev)
        pt_stride = page_table.stride(0) if page_table is not None else 0
        topk = topk_indices.shape[1] if topk_indices is not None else 0
        if topk_indices is not None and topk_indices.stride(1) != 1:
            raise ValueError("topk_indices rows must be contiguous")
        args = (_ptr(q), B, H, _ptr(cache), cache.shape[0], cache.shape[1], _ptr(page_table), pt_stride,
                page_size, _ptr(seq_lens), _ptr(topk_indices), topk, float(softmax_scale), _ptr(global_scale))
        tail = (_ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() if workspace is not None else 0,
                num_splits, _ptr(error_word), _stream(q))
        if _q_global_scale is None:
            _check("mla_nvfp4_decode", lib.mla_nvfp4_decode(*args, *tail))
        else:
            _need(_q_global_scale, "q_global_scale", torch.float32, dev)
            _check("mla_nvfp4_decode_q4", lib.mla_nvfp4_decode_q4(*args, _ptr(_q_global_scale), *tail))
    return (out, lse) if return_lse else out


def _host_dev_pair(h, d, name, dtype, dev, shape):
    """A host tensor and its device buffer: both or neither, same shape."""
    if (h is None) != (d is None):
        raise ValueError(f"{name}_host and {name}_dev go together")
    if h is None:
        return
    if h.device.type != "cpu" or not h.is_contiguous() or h.dtype != dtype:
        raise ValueError(f"{name}_host must be a contiguous {dtype} CPU tensor")
    if d.device != dev or not d.is_contiguous() or d.dtype != dtype:
        raise ValueError(f"{name}_dev must be a contiguous {dtype} tensor on {dev}")
    if tuple(h.shape) != tuple(d.shape) or (shape is not None and tuple(h.shape) != tuple(shape)):
        raise ValueError(f"{name}_host and {name}_dev must both have shape {shape or tuple(h.shape)}")


def mla_nvfp4_decode_host(q_host, q_dev, cache, global_scale, softmax_scale, out_host, out_dev, *,
                          page_table_host=None, page_table_dev=None, seq_lens_host=None,
                          seq_lens_dev=None, page_size=64, topk_host=None, topk_dev=None,
                          lse_host=None, lse_dev=None, workspace=None, num_splits=0,
                          error_word=None):
    """mla_nvfp4_decode from host tensors to host tensors through one C-ABI
    call: the library copies the inputs into the given device buffers, runs
    the decode and copies ``out`` (and ``lse``) back, all on the current
    stream of ``cache``'s device.  Use pinned host tensors for asynchronous
    copies and synchronise the stream before reading ``out_host``."""
    dev = cache.device
    _need(cache, "cache", torch.uint8, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    if q_host.dim() != 3 or q_host.shape[2] != 576:
        raise ValueError("q_host must be [B, H, 576]")
    B, H, _ = q_host.shape
    _host_dev_pair(q_host, q_dev, "q", torch.bfloat16, dev, (B, H, 576))
    _host_dev_pair(out_host, out_dev, "out", torch.bfloat16, dev, (B, H, 512))
    for t, name in ((page_table_host, "page_table_host"), (topk_host, "topk_host")):
        if t is not None and (t.dim() != 2 or t.shape[0] != B):
            raise ValueError(f"{name} must be [B, n]")
    _host_dev_pair(page_table_host, page_table_dev, "page_table", torch.int32, dev, None)
    _host_dev_pair(seq_lens_host, seq_lens_dev, "seq_lens", torch.int32, dev, (B,))
    _host_dev_pair(topk_host, topk_dev, "topk", torch.int32, dev, None)
    _host_dev_pair(lse_host, lse_dev, "lse", torch.float32, dev, (B, H))
    lib = load_library()
    with torch.cuda.device(dev):
        need = int(lib.mla_nvfp4_decode_workspace_size(B, H, num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, dev)
        pt_stride = page_table_host.shape[1] if page_table_host is not None else 0
        topk = topk_host.shape[1] if topk_host is not None else 0
        _check("mla_nvfp4_decode_host", lib.mla_nvfp4_decode_host(
            _ptr(q_host), _ptr(q_dev), B, H, _ptr(cache), cache.shape[0], cache.shape[1],
            _ptr(page_table_host), _ptr(page_table_dev), pt_stride, page_size, _ptr(seq_lens_host),
            _ptr(seq_lens_dev), _ptr(topk_host), _ptr(topk_dev), topk, float(softmax_scale),
            _ptr(global_scale), _ptr(out_host), _ptr(out_dev), _ptr(lse_host), _ptr(lse_dev),
            _ptr(workspace), workspace.numel() if workspace is not None else 0, num_splits,
            _ptr(error_word), _stream(cache)))
    return out_host


def mla_nvfp4_selftest_wait(error_word, limit_ns, elapsed_ns=None):
    """Test hook: one CTA whose wait on a barrier nothing arrives on runs
    out after ``limit_ns`` (flagging DEVERR_TIMEOUT in ``error_word``) and
    whose second, 2-second wait then ends through the CTA's abort flag;
    ``elapsed_ns`` (int64 [2] on the device) receives both waits' times."""
    _need(error_word, "error_word", torch.int32)
    _need(elapsed_ns, "elapsed_ns", torch.int64, error_word.device)
    lib = load_library()
    with torch.cuda.device(error_word.device):
        _check("mla_nvfp4_selftest_wait", lib.mla_nvfp4_selftest_wait(
            _ptr(error_word), int(limit_ns), _ptr(elapsed_ns), _stream(error_word)))


def mla_nvfp4_decode_noalloc(q, cache, global_scale, softmax_scale, out, *, page_table=None,
                             seq_lens=None, page_size=64, topk_indices=None, lse=None, num_splits=0,
                             error_word=None):
    """mla_nvfp4_decode with the library's built-in scratch instead of a
    workspace; the caller passes ``out`` (and ``lse`` if wanted), so nothing
    is allocated.  Returns ``out``."""
    dev = q.device
    _need(q, "q", torch.bfloat16)
    _need(cache, "cache", torch.uint8, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(page_table, "page_table", torch.int32, dev)
    _need(seq_lens, "seq_lens", torch.int32, dev)
    _need(topk_indices, "topk_indices", torch.int32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    if out is None:
        raise ValueError("out must be given: this entry point allocates nothing")
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    if q.dim() != 3 or q.shape[2] != 576 or not q.is_contiguous():
        raise ValueError("q must be contiguous [B, H, 576]")
    B, H, _ = q.shape
    if out.shape != (B, H, 512) or not out.is_contiguous():
        raise ValueError("out must be contiguous [B, H, 512]")
    if lse is not None and (lse.shape != (B, H) or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous [B, H]")
    if topk_indices is not None and topk_indices.stride(1) != 1:
        raise ValueError("topk_indices rows must be contiguous")
    lib = load_library()
    pt_stride = page_table.stride(0) if page_table is not None else 0
    topk = topk_indices.shape[1] if topk_indices is not None else 0
    with torch.cuda.device(dev):
        st = lib.mla_nvfp4_decode_noalloc(
            _ptr(q), B, H, _ptr(cache), cache.shape[0], cache.shape[1], _ptr(page_table), pt_stride,
            page_size, _ptr(seq_lens), _ptr(topk_indices), topk, float(softmax_scale),
            _ptr(global_scale), _ptr(out), _ptr(lse), num_splits, _ptr(error_word), _stream(q))
    if st != 0:
        detail = lib.mla_nvfp4_last_error().decode() if st in (5, 6) else None
        raise MLAError("mla_nvfp4_decode_noalloc", st, detail)
    return out


def prefill_scale_bytes(total_tokens: int, num_heads: int) -> int:
    return ((total_tokens + 127) // 128 * 128) * ((num_heads * 8 + 3) // 4 * 4)


def mla_nvfp4_prefill_fused_out(q, k, v, cu_seqlens, max_seqlen, softmax_scale, global_scale, *,
                                out_codes=None, out_scales=None, lse=None, return_lse=False,
                                error_word=None):
    """Causal varlen prefill -> (codes [T, H*64] uint8, swizzled scales uint8[, lse [H, T]])."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, dev)
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError(f"{n} must be [T, H, D] with a contiguous last dimension")
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    T, H, dq = q.shape
    if dq != 192 or k.shape != (T, H, 192) or v.shape != (T, H, 128):
        raise ValueError("expected q, k [T,H,192] and v [T,H,128]")
    if out_codes is None:
        out_codes = torch.empty((T, H * 64), dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty(prefill_scale_bytes(T, H), dtype=torch.uint8, device=dev)
    _need(out_codes, "out_codes", torch.uint8, dev)
    _need(out_scales, "out_scales", torch.uint8, dev)
    if return_lse and lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    _need(lse, "lse", torch.float32, dev)
    with torch.cuda.device(dev):
        _check("mla_nvfp4_prefill_fused_out", load_library().mla_nvfp4_prefill_fused_out(
            _ptr(q), _ptr(k), _ptr(v), q.stride(0), q.stride(1), k.stride(0), k.stride(1),
            v.stride(0), v.stride(1), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen), H,
            float(softmax_scale), _ptr(global_scale), _ptr(out_codes), _ptr(out_scales), _ptr(lse),
            _ptr(error_word), _stream(q)))
    return (out_codes, out_scales, lse) if return_lse else (out_codes, out_scales)


def mla_nvfp4_quantize_rows(x, global_scale, *, codes=None, scales=None, error_word=None):
    """fp32 [M, N] -> (packed codes [M, N/2] uint8, swizzled scales uint8)."""
    dev = x.device
    _need(x, "x", torch.float32)
    _need(global_scale, "global_scale", torch.float32, dev)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    M, N = x.shape
    if codes is None:
        codes = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(((M + 127) // 128 * 128) * ((N // 16 + 3) // 4 * 4), dtype=torch.uint8,
                             device=dev)
    with torch.cuda.device(dev):
        _check("mla_nvfp4_quantize_rows", load_library().mla_nvfp4_quantize_rows(
            _ptr(x), M, N, _ptr(global_scale), _ptr(codes), _ptr(scales), _ptr(error_word),
            _stream(x)))
    return codes, scales


def mla_nvfp4_gemm(a_codes, a_scales, w_codes, w_scales, gs_a, gs_w, *, out=None):
    """NVFP4 x NVFP4 -> bf16: a_codes [M, K/2] / w_codes [N, K/2] (uint8)
    with their 128x4-swizzled scale buffers and device fp32 global scales;
    returns out [M, N] bf16."""
    dev = a_codes.device
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"), (w_scales, "w_scales")):
        _need(t, n, torch.uint8, dev)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _need(gs_a, "gs_a", torch.float32, dev)
    _need(gs_w, "gs_w", torch.float32, dev)
    if a_codes.dim() != 2 or w_codes.dim() != 2 or a_codes.shape[1] != w_codes.shape[1]:
        raise ValueError("a_codes [M, K/2] and w_codes [N, K/2] must share K")
    M, N, K = a_codes.shape[0], w_codes.shape[0], 2 * a_codes.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    if out.dim() != 2 or out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with a contiguous last dimension")
    with torch.cuda.device(dev):
        _check("mla_nvfp4_gemm", load_library().mla_nvfp4_gemm(
            _ptr(a_codes), _ptr(a_scales), M, _ptr(w_codes), _ptr(w_scales), N, K, _ptr(gs_a), _ptr(gs_w),
            _ptr(out), out.stride(0), None, _stream(a_codes)))
    return out


def mla_nvfp4_gather_latent(cache, global_scale, slots, *, kv_c=None, k_pe=None, error_word=None):
    """Records of ``slots`` (int64 [n]) read back: kv_c bf16 [n, 512] (the
    dequantised latent rounded to bf16) and k_pe bf16 [n, 64]."""
    dev = cache.device
    _need(cache, "cache", torch.uint8, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(slots, "slots", torch.int64, dev)
    _need(error_word, "error_word", torch.int32, dev)
    if cache.dim() != 2 or not cache.is_contiguous() or not slots.is_contiguous():
        raise ValueError("cache [num_slots, record_bytes] and slots must be contiguous")
    n = slots.numel()
    if kv_c is None:
        kv_c = torch.empty((n, 512), dtype=torch.bfloat16, device=dev)
    if k_pe is None:
        k_pe = torch.empty((n, 64), dtype=torch.bfloat16, device=dev)
    for t, name, d in ((kv_c, "kv_c", 512), (k_pe, "k_pe", 64)):
        _need(t, name, torch.bfloat16, dev)
        if t.shape != (n, d) or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [n, {d}]")
    with torch.cuda.device(dev):
        _check("mla_nvfp4_gather_latent", load_library().mla_nvfp4_gather_latent(
            _ptr(cache), cache.shape[0], cache.shape[1], _ptr(global_scale), _ptr(slots), n, _ptr(kv_c), _ptr(k_pe),
            _ptr(error_word), _stream(cache)))
    return kv_c, k_pe


def mla_nvfp4_prefill_partial(q, k, v, cu_seqlens, max_seqlen, softmax_scale, *, cu_seqlens_k=None, out=None,
                              lse=None, error_word=None):
    """Prefill attention with an unquantised result: causal over the
    sequence's own tokens (cu_seqlens_k None) or over all keys of its chunk
    of k / v (cu_seqlens_k given).  Returns (out fp32 [T, H, 128], lse fp32
    [H, T])."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, dev)
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError(f"{n} must be [T, H, D] with a contiguous last dimension")
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    T, H, dq = q.shape
    if dq != 192 or k.shape[1:] != (H, 192) or v.shape[1:] != (H, 128) or k.shape[0] != v.shape[0]:
        raise ValueError("expected q [T,H,192], k [Tk,H,192], v [Tk,H,128]")
    if cu_seqlens_k is None and k.shape[0] != T:
        raise ValueError("without cu_seqlens_k, k and v hold the queries' own tokens")
    if out is None:
        out = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    _need(lse, "lse", torch.float32, dev)
    with torch.cuda.device(dev):
        _check("mla_nvfp4_prefill_partial", load_library().mla_nvfp4_prefill_partial(
            _ptr(q), _ptr(k), _ptr(v), q.stride(0), q.stride(1), k.stride(0), k.stride(1), v.stride(0), v.stride(1),
            _ptr(cu_seqlens), _ptr(cu_seqlens_k), cu_seqlens.numel() - 1, T, k.shape[0], int(max_seqlen), H,
            float(softmax_scale), _ptr(out), _ptr(lse), _ptr(error_word), _stream(q)))
    return out, lse


def mla_nvfp4_merge_fused_out(o_parts, lse_parts, global_scale, *, out_codes=None, out_scales=None, lse=None,
                              error_word=None):
    """Merge partials o_parts fp32 [P, T, H, 128] / lse_parts fp32 [P, H, T]
    by LSE into the fused NVFP4 output: (codes [T, H*64], swizzled scales)."""
    dev = o_parts.device
    _need(o_parts, "o_parts", torch.float32, dev)
    _need(lse_parts, "lse_parts", torch.float32, dev)
    _need(global_scale, "global_scale", torch.float32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    if o_parts.dim() != 4 or o_parts.shape[3] != 128 or not o_parts.is_contiguous() or not lse_parts.is_contiguous():
        raise ValueError("o_parts must be contiguous [P, T, H, 128]")
    P, T, H, _ = o_parts.shape
    if lse_parts.shape != (P, H, T):
        raise ValueError("lse_parts must be [P, H, T]")
    if out_codes is None:
        out_codes = torch.empty((T, H * 64), dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty(prefill_scale_bytes(T, H), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("mla_nvfp4_merge_fused_out", load_library().mla_nvfp4_merge_fused_out(
            _ptr(o_parts), _ptr(lse_parts), P, T, H, _ptr(global_scale), _ptr(out_codes), _ptr(out_scales),
            _ptr(lse), _ptr(error_word), _stream(o_parts)))
    return out_codes, out_scales


def mla_nvfp4_prefill_qdq(q, k, v, cu_seqlens, max_seqlen, gs_q, gs_k, gs_v, *, error_word=None):
    """NVFP4 fake quantisation of the prefill operands along their
    contraction axes: (q_cs f16 [T,H,192], k_cs f16 [T,H,192], v_cs f16
    [T,H,128]) holding code * e4m3 scale (global scales left out)."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, dev)
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError(f"{n} must be [T, H, D] with a contiguous last dimension")
    for t, n in ((gs_q, "gs_q"), (gs_k, "gs_k"), (gs_v, "gs_v")):
        _need(t, n, torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    T, H, _ = q.shape
    if q.shape[2] != 192 or k.shape != (T, H, 192) or v.shape != (T, H, 128):
        raise ValueError("expected q, k [T,H,192] and v [T,H,128]")
    q_out = torch.empty((T, H, 192), dtype=torch.float16, device=dev)
    k_out = torch.empty((T, H, 192), dtype=torch.float16, device=dev)
    v_out = torch.empty((T, H, 128), dtype=torch.float16, device=dev)
    with torch.cuda.device(dev):
        _check("mla_nvfp4_prefill_qdq", load_library().mla_nvfp4_prefill_qdq(
            _ptr(q), _ptr(k), _ptr(v), q.stride(0), q.stride(1), k.stride(0), k.stride(1), v.stride(0), v.stride(1),
            _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen), H, _ptr(gs_q), _ptr(gs_k), _ptr(gs_v),
            _ptr(q_out), _ptr(k_out), _ptr(v_out), _ptr(error_word), _stream(q)))
    return q_out, k_out, v_out


def mla_nvfp4_prefill_fakequant(q_cs, k_cs, v_cs, cu_seqlens, max_seqlen, softmax_scale, gs_q, gs_k, gs_v,
                                global_scale, *, sparse24=False, out_codes=None, out_scales=None,
                                return_lse=False, lse=None, error_word=None):
    """Causal prefill over fake-quantised operands (mla_nvfp4_prefill_qdq's
    outputs), P quantised to NVFP4, optional 2:4 score sparsity; the output
    as mla_nvfp4_prefill_fused_out writes it."""
    dev = q_cs.device
    for t, n in ((q_cs, "q_cs"), (k_cs, "k_cs"), (v_cs, "v_cs")):
        _need(t, n, torch.float16, dev)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((gs_q, "gs_q"), (gs_k, "gs_k"), (gs_v, "gs_v"), (global_scale, "global_scale")):
        _need(t, n, torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(error_word, "error_word", torch.int32, dev)
    T, H, _ = q_cs.shape
    if q_cs.shape[2] != 192 or k_cs.shape != (T, H, 192) or v_cs.shape != (T, H, 128):
        raise ValueError("expected q_cs, k_cs [T,H,192] and v_cs [T,H,128]")
    if out_codes is None:
        out_codes = torch.empty((T, H * 64), dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty(prefill_scale_bytes(T, H), dtype=torch.uint8, device=dev)
    if return_lse and lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check("mla_nvfp4_prefill_fakequant", load_library().mla_nvfp4_prefill_fakequant(
            _ptr(q_cs), _ptr(k_cs), _ptr(v_cs), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen), H,
            float(softmax_scale), _ptr(gs_q), _ptr(gs_k), _ptr(gs_v), 1 if sparse24 else 0, _ptr(global_scale),
            _ptr(out_codes), _ptr(out_scales), _ptr(lse), _ptr(error_word), _stream(q_cs)))
    return (out_codes, out_scales, lse) if return_lse else (out_codes, out_scales)


def mla_nvfp4_prefill_quantized(q, k, v, cu_seqlens, max_seqlen, softmax_scale, global_scale, *, sparse24=False,
                                return_lse=False, error_word=None):
    """The fake-quantised prefill end to end: the global scales of q, k, v
    (amax/2688 each), their NVFP4 fake quantisation, and the prefill with P
    quantised (and optional 2:4 sparsity) writing the NVFP4 output."""
    gs = [mla_nvfp4_global_scale(t) for t in (q, k, v)]
    q_cs, k_cs, v_cs = mla_nvfp4_prefill_qdq(q, k, v, cu_seqlens, max_seqlen, *gs, error_word=error_word)
    return mla_nvfp4_prefill_fakequant(q_cs, k_cs, v_cs, cu_seqlens, max_seqlen, softmax_scale, *gs, global_scale,
                                       sparse24=sparse24, return_lse=return_lse, error_word=error_word)
