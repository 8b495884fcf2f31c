"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point include/mla_nvfp4.h declares, and rejects bad arguments on the
host before touching a device."""
import ctypes
import os
import re

import pytest

import mla_attention_nvfp4_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "mla_nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_nvfp4_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = mla.load_library()
    declared = _header_functions()
    assert len(declared) >= 7
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(mla.abi_symbols()) == declared
    assert lib.mla_nvfp4_abi_version() == 2


def test_status_strings():
    assert mla.status_string(0) == "MLA_OK"
    assert "368 or 432" in mla.status_string(2)
    assert mla.status_string(99) == "MLA_ERR_UNKNOWN"


def test_record_width_rejected_before_launch():
    lib = mla.load_library()
    for rb in (0, 400, 431, 433, 367, 369, 512):
        assert lib.mla_nvfp4_cache_write(None, 512, None, 64, None, 1, None, 1, rb, None, None, None) == 2
        assert lib.mla_nvfp4_decode(None, 1, 1, None, 1, rb, None, 0, 64, None, None, 0, 1.0, None,
                                    None, None, None, 0, 0, None, None) == 2


def test_mode_mix_rejected():
    lib = mla.load_library()
    p = ctypes.c_void_p(16)
    # both paged and top-k
    assert lib.mla_nvfp4_decode(p, 1, 1, p, 1, 432, p, 1, 64, p, p, 4, 1.0, p, p, None, p, 1 << 20, 1,
                                None, None) == 1
    # neither
    assert lib.mla_nvfp4_decode(p, 1, 1, p, 1, 432, None, 0, 64, None, None, 0, 1.0, p, p, None, p,
                                1 << 20, 1, None, None) == 1


def test_bad_sizes_rejected():
    lib = mla.load_library()
    p = ctypes.c_void_p(16)
    assert lib.mla_nvfp4_quantize_rows(p, 4, 17, p, p, p, None, None) == 1   # N % 16
    assert lib.mla_nvfp4_quantize_rows(p, 0, 32, p, p, p, None, None) == 0   # empty is a no-op
    assert lib.mla_nvfp4_cache_write(p, 500, p, 64, p, 1, p, 1, 432, p, None, None) == 1  # stride < 512
    assert lib.mla_nvfp4_cache_write(p, 516, p, 64, p, 1, p, 1, 432, p, None, None) == 3  # 1032 B stride
    assert lib.mla_nvfp4_cache_write(ctypes.c_void_p(8), 512, p, 64, p, 1, p, 1, 432, p, None, None) == 3
    assert lib.mla_nvfp4_decode_workspace_size(0, 128, 4) == 0
    assert lib.mla_nvfp4_decode_workspace_size(2, 16, 4) > 0
    # prefill: bad head stride, zero tokens is a no-op
    assert lib.mla_nvfp4_prefill_fused_out(p, p, p, 192 * 2, 100, 192 * 2, 192, 128 * 2, 128, p, 1, 4, 4,
                                           2, 1.0, p, p, p, None, None, None) == 1
    assert lib.mla_nvfp4_prefill_fused_out(p, p, p, 192, 192, 192, 192, 128, 128, p, 1, 0, 0, 1, 1.0, p,
                                           p, p, None, None, None) == 0
    # non-positive softmax scale
    assert lib.mla_nvfp4_prefill_fused_out(p, p, p, 192, 192, 192, 192, 128, 128, p, 1, 4, 4, 1, 0.0, p,
                                           p, p, None, None, None) == 1


def test_decode_split_modes_launch_count_and_workspace():
    # an explicit split count is returned as given, num_splits <= 0 gives
    # the default that fills the SMs (at least 1), invalid sizes give 0
    assert mla.mla_nvfp4_decode_default_splits(4, 128, 5) == 5
    assert mla.mla_nvfp4_decode_default_splits(64, 128, 0) >= 1
    assert mla.mla_nvfp4_decode_default_splits(2, 128, 0) > 1
    assert mla.mla_nvfp4_decode_default_splits(0, 128, 0) == 0
    assert mla.mla_nvfp4_decode_default_splits(4, 0, 0) == 0
    # launches: one split = the decode alone; uniform splits add the merge;
    # a planned call (paged, num_splits <= 0, a workspace) adds the plan
    assert mla.decode_launches(64, 128, 1) == 1
    assert mla.decode_launches(64, 128, 3) == 2
    assert mla.decode_launches(64, 128, 0) == 3
    assert mla.decode_launches(2, 128, 0, paged=False) == 2
    assert mla.decode_launches(2, 128, 0, workspace=False) == 2
    # workspace: none for one split, rows for uniform splits, the plan's
    # tables plus one chunk row per possible item (batch + one per SM pair)
    lib = mla.load_library()
    assert lib.mla_nvfp4_decode_workspace_size(64, 128, 1) == 0
    assert lib.mla_nvfp4_decode_workspace_size(64, 128, 3) >= 64 * 3 * 128 * 2052
    planned = lib.mla_nvfp4_decode_workspace_size(64, 128, 0)
    items = 64 + 76  # batch + one per SM pair (152 SMs assumed when no device is visible)
    assert items * 128 * 2052 <= planned <= items * 128 * 2052 + items * 8 + 64 * 8 + 2048


def test_decode_host_pairs_checked_before_any_copy():
    # every host buffer needs its device buffer: a missing one is rejected on
    # the host, as is a bad record width, before anything is enqueued
    lib = mla.load_library()
    p = ctypes.c_void_p(16)

    def call(q_host=p, q_dev=p, rb=432, out_dev=p, lse_host=None, lse_dev=None):
        return lib.mla_nvfp4_decode_host(q_host, q_dev, 1, 1, p, 1, rb, p, p, 1, 64, p, p, None, None,
                                         0, 1.0, p, p, out_dev, lse_host, lse_dev, p, 1 << 20, 1,
                                         None, None)

    assert call(q_dev=None) == 1
    assert call(out_dev=None) == 1
    assert call(lse_host=p) == 1
    assert call(lse_dev=p) == 1
    assert call(q_dev=None, rb=400) == 2
    assert call(rb=433) == 2


def test_selftest_wait_arguments_checked():
    lib = mla.load_library()
    p = ctypes.c_void_p(16)
    assert lib.mla_nvfp4_selftest_wait(None, 50_000_000, None, None) == 1   # no error word
    assert lib.mla_nvfp4_selftest_wait(p, 0, None, None) == 1               # limit below 1 us
    assert lib.mla_nvfp4_selftest_wait(p, 2_000_000_000, None, None) == 1   # limit above 1 s


def test_extension_entry_points_reject_bad_arguments():
    """The chunked-context, fake-quant and NVFP4-query entry points check
    their arguments on the host (status codes: 1 invalid, 2 record width,
    3 alignment) before any launch; empty work is a no-op."""
    lib = mla.load_library()
    p = ctypes.c_void_p(16)
    odd = ctypes.c_void_p(8)
    # gather: record width, negative count, empty, misaligned cache
    assert lib.mla_nvfp4_gather_latent(p, 10, 400, p, p, 4, p, p, None, None) == 2
    assert lib.mla_nvfp4_gather_latent(p, 10, 432, p, p, -1, p, p, None, None) == 1
    assert lib.mla_nvfp4_gather_latent(p, 10, 432, p, p, 0, p, p, None, None) == 0
    assert lib.mla_nvfp4_gather_latent(odd, 10, 432, p, p, 4, p, p, None, None) == 3
    # partial prefill: no heads, null lse, short head stride, misaligned out, empty
    H = 2
    args = [p, p, p, H * 192, 192, H * 192, 192, H * 128, 128, p, None, 1, 4, 0, 4, H, 0.1, p, p, None, None]
    bad = list(args); bad[15] = 0
    assert lib.mla_nvfp4_prefill_partial(*bad) == 1
    bad = list(args); bad[18] = None
    assert lib.mla_nvfp4_prefill_partial(*bad) == 1
    bad = list(args); bad[4] = 100
    assert lib.mla_nvfp4_prefill_partial(*bad) == 1
    bad = list(args); bad[17] = odd
    assert lib.mla_nvfp4_prefill_partial(*bad) == 3
    bad = list(args); bad[12] = 0; bad[11] = 0
    assert lib.mla_nvfp4_prefill_partial(*bad) == 0
    # merge: no parts, null scale, empty
    assert lib.mla_nvfp4_merge_fused_out(p, p, 0, 4, H, p, p, p, None, None, None) == 1
    assert lib.mla_nvfp4_merge_fused_out(p, p, 2, 4, H, None, p, p, None, None, None) == 1
    assert lib.mla_nvfp4_merge_fused_out(p, p, 2, 0, H, p, p, p, None, None, None) == 0
    # operand fake quant: a missing global scale, a short v stride
    q = [p, p, p, H * 192, 192, H * 192, 192, H * 128, 128, p, 1, 4, 4, H, p, p, p, p, p, p, None, None]
    bad = list(q); bad[16] = None
    assert lib.mla_nvfp4_prefill_qdq(*bad) == 1
    bad = list(q); bad[7] = 100
    assert lib.mla_nvfp4_prefill_qdq(*bad) == 1
    # fake-quant prefill: sparse24 must be 0 or 1, global scales required
    f = [p, p, p, p, 1, 4, 4, H, 0.1, p, p, p, 2, p, p, p, None, None, None]
    assert lib.mla_nvfp4_prefill_fakequant(*f) == 1
    f[12] = 0
    f[10] = None
    assert lib.mla_nvfp4_prefill_fakequant(*f) == 1
    # NVFP4-query decode: the query's global scale is required
    assert lib.mla_nvfp4_decode_q4(p, 1, 1, p, 1, 432, p, 1, 64, p, None, 0, 1.0, p, None, p, None, None, 0, 1,
                                   None, None) == 1
