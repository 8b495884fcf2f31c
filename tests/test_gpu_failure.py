"""Failure detection on the GPU without a fault: a bounded wait on a barrier
nothing arrives on runs out, the kernel ends with MLA_DEVERR_TIMEOUT in the
error word, the CTA's other (2-second) wait ends through the abort flag,
and the context stays usable for the library's kernels afterwards."""
import time

import numpy as np
import pytest
import torch

import mla_attention_nvfp4_gb300 as mla
from mla_attention_nvfp4_gb300 import workloads
from tests.helpers import oracle_cache, oracle_gs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]
DEV = "cuda:0"


def test_wait_timeout_is_flagged_and_aborts_the_cta():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    elapsed = torch.zeros(2, dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mla.mla_nvfp4_selftest_wait(err, 50_000_000, elapsed)  # 50 ms
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert int(err.item()) == mla.DEVERR_TIMEOUT
    short_ns, long_ns = elapsed.cpu().tolist()
    assert 50_000_000 <= short_ns < 1_000_000_000   # ran to its limit, then gave up
    assert 0 < long_ns < 1_000_000_000              # ended by the abort flag, far inside its 2 s
    assert wall < 1.5
    # the context still runs the library's kernels: a cache write after the
    # timed-out kernel is bit-exact
    w = workloads.decode_tiny(record_bytes=432)
    gs = oracle_gs(w.kv_c)
    cache = torch.zeros((w.num_slots, 432), dtype=torch.uint8, device=DEV)
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.mla_nvfp4_cache_write(w.kv_c.to(DEV), w.k_pe.to(DEV), w.slot_mapping.to(DEV), cache,
                              torch.tensor([gs], device=DEV), err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    assert np.array_equal(cache.cpu().numpy(), oracle_cache(w, gs))
