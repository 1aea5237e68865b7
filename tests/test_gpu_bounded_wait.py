"""Failure detection without a GPU fault: a wait that is never satisfied must
give up after its limit, report DEV_TIMEOUT through the status word and leave
the context usable (tvl_selftest_bounded_wait runs the same bounded mbarrier
wait the kernels use, on a barrier nothing arrives at)."""
import time

import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status, assert_close

pytestmark = pytest.mark.gpu


def test_unsatisfied_wait_times_out_and_the_context_survives():
    tvl.get_device_status()                              # start from a clean word
    t0 = time.time()
    tvl.selftest_bounded_wait()
    bits = tvl.get_device_status()                       # synchronises
    elapsed = time.time() - t0
    assert bits & tvl.DEV_TIMEOUT
    assert elapsed < 30.0
    # the context still works: a decode step right after matches the oracle
    wl = W.named("tiny")
    t = W.to_device(wl, DEV)
    out = torch.empty(tuple(wl.q.shape), dtype=torch.float32, device=DEV)
    tvl.paged_decode_step(out, t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                          t["block_tables"], t["context_lens"], wl.scale)
    torch.cuda.synchronize()
    kw, vw = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    ref = oracle.decode(wl.q, kw, vw, wl.block_tables, wl.context_lens, wl.scale)
    assert_close(out.double().cpu().numpy(), ref, "after the timeout")
    assert_clean_status()
