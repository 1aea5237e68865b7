"""tvl_paged_attention_decode_noalloc, the decode for callers that cannot
allocate device memory at the call site (an engine whose device memory all
went to its KV pool, a plugin interface that passes only input and output
pointers, a thread that must not take the driver's allocation lock).  It is
called here through the C ABI on two calls in a row that share its built-in
scratch array.  Each must give exactly the bits of tvl_paged_attention_decode
with a caller workspace (the same kernels run; only where the split-K records
live differs) and agree with the CPU oracle within the parity tolerance.
This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_close, oracle_decode

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    from paged_kv_cache_198_gb300 import _build

    lib = ctypes.CDLL(_build.build())
    fn = lib.tvl_paged_attention_decode_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_float, I, P]
    fn.restype = I
    return fn


def _run_noalloc(fn, wl, t, part):
    s, hq, d = wl.q.shape
    out = torch.full((s, hq, d), float("nan"), dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(t["q"].data_ptr()),
            ctypes.c_void_p(t["k_cache"].data_ptr()), ctypes.c_void_p(t["v_cache"].data_ptr()),
            ctypes.c_void_p(t["block_tables"].data_ptr()),
            ctypes.c_void_p(t["context_lens"].data_ptr()), s, hq, wl.num_kv_heads, d,
            wl.block_size, wl.num_blocks, wl.max_blocks_per_seq, wl.scale, part, stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def _run_with_workspace(wl, t, part):
    out = torch.empty(tuple(wl.q.shape), dtype=torch.float32, device=DEV)
    tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                               t["context_lens"], wl.scale, partition_size=part)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


# partition 0: balanced split (2 records per SM); 1024: fixed windows, 4 per
# sequence of up to 4096 tokens (64 * 4 records of 32 heads = 2.2 MB).
@pytest.mark.parametrize("part", [0, 1024])
def test_noalloc_matches_workspace_decode_two_calls_in_a_row(part):
    fn = _noalloc_fn()
    first = W.named("llama1b_decode", 0)
    second = W.make_decode(911, [3000, 17, 700, 1, 4095, 2048], block_size=16,
                           max_blocks_per_seq=256)
    for wl in (first, second):
        t = W.to_device(wl, DEV)              # the cache as drawn: no write this step
        got = _run_noalloc(fn, wl, t, part)
        ws_out = _run_with_workspace(wl, t, part)
        assert np.array_equal(got, ws_out), "differs from the workspace decode"
        assert_close(got, oracle_decode(wl, write=False), f"no-alloc P{part}")


def test_noalloc_rejects_scratch_beyond_its_limit():
    fn = _noalloc_fn()
    wl = W.make_decode(912, [64, 64], block_size=16, max_blocks_per_seq=8192, write=False)
    t = W.to_device(wl, DEV)
    s, hq, d = wl.q.shape
    out = torch.empty((s, hq, d), dtype=torch.float32, device=DEV)
    # 16-token windows over 8192 blocks: 2 * 8192 records of 32 heads -> ~138 MB > 4 MiB
    rc = fn(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(t["q"].data_ptr()),
            ctypes.c_void_p(t["k_cache"].data_ptr()), ctypes.c_void_p(t["v_cache"].data_ptr()),
            ctypes.c_void_p(t["block_tables"].data_ptr()),
            ctypes.c_void_p(t["context_lens"].data_ptr()), s, hq, wl.num_kv_heads, d,
            wl.block_size, wl.num_blocks, wl.max_blocks_per_seq, wl.scale, 16,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == tvl.ERR_WORKSPACE
