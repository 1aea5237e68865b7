"""Prefix caching: several sequences' block tables name the same physical
blocks for a shared prefix [nano-vLLM guide ch. 7 "Prefix Caching"].  The
kernels read through the tables, so sharing needs no change to them; these
tests pin that contract on decode and prefill."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status, assert_close, gpu_decode, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("part", [0, 64])
def test_decode_with_shared_prefix_blocks(part):
    wl = W.make_decode(801, [700, 650, 900, 513], num_q_heads=32, num_kv_heads=8,
                       block_size=16)
    W.share_prefix(wl, 32)                    # 512 shared tokens
    got, _ = gpu_decode(wl, partition_size=part)
    assert_close(got, oracle_decode(wl), f"shared prefix P{part}")
    assert_clean_status()


def test_decode_identical_sequences_on_shared_blocks_agree():
    wl = W.make_decode(802, [300, 300, 300], num_q_heads=8, num_kv_heads=2, block_size=16,
                       write=False)
    W.share_prefix(wl, 18)                    # everything but the last partial block
    wl.block_tables[1:, 18] = wl.block_tables[0, 18]
    wl.q[1:] = wl.q[0]
    # a single pass per sequence (window >= context) gives each sequence the
    # same summation order, so equal inputs must give bit-equal outputs
    got, _ = gpu_decode(wl, partition_size=4096, write=False)
    assert np.array_equal(got[0], got[1]) and np.array_equal(got[0], got[2])


def test_prefill_over_shared_prefix():
    wl = W.make_prefill(803, [256, 256, 256], [64, 100, 1], num_q_heads=8, num_kv_heads=2,
                        block_size=16)
    W.share_prefix(wl, 16)                    # the 256-token prefix is one set of blocks
    t = W.to_device(wl, DEV)
    tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.full(tuple(wl.q.shape), float("nan"), dtype=torch.float32, device=DEV)
    tvl.paged_attention_prefill(out, t["q"], t["query_start_loc"], t["k_cache"], t["v_cache"],
                                t["block_tables"], t["context_lens"], wl.scale, wl.max_q_len)
    torch.cuda.synchronize()
    kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    ref = oracle.prefill(wl.q, wl.query_start_loc, kc, vc, wl.block_tables, wl.context_lens,
                         wl.scale)
    assert_close(out.double().cpu().numpy(), ref, "prefill shared prefix")
