"""GPU parity of the one-call decode step (tvl_paged_decode_step): the new
token of each sequence is written at position context_lens[s] - 1, then the
decode runs over the updated cache [tiny-vllm README, curriculum "Why KV cache
exists", "Paged KV cache", "Paged Attention"; nano-vLLM guide ch. 4, ch. 5].
The cache must equal the oracle's write bit for bit, the output must match the
oracle's decode within the parity tolerance and equal, bit for bit, the
two-call path (tvl_paged_kv_write, then tvl_paged_attention_decode)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status, assert_close, bits_of

pytestmark = pytest.mark.gpu


def _full_new(wl, gen):
    """k_new / v_new with one row per sequence (rows of ctx-0 sequences are
    arbitrary and never written)."""
    s = wl.q.shape[0]
    kn = torch.randn(s, wl.num_kv_heads, wl.head_dim, generator=gen).to(torch.bfloat16)
    vn = torch.randn(s, wl.num_kv_heads, wl.head_dim, generator=gen).to(torch.bfloat16)
    rows = [i for i in range(s) if int(wl.context_lens[i]) > 0]
    kn[rows] = wl.k_new
    vn[rows] = wl.v_new
    return kn, vn


CASES = [
    # (context lengths, Hq, Hkv, bs, partition)
    ([40, 700, 1500, 3, 1, 4096, 2048, 17], 32, 8, 16, 0),
    ([40, 700, 1500, 3, 1, 4096, 2048, 17], 32, 8, 16, 256),
    ([300, 1, 33, 2000, 64, 65], 32, 8, 32, 0),
    ([900, 5, 1024, 2500], 64, 8, 16, 0),       # G = 8: two KV-head groups per sequence
    ([129, 7, 3000], 8, 8, 16, 0),              # G = 1
    ([129, 7, 3000, 0, 44], 16, 8, 32, 512),    # G = 2, an empty sequence
    ([1, 64, 65, 700, 2047], 32, 8, 64, 0),     # blocks of 64
    ([128, 129, 5, 1000], 64, 8, 128, 256),     # G = 8, blocks of 128, fixed windows
    # more windows than SMs: the windows are walked by a persistent grid
    ([0 if i % 7 == 0 else (i * 37) % 300 + 1 for i in range(200)], 32, 8, 16, 64),
    ([0 if i % 5 == 0 else (i * 53) % 400 + 1 for i in range(120)], 64, 8, 16, 32),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_step_matches_oracle_and_two_calls(case):
    ctx, hq, hkv, bs, part = CASES[case]
    wl = W.make_decode(500 + case, ctx, num_q_heads=hq, num_kv_heads=hkv, block_size=bs,
                       partition_size=part)
    gen = torch.Generator().manual_seed(600 + case)
    kn, vn = _full_new(wl, gen)
    t = W.to_device(wl, DEV)
    s, _, d = wl.q.shape
    # fused step
    k1, v1 = t["k_cache"].clone(), t["v_cache"].clone()
    out1 = torch.empty(s, hq, d, dtype=torch.float32, device=DEV)
    tvl.paged_decode_step(out1, t["q"], kn.to(DEV), vn.to(DEV), k1, v1, t["block_tables"],
                          t["context_lens"], wl.scale, partition_size=part)
    # two calls
    k2, v2 = t["k_cache"].clone(), t["v_cache"].clone()
    out2 = torch.empty_like(out1)
    if wl.slot_mapping.numel():
        tvl.paged_kv_write(t["k_new"], t["v_new"], k2, v2, t["slot_mapping"])
    tvl.paged_attention_decode(out2, t["q"], k2, v2, t["block_tables"], t["context_lens"],
                               wl.scale, partition_size=part)
    torch.cuda.synchronize()
    kw, vw = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    assert np.array_equal(bits_of(k1), kw)
    assert np.array_equal(bits_of(v1), vw)
    assert torch.equal(out1, out2)
    ref = oracle.decode(wl.q, kw.reshape(wl.k_cache.shape), vw.reshape(wl.v_cache.shape),
                        wl.block_tables, wl.context_lens, wl.scale)
    assert_close(out1.double().cpu().numpy(), ref, "decode step")
    assert_clean_status()


def test_decode_step_bad_last_block_is_reported_and_not_written():
    wl = W.make_decode(520, [100, 200], num_q_heads=32, num_kv_heads=8, block_size=16)
    t = W.to_device(wl, DEV)
    tables = t["block_tables"].clone()
    last = (200 - 1) // 16
    tables[1, last] = wl.num_blocks + 5                 # out of range
    k1, v1 = t["k_cache"].clone(), t["v_cache"].clone()
    out = torch.empty(2, 32, 64, dtype=torch.float32, device=DEV)
    tvl.paged_decode_step(out, t["q"], t["k_new"], t["v_new"], k1, v1, tables,
                          t["context_lens"], wl.scale)
    torch.cuda.synchronize()
    assert tvl.get_device_status() & tvl.DEV_BAD_BLOCK_ID
    # sequence 0's row written, nothing else changed
    kw, _ = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new[:1], wl.v_new[:1],
                            wl.slot_mapping[:1])
    assert np.array_equal(bits_of(k1), kw)


@pytest.mark.parametrize("name", ["llama1b_decode", "continuous_batch"])
def test_decode_step_full_size_as_benchmarked(name):
    """The benchmarked call at full size: the Llama-1B-shaped batch and the
    continuous batch, balanced split, one new token per sequence."""
    wl = W.named(name, 0)
    assert wl.k_new.shape[0] == wl.q.shape[0]
    t = W.to_device(wl, DEV)
    s, hq, d = wl.q.shape
    out = torch.empty(s, hq, d, dtype=torch.float32, device=DEV)
    tvl.paged_decode_step(out, t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                          t["block_tables"], t["context_lens"], wl.scale)
    torch.cuda.synchronize()
    kw, vw = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    assert np.array_equal(bits_of(t["k_cache"]), kw)
    assert np.array_equal(bits_of(t["v_cache"]), vw)
    ref = oracle.decode(wl.q, kw.reshape(wl.k_cache.shape), vw.reshape(wl.v_cache.shape),
                        wl.block_tables, wl.context_lens, wl.scale)
    assert_close(out.double().cpu().numpy(), ref, name)
    assert_clean_status()
