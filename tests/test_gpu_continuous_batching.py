"""A continuous-batching trace driven by the host block allocator
[nano-vLLM guide ch. 5 "The Scheduler", ch. 7 "Prefix Caching"]: sequences
arrive with prompts, fork (sharing their prefix blocks), decode one token per
step and finish; the allocator hands out slots and copy-on-write block copies,
the GPU runs copy_blocks + paged_kv_write + decode.  A CPU mirror of the cache
gets the same copies and writes through the oracle; every step's decode must
match the oracle, and the caches must stay bit-identical to the mirror."""
import random

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from gpu_common import DEV, assert_clean_status, assert_close, bits_of

pytestmark = pytest.mark.gpu

NB, BS, HQ, HKV, D, MB = 400, 16, 32, 8, 64, 64
SCALE = 0.125


def _rand(gen, *shape):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("part", [0, 128])
def test_continuous_batching_trace(seed, part):
    rng = random.Random(seed)
    gen = torch.Generator().manual_seed(1234 + seed)
    alloc = tvl.BlockAllocator(NB, BS)
    k_dev = _rand(gen, NB, BS, HKV, D).to(DEV)
    v_dev = _rand(gen, NB, BS, HKV, D).to(DEV)
    k_mir = bits_of(k_dev).copy()
    v_mir = bits_of(v_dev).copy()
    live = []

    def write(seq_slots, kn, vn):
        nonlocal k_mir, v_mir
        slots = torch.from_numpy(np.concatenate(seq_slots).astype(np.int32))
        tvl.paged_kv_write(kn.to(DEV), vn.to(DEV), k_dev, v_dev, slots.to(DEV))
        k_mir, v_mir = oracle.kv_write(k_mir, v_mir, kn, vn, slots)

    def run_copies():
        src, dst = alloc.take_copies()
        if src.size:
            tvl.copy_blocks(k_dev, v_dev, torch.from_numpy(src).to(DEV),
                            torch.from_numpy(dst).to(DEV))
            k_mir[dst] = k_mir[src]
            v_mir[dst] = v_mir[src]

    copies_seen = 0
    for step in range(14):
        # arrivals with a prompt written in one go
        for _ in range(rng.randint(0, 3) if step else 4):
            if len(live) >= 24:
                break
            s = alloc.new_sequence()
            n = rng.randint(1, 300)
            try:
                slots = alloc.append(s, n)
            except tvl.TvlError:
                alloc.free(s)
                continue
            live.append(s)
            write([slots], _rand(gen, n, HKV, D), _rand(gen, n, HKV, D))
        # forks share the parent's blocks
        if live and rng.random() < 0.6:
            live.append(alloc.fork(rng.choice(live)))
        # one decode step: every live sequence appends one token
        slots = []
        for s in live:
            slots.append(alloc.append(s, 1))
        src_dst = alloc.take_copies()
        copies_seen += src_dst[0].size
        if src_dst[0].size:
            src, dst = src_dst
            tvl.copy_blocks(k_dev, v_dev, torch.from_numpy(src).to(DEV),
                            torch.from_numpy(dst).to(DEV))
            k_mir[dst] = k_mir[src]
            v_mir[dst] = v_mir[src]
        t = len(live)
        write(slots, _rand(gen, t, HKV, D), _rand(gen, t, HKV, D))
        run_copies()
        tables, ctx = alloc.build_tables(live, MB)
        q = _rand(gen, t, HQ, D)
        out = torch.empty(t, HQ, D, dtype=torch.float32, device=DEV)
        tvl.paged_attention_decode(out, q.to(DEV), k_dev, v_dev,
                                   torch.from_numpy(tables).to(DEV),
                                   torch.from_numpy(ctx).to(DEV), SCALE, partition_size=part)
        torch.cuda.synchronize()
        ref = oracle.decode(q, k_mir.reshape(NB, BS, HKV, D), v_mir.reshape(NB, BS, HKV, D),
                            tables, ctx, SCALE)
        assert_close(out.double().cpu().numpy(), ref, f"step {step}")
        # departures
        for s in list(live):
            if rng.random() < 0.15:
                alloc.free(s)
                live.remove(s)
    assert np.array_equal(bits_of(k_dev), k_mir)
    assert np.array_equal(bits_of(v_dev), v_mir)
    assert copies_seen > 0, "the trace never exercised copy-on-write"
    assert_clean_status()
    for s in live:
        alloc.free(s)
    assert alloc.stats()["free_blocks"] == NB


def test_copy_blocks_bit_exact_and_reports_bad_ids():
    gen = torch.Generator().manual_seed(9)
    kc = _rand(gen, 10, BS, HKV, D).to(DEV)
    vc = _rand(gen, 10, BS, HKV, D).to(DEV)
    k0, v0 = kc.clone(), vc.clone()
    src = torch.tensor([1, 4, 7], dtype=torch.int32, device=DEV)
    dst = torch.tensor([2, 5, 12], dtype=torch.int32, device=DEV)   # 12 is out of range
    tvl.copy_blocks(kc, vc, src, dst)
    assert tvl.get_device_status() & tvl.DEV_BAD_BLOCK_ID
    exp_k, exp_v = k0.clone(), v0.clone()
    exp_k[2], exp_v[2] = k0[1], v0[1]
    exp_k[5], exp_v[5] = k0[4], v0[4]
    assert torch.equal(kc.view(torch.int16), exp_k.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), exp_v.view(torch.int16))
