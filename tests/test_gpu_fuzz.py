"""Seeded random sweep of shapes against the oracle: decode (every split mode)
and the one-call decode step over random GQA groups, block sizes, context
lengths (empty, single-token, block-aligned, ragged) and batch sizes; prefill
over random prefixes and chunk lengths.  Each case is small enough for the
oracle and draws its own inputs from its seed."""
import random

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status, assert_close, bits_of

pytestmark = pytest.mark.gpu

GROUPS = [(8, 8), (16, 8), (32, 8), (64, 8), (4, 4), (8, 2), (32, 4), (16, 16)]


def _ctx_list(rng, n, cap):
    out = []
    for _ in range(n):
        kind = rng.random()
        if kind < 0.1:
            out.append(0)
        elif kind < 0.2:
            out.append(1)
        elif kind < 0.35:
            out.append(rng.choice([16, 32, 64, 128, 512]))
        else:
            out.append(rng.randint(2, cap))
    if all(c == 0 for c in out):
        out[0] = 5
    return out


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_decode_and_step(seed):
    rng = random.Random(9000 + seed)
    hq, hkv = rng.choice(GROUPS)
    bs = rng.choice([16, 32, 16, 32, 64, 128])
    ctx = _ctx_list(rng, rng.randint(1, 40), rng.choice([64, 700, 3000]))
    part = rng.choice([0, 0, bs, 4 * bs, max(bs, 256 // bs * bs), 1024])
    wl = W.make_decode(9100 + seed, ctx, num_q_heads=hq, num_kv_heads=hkv, block_size=bs)
    t = W.to_device(wl, DEV)
    s, _, d = wl.q.shape
    # two calls: write, then decode
    if wl.slot_mapping.numel():
        tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.empty(s, hq, d, dtype=torch.float32, device=DEV)
    tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                               t["context_lens"], wl.scale, partition_size=part)
    torch.cuda.synchronize()
    kw, vw = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    ref = oracle.decode(wl.q, kw.reshape(wl.k_cache.shape), vw.reshape(wl.v_cache.shape),
                        wl.block_tables, wl.context_lens, wl.scale)
    assert_close(out.double().cpu().numpy(), ref, f"seed {seed} decode")
    assert np.array_equal(bits_of(t["k_cache"]), kw)
    # the one-call step on fresh caches gives the same bits
    t2 = W.to_device(wl, DEV)
    kn = torch.zeros(s, hkv, d, dtype=torch.bfloat16)
    vn = torch.zeros(s, hkv, d, dtype=torch.bfloat16)
    rows = [i for i in range(s) if ctx[i] > 0]
    kn[rows], vn[rows] = wl.k_new, wl.v_new
    out2 = torch.empty_like(out)
    tvl.paged_decode_step(out2, t2["q"], kn.to(DEV), vn.to(DEV), t2["k_cache"], t2["v_cache"],
                          t2["block_tables"], t2["context_lens"], wl.scale, partition_size=part)
    torch.cuda.synchronize()
    assert torch.equal(out2, out)
    assert np.array_equal(bits_of(t2["k_cache"]), kw)
    assert np.array_equal(bits_of(t2["v_cache"]), vw)
    assert_clean_status()


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_prefill(seed):
    rng = random.Random(9500 + seed)
    hq, hkv = rng.choice(GROUPS)
    bs = rng.choice([16, 32, 64, 128])
    n = rng.randint(1, 6)
    prefix = [rng.choice([0, 1, rng.randint(0, 600), 128, 255]) for _ in range(n)]
    lq = [rng.choice([1, 2, rng.randint(1, 300), 128, 129]) for _ in range(n)]
    wl = W.make_prefill(9600 + seed, prefix, lq, num_q_heads=hq, num_kv_heads=hkv,
                        block_size=bs)
    t = W.to_device(wl, DEV)
    tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.full(tuple(wl.q.shape), float("nan"), dtype=torch.float32, device=DEV)
    tvl.paged_attention_prefill(out, t["q"], t["query_start_loc"], t["k_cache"], t["v_cache"],
                                t["block_tables"], t["context_lens"], wl.scale, wl.max_q_len)
    torch.cuda.synchronize()
    kw, vw = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    ref = oracle.prefill(wl.q, wl.query_start_loc, kw.reshape(wl.k_cache.shape),
                         vw.reshape(wl.v_cache.shape), wl.block_tables, wl.context_lens,
                         wl.scale)
    assert_close(out.double().cpu().numpy(), ref, f"seed {seed} prefill")
    assert_clean_status()
