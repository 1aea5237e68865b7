"""GPU parity of the paged KV write and PagedAttention decode (all split
modes) against the CPU oracle, element by element, plus the invariants the
method guarantees (physical placement, determinism, over-read poisoning)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import (DEV, assert_clean_status, assert_close, bits_of, gpu_decode,
                        oracle_caches, oracle_decode)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ KV write


@pytest.mark.parametrize("name", ["tiny", "continuous_batch", "chunked_prefill"])
def test_kv_write_bit_exact(name):
    wl = W.named(name)
    t = W.to_device(wl, DEV)
    tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    torch.cuda.synchronize()
    kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    assert np.array_equal(bits_of(t["k_cache"]), kc)
    assert np.array_equal(bits_of(t["v_cache"]), vc)
    assert_clean_status()


def test_kv_write_skips_negative_slots_and_reports_out_of_range():
    gen = torch.Generator().manual_seed(3)
    nb, bs, hkv, d = 4, 16, 8, 64
    kc = torch.randn(nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    kn = torch.randn(5, hkv, d, generator=gen).to(torch.bfloat16)
    vn = torch.randn(5, hkv, d, generator=gen).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 63, nb * bs, 17], dtype=torch.int32)   # one past the pool
    gk, gv = kc.to(DEV), vc.to(DEV)
    tvl.paged_kv_write(kn.to(DEV), vn.to(DEV), gk, gv, slots.to(DEV))
    bits = tvl.get_device_status()
    assert bits & tvl.DEV_BAD_SLOT
    keep = torch.tensor([True, False, True, False, True])
    ek, ev = oracle.kv_write(kc, vc, kn[keep], vn[keep], slots[keep])
    assert np.array_equal(bits_of(gk), ek)
    assert np.array_equal(bits_of(gv), ev)


def test_kv_write_zero_tokens_is_a_no_op():
    kc = torch.zeros(2, 16, 8, 64, dtype=torch.bfloat16, device=DEV)
    e = torch.empty(0, 8, 64, dtype=torch.bfloat16, device=DEV)
    tvl.paged_kv_write(e, e, kc, kc, torch.empty(0, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert int(kc.abs().sum()) == 0


# ------------------------------------------------------- decode, named configs


@pytest.mark.parametrize("replica", [0, 1, 2])
@pytest.mark.parametrize("part", [0, 16, 32, 4096])
def test_decode_tiny(replica, part):
    wl = W.named("tiny", replica)
    got, _ = gpu_decode(wl, partition_size=part)
    assert_close(got, oracle_decode(wl), f"tiny r{replica} P{part}")
    assert_clean_status()


@pytest.mark.parametrize("replica", [0, 1, 2])
@pytest.mark.parametrize("part", [0, 512])
def test_decode_llama1b(replica, part):
    wl = W.named("llama1b_decode", replica)
    got, _ = gpu_decode(wl, partition_size=part)
    assert_close(got, oracle_decode(wl), f"llama1b r{replica} P{part}")
    assert_clean_status()


@pytest.mark.parametrize("replica", [0, 1, 2])
def test_decode_continuous_batch(replica):
    wl = W.named("continuous_batch", replica)
    got, _ = gpu_decode(wl, partition_size=0)
    assert_close(got, oracle_decode(wl), f"continuous r{replica}")
    assert_clean_status()


@pytest.mark.parametrize("replica", [0, 1, 2])
def test_decode_long_splitk(replica):
    """8 sequences of 32k-128k tokens: 512-token windows merged by
    log-sum-exp, and the balanced split, on the same written cache."""
    wl = W.named("long_splitk", replica)
    ref = oracle_decode(wl)
    got, t = gpu_decode(wl, partition_size=512)
    assert_close(got, ref, f"long r{replica} P512")
    got, _ = gpu_decode(wl, partition_size=0, write=False, tensors=t)
    assert_close(got, ref, f"long r{replica} balanced")
    assert_clean_status()


# ------------------------------------------------------------- random shapes


CASES = [
    # (ctx list, Hq, Hkv, bs)
    ([1, 2, 15, 16, 17, 31, 33, 100], 4, 2, 16),
    ([5, 300, 47, 1000, 1], 8, 8, 16),     # MHA-like G = 1
    ([129, 64, 640, 3], 16, 8, 32),        # G = 2, bs 32
    ([700, 250, 1], 32, 4, 16),            # G = 8
    ([77, 513, 2049], 32, 16, 16),         # 16 KV heads: two KV-head groups
    ([0, 40, 0, 9], 8, 2, 32),             # empty contexts give zeros
    ([1, 63, 64, 65, 700, 2048], 32, 8, 64),   # blocks of 64: two stages each
    ([1, 127, 128, 129, 900], 16, 4, 128),     # blocks of 128: four stages each
    ([300, 5, 1500], 64, 8, 128),              # G = 8 (two KV-head groups), blocks of 128
]


@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8)])
def test_decode_window_walk_with_empty_sequences(hq, hkv):
    """More windows than SMs: a persistent grid walks the fixed windows, a
    segment and a record each (the merge then zeroes the empty sequences,
    which no CTA owns)."""
    gen = np.random.default_rng(77)
    ctx = [int(c) for c in gen.integers(0, 600, 300)]
    for i in range(0, 300, 9):
        ctx[i] = 0
    wl = W.make_decode(777, ctx, num_q_heads=hq, num_kv_heads=hkv, block_size=16)
    got, _ = gpu_decode(wl, partition_size=64)
    ref = oracle_decode(wl)
    assert_close(got, ref, f"window walk G{hq // hkv}")
    zero = np.array(ctx) == 0
    assert np.array_equal(got[zero], np.zeros_like(got[zero]))
    assert_clean_status()


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("part", [0, 32, 256])
def test_decode_random_shapes(case, part):
    ctx, hq, hkv, bs = CASES[case]
    if part % bs:
        part = bs                   # windows must be whole blocks: one block each
    wl = W.make_decode(500 + case, ctx, num_q_heads=hq, num_kv_heads=hkv, block_size=bs)
    got, _ = gpu_decode(wl, partition_size=part)
    ref = oracle_decode(wl)
    assert_close(got, ref, f"case {case} P{part}")
    zero = np.array(ctx) == 0
    if zero.any():
        assert np.array_equal(got[zero], np.zeros_like(got[zero]))
    assert_clean_status()


def test_decode_many_short_sequences_balanced():
    gen = torch.Generator().manual_seed(77)
    ctx = torch.randint(1, 40, (1000,), generator=gen).tolist()
    wl = W.make_decode(78, ctx, num_q_heads=32, num_kv_heads=8, block_size=16)
    got, _ = gpu_decode(wl, partition_size=0)
    assert_close(got, oracle_decode(wl), "1000 short")
    assert_clean_status()


@pytest.mark.parametrize("num_seqs,max_ctx", [(1500, 300), (4096, 64)])
def test_decode_large_batches_balanced(num_seqs, max_ctx):
    """Balanced batches beyond 512 sequences, where the merge reads the
    per-sequence block offsets the decode recorded instead of scanning every
    length: 1500 sequences of up to 300 tokens (many cut between CTAs) and
    4096 short ones, against the oracle."""
    gen = torch.Generator().manual_seed(num_seqs)
    ctx = torch.randint(1, max_ctx + 1, (num_seqs,), generator=gen).tolist()
    wl = W.make_decode(79 + num_seqs, ctx, num_q_heads=32, num_kv_heads=8, block_size=16)
    got, _ = gpu_decode(wl, partition_size=0)
    assert_close(got, oracle_decode(wl), f"{num_seqs} sequences")
    assert_clean_status()


# ------------------------------------------------------------------ invariants


@pytest.mark.parametrize("part", [0, 512])
def test_decode_bit_identical_under_block_permutation(part):
    wl = W.named("llama1b_decode", 0)
    base, _ = gpu_decode(wl, partition_size=part, write=False)
    gen = torch.Generator().manual_seed(99)
    perm = torch.randperm(wl.num_blocks, generator=gen)
    kc2 = torch.empty_like(wl.k_cache)
    vc2 = torch.empty_like(wl.v_cache)
    kc2[perm] = wl.k_cache
    vc2[perm] = wl.v_cache
    t2 = wl.block_tables.clone()
    valid = t2 >= 0
    t2[valid] = perm[t2[valid].long()].to(torch.int32)
    wl.k_cache, wl.v_cache, wl.block_tables = kc2, vc2, t2
    moved, _ = gpu_decode(wl, partition_size=part, write=False)
    assert np.array_equal(base, moved)


def test_decode_deterministic():
    wl = W.named("continuous_batch", 0)
    a, t = gpu_decode(wl, partition_size=0)
    b, _ = gpu_decode(wl, partition_size=0, write=False, tensors=t)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("part", [0, 64])
def test_decode_poisoned_unused_slots(part):
    wl = W.make_decode(601, [3, 17, 40, 129, 250], num_q_heads=32, num_kv_heads=8,
                       block_size=32)
    W.poison_unused(wl, 1.0e4)
    got, _ = gpu_decode(wl, partition_size=part)
    assert_close(got, oracle_decode(wl), "poisoned")


def test_decode_context_one_returns_v():
    wl = W.make_decode(602, [1, 1, 1], num_q_heads=8, num_kv_heads=2, block_size=16,
                       write=False)
    got, _ = gpu_decode(wl, partition_size=0, write=False)
    for s in range(3):
        blk = int(wl.block_tables[s, 0])
        for h in range(8):
            v = wl.v_cache[blk, 0, h // 4].double().numpy()
            np.testing.assert_allclose(got[s, h], v, rtol=1e-6, atol=1e-6)


def test_decode_bad_block_id_is_reported_not_faulted():
    wl = W.make_decode(603, [40, 20], num_q_heads=8, num_kv_heads=2, block_size=16,
                       write=False)
    wl.block_tables[0, 1] = wl.num_blocks + 5
    gpu_decode(wl, partition_size=0, write=False)
    bits = tvl.get_device_status()
    assert bits & tvl.DEV_BAD_BLOCK_ID
    assert_clean_status()


def test_decode_workspace_too_small_is_rejected():
    wl = W.named("tiny")
    t = W.to_device(wl, DEV)
    out = torch.empty(wl.q.shape, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tvl.TvlError) as ei:
        tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], wl.scale, partition_size=0, workspace=ws)
    assert ei.value.status == tvl.ERR_WORKSPACE


@pytest.mark.parametrize("part", [0, 256])
def test_decode_ignores_workspace_contents(part):
    """Every partial record the merge reads is written by the same call's
    decode first, so a workspace full of arbitrary bytes gives the same
    result as a zeroed one, and reusing it for a second call changes
    nothing."""
    wl = W.make_decode(77, [5000, 17, 3000, 1, 700, 4096], num_q_heads=32, num_kv_heads=8,
                       block_size=16)
    t = W.to_device(wl, DEV)
    s, hq, d = wl.q.shape
    size = tvl.paged_attention_decode_workspace_size(s, hq, wl.num_kv_heads, d,
                                                     wl.max_blocks_per_seq, wl.block_size, part)
    assert size > 0
    outs = []
    for fill in ("zeros", "random", "random"):
        if fill == "zeros":
            ws = torch.zeros(size, dtype=torch.uint8, device=DEV)
        else:
            ws = torch.randint(0, 256, (size,), dtype=torch.uint8, device=DEV)
        for _ in range(2):
            out = torch.empty(s, hq, d, dtype=torch.float32, device=DEV)
            tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                       t["context_lens"], wl.scale, partition_size=part,
                                       workspace=ws)
            torch.cuda.synchronize()
            outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    assert_close(outs[0].double().numpy(), ref, "decode")
    assert_clean_status()
