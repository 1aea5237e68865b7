"""Host block allocator (tvl_allocator_*): invariants under random
operations, copy-on-write of shared partial blocks, all-or-nothing failure.
Host code only -- runs without a GPU."""
import random

import numpy as np
import pytest

pytest.importorskip("ctypes")


@pytest.fixture(scope="module")
def tvl():
    from paged_kv_cache_198_gb300 import _build

    _build.build()
    import paged_kv_cache_198_gb300 as t

    return t


def _owners(alloc, live, mb):
    """physical block -> set of sequences whose table names it"""
    tables, ctx = alloc.build_tables(sorted(live), mb)
    owners = {}
    for seq, row, c in zip(sorted(live), tables, ctx):
        nb = (int(c) + alloc.block_size - 1) // alloc.block_size
        assert (row[:nb] >= 0).all() and (row[nb:] == -1).all()
        for b in row[:nb]:
            owners.setdefault(int(b), set()).add(seq)
    return owners, dict(zip(sorted(live), ctx.tolist()))


def test_append_hands_out_consecutive_slots_in_fresh_blocks(tvl):
    a = tvl.BlockAllocator(8, 16)
    s = a.new_sequence()
    slots = a.append(s, 40)
    blocks = slots // 16
    assert list(slots % 16) == [i % 16 for i in range(40)]
    assert len(set(blocks.tolist())) == 3
    assert a.context_len(s) == 40
    st = a.stats()
    assert st["free_blocks"] == 5 and st["slack_slots"] == 8 and st["tokens"] == 40


def test_out_of_blocks_changes_nothing(tvl):
    a = tvl.BlockAllocator(2, 16)
    s = a.new_sequence()
    a.append(s, 20)
    before = a.stats()
    with pytest.raises(tvl.TvlError) as ei:
        a.append(s, 13)                      # needs a third block
    assert ei.value.status == tvl.ERR_OUT_OF_BLOCKS
    assert a.stats() == before and a.context_len(s) == 20
    a.append(s, 12)                          # fills the second block exactly
    assert a.stats()["free_blocks"] == 0


def test_fork_shares_blocks_and_copies_on_write(tvl):
    a = tvl.BlockAllocator(16, 16)
    p = a.new_sequence()
    a.append(p, 40)                          # blocks b0 b1 (full) + b2 (8 tokens)
    c = a.fork(p)
    assert a.stats()["shared_blocks"] == 3
    (tp, tc), _ = a.build_tables([p, c], 4)
    assert list(tp[:3]) == list(tc[:3])
    slot = a.append(c, 1)[0]                 # writes into the shared partial block
    src, dst = a.take_copies()
    assert list(src) == [tp[2]] and dst[0] != tp[2]
    assert slot == dst[0] * 16 + 8
    (tp2, tc2), _ = a.build_tables([p, c], 4)
    assert list(tp2[:3]) == list(tp[:3]) and tc2[2] == dst[0] and list(tc2[:2]) == list(tp[:2])
    assert a.take_copies()[0].size == 0
    a.append(p, 8)                           # parent's block is private again: no copy
    assert a.take_copies()[0].size == 0


def test_fork_at_a_block_boundary_needs_no_copy(tvl):
    a = tvl.BlockAllocator(8, 16)
    p = a.new_sequence()
    a.append(p, 32)
    c = a.fork(p)
    a.append(c, 5)
    assert a.take_copies()[0].size == 0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_keep_the_pool_consistent(tvl, seed):
    rng = random.Random(seed)
    nb, bs, mb = 64, 16, 64
    a = tvl.BlockAllocator(nb, bs)
    live = set()
    for _ in range(400):
        op = rng.random()
        if op < 0.15 or not live:
            live.add(a.new_sequence())
        elif op < 0.25:
            live.add(a.fork(rng.choice(sorted(live))))
        elif op < 0.40:
            s = rng.choice(sorted(live))
            a.free(s)
            live.discard(s)
        else:
            s = rng.choice(sorted(live))
            n = rng.randint(1, 40)
            try:
                slots = a.append(s, n)
                assert len(set(slots.tolist())) == n
            except tvl.TvlError as e:
                assert e.status == tvl.ERR_OUT_OF_BLOCKS
        a.take_copies()
        owners, ctx = _owners(a, live, mb)
        st = a.stats()
        assert st["free_blocks"] + len(owners) == nb          # every block owned or free
        assert st["live_sequences"] == len(live)
        assert st["shared_blocks"] == sum(1 for v in owners.values() if len(v) > 1)
        assert st["tokens"] == sum(ctx.values())
    for s in list(live):
        a.free(s)
    assert a.stats()["free_blocks"] == nb


def test_bad_ids_are_rejected(tvl):
    a = tvl.BlockAllocator(4, 16)
    with pytest.raises(tvl.TvlError):
        a.append(3, 1)
    s = a.new_sequence()
    a.free(s)
    with pytest.raises(tvl.TvlError):
        a.free(s)
    with pytest.raises(tvl.TvlError):
        tvl.BlockAllocator(0, 16)
