"""GPU parity of the tcgen05 chunked causal prefill against the CPU oracle,
plus the causal and placement invariants."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import (DEV, MAX_ABS, MEAN_ABS, assert_clean_status, assert_close,
                        oracle_caches)

pytestmark = pytest.mark.gpu


def gpu_prefill(wl, write=True, tensors=None):
    t = tensors if tensors is not None else W.to_device(wl, DEV)
    if write:
        tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.full(tuple(wl.q.shape), float("nan"), dtype=torch.float32, device=DEV)
    tvl.paged_attention_prefill(out, t["q"], t["query_start_loc"], t["k_cache"], t["v_cache"],
                                t["block_tables"], t["context_lens"], wl.scale, wl.max_q_len)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), t


def oracle_prefill(wl, write=True, row_mask=None):
    kc, vc = oracle_caches(wl, write)
    return oracle.prefill(wl.q, wl.query_start_loc, kc, vc, wl.block_tables, wl.context_lens,
                          wl.scale, row_mask=row_mask)


CASES = [
    # (prefix lens, q lens, Hq, Hkv, bs)
    ([0], [1], 4, 1, 16),
    ([0], [100], 4, 2, 16),              # one partial tile, causal from row 0
    ([0, 0], [128, 129], 8, 2, 16),      # exact tile and one row over
    ([5, 300, 47], [20, 64, 200], 8, 2, 16),
    ([130, 0, 1000], [1, 255, 77], 32, 8, 32),
    ([17, 2000], [300, 3], 8, 1, 64),    # G = 8
    ([64, 0], [70, 33], 4, 4, 128),      # G = 1, block = one whole KV tile
    ([1, 2, 3, 129, 257], [128, 127, 129, 1, 2], 16, 8, 16),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_random_shapes(case):
    prefix, lq, hq, hkv, bs = CASES[case]
    wl = W.make_prefill(700 + case, prefix, lq, num_q_heads=hq, num_kv_heads=hkv, block_size=bs)
    got, _ = gpu_prefill(wl)
    assert_close(got, oracle_prefill(wl), f"case {case}")
    assert_clean_status()


@pytest.mark.parametrize("hkv", [2, 8])    # two query heads per CTA / one
def test_prefill_more_items_than_threads(hkv):
    """400 (sequence, query tile) items: more than a CTA has threads, so the
    CTAs take the items in item order instead of longest first.  Every row of
    every sequence is still written once (the output starts as NaN)."""
    gen = np.random.default_rng(31)
    lq = gen.integers(1, 40, 200).tolist()
    lq[7] = 200                                  # two query tiles for every sequence
    prefix = gen.integers(0, 300, 200).tolist()
    wl = W.make_prefill(731, prefix, lq, num_q_heads=8, num_kv_heads=hkv, block_size=16)
    got, _ = gpu_prefill(wl)
    assert_close(got, oracle_prefill(wl), f"400 items hkv {hkv}")
    assert_clean_status()


@pytest.mark.parametrize("replica", [0, 1, 2])
def test_prefill_chunked_config_every_row(replica):
    """The full chunked-prefill batch (16 sequences, cached prefix U{0..2048}
    + 512 new tokens, 32/8 heads, bs 16): every one of its 8192 x 32 output
    rows against the oracle."""
    wl = W.named("chunked_prefill", replica)
    got, _ = gpu_prefill(wl)
    ref = oracle_prefill(wl)
    assert not np.isnan(ref).any()
    assert_close(got, ref, f"chunked r{replica}")
    assert np.isfinite(got).all()
    assert_clean_status()


def test_prefill_short_rows_with_large_values():
    """Rows with one to a few visible keys, K scaled by 3 and V by 8.  The
    error of the fp16 P.V path is linear in |v| (P is rounded to 2^-11
    relative), so the N(0,1) bound is scaled by the factor on V."""
    wl = W.make_prefill(720, [0, 0], [8, 130], num_q_heads=8, num_kv_heads=2, block_size=16)
    wl.k_new = (wl.k_new.float() * 3).to(torch.bfloat16)
    wl.v_new = (wl.v_new.float() * 8).to(torch.bfloat16)
    got, _ = gpu_prefill(wl)
    ref = oracle_prefill(wl)
    err = np.abs(got - ref)
    assert err.max() <= 8 * MAX_ABS and err.mean() <= 8 * MEAN_ABS, (err.max(), err.mean())


def test_prefill_short_rows_unit_variance():
    """The same short rows (prefix 0, rows with 1..8 keys) with N(0,1) inputs
    meet the stated bound itself."""
    wl = W.make_prefill(725, [0, 0, 0], [8, 3, 130], num_q_heads=8, num_kv_heads=2,
                        block_size=16)
    got, _ = gpu_prefill(wl)
    assert_close(got, oracle_prefill(wl), "short rows N(0,1)")


@pytest.mark.parametrize("rise", [20.0, -20.0])
def test_prefill_scores_rising_along_the_context(rise):
    """Scores that grow (or fall) by ~20 along each row: later key tiles beat
    the first tile's maximum by far more than fp16 P can absorb, so the kernel
    must move its reference maximum (and rescale O) on later tiles; falling
    scores drive P of later tiles toward 0 instead."""
    wl = W.make_prefill(726, [1000, 37], [130, 300], num_q_heads=8, num_kv_heads=2,
                        block_size=16)
    bs = wl.block_size
    q = wl.q.float()
    q[:, :, 0] = 8.0
    wl.q = q.to(torch.bfloat16)
    kc = wl.k_cache.float().view(-1, wl.num_kv_heads, wl.head_dim)
    kn = wl.k_new.float()
    for s in range(wl.num_seqs):
        ctx = int(wl.context_lens[s])
        pre = int(wl.prefix_lens[s])
        q0 = int(wl.query_start_loc[s])
        for j in range(ctx):
            val = rise * j / ctx / (8.0 * wl.scale)     # score component = rise * j / ctx
            if j < pre:
                kc[W.slot_of(wl.block_tables, s, j, bs), :, 0] = val
            else:
                kn[q0 + j - pre, :, 0] = val
    wl.k_cache = kc.view(wl.k_cache.shape).to(torch.bfloat16)
    wl.k_new = kn.to(torch.bfloat16)
    got, _ = gpu_prefill(wl)
    assert_close(got, oracle_prefill(wl), f"rising {rise}")
    assert_clean_status()


@pytest.mark.parametrize("hkv", [2, 8])     # two query heads per unit / one
def test_prefill_inconsistent_lengths_are_reported_and_skipped(hkv):
    """One sequence whose context is shorter than its chunk, one whose context
    runs past its block table: their rows are left alone and the status word
    says why, while the other sequence is computed as usual."""
    wl = W.make_prefill(732, [30, 50, 70], [40, 20, 130], num_q_heads=8, num_kv_heads=hkv,
                        block_size=16)
    t = W.to_device(wl, DEV)
    tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    ctx = t["context_lens"].clone()
    ctx[1] = 19                                   # < Lq = 20
    ctx[2] = wl.max_blocks_per_seq * wl.block_size + 1
    out = torch.full(tuple(wl.q.shape), float("nan"), dtype=torch.float32, device=DEV)
    tvl.paged_attention_prefill(out, t["q"], t["query_start_loc"], t["k_cache"], t["v_cache"],
                                t["block_tables"], ctx, wl.scale, wl.max_q_len)
    torch.cuda.synchronize()
    bits = tvl.get_device_status()
    assert bits & tvl.DEV_BAD_QUERY_LEN
    assert bits & tvl.DEV_BAD_CONTEXT_LEN
    got = out.double().cpu().numpy()
    qsl = wl.query_start_loc.tolist()
    ref = oracle_prefill(wl)
    assert_close(got[qsl[0]:qsl[1]], ref[qsl[0]:qsl[1]], "valid sequence")
    assert np.isnan(got[qsl[1]:qsl[3]]).all()
    assert_clean_status()


def test_prefill_bad_query_start_loc_is_reported_and_contained():
    """query_start_loc entries that would put rows outside [0, Tq) -- a
    decreasing entry, an end past total_q_tokens -- and a chunk longer than
    max_q_len: those sequences are reported and skipped, nothing outside the
    Tq rows of `out` is written (the buffer is allocated larger and its extra
    rows must stay NaN), and the consistent sequence is computed as usual."""
    wl = W.make_prefill(733, [30, 50, 70, 10], [40, 20, 30, 100], num_q_heads=8,
                        num_kv_heads=2, block_size=16)
    t = W.to_device(wl, DEV)
    tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    tq = wl.total_q                                    # 190; the chunks start at 0, 40, 60, 90
    # seq 1: [40, 30) decreasing; seq 2: [30, 180) has 150 rows, more than the
    # 128 that max_q_len 100 provides; seq 3: [180, 190) is consistent -- the
    # last 10 positions of its 110-token context, whose queries are rows
    # 180..189 of q in the workload's own packing too.
    qsl = torch.tensor([0, 40, 30, tq - 10, tq], dtype=torch.int32)
    ctx = t["context_lens"].clone()
    ref_rows = 40
    extra = 64
    out_big = torch.full((tq + extra, wl.num_q_heads, wl.head_dim), float("nan"),
                         dtype=torch.float32, device=DEV)
    out = out_big[:tq]
    tvl.paged_attention_prefill(out, t["q"], qsl.to(DEV), t["k_cache"], t["v_cache"],
                                t["block_tables"], ctx, wl.scale, 100)
    torch.cuda.synchronize()
    bits = tvl.get_device_status()
    assert bits & tvl.DEV_BAD_QUERY_LEN
    got = out_big.double().cpu().numpy()
    assert np.isnan(got[tq:]).all(), "rows past total_q_tokens were written"
    ref = oracle_prefill(wl)
    assert_close(got[:ref_rows], ref[:ref_rows], "consistent sequence 0")
    assert np.isnan(got[ref_rows:tq - 10]).all()
    assert_close(got[tq - 10:tq], ref[tq - 10:tq], "consistent sequence 3")

    # an end past total_q_tokens
    qsl2 = torch.tensor([0, 40, 60, 90, tq + 5], dtype=torch.int32)
    out_big.fill_(float("nan"))
    tvl.paged_attention_prefill(out, t["q"], qsl2.to(DEV), t["k_cache"], t["v_cache"],
                                t["block_tables"], ctx, wl.scale, 128)
    torch.cuda.synchronize()
    assert tvl.get_device_status() & tvl.DEV_BAD_QUERY_LEN
    got = out_big.double().cpu().numpy()
    assert np.isnan(got[tq:]).all(), "rows past total_q_tokens were written"
    assert np.isnan(got[90:tq]).all()
    assert_close(got[:90], ref[:90], "consistent sequences 0-2 (second call)")
    assert_clean_status()


def test_prefill_v_within_fp16_range():
    """V entries of magnitude 3e4 (inside the fp16 range the P.V product
    uses) give results as close to the oracle as N(0,1) ones, relative to
    the largest |v|; nothing is reported."""
    wl = W.make_prefill(734, [100, 0], [60, 130], num_q_heads=8, num_kv_heads=2, block_size=16)
    vn = wl.v_new.float()
    vn[5, 0, 3] = 30000.0
    vn[70, 1, 10] = -30000.0
    wl.v_new = vn.to(torch.bfloat16)
    got, _ = gpu_prefill(wl)
    ref = oracle_prefill(wl)
    vmax = 30000.0
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= MAX_ABS * vmax and err.mean() <= MEAN_ABS * vmax, (err.max(), err.mean())
    assert_clean_status()


def test_prefill_v_beyond_fp16_range_is_reported():
    """A V value of 1e5 (a bf16 value beyond fp16's 65504) leaves output
    rows that are not finite, which sets DEV_NONFINITE; a sequence whose keys
    do not include it is unaffected."""
    wl = W.make_prefill(735, [50, 20], [30, 40], num_q_heads=8, num_kv_heads=2, block_size=16)
    vn = wl.v_new.float()
    vn[45, 0, 7] = 1.0e5                              # a token of sequence 1
    wl.v_new = vn.to(torch.bfloat16)
    got, _ = gpu_prefill(wl)
    bits = tvl.get_device_status()
    assert bits & tvl.DEV_NONFINITE
    ref = oracle_prefill(wl)
    assert_close(got[:30], ref[:30], "sequence 0")
    assert_clean_status()


def test_prefill_poisoned_unused_slots():
    wl = W.make_prefill(721, [3, 40, 200], [10, 100, 60], num_q_heads=8, num_kv_heads=2,
                        block_size=32)
    W.poison_unused(wl, 1.0e4)
    got, _ = gpu_prefill(wl)
    assert_close(got, oracle_prefill(wl), "poisoned")


def test_prefill_bit_identical_under_block_permutation():
    wl = W.make_prefill(722, [100, 700], [200, 129], num_q_heads=8, num_kv_heads=2,
                        block_size=16)
    base, t = gpu_prefill(wl)
    kc = t["k_cache"].cpu()
    vc = t["v_cache"].cpu()
    gen = torch.Generator().manual_seed(5)
    perm = torch.randperm(wl.num_blocks, generator=gen)
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = wl.block_tables.clone()
    valid = t2 >= 0
    t2[valid] = perm[t2[valid].long()].to(torch.int32)
    wl.k_cache, wl.v_cache, wl.block_tables = kc2, vc2, t2
    moved, _ = gpu_prefill(wl, write=False)
    assert np.array_equal(base, moved)


def test_prefill_causal_rows_ignore_later_keys():
    wl = W.make_prefill(723, [50], [200], num_q_heads=4, num_kv_heads=1, block_size=16)
    base, t = gpu_prefill(wl)
    i = 90                                    # row 90 sits at position 140
    pos = 50 + i
    kc = t["k_cache"]
    vc = t["v_cache"]
    for j in range(pos + 1, 250):
        b, o = int(wl.block_tables[0, j // 16]), j % 16
        kc[b, o] = 5.0
        vc[b, o] = -5.0
    out = torch.full(tuple(wl.q.shape), float("nan"), dtype=torch.float32, device=DEV)
    tvl.paged_attention_prefill(out, t["q"], t["query_start_loc"], kc, vc, t["block_tables"],
                                t["context_lens"], wl.scale, wl.max_q_len)
    pert = out.double().cpu().numpy()
    assert np.array_equal(base[:i + 1], pert[:i + 1])
    assert not np.array_equal(base[i + 1], pert[i + 1])


def test_prefill_matches_decode_for_single_token_chunks():
    """A prefill chunk of one token per sequence is a decode step."""
    wl = W.make_prefill(724, [33, 500, 1], [1, 1, 1], num_q_heads=32, num_kv_heads=8,
                        block_size=16)
    got, t = gpu_prefill(wl)
    out = torch.empty(tuple(wl.q.shape), dtype=torch.float32, device=DEV)
    tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                               t["context_lens"], wl.scale, partition_size=0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(got, out.double().cpu().numpy(), rtol=0, atol=2e-3)
