"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a library routine (torch
scaled_dot_product_attention, numpy row assignment), a closed form, an
invariant the method guarantees, or brute force on tiny inputs, so that a
plausible slip in the oracle (a dropped scale, a wrong GQA head, a transposed
operand, an off-by-one in the causal limit or the block-table index) fails at
least one of them.  The mutation tests at the end plant such slips in a copy
of the oracle's C source and check that these pins catch them.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_198_gb300 import workloads as W
from _helpers import bits, contiguous_tables, f64

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _rand_bf16(gen, *shape):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


# ----------------------------------------------------------------- KV write


def test_kv_write_equals_numpy_row_assignment():
    gen = torch.Generator().manual_seed(7)
    nb, bs, hkv, d = 6, 16, 2, 64
    kc = _rand_bf16(gen, nb, bs, hkv, d)
    vc = _rand_bf16(gen, nb, bs, hkv, d)
    t = 11
    kn = _rand_bf16(gen, t, hkv, d)
    vn = _rand_bf16(gen, t, hkv, d)
    slots = torch.randperm(nb * bs, generator=gen)[:t].to(torch.int32)
    slots[3] = -1
    slots[7] = -5
    k2, v2 = oracle.kv_write(kc, vc, kn, vn, slots)
    # independent: numpy fancy-index assignment on the flat [NB*bs, Hkv*D] view
    ek = bits(kc).reshape(nb * bs, hkv * d).copy()
    ev = bits(vc).reshape(nb * bs, hkv * d).copy()
    keep = slots.numpy() >= 0
    ek[slots.numpy()[keep]] = bits(kn).reshape(t, -1)[keep]
    ev[slots.numpy()[keep]] = bits(vn).reshape(t, -1)[keep]
    assert np.array_equal(k2.reshape(nb * bs, -1), ek)
    assert np.array_equal(v2.reshape(nb * bs, -1), ev)
    # untouched rows keep their exact bits
    untouched = np.ones(nb * bs, bool)
    untouched[slots.numpy()[keep]] = False
    assert np.array_equal(k2.reshape(nb * bs, -1)[untouched],
                          bits(kc).reshape(nb * bs, -1)[untouched])


def test_kv_write_rejects_out_of_range_slot():
    gen = torch.Generator().manual_seed(8)
    kc = _rand_bf16(gen, 2, 16, 1, 64)
    kn = _rand_bf16(gen, 1, 1, 64)
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(kc, kc, kn, kn, torch.tensor([32], dtype=torch.int32))


# ------------------------------------------------ library special cases (SDPA)


@pytest.mark.parametrize("hq,hkv,bs", [(4, 2, 16), (8, 2, 16), (8, 8, 32), (32, 8, 16)])
def test_decode_matches_sdpa_on_contiguous_tables(hq, hkv, bs):
    gen = torch.Generator().manual_seed(100 + hq + hkv + bs)
    d = 64
    ctx = [1, 17, 40, 95]
    tables, starts, nb = contiguous_tables(ctx, bs)
    kc = _rand_bf16(gen, nb, bs, hkv, d)
    vc = _rand_bf16(gen, nb, bs, hkv, d)
    q = _rand_bf16(gen, len(ctx), hq, d)
    scale = 0.125
    out = oracle.decode(q, kc, vc, tables, torch.tensor(ctx, dtype=torch.int32), scale)
    kflat = f64(kc).reshape(nb * bs, hkv, d)
    vflat = f64(vc).reshape(nb * bs, hkv, d)
    for s, c in enumerate(ctx):
        k = kflat[starts[s] * bs: starts[s] * bs + c].permute(1, 0, 2)[None]
        v = vflat[starts[s] * bs: starts[s] * bs + c].permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(f64(q[s])[None, :, None, :], k, v, scale=scale,
                                             enable_gqa=True)[0, :, 0, :]
        np.testing.assert_allclose(out[s], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_matches_sdpa_is_causal_without_prefix():
    gen = torch.Generator().manual_seed(5)
    hq, hkv, d, bs = 8, 2, 64, 16
    lq = [37, 1, 64]
    tables, starts, nb = contiguous_tables(lq, bs)
    kc = _rand_bf16(gen, nb, bs, hkv, d)
    vc = _rand_bf16(gen, nb, bs, hkv, d)
    qsl = torch.tensor([0] + list(np.cumsum(lq)), dtype=torch.int32)
    q = _rand_bf16(gen, int(qsl[-1]), hq, d)
    scale = 0.2
    out = oracle.prefill(q, qsl, kc, vc, tables, torch.tensor(lq, dtype=torch.int32), scale)
    kflat = f64(kc).reshape(nb * bs, hkv, d)
    vflat = f64(vc).reshape(nb * bs, hkv, d)
    for s, n in enumerate(lq):
        k = kflat[starts[s] * bs: starts[s] * bs + n].permute(1, 0, 2)[None]
        v = vflat[starts[s] * bs: starts[s] * bs + n].permute(1, 0, 2)[None]
        qs = f64(q[int(qsl[s]):int(qsl[s + 1])]).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qs, k, v, is_causal=True, scale=scale,
                                             enable_gqa=True)[0].permute(1, 0, 2)
        np.testing.assert_allclose(out[int(qsl[s]):int(qsl[s + 1])], ref.numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_prefill_matches_sdpa_lower_right_causal_with_prefix():
    from torch.nn.attention.bias import causal_lower_right

    gen = torch.Generator().manual_seed(6)
    hq, hkv, d, bs = 4, 1, 64, 16
    prefix = [0, 5, 48, 100]
    lq = [3, 20, 16, 33]
    ctx = [p + n for p, n in zip(prefix, lq)]
    tables, starts, nb = contiguous_tables(ctx, bs)
    kc = _rand_bf16(gen, nb, bs, hkv, d)
    vc = _rand_bf16(gen, nb, bs, hkv, d)
    qsl = torch.tensor([0] + list(np.cumsum(lq)), dtype=torch.int32)
    q = _rand_bf16(gen, int(qsl[-1]), hq, d)
    scale = 0.125
    out = oracle.prefill(q, qsl, kc, vc, tables, torch.tensor(ctx, dtype=torch.int32), scale)
    kflat = f64(kc).reshape(nb * bs, hkv, d)
    vflat = f64(vc).reshape(nb * bs, hkv, d)
    for s in range(len(ctx)):
        k = kflat[starts[s] * bs: starts[s] * bs + ctx[s], 0][None, None]
        v = vflat[starts[s] * bs: starts[s] * bs + ctx[s], 0][None, None]
        for h in range(hq):
            qs = f64(q[int(qsl[s]):int(qsl[s + 1]), h])[None, None]
            bias = causal_lower_right(lq[s], ctx[s])
            ref = F.scaled_dot_product_attention(qs, k, v, attn_mask=bias, scale=scale)[0, 0]
            np.testing.assert_allclose(out[int(qsl[s]):int(qsl[s + 1]), h], ref.numpy(),
                                       rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- closed forms


def _single_seq(gen, ctx, hq=2, hkv=1, d=64, bs=16, nb=None):
    nblk = (ctx + bs - 1) // bs
    nb = nb or nblk + 2
    tables = torch.full((1, max(nblk, 1)), -1, dtype=torch.int32)
    tables[0, :nblk] = torch.randperm(nb, generator=gen)[:nblk].to(torch.int32)
    kc = _rand_bf16(gen, nb, bs, hkv, d)
    vc = _rand_bf16(gen, nb, bs, hkv, d)
    q = _rand_bf16(gen, 1, hq, d)
    return q, kc, vc, tables, torch.tensor([ctx], dtype=torch.int32)


def _logical_row(cache, tables, s, j, bs, g):
    return f64(cache[int(tables[s, j // bs]), j % bs, g])


def test_context_one_returns_v_exactly():
    gen = torch.Generator().manual_seed(11)
    q, kc, vc, tables, cl = _single_seq(gen, 1, hq=4, hkv=2)
    out = oracle.decode(q, kc, vc, tables, cl, 0.125)
    for h in range(4):
        assert np.array_equal(out[0, h], _logical_row(vc, tables, 0, 0, 16, h // 2).numpy())


def test_identical_keys_give_mean_of_v():
    gen = torch.Generator().manual_seed(12)
    ctx = 37
    q, kc, vc, tables, cl = _single_seq(gen, ctx)
    for j in range(ctx):
        kc[int(tables[0, j // 16]), j % 16, 0] = kc[int(tables[0, 0]), 0, 0]
    out = oracle.decode(q, kc, vc, tables, cl, 0.125)
    mean_v = torch.stack([_logical_row(vc, tables, 0, j, 16, 0) for j in range(ctx)]).mean(0)
    np.testing.assert_allclose(out[0, 0], mean_v.numpy(), rtol=0, atol=1e-13)


def test_scale_zero_gives_mean_of_v():
    gen = torch.Generator().manual_seed(13)
    ctx = 29
    q, kc, vc, tables, cl = _single_seq(gen, ctx)
    out = oracle.decode(q, kc, vc, tables, cl, 0.0)
    mean_v = torch.stack([_logical_row(vc, tables, 0, j, 16, 0) for j in range(ctx)]).mean(0)
    np.testing.assert_allclose(out[0, 1], mean_v.numpy(), rtol=0, atol=1e-13)


@pytest.mark.parametrize("a", [0.5, 3.0, -2.0])
def test_two_keys_closed_form(a):
    # q = e_0, k_0 = 0, k_1 = a e_0, scale c: weights (1, e^{ca}) / (1 + e^{ca}).
    # block_size 1 puts token 0 in physical block 3 and token 1 in block 1.
    d, bs, c = 64, 1, 0.25
    kc = torch.zeros(5, bs, 1, d, dtype=torch.bfloat16)
    vc = torch.zeros(5, bs, 1, d, dtype=torch.bfloat16)
    tables = torch.tensor([[3, 1]], dtype=torch.int32)
    kc[1, 0, 0, 0] = a
    vc[3, 0, 0] = torch.arange(d, dtype=torch.float32).to(torch.bfloat16)
    vc[1, 0, 0] = (-torch.arange(d, dtype=torch.float32) / 4).to(torch.bfloat16)
    q = torch.zeros(1, 1, d, dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    out = oracle.decode(q, kc, vc, tables, torch.tensor([2], dtype=torch.int32), c)
    w1 = math.exp(c * a) / (1.0 + math.exp(c * a))
    expect = (1 - w1) * np.arange(d) + w1 * (-np.arange(d) / 4)
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-14, atol=1e-14)


def test_zero_context_gives_zeros():
    gen = torch.Generator().manual_seed(14)
    q, kc, vc, tables, cl = _single_seq(gen, 0)
    out = oracle.decode(q, kc, vc, tables, cl, 0.125)
    assert np.array_equal(out, np.zeros_like(out))


# ---------------------------------------------------------------- invariants


def test_physical_block_permutation_invariance():
    wl = W.make_decode(21, [5, 16, 33, 70], num_q_heads=8, num_kv_heads=2, block_size=16,
                       write=False)
    out = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                        wl.scale)
    gen = torch.Generator().manual_seed(22)
    perm = torch.randperm(wl.num_blocks, generator=gen)      # new place of old block b
    kc2 = torch.empty_like(wl.k_cache)
    vc2 = torch.empty_like(wl.v_cache)
    kc2[perm] = wl.k_cache
    vc2[perm] = wl.v_cache
    t2 = wl.block_tables.clone()
    valid = t2 >= 0
    t2[valid] = perm[t2[valid].long()].to(torch.int32)
    out2 = oracle.decode(wl.q, kc2, vc2, t2, wl.context_lens, wl.scale)
    assert np.array_equal(out, out2)


def test_causal_row_independent_of_later_keys():
    wl = W.make_prefill(31, [20, 3], 24, num_q_heads=4, num_kv_heads=2, block_size=16)
    base = oracle.prefill(wl.q, wl.query_start_loc, wl.k_cache, wl.v_cache, wl.block_tables,
                          wl.context_lens, wl.scale)
    s, i = 0, 9                       # row 9 of seq 0 sits at position 20 + 9 = 29
    pos = int(wl.context_lens[s]) - 24 + i
    kc = wl.k_cache.clone()
    vc = wl.v_cache.clone()
    for j in range(pos + 1, int(wl.context_lens[s])):
        b, o = int(wl.block_tables[s, j // 16]), j % 16
        kc[b, o] = 7.0
        vc[b, o] = -7.0
    pert = oracle.prefill(wl.q, wl.query_start_loc, kc, vc, wl.block_tables, wl.context_lens,
                          wl.scale)
    rows = slice(0, i + 1)
    assert np.array_equal(base[rows], pert[rows])
    assert not np.array_equal(base[i + 1], pert[i + 1])   # the next row does see position 30


def test_prefill_of_one_token_equals_decode():
    wl = W.make_decode(41, [1, 33, 64], num_q_heads=8, num_kv_heads=4, block_size=16,
                       write=False)
    dec = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                        wl.scale)
    qsl = torch.arange(0, 4, dtype=torch.int32)
    pre = oracle.prefill(wl.q, qsl, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                         wl.scale)
    assert np.array_equal(dec, pre)


# --------------------------------------------- brute force and reformulations


def _brute_force_decode(wl):
    """Direct float64 formula with per-token python indexing (tiny inputs)."""
    s_n, hq, d = wl.q.shape
    g = hq // wl.num_kv_heads
    out = np.zeros((s_n, hq, d))
    for s in range(s_n):
        c = int(wl.context_lens[s])
        for h in range(hq):
            qv = f64(wl.q[s, h]).numpy()
            ks = np.stack([_logical_row(wl.k_cache, wl.block_tables, s, j, wl.block_size,
                                        h // g).numpy() for j in range(c)])
            vs = np.stack([_logical_row(wl.v_cache, wl.block_tables, s, j, wl.block_size,
                                        h // g).numpy() for j in range(c)])
            sc = wl.scale * (ks @ qv)
            p = np.exp(sc - sc.max())
            out[s, h] = (p[:, None] * vs).sum(0) / p.sum()
    return out


def test_brute_force_tiny_workload():
    wl = W.named("tiny")
    kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    out = oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    wl.k_cache = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    wl.v_cache = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    np.testing.assert_allclose(out, _brute_force_decode(wl), rtol=1e-12, atol=1e-12)


def _online_decode(q, k, v, scale, chunk):
    """Running max / running sum over chunks of keys (the online softmax)."""
    m, l, acc = -np.inf, 0.0, np.zeros(q.shape[-1])
    for j0 in range(0, k.shape[0], chunk):
        s = scale * (k[j0:j0 + chunk] @ q)
        m_new = max(m, s.max())
        alpha = math.exp(m - m_new) if m > -np.inf else 0.0
        p = np.exp(s - m_new)
        l = l * alpha + p.sum()
        acc = acc * alpha + p @ v[j0:j0 + chunk]
        m = m_new
    return acc / l


def _split_merge_decode(q, k, v, scale, part):
    """Independent partials per window, merged by log-sum-exp."""
    ms, ls, accs = [], [], []
    for j0 in range(0, k.shape[0], part):
        s = scale * (k[j0:j0 + part] @ q)
        m = s.max()
        p = np.exp(s - m)
        ms.append(m)
        ls.append(p.sum())
        accs.append(p @ v[j0:j0 + part])
    big = max(ms)
    w = [math.exp(m - big) for m in ms]
    return sum(wi * a for wi, a in zip(w, accs)) / sum(wi * li for wi, li in zip(w, ls))


@pytest.mark.parametrize("chunk", [1, 16, 100])
def test_online_and_split_forms_agree_with_oracle(chunk):
    wl = W.make_decode(51, [300, 47], num_q_heads=4, num_kv_heads=2, block_size=16,
                       write=False)
    out = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                        wl.scale)
    for s in range(2):
        c = int(wl.context_lens[s])
        for h in range(4):
            k = np.stack([_logical_row(wl.k_cache, wl.block_tables, s, j, 16, h // 2).numpy()
                          for j in range(c)])
            v = np.stack([_logical_row(wl.v_cache, wl.block_tables, s, j, 16, h // 2).numpy()
                          for j in range(c)])
            qv = f64(wl.q[s, h]).numpy()
            np.testing.assert_allclose(_online_decode(qv, k, v, wl.scale, chunk), out[s, h],
                                       rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(_split_merge_decode(qv, k, v, wl.scale, chunk * 16),
                                       out[s, h], rtol=1e-12, atol=1e-13)


# -------------------------------------------------------- stored golden values


def test_golden_tiny_decode_fixture():
    """tests/golden/tiny_decode.txt was written by tests/golden/make_golden.py,
    which calls only the oracle; it freezes the oracle's tiny-workload output
    so a later change to its arithmetic cannot pass silently."""
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_decode.txt")
    rows = np.loadtxt(path)
    wl = W.named("tiny")
    kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    out = oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    np.testing.assert_allclose(out.reshape(-1, out.shape[-1]), rows, rtol=0, atol=1e-15)


# ------------------------------------------------------------ planted slips


_PLANTS = {
    # a dropped scale
    "drop_scale": ("scores[j] = scale * dot;", "scores[j] = dot;"),
    # GQA: h % G instead of h / G style mapping (heads of a group read other KV heads)
    "gqa_mapping": ("for (int h = g * group; h < (g + 1) * group; ++h) {\n"
                    "        const uint16_t* qsrc = q + ((long long)s * hq + h) * d;",
                    "for (int h = g; h < hq; h += hkv) {\n"
                    "        const uint16_t* qsrc = q + ((long long)s * hq + h) * d;"),
    # causal limit off by one (row sees one key too few)
    "causal_off_by_one": ("attend(out + (t * hq + h) * d, qv, kc, vc, pos + 1, d, scale,",
                          "attend(out + (t * hq + h) * d, qv, kc, vc, pos, d, scale,"),
    # wrong offset inside a physical block
    "block_offset": ("long long offset = j % bs;", "long long offset = (j + 1) % bs;"),
    # softmax max not subtracted consistently (exp of raw score, max used in sum)
    "softmax_norm": ("for (int e = 0; e < d; ++e) out[e] /= l;",
                     "for (int e = 0; e < d; ++e) out[e] /= (l + 1.0);"),
}


_PIN_RUNNER = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[2])
import oracle
real = oracle._load()
planted = ctypes.CDLL(sys.argv[3])
for name in ("oracle_kv_write", "oracle_decode", "oracle_prefill", "oracle_set_threads",
             "oracle_max_threads"):
    getattr(planted, name).argtypes = getattr(real, name).argtypes
    getattr(planted, name).restype = getattr(real, name).restype
oracle._lib = planted
import test_oracle as T
pins = [
    lambda: T.test_decode_matches_sdpa_on_contiguous_tables(32, 8, 16),
    lambda: T.test_prefill_matches_sdpa_lower_right_causal_with_prefix(),
    lambda: T.test_two_keys_closed_form(3.0),
    lambda: T.test_brute_force_tiny_workload(),
    lambda: T.test_scale_zero_gives_mean_of_v(),
    lambda: T.test_physical_block_permutation_invariance(),
]
caught = 0
for pin in pins:
    try:
        pin()
    except (AssertionError, oracle.OracleError):
        caught += 1
print("CAUGHT", caught)
"""


@pytest.mark.parametrize("plant", sorted(_PLANTS))
def test_pins_catch_planted_oracle_slips(plant, tmp_path):
    """Compile a copy of the oracle with one planted slip and check, in a
    separate process, that at least one pin above fails on it (planting
    happens on the CPU only)."""
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    with open(os.path.join(root, "oracle", "oracle.c")) as fh:
        src = fh.read()
    old, new = _PLANTS[plant]
    assert src.count(old) >= 1, plant
    lib = tmp_path / "libplant.so"
    csrc = tmp_path / "plant.c"
    csrc.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(csrc), "-o", str(lib),
                    "-lm"], check=True, capture_output=True)
    res = subprocess.run([sys.executable, "-c", _PIN_RUNNER, root, here, str(lib)],
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    caught = int(res.stdout.split("CAUGHT")[-1])
    assert caught >= 1, f"no pin caught the planted slip {plant}"
