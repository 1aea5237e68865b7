"""Pins of the oracle's rotary embedding and of its double -> bf16 rounding.

RoPE [tiny-vllm README, curriculum "RoPE"]: pairs (x_i, x_{i+D/2}) rotated by
pos * theta^(-2i/D).  Pinned by: position 0 is the identity, rotations keep
each pair's length, the rotated dot product depends only on the relative
position, two rotations compose, and a hand-computed D = 4 case."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _bf16_value(bits: int) -> Fraction:
    import struct

    return Fraction(struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0])


def test_round_bf16_exact_values_ties_and_neighbours():
    rng = np.random.default_rng(3)
    samples = []
    for bits in rng.integers(0x0080, 0x7F7F, 3000).tolist() + [0x3F80, 0x0001, 0x7F00]:
        for sign in (0, 0x8000):
            b = bits | sign
            lo, hi = _bf16_value(b), _bf16_value(b + 1)
            mid = (lo + hi) / 2
            eps = (hi - lo) / 1000
            samples += [(float(lo), b), (float(mid), b if (b & 1) == 0 else b + 1),
                        (float(mid - eps), b), (float(mid + eps), b + 1)]
    vals = np.array([v for v, _ in samples])
    want = np.array([w for _, w in samples], dtype=np.uint16)
    assert np.array_equal(oracle.round_bf16(vals), want)


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal(64)
    assert np.array_equal(oracle.rope_double(x, 0, 10000.0), x)


@pytest.mark.parametrize("pos", [1, 17, 4095, 131071])
def test_rope_keeps_pair_lengths(pos):
    x = np.random.default_rng(pos).standard_normal(64)
    y = oracle.rope_double(x, pos, 500000.0)
    np.testing.assert_allclose(np.hypot(y[:32], y[32:]), np.hypot(x[:32], x[32:]), rtol=1e-12)


def test_rope_dot_product_depends_on_relative_position_only():
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    base = oracle.rope_double(q, 300, 1e4) @ oracle.rope_double(k, 200, 1e4)
    for shift in (1, 37, 1000):
        moved = oracle.rope_double(q, 300 + shift, 1e4) @ oracle.rope_double(k, 200 + shift, 1e4)
        assert abs(moved - base) <= 1e-9 * (1 + abs(base))


def test_rope_rotations_compose():
    x = np.random.default_rng(9).standard_normal(64)
    twice = oracle.rope_double(oracle.rope_double(x, 5, 1e4), 7, 1e4)
    np.testing.assert_allclose(twice, oracle.rope_double(x, 12, 1e4), rtol=1e-12, atol=1e-12)


def test_rope_hand_computed_d4():
    # D = 4, theta = 100: pair (x0, x2) turns by pos, pair (x1, x3) by pos / 10
    x = np.array([1.0, 2.0, 3.0, 4.0])
    pos = 3
    a0, a1 = pos * 1.0, pos * 100.0 ** -0.5
    want = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
            3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    np.testing.assert_allclose(oracle.rope_double(x, pos, 100.0), want, rtol=1e-14)


def test_rope_kv_write_rotates_q_and_k_and_copies_v():
    gen = torch.Generator().manual_seed(4)
    nb, bs, hkv, hq, d, t = 4, 16, 2, 4, 64, 5
    kc = torch.randn(nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    kn = torch.randn(t, hkv, d, generator=gen).to(torch.bfloat16)
    vn = torch.randn(t, hkv, d, generator=gen).to(torch.bfloat16)
    q = torch.randn(t, hq, d, generator=gen).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 20, 63, 40], dtype=torch.int32)
    pos = torch.tensor([0, 5, 77, 1000, 2], dtype=torch.int32)
    q2, k2, v2 = oracle.rope_kv_write(q, kc, vc, kn, vn, slots, pos, 10000.0)
    qd = q.double().numpy()
    for tt in range(t):
        for h in range(hq):
            want = oracle.round_bf16(oracle.rope_double(qd[tt, h], int(pos[tt]), 1e4))
            assert np.array_equal(q2[tt, h], want)
    kflat = k2.reshape(nb * bs, hkv, d)
    vflat = v2.reshape(nb * bs, hkv, d)
    for tt in range(t):
        s = int(slots[tt])
        if s < 0:
            continue
        for h in range(hkv):
            want = oracle.round_bf16(oracle.rope_double(kn[tt, h].double().numpy(), int(pos[tt]), 1e4))
            assert np.array_equal(kflat[s, h], want)
        assert np.array_equal(vflat[s], vn[tt].view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(q2[0], q[0].view(torch.int16).numpy().view(np.uint16))  # position 0
