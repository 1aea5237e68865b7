"""GPU parity of the fused RoPE + paged KV write (tvl_rope_paged_kv_write)
against the oracle's double-precision rotation [tiny-vllm README, curriculum
"RoPE", "Paged KV cache"].  The GPU rotates in fp32 after reducing the angle
in double precision, the oracle in double; both round to bf16 once.  The
results agree to one bf16 ulp plus the fp32 rounding of the rotation (which
shows only where the two products cancel), and almost all bit for bit.  The
V rows and every untouched slot are bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status, assert_close, bits_of

pytestmark = pytest.mark.gpu


def _value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_rotated(got, want, src_bits, what):
    """Each result within one bf16 ulp of the double-precision value plus the
    fp32 rounding of the rotation, 2^-21 * (|x_i| + |x_{i+D/2}|) (it matters
    only where the two products cancel); almost all bit-identical."""
    g, w = _value(got), _value(want)
    x = np.abs(_value(src_bits))
    pair = x[..., :32] + x[..., 32:]
    scale = np.concatenate([pair, pair], axis=-1)
    ulp = np.maximum(np.abs(w), 1e-30) * 2.0 ** -7
    assert (np.abs(g - w) <= ulp + scale * 2.0 ** -21).all(), what
    assert (got != want).mean() < 1e-3, f"{what}: {(got != want).mean():.2e} of elements differ"


@pytest.mark.parametrize("theta", [10000.0, 500000.0])
def test_rope_write_matches_oracle(theta):
    gen = torch.Generator().manual_seed(31)
    nb, bs, hkv, hq, d, t = 64, 16, 8, 32, 64, 300
    kc = torch.randn(nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    kn = torch.randn(t, hkv, d, generator=gen).to(torch.bfloat16)
    vn = torch.randn(t, hkv, d, generator=gen).to(torch.bfloat16)
    q = torch.randn(t, hq, d, generator=gen).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=gen)[:t].to(torch.int32)
    slots[::17] = -1
    pos = torch.randint(0, 131072, (t,), generator=gen).to(torch.int32)
    pos[:4] = torch.tensor([0, 1, 2, 131071], dtype=torch.int32)
    dq, dk, dv = q.to(DEV), kc.to(DEV), vc.to(DEV)
    tvl.rope_paged_kv_write(dq, kn.to(DEV), vn.to(DEV), dk, dv, slots.to(DEV), pos.to(DEV),
                            rope_theta=theta)
    torch.cuda.synchronize()
    q2, k2, v2 = oracle.rope_kv_write(q, kc, vc, kn, vn, slots, pos, theta)
    _check_rotated(bits_of(dq), q2, bits_of(q), "q")
    # rows of the cache that received a rotated K: compare with their source rows
    flat_got = bits_of(dk).reshape(nb * bs, hkv, d)
    flat_want = k2.reshape(nb * bs, hkv, d)
    keep = slots.numpy() >= 0
    rows = slots.numpy()[keep]
    _check_rotated(flat_got[rows], flat_want[rows], bits_of(kn)[keep], "k_cache")
    untouched = np.ones(nb * bs, bool)
    untouched[rows] = False
    assert np.array_equal(flat_got[untouched], flat_want[untouched])
    assert np.array_equal(bits_of(dv), v2)
    # position 0 leaves q unchanged, bit for bit
    assert np.array_equal(bits_of(dq)[0], bits_of(q)[0])
    assert_clean_status()


def test_rope_write_then_decode_matches_oracle():
    """A decode step with RoPE: rotate q and the new K at position ctx-1,
    write, then decode over the cache (whose older K rows are taken as
    already rotated)."""
    wl = W.make_decode(33, [40, 700, 1500, 3], num_q_heads=32, num_kv_heads=8, block_size=16)
    pos = (wl.context_lens - 1).to(torch.int32)
    t = W.to_device(wl, DEV)
    tvl.rope_paged_kv_write(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                            t["slot_mapping"], pos.to(DEV), rope_theta=500000.0)
    out = torch.empty(tuple(wl.q.shape), dtype=torch.float32, device=DEV)
    tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                               t["context_lens"], wl.scale)
    torch.cuda.synchronize()
    q2, k2, v2 = oracle.rope_kv_write(wl.q, wl.k_cache, wl.v_cache, wl.k_new, wl.v_new,
                                      wl.slot_mapping, pos, 500000.0)
    ref = oracle.decode(q2, k2, v2, wl.block_tables, wl.context_lens, wl.scale)
    assert_close(out.double().cpu().numpy(), ref, "rope + decode")
    assert_clean_status()


def test_rope_write_without_q_and_bad_slot():
    gen = torch.Generator().manual_seed(32)
    kc = torch.zeros(2, 16, 8, 64, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kn = torch.randn(2, 8, 64, generator=gen).to(torch.bfloat16).to(DEV)
    slots = torch.tensor([5, 32], dtype=torch.int32, device=DEV)      # 32 = one past the pool
    pos = torch.tensor([0, 9], dtype=torch.int32, device=DEV)
    tvl.rope_paged_kv_write(None, kn, kn, kc, vc, slots, pos)
    assert tvl.get_device_status() & tvl.DEV_BAD_SLOT
    flat = kc.view(-1, 8, 64)
    assert torch.equal(flat[5].view(torch.int16), kn[0].view(torch.int16))   # position 0
    assert int((flat[:5].float().abs().sum() + flat[6:].float().abs().sum())) == 0
