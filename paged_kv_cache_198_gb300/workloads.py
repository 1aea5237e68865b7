"""Seeded synthetic workloads for the paged-attention hot path.

This module only draws inputs: context lengths, a scattered physical block
assignment, bf16 q / K / V ~ N(0, 1) and the slot mapping of the tokens a step
writes.  It holds none of the attention arithmetic, so the CUDA library and
the CPU oracle can both be fed from it.

Draw order for one seed (``torch.Generator().manual_seed(seed)``, CPU):
  1. lengths (context lengths for decode, cached-prefix lengths for prefill)
  2. ``randperm(NB)``: physical blocks, dealt to sequences in order
  3. q, 4. k_cache, 5. v_cache (drawn in chunks of 4096 blocks), 6. k_new,
  7. v_new -- all fp32 N(0, 1) rounded to bf16 (round-to-nearest-even).

The five named workloads are the Llama-3.2-1B-shaped cases of the method
(32 query heads, 8 KV heads, head_dim 64) plus a tiny GQA-2 case:
  tiny              2 seqs, ctx [17, 40], 4/2 heads, bs 16, pool of 8 blocks
  llama1b_decode    64 seqs, ctx ~ U{512..4096}, bs 16, pool 1.5x
  continuous_batch  256 seqs, ctx = round(exp(U(ln 16, ln 8192))), bs 32
  long_splitk       8 seqs, ctx ~ U{32768..131072}, bs 16, 512-token splits
  chunked_prefill   16 seqs, prefix ~ U{0..2048} + 512 new tokens, bs 16
Every decode workload writes one new token per sequence (at position ctx-1,
so the context includes it); the prefill workload writes its whole chunk.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

HEAD_DIM = 64
BF16 = torch.bfloat16

# name -> (index, builder kwargs); seeds are 1000 * index + replica.
NAMED = {
    "tiny": 1,
    "llama1b_decode": 2,
    "continuous_batch": 3,
    "long_splitk": 4,
    "chunked_prefill": 5,
}


def _randn_bf16(gen: torch.Generator, shape, chunk_rows: Optional[int] = None) -> torch.Tensor:
    """N(0,1) fp32 rounded to bf16; large tensors are drawn in row chunks."""
    if chunk_rows is None or shape[0] <= chunk_rows:
        return torch.randn(*shape, generator=gen).to(BF16)
    out = torch.empty(*shape, dtype=BF16)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        out[r0:r1] = torch.randn(r1 - r0, *shape[1:], generator=gen).to(BF16)
    return out


def _deal_blocks(gen, context_lens, block_size, num_blocks, max_blocks, pool_factor):
    nblk = [(int(c) + block_size - 1) // block_size for c in context_lens.tolist()]
    needed = sum(nblk)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * needed))
    if needed > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {needed}")
    if max_blocks is None:
        max_blocks = max(1, max(nblk) if nblk else 1)
    if nblk and max(nblk) > max_blocks:
        raise ValueError("max_blocks_per_seq too small")
    perm = torch.randperm(num_blocks, generator=gen)
    tables = torch.full((len(nblk), max_blocks), -1, dtype=torch.int32)
    at = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[at:at + n].to(torch.int32)
        at += n
    return tables, num_blocks, max_blocks


def slot_of(block_tables: torch.Tensor, seq: int, pos: int, block_size: int) -> int:
    """Cache slot of logical position pos of a sequence (what a host block
    allocator hands to the write)."""
    return int(block_tables[seq, pos // block_size]) * block_size + pos % block_size


@dataclass
class DecodeWorkload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    partition_size: int
    context_lens: torch.Tensor      # int32 [S]
    block_tables: torch.Tensor      # int32 [S, MB], -1 padded
    q: torch.Tensor                 # bf16 [S, Hq, D]
    k_cache: torch.Tensor           # bf16 [NB, bs, Hkv, D]
    v_cache: torch.Tensor
    k_new: torch.Tensor             # bf16 [T, Hkv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # int32 [T]
    meta: Dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    def kv_bytes(self) -> int:
        """K and V bytes the decode must read once (each cached token once)."""
        return int(self.context_lens.sum()) * self.num_kv_heads * self.head_dim * 2 * 2


@dataclass
class PrefillWorkload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    prefix_lens: torch.Tensor       # int32 [S]
    context_lens: torch.Tensor      # int32 [S] = prefix + Lq
    query_start_loc: torch.Tensor   # int32 [S + 1]
    block_tables: torch.Tensor
    q: torch.Tensor                 # bf16 [Tq, Hq, D]
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor             # bf16 [Tq, Hkv, D] (the chunk's K/V)
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # int32 [Tq]
    meta: Dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_q_len(self) -> int:
        q = self.query_start_loc
        return int((q[1:] - q[:-1]).max()) if self.num_seqs else 0

    def causal_pairs(self) -> int:
        """Visible (query, key) pairs: sum over rows of (position + 1)."""
        total = 0
        for s in range(self.num_seqs):
            lq = int(self.query_start_loc[s + 1] - self.query_start_loc[s])
            p = int(self.context_lens[s]) - lq
            total += lq * p + lq * (lq + 1) // 2
        return total


def make_decode(seed: int, context_lens, num_q_heads=32, num_kv_heads=8, head_dim=HEAD_DIM,
                block_size=16, num_blocks=None, max_blocks_per_seq=None, pool_factor=1.5,
                scale=None, partition_size=0, write=True, name="custom",
                lengths_fn=None) -> DecodeWorkload:
    """Decode workload.  context_lens: list/tensor, or None with lengths_fn(gen)."""
    gen = torch.Generator().manual_seed(seed)
    if lengths_fn is not None:
        ctx = lengths_fn(gen).to(torch.int32)
    else:
        ctx = torch.as_tensor(context_lens, dtype=torch.int32)
    tables, nb, mb = _deal_blocks(gen, ctx, block_size, num_blocks, max_blocks_per_seq,
                                  pool_factor)
    s = int(ctx.shape[0])
    q = _randn_bf16(gen, (s, num_q_heads, head_dim))
    kc = _randn_bf16(gen, (nb, block_size, num_kv_heads, head_dim), 4096)
    vc = _randn_bf16(gen, (nb, block_size, num_kv_heads, head_dim), 4096)
    writers = [i for i in range(s) if write and int(ctx[i]) > 0]
    kn = _randn_bf16(gen, (len(writers), num_kv_heads, head_dim))
    vn = _randn_bf16(gen, (len(writers), num_kv_heads, head_dim))
    slots = torch.tensor([slot_of(tables, i, int(ctx[i]) - 1, block_size) for i in writers],
                         dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return DecodeWorkload(name, seed, num_q_heads, num_kv_heads, head_dim, block_size, nb, mb,
                          float(scale), int(partition_size), ctx, tables, q, kc, vc, kn, vn,
                          slots)


def make_prefill(seed: int, prefix_lens, q_lens, num_q_heads=32, num_kv_heads=8,
                 head_dim=HEAD_DIM, block_size=16, num_blocks=None, max_blocks_per_seq=None,
                 pool_factor=1.5, scale=None, name="custom", prefix_fn=None) -> PrefillWorkload:
    """Chunked prefill: each sequence has a cached prefix plus q_lens[s] new
    tokens whose K/V the step writes (positions prefix .. prefix + Lq - 1)."""
    gen = torch.Generator().manual_seed(seed)
    if prefix_fn is not None:
        prefix = prefix_fn(gen).to(torch.int32)
    else:
        prefix = torch.as_tensor(prefix_lens, dtype=torch.int32)
    s = int(prefix.shape[0])
    lq = torch.as_tensor(q_lens, dtype=torch.int32)
    if lq.dim() == 0:
        lq = lq.repeat(s)
    ctx = (prefix + lq).to(torch.int32)
    tables, nb, mb = _deal_blocks(gen, ctx, block_size, num_blocks, max_blocks_per_seq,
                                  pool_factor)
    qsl = torch.zeros(s + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(lq, 0).to(torch.int32)
    tq = int(qsl[-1])
    q = _randn_bf16(gen, (tq, num_q_heads, head_dim), 4096)
    kc = _randn_bf16(gen, (nb, block_size, num_kv_heads, head_dim), 4096)
    vc = _randn_bf16(gen, (nb, block_size, num_kv_heads, head_dim), 4096)
    kn = _randn_bf16(gen, (tq, num_kv_heads, head_dim), 4096)
    vn = _randn_bf16(gen, (tq, num_kv_heads, head_dim), 4096)
    slots = torch.empty(tq, dtype=torch.int32)
    for i in range(s):
        p0 = int(prefix[i])
        for r in range(int(lq[i])):
            slots[int(qsl[i]) + r] = slot_of(tables, i, p0 + r, block_size)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PrefillWorkload(name, seed, num_q_heads, num_kv_heads, head_dim, block_size, nb, mb,
                           float(scale), prefix, ctx, qsl, tables, q, kc, vc, kn, vn, slots)


def _uniform_int(lo, hi, n):
    return lambda gen: torch.randint(lo, hi + 1, (n,), generator=gen)


def _log_uniform(lo, hi, n):
    def draw(gen):
        u = torch.rand(n, generator=gen, dtype=torch.float64)
        x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        return torch.round(x).clamp(lo, hi).to(torch.int32)
    return draw


def named(name: str, replica: int = 0):
    """One of the five named workloads; seed = 1000 * index + replica."""
    idx = NAMED[name]
    seed = 1000 * idx + replica
    if name == "tiny":
        return make_decode(seed, [17, 40], num_q_heads=4, num_kv_heads=2, block_size=16,
                           num_blocks=8, max_blocks_per_seq=3, scale=0.125, name=name)
    if name == "llama1b_decode":
        return make_decode(seed, None, lengths_fn=_uniform_int(512, 4096, 64), block_size=16,
                           max_blocks_per_seq=256, scale=0.125, name=name)
    if name == "continuous_batch":
        return make_decode(seed, None, lengths_fn=_log_uniform(16, 8192, 256), block_size=32,
                           max_blocks_per_seq=256, scale=0.125, name=name)
    if name == "long_splitk":
        return make_decode(seed, None, lengths_fn=_uniform_int(32768, 131072, 8), block_size=16,
                           max_blocks_per_seq=8192, scale=0.125, partition_size=512, name=name)
    if name == "chunked_prefill":
        return make_prefill(seed, None, 512, prefix_fn=_uniform_int(0, 2048, 16), block_size=16,
                            max_blocks_per_seq=160, scale=0.125, name=name)
    raise KeyError(name)


def share_prefix(wl, prefix_blocks: int) -> None:
    """Prefix caching [nano-vLLM guide ch. 7]: make every sequence's first
    `prefix_blocks` logical blocks the same physical blocks as sequence 0's
    (in place).  Sequences must all have more than prefix_blocks blocks.  The
    blocks a sequence gave up stay in the pool, unused."""
    bs = wl.block_size
    nb = [(int(c) + bs - 1) // bs for c in wl.context_lens.tolist()]
    if min(nb) <= prefix_blocks:
        raise ValueError("every sequence must extend past the shared prefix")
    wl.block_tables[1:, :prefix_blocks] = wl.block_tables[0, :prefix_blocks]
    if hasattr(wl, "slot_mapping") and wl.slot_mapping.numel():
        # the new tokens live past the prefix, in private blocks: slots unchanged
        pass


def poison_unused(wl, value: float = 1.0e4) -> None:
    """Fill every cache slot that no sequence reads (whole unused blocks and
    the tail of each sequence's last block) with a large finite value, in
    place.  Any over-read then shows up as a large error."""
    bs = wl.block_size
    used = torch.zeros(wl.num_blocks, bs, dtype=torch.bool)
    for s in range(int(wl.context_lens.shape[0])):
        c = int(wl.context_lens[s])
        nfull, rem = c // bs, c % bs
        if nfull:
            used[wl.block_tables[s, :nfull].long()] = True
        if rem:
            used[int(wl.block_tables[s, nfull]), :rem] = True
    mask = ~used
    for cache in (wl.k_cache, wl.v_cache):
        cache[mask] = torch.tensor(value, dtype=BF16)


def to_device(wl, device) -> Dict[str, torch.Tensor]:
    """Device copies of every tensor field."""
    out = {}
    for k, v in vars(wl).items():
        if isinstance(v, torch.Tensor):
            out[k] = v.to(device).contiguous()
    return out
