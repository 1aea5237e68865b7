"""Shared pieces of the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W

MAX_ABS = 2e-3
MEAN_ABS = 2e-4
DEV = "cuda:0"


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def gpu_decode(wl, partition_size=None, write=True, dev=DEV, tensors=None):
    """Paged write (optional) + decode on the GPU; returns (out float64, device tensors)."""
    t = tensors if tensors is not None else W.to_device(wl, dev)
    if write and t["slot_mapping"].numel():
        tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = torch.full(tuple(wl.q.shape), float("nan"), dtype=torch.float32, device=dev)
    part = wl.partition_size if partition_size is None else partition_size
    tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                               t["context_lens"], wl.scale, partition_size=part)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), t


def oracle_caches(wl, write=True):
    if write and wl.slot_mapping.numel():
        return oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    return bits_of(wl.k_cache), bits_of(wl.v_cache)


def oracle_decode(wl, write=True, seq_mask=None):
    kc, vc = oracle_caches(wl, write)
    return oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale,
                         seq_mask=seq_mask)


def assert_close(got, ref, what=""):
    keep = ~np.isnan(ref).any(axis=-1)
    assert keep.any(), "nothing to compare"
    err = np.abs(got[keep] - ref[keep])
    assert np.isfinite(got[keep]).all(), f"{what}: non-finite output"
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (
        f"{what}: max abs {err.max():.3e} (<= {MAX_ABS}), mean abs {err.mean():.3e} "
        f"(<= {MEAN_ABS})")
    return float(err.max()), float(err.mean())


def assert_clean_status():
    bits = tvl.get_device_status()
    assert bits == 0, f"device status bits 0x{bits:x}"
