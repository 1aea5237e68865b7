"""Writes tests/golden/tiny_decode.txt from the CPU oracle alone.

The fixture is the oracle's float64 decode output for the "tiny" workload
(2 sequences, context lengths 17 and 40, 4 query / 2 KV heads, head_dim 64,
block_size 16, 8 physical blocks, scale 1/8) after the paged write of one new
token per sequence; one row per (sequence, query head), 64 columns.
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_cache_198_gb300 import workloads as W  # noqa: E402


def main():
    wl = W.named("tiny")
    kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
    out = oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.txt")
    header = ("oracle float64 decode of the tiny workload (seed 1000); rows = (seq, head), "
              "cols = head_dim")
    np.savetxt(path, out.reshape(-1, out.shape[-1]), fmt="%.17g", header=header)
    print("wrote", path)


if __name__ == "__main__":
    main()
