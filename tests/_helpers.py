"""Small shared helpers for the tests (no attention arithmetic here)."""
import numpy as np
import torch


def f64(x: torch.Tensor) -> torch.Tensor:
    """bf16/float tensor -> float64 (exact for bf16)."""
    return x.detach().cpu().to(torch.float64)


def bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def contiguous_tables(ctx_list, block_size, max_blocks=None):
    """Block tables that place sequence s in consecutive physical blocks,
    sequence after sequence (the layout in which paging is a plain slice)."""
    nblk = [(c + block_size - 1) // block_size for c in ctx_list]
    mb = max_blocks or max(1, max(nblk))
    tables = torch.full((len(ctx_list), mb), -1, dtype=torch.int32)
    starts = []
    at = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = torch.arange(at, at + n, dtype=torch.int32)
        starts.append(at)
        at += n
    return tables, starts, max(at, 1)
