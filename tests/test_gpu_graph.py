"""CUDA-graph capture of a decode step [nano-vLLM guide ch. 10 "The
Optimization Stack": CUDA Graphs]: the paged KV write and the decode (with
its split-K merge) are captured once and replayed; every replay must give
exactly the eager result for the inputs present at replay time.  The first
(eager) call on a device does the library's per-device set-up, so it comes
before the capture."""
import numpy as np
import pytest
import torch

import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("part", [0, 512])
def test_graph_replay_equals_eager(part):
    wl = W.named("llama1b_decode", 0)
    t = W.to_device(wl, DEV)
    s, hq, d = wl.q.shape
    out = torch.empty(s, hq, d, dtype=torch.float32, device=DEV)
    ws = torch.zeros(tvl.paged_attention_decode_workspace_size(
        s, hq, wl.num_kv_heads, d, wl.max_blocks_per_seq, wl.block_size, part) or 16,
        dtype=torch.uint8, device=DEV)

    def step():
        tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
        tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], wl.scale, partition_size=part,
                                   workspace=ws)

    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        step()                                    # eager: per-device set-up happens here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    gen = torch.Generator().manual_seed(5)
    for _ in range(3):
        # new inputs in the same buffers, then replay vs eager
        t["q"].copy_(torch.randn(s, hq, d, generator=gen).to(torch.bfloat16))
        t["k_new"].copy_(torch.randn(*t["k_new"].shape, generator=gen).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        assert torch.equal(replayed, out)
    assert_clean_status()
