"""CUDA-graph capture of a decode step [nano-vLLM guide ch. 10 "The
Optimization Stack": CUDA Graphs]: the paged KV write and the decode (with
its split-K merge) are captured once and replayed with new inputs in the
same buffers.  Every replay is checked against the CPU oracle on the inputs
present at replay time -- the cache bit for bit, the output within the
parity tolerance -- and against an eager call on the same inputs, bit for
bit.  The first (eager) call on a device does the library's per-device
set-up, so it comes before the capture."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_198_gb300 as tvl
from paged_kv_cache_198_gb300 import workloads as W
from gpu_common import DEV, assert_clean_status, assert_close, bits_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("part", [0, 512])
def test_graph_replay_matches_oracle(part, fused):
    wl = W.named("llama1b_decode", 0)
    t = W.to_device(wl, DEV)
    s, hq, d = wl.q.shape
    out = torch.empty(s, hq, d, dtype=torch.float32, device=DEV)
    ws = torch.zeros(tvl.paged_attention_decode_workspace_size(
        s, hq, wl.num_kv_heads, d, wl.max_blocks_per_seq, wl.block_size, part) or 16,
        dtype=torch.uint8, device=DEV)

    def step():
        if fused:       # one call: the write fused into the decode
            tvl.paged_decode_step(out, t["q"], t["k_new"], t["v_new"], t["k_cache"],
                                  t["v_cache"], t["block_tables"], t["context_lens"], wl.scale,
                                  partition_size=part, workspace=ws)
        else:
            tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                               t["slot_mapping"])
            tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"],
                                       t["block_tables"], t["context_lens"], wl.scale,
                                       partition_size=part, workspace=ws)

    stream = torch.cuda.Stream(DEV)
    with torch.cuda.stream(stream):
        step()                                    # eager: per-device set-up happens here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    gen = torch.Generator().manual_seed(5)
    for _ in range(3):
        # new inputs in the same buffers, then replay
        q = torch.randn(s, hq, d, generator=gen).to(torch.bfloat16)
        kn = torch.randn(*wl.k_new.shape, generator=gen).to(torch.bfloat16)
        vn = torch.randn(*wl.v_new.shape, generator=gen).to(torch.bfloat16)
        t["q"].copy_(q)
        t["k_new"].copy_(kn)
        t["v_new"].copy_(vn)
        graph.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        # the oracle on the inputs present at replay: the step writes the new
        # rows at each sequence's last position (the same slots every step,
        # so earlier steps' rows are overwritten), then decodes
        kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, kn, vn, wl.slot_mapping)
        assert np.array_equal(bits_of(t["k_cache"]), kc), "replayed write: K cache"
        assert np.array_equal(bits_of(t["v_cache"]), vc), "replayed write: V cache"
        ref = oracle.decode(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        assert_close(replayed.double().cpu().numpy(), ref, f"replay P{part} fused {fused}")
        # and an eager call on the same inputs gives the same bits
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        assert torch.equal(replayed, out)
    assert_clean_status()
