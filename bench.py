"""Benchmark of the paged-attention hot path on GB300.

Default: the Llama-3.2-1B-shaped single-layer decode step (64 sequences, 32
query / 8 KV heads, head_dim 64, block_size 16, context ~ U{512..4096},
blocks scattered over a 1.5x pool).  One step = the paged KV write of the
batch's 64 new tokens + PagedAttention decode (balanced split-K + merge).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--config NAME]

Prints one JSON line.  `value` is achieved HBM GB/s of the step's algorithmic
bytes (each cached K/V byte counted once, plus q, out, the written rows and
the metadata) over the device-timed step; `seq_steps_per_s` is sequences
decoded per second.  The reference arm (`--impl reference`) times the CPU
oracle on the host cores on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_198_gb300 import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CSRC = os.path.join(ROOT, "paged_kv_cache_198_gb300", "csrc")


# ------------------------------------------------------------------ helpers


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name, files):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        kv = {}
        with open(path) as fh:
            for line in fh:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != source_sha(files):
            return None
        return int(float(kv["traffic_bytes_per_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock and active throttle reasons of the samples taken
        between host times t0 and t1 (all samples when not given)."""
        import datetime

        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if t0 is not None:
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if not (t0 <= ts <= t1):
                    continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def combine_ranks(times_ms, units, world, device):
    """Whole-job view of a weak-scaling run: the slowest rank's times (MAX)
    and the units every rank processed (SUM).  Identity when world == 1."""
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    u = torch.tensor([float(x) for x in units], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], [float(x) for x in u.tolist()]


def rank_workload(name, rank):
    """Each rank decodes its own independent batch (replica seed = rank)."""
    return W.named(name, rank)


# --------------------------------------------------------------- workloads


def decode_algorithmic_bytes(wl):
    s, hq, d = wl.q.shape
    nblk = [(int(c) + wl.block_size - 1) // wl.block_size for c in wl.context_lens.tolist()]
    return (wl.kv_bytes() + s * hq * d * 2 + s * hq * d * 4 + 4 * sum(nblk) + 4 * s)


def write_algorithmic_bytes(wl):
    t = int(wl.slot_mapping.numel())
    return 2 * 2 * t * wl.num_kv_heads * wl.head_dim + 4 * t   # read new + write cache


def prefill_flops(wl):
    return 4.0 * wl.head_dim * wl.num_q_heads * wl.causal_pairs()


# ------------------------------------------------------------ native decode


def pack_pinned(tensors):
    """The step's host inputs in one pinned buffer (each 256-byte aligned), so
    one copy moves them all; returns {"buf", "nbytes", "layout"}."""
    layout, off = {}, 0
    for k, v in tensors.items():
        n = v.numel() * v.element_size()
        layout[k] = (off, v.dtype, tuple(v.shape))
        off += (n + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    for k, v in tensors.items():
        o, _, _ = layout[k]
        n = v.numel() * v.element_size()
        buf[o:o + n].copy_(v.contiguous().view(-1).view(torch.uint8))
    return {"buf": buf, "nbytes": sum(v.numel() * v.element_size() for v in tensors.values()),
            "layout": layout}


def unpack_views(packed, dev_buf):
    """Typed device views into a copy of a pack_pinned buffer."""
    out = {"buf": dev_buf}
    for k, (o, dt, shape) in packed["layout"].items():
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.empty(0, dtype=dt).element_size()
        out[k] = dev_buf[o:o + nbytes].view(dt).view(shape)
    return out


def bench_decode(wl, args, rank, world, device):
    import paged_kv_cache_198_gb300 as tvl

    part = wl.partition_size
    copies = max(1, math.ceil(3 * L2_BYTES / max(1, wl.kv_bytes())) + 1)
    copies = min(copies, 4)
    base = W.to_device(wl, device)
    sets = [base]
    for _ in range(copies - 1):
        sets.append({k: (v.clone() if k in ("k_cache", "v_cache") else v)
                     for k, v in base.items()})
    s, hq, d = wl.q.shape
    out = torch.empty(s, hq, d, dtype=torch.float32, device=device)
    ws_bytes = tvl.paged_attention_decode_workspace_size(
        s, hq, wl.num_kv_heads, d, wl.max_blocks_per_seq, wl.block_size, part)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    if wl.k_new.shape[0] != s:
        raise SystemExit("the decode step needs a new token for every sequence")

    def step(t):
        # one call: the new tokens' paged write fused into the decode (+ merge)
        tvl.paged_decode_step(out, t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                              t["block_tables"], t["context_lens"], wl.scale,
                              partition_size=part, workspace=ws)

    for i in range(args.warmup):
        step(sets[i % copies])
    torch.cuda.synchronize(device)
    if tvl.get_device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    # The timed steps run back to back (each step is one call, so its average
    # duration is the call's); no event sits between the calls, which would
    # break the programmatic overlap of one call's launch with the previous.
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        time.sleep(0.5)                     # let the sampler start
        for i in range(args.warmup):
            step(sets[i % copies])
        torch.cuda.synchronize(device)
        host_t0 = time.time()
        start.record(stream)
        for i in range(args.steps):
            step(sets[i % copies])
        stop.record(stream)
        torch.cuda.synchronize(device)
        host_t1 = time.time()
        time.sleep(0.1)
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = start.elapsed_time(stop)

    # the decode alone (tvl_paged_attention_decode over the written caches),
    # back to back, for the decode-only figure
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    n_dec = max(1, min(args.steps, 2000))
    d0.record(stream)
    for i in range(n_dec):
        t = sets[i % copies]
        tvl.paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], wl.scale, partition_size=part,
                                   workspace=ws)
    d1.record(stream)
    torch.cuda.synchronize(device)
    decode_only_ms = d0.elapsed_time(d1) / n_dec

    # End to end through the public API: every step copies its inputs from
    # pinned host memory (one packed H2D), makes the call and reads its output
    # back.  H2D and D2H run on two copy streams (separate copy engines) with
    # two buffer sets, so the H2D of step i+1 and the D2H of step i-1 overlap
    # step i (double buffering).
    host = pack_pinned({k: v for k, v in W.to_device(wl, "cpu").items()
                        if k in ("q", "k_new", "v_new", "block_tables", "context_lens")})
    out_host = [torch.empty(s, hq, d, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = host["nbytes"]
    d2h = out_host[0].numel() * out_host[0].element_size()
    dev_in = [unpack_views(host, torch.empty_like(host["buf"], device=device)) for _ in range(2)]
    outs = [torch.empty(s, hq, d, dtype=torch.float32, device=device) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device)
    d2h_stream = torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()                      # noqa: E731
    in_ready, done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if used[b]:
                copy_stream.wait_event(done[b])          # step i-2 has read these inputs
            dev_in[b]["buf"].copy_(host["buf"], non_blocking=True)   # one H2D of all inputs
            in_ready[b].record(copy_stream)
        stream.wait_event(in_ready[b])
        if used[b]:
            stream.wait_event(out_read[b])               # step i-2's output was read back
        t = sets[i % copies]
        tvl.paged_decode_step(outs[b], dev_in[b]["q"], dev_in[b]["k_new"], dev_in[b]["v_new"],
                              t["k_cache"], t["v_cache"], dev_in[b]["block_tables"],
                              dev_in[b]["context_lens"], wl.scale, partition_size=part,
                              workspace=ws)
        done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(done[b])
            out_host[b].copy_(outs[b], non_blocking=True)
            out_read[b].record(d2h_stream)
        used[b] = True

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    for i in range(args.steps):
        e2e_step(args.warmup + i)
    stream.wait_event(out_read[(args.warmup + args.steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = e0.elapsed_time(e1)
    if tvl.get_device_status() != 0:
        raise RuntimeError("device status word set during timing")
    return {
        "elapsed_ms": elapsed_ms, "decode_ms": elapsed_ms / args.steps, "e2e_ms": e2e_ms,
        "decode_only_ms": decode_only_ms,
        "h2d": h2d, "d2h": d2h, "copies": copies, "clocks": clocks.summary(host_t0, host_t1),
        "launches_per_step": 2 if (part == 0 or wl.max_blocks_per_seq * wl.block_size > part)
        else 1,
    }


def bench_prefill(wl, args, device):
    """Chunked prefill step: paged write of the chunk's K/V + causal prefill."""
    import paged_kv_cache_198_gb300 as tvl

    base = W.to_device(wl, device)
    cache_bytes = 2 * base["k_cache"].numel() * 2
    copies = min(4, max(1, math.ceil(3 * L2_BYTES / max(1, cache_bytes)) + 1))
    sets = [base] + [{k: (v.clone() if k in ("k_cache", "v_cache", "q") else v)
                      for k, v in base.items()} for _ in range(copies - 1)]
    out = torch.empty(tuple(wl.q.shape), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def prefill(t):
        tvl.paged_attention_prefill(out, t["q"], t["query_start_loc"], t["k_cache"],
                                    t["v_cache"], t["block_tables"], t["context_lens"], wl.scale,
                                    wl.max_q_len)

    def step(t):
        tvl.paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
        prefill(t)

    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    k0 = torch.cuda.Event(enable_timing=True)
    k1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        time.sleep(0.5)
        for i in range(args.warmup):
            step(sets[i % copies])
        torch.cuda.synchronize(device)
        host_t0 = time.time()
        # the step (write + prefill), back to back
        start.record(stream)
        for i in range(args.steps):
            step(sets[i % copies])
        stop.record(stream)
        # the prefill kernel alone, back to back, for its roofline
        k0.record(stream)
        for i in range(args.steps):
            prefill(sets[i % copies])
        k1.record(stream)
        torch.cuda.synchronize(device)
        host_t1 = time.time()
        time.sleep(0.1)
    if tvl.get_device_status() != 0:
        raise RuntimeError("device status word set during timing")
    # End to end: each step copies its inputs from pinned host memory (one
    # packed H2D), writes the chunk, runs the prefill and reads the output
    # back.  H2D and D2H run on two copy streams (the two directions use
    # separate copy engines) with two buffer sets, so step i's compute
    # overlaps the H2D of step i+1 and the D2H of step i-1.
    host = pack_pinned({k: base[k].cpu() for k in ("q", "k_new", "v_new", "slot_mapping",
                                                   "query_start_loc", "block_tables",
                                                   "context_lens")})
    out_host = [torch.empty(tuple(wl.q.shape), dtype=torch.float32).pin_memory()
                for _ in range(2)]
    dev_in = [unpack_views(host, torch.empty_like(host["buf"], device=device)) for _ in range(2)]
    outs = [torch.empty(tuple(wl.q.shape), dtype=torch.float32, device=device) for _ in range(2)]
    h2d_stream = torch.cuda.Stream(device)
    d2h_stream = torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()                      # noqa: E731
    in_ready, done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d_stream):
            if used[b]:
                h2d_stream.wait_event(done[b])           # step i-2 has read these inputs
            dev_in[b]["buf"].copy_(host["buf"], non_blocking=True)
            in_ready[b].record(h2d_stream)
        stream.wait_event(in_ready[b])
        if used[b]:
            stream.wait_event(out_read[b])               # step i-2's output was read back
        t, d = sets[i % copies], dev_in[b]
        tvl.paged_kv_write(d["k_new"], d["v_new"], t["k_cache"], t["v_cache"], d["slot_mapping"])
        tvl.paged_attention_prefill(outs[b], d["q"], d["query_start_loc"], t["k_cache"],
                                    t["v_cache"], d["block_tables"], d["context_lens"],
                                    wl.scale, wl.max_q_len)
        done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(done[b])
            out_host[b].copy_(outs[b], non_blocking=True)
            out_read[b].record(d2h_stream)
        used[b] = True

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    e2e_steps = max(2, min(args.steps, 200))
    for i in range(e2e_steps):
        e2e_step(args.warmup + i)
    stream.wait_event(out_read[(args.warmup + e2e_steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(device)
    return {
        "elapsed_ms": start.elapsed_time(stop),
        "kernel_ms": k0.elapsed_time(k1) / args.steps,
        "e2e_ms_per_step": e0.elapsed_time(e1) / e2e_steps,
        "h2d": host["nbytes"],
        "d2h": out_host[0].numel() * out_host[0].element_size(), "copies": copies,
        "clocks": clocks.summary(host_t0, host_t1),
    }


def prefill_line(wl, args, r, bf16_sus, peak_src):
    flops = prefill_flops(wl)
    per_step_ms = r["elapsed_ms"] / args.steps
    achieved = flops / (r["kernel_ms"] / 1e3) / 1e12
    return {
        "metric": "chunked causal prefill TFLOP/s (causal-visible pairs, % of bf16 tensor peak)",
        "value": round(flops / (per_step_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "num_seqs": wl.num_seqs,
                   "heads": f"{wl.num_q_heads}/{wl.num_kv_heads}", "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "query_tokens": wl.total_q,
                   "context_tokens": int(wl.context_lens.sum()),
                   "causal_pairs": wl.causal_pairs(), "flops_per_step": flops,
                   "step": "paged KV write of the chunk + causal prefill",
                   "l2": f"{r['copies']} rotating copies of q and the caches"},
        "roofline": {"kernel": "prefill_kernel", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": bf16_sus, "unit": "TFLOP/s", "frac": round(achieved / bf16_sus, 4),
                     "traffic": recorded_traffic("prefill_chunked_prefill.txt",
                                                 ["prefill.cu", "tc.cuh", "device.cuh"]),
                     "peak_source": f"{peak_src} bf16_tflops_sustained (the kernel runs in a "
                                    f"seconds-long loop)",
                     "launch_ms_mean": round(r["kernel_ms"], 5),
                     "launch_timing": "prefill calls back to back over a timed region of "
                                      "their own, CUDA events around it"},
        "e2e": {"value": round(flops / (r["e2e_ms_per_step"] / 1e3) / 1e12, 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": 2 * args.steps,     # the step's region; the kernel-only one adds K more
        "clocks": r["clocks"],
    }


def cpu_baseline_decode(wl, budget_s=10.0):
    """The oracle (write + decode of the whole batch) on the host cores,
    repeated until about budget_s seconds have passed."""
    import oracle

    oracle.build()
    cores = oracle.max_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new, wl.slot_mapping)
        oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    per_step = (time.perf_counter() - t0) / reps
    return per_step, cores, reps


ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
             "0xd8e": "Arm Neoverse N3", "0xd84": "Arm Neoverse V3"}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    v = line.split(":", 1)[1].strip()
                    return f"{ARM_PARTS[v]} ({v})" if v in ARM_PARTS else v
    except Exception:
        pass
    return os.uname().machine


# -------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="llama1b_decode",
                    choices=["llama1b_decode", "continuous_batch", "long_splitk", "tiny",
                             "chunked_prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()
    metric = "paged-attn decode achieved HBM GB/s (% of GB300 peak); seq-steps/sec"

    if args.impl == "reference":
        if rank != 0:
            return
        wl = W.named(args.config, 0)
        import oracle

        oracle.build()
        for _ in range(args.warmup if args.warmup <= 3 else 3):
            pass
        step_bytes = decode_algorithmic_bytes(wl) + write_algorithmic_bytes(wl)
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new,
                                     wl.slot_mapping)
            oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        per = sum(times) / len(times)
        val = step_bytes / per / 1e9
        line = {
            "impl": "reference", "metric": metric, "value": round(val, 3), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "seq_steps_per_s": round(wl.num_seqs / per, 1),
            "config": {"workload": wl.name, "num_seqs": wl.num_seqs,
                       "heads": f"{wl.num_q_heads}/{wl.num_kv_heads}",
                       "head_dim": wl.head_dim, "block_size": wl.block_size,
                       "partition_size": wl.partition_size},
            "cpu_baseline": {"value": round(val, 3), "unit": "GB/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": "the whole workload (paged write + decode of every "
                                       "sequence) per step; " + cpu_model()},
            "e2e": {"value": round(val, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_cache_198_gb300 import _build

    if rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()

    wl = rank_workload(args.config, rank)
    if args.config == "chunked_prefill":
        if world > 1:
            raise SystemExit("the prefill line is measured on one GPU")
        print(json.dumps(prefill_line(wl, args, bench_prefill(wl, args, device), bf16_sus,
                                      peak_src)))
        return
    r = bench_decode(wl, args, rank, world, device)
    step_bytes = decode_algorithmic_bytes(wl) + write_algorithmic_bytes(wl)
    (t_ms, e2e_ms), (total_bytes, total_seqs) = combine_ranks(
        [r["elapsed_ms"], r["e2e_ms"]], [float(step_bytes), float(wl.num_seqs)], world, device)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    per_step_ms = t_ms / args.steps
    value = total_bytes * args.steps / (t_ms / 1e3) / 1e9
    e2e_val = total_bytes * args.steps / (e2e_ms / 1e3) / 1e9

    dec_bytes = step_bytes            # the call writes the new tokens and decodes
    achieved = dec_bytes / (r["decode_ms"] / 1e3) / 1e9
    traffic = recorded_traffic("decode_llama1b_decode.txt", ["decode.cu", "device.cuh"])
    line = {
        "metric": metric, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "seq_steps_per_s": round(total_seqs * args.steps / (t_ms / 1e3), 1),
        "config": {
            "workload": wl.name, "num_seqs": wl.num_seqs,
            "heads": f"{wl.num_q_heads}/{wl.num_kv_heads}", "head_dim": wl.head_dim,
            "block_size": wl.block_size, "num_blocks": wl.num_blocks,
            "context_tokens": int(wl.context_lens.sum()),
            "partition_size": wl.partition_size,
            "step": "one tvl_paged_decode_step call: paged KV write of the new tokens fused "
                    "into the paged decode (+ split-K merge)",
            "bytes_per_step": step_bytes,
            "l2": f"inputs larger than L2: {r['copies']} rotating cache copies, "
                  f"{wl.kv_bytes() / 1e6:.0f} MB K/V read per step vs 129 MB L2",
        },
        "roofline": {
            "kernel": "decode step (decode_kernel with the fused write + merge_kernel, one "
                      "C-ABI call)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": dec_bytes,
            "launch_ms_mean": round(r["decode_ms"], 5),
            "launch_timing": "calls back to back over the timed region, CUDA events around it",
        },
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": round(e2e_ms / args.steps, 4),
                "copies": "pinned host buffers, H2D and D2H streams and two device buffer "
                          "sets: the H2D of step i+1 and the D2H of step i-1 overlap step i"},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
        "decode_only": {
            "call": "tvl_paged_attention_decode (decode + merge, the write not included)",
            "ms_per_call": round(r["decode_only_ms"], 5),
            "achieved_gbs": round(decode_algorithmic_bytes(wl) / (r["decode_only_ms"] / 1e3)
                                  / 1e9, 1),
            "frac": round(decode_algorithmic_bytes(wl) / (r["decode_only_ms"] / 1e3) / 1e9
                          / hbm_peak, 4)},
    }
    if not args.no_cpu_baseline and world == 1:
        per, cores, reps = cpu_baseline_decode(wl)
        line["cpu_baseline"] = {
            "value": round(step_bytes / per / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} full steps (paged write + fp64 decode of all {wl.num_seqs} "
                      f"sequences), {per:.3f} s each; {cpu_model()}"}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
