"""Benchmark of the paged-attention hot path on GB300.

Default: the Llama-3.2-1B-shaped single-layer decode step (64 sequences, 32
query / 8 KV heads, head_dim 64, block_size 16, context ~ U{512..4096},
blocks scattered over a 1.5x pool).  One step = the paged KV write of the
batch's 64 new tokens + PagedAttention decode (balanced split-K + merge), one
tvl_paged_decode_step call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--config NAME] [--no-extras] [--no-cpu-baseline]

Prints one JSON line.  `value` is achieved HBM GB/s of the step's algorithmic
bytes (each cached K/V byte counted once, plus q, out, the written rows and
the metadata) over the device-timed step; `seq_steps_per_s` is sequences
decoded per second.  With the default config on one GPU the same line also
carries the other measured workloads under their names -- `continuous_batch`
(256 sequences, log-uniform lengths, bs 32), `long_splitk` (8 sequences of
32k-128k tokens, 512-token windows) and `chunked_prefill` (16 x (prefix
U{0..2048} + 512), tensor-core prefill) -- each with its own roofline,
end-to-end figure, clock record and CPU-oracle sample.  The reference arm
(`--impl reference`) times the CPU oracle on the host cores on the same
workload.

Timing: W untimed warm-up steps; then, after a synchronize (and a barrier
when N > 1), a short GPU hold kernel is queued so that the host has queued
the first steps before the start event fires, and exactly K steps run back
to back between two CUDA events on the launching stream.  Inputs are larger
than L2 (rotating cache copies).  After the K steps the same step runs back
to back for at least a second while nvidia-smi samples the SM clock; that
region's per-step time and clocks are reported beside the K-step figure.
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
HOLD_CYCLES = 400_000            # ~0.2 ms GPU hold before each timed region
SUSTAIN_S = 1.0                  # length of the clock-sampled region
DECODE_SOURCES = ["decode.cu", "device.cuh"]
PREFILL_SOURCES = ["prefill.cu", "tc.cuh", "device.cuh"]


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


def recorded_profile(profile_name, files):
    """key: value pairs of a committed ncu summary, if it was taken on the
    current kernel source (else None)."""
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
        return kv
    except Exception:
        return None


def recorded_traffic(profile_name, files):
    """DRAM bytes per launch from a committed ncu summary taken on the
    current kernel source (else None)."""
    kv = recorded_profile(profile_name, files)
    try:
        return int(float(kv["traffic_bytes_per_launch"])) if kv else None
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.samples = []         # (host time, sm MHz, max MHz, power W, active reasons)
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
        import datetime

        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = None
            active = [n for n, v in zip(self.NAMES, parts[5:9]) if v.lower() == "active"]
            self.samples.append((ts, sm, mx, pw, active))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0, t1):
        """Median SM clock and the throttle reasons of the samples taken
        between host times t0 and t1.  A window shorter than the sampling
        period may hold none: then the last sample before t0 and the first
        after t1 stand in for it (window "nearest")."""
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        window = "timed region"
        if not inside:
            before = [x for x in self.samples if x[0] < t0]
            after = [x for x in self.samples if x[0] > t1]
            inside = ([before[-1]] if before else []) + ([after[0]] if after else [])
            window = "nearest"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for x in inside for r in x[4]})
        powers = [x[3] for x in inside if x[3] is not None]
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "reasons": reasons,
                "samples": len(inside), "window": window,
                "power_w_median": statistics.median(powers) if powers else None}


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


def warm_up(run, w, min_s=0.2):
    """At least w untimed calls, and more until min_s seconds have passed
    (a GPU that sat idle while the host drew inputs runs its first
    milliseconds slower).  Returns the number of calls made."""
    t0 = time.perf_counter()
    i = 0
    while i < w or time.perf_counter() - t0 < min_s:
        run(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    return i


def timed_region(run, n, stream):
    """ms of n back-to-back run(i) calls between two CUDA events on `stream`.
    A GPU hold kernel is queued first, so the start event fires only after
    the host has queued the first calls (the region then measures the GPU,
    not the host's first enqueue)."""
    torch.cuda.synchronize()
    torch.cuda._sleep(HOLD_CYCLES)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(n):
        run(i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def sustained_region(run, ms_per_call, stream, device):
    """The same calls back to back for at least SUSTAIN_S seconds while
    nvidia-smi samples: (ms per call, clock summary of the region, calls)."""
    n = int(min(200_000, max(20, math.ceil(SUSTAIN_S * 1e3 / max(ms_per_call, 1e-3)))))
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        time.sleep(0.3)                      # let the sampler start
        t0 = time.time()
        ms = timed_region(run, n, stream)
        t1 = time.time()
        time.sleep(0.1)
    summ = clocks.summary(t0, t1)
    return ms / n, summ, n


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


class E2E:
    """End-to-end steps through the public API: each step copies its inputs
    from pinned host memory (one packed H2D), makes the library call(s) and
    reads its output back.  H2D and D2H run on their own streams with two
    device buffer sets, so the H2D of step i+1 and the D2H of step i-1
    overlap step i (double buffering)."""

    def __init__(self, host_inputs, out_shape, device, bind, period):
        """bind(buffer_views, out, i) -> callable issuing step i's library
        call(s) on the current stream with the inputs in buffer_views; the
        call of step i is that of step i + 2 * period (the rotating cache
        copies repeat every `period` steps)."""
        self.host = pack_pinned(host_inputs)
        self.out_host = [torch.empty(out_shape, dtype=torch.float32).pin_memory()
                         for _ in range(2)]
        self.dev_in = [unpack_views(self.host, torch.empty_like(self.host["buf"], device=device))
                       for _ in range(2)]
        self.outs = [torch.empty(out_shape, dtype=torch.float32, device=device)
                     for _ in range(2)]
        self.stream = torch.cuda.current_stream(device)
        self.h2d_stream = torch.cuda.Stream(device)
        self.d2h_stream = torch.cuda.Stream(device)
        ev = torch.cuda.Event
        self.in_ready, self.done, self.out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        self.used = [False, False]
        self.bind = bind
        self.period = period
        self.calls = {}
        self.h2d_bytes = self.host["nbytes"]
        self.d2h_bytes = self.out_host[0].numel() * 4

    def step(self, i):
        b = i % 2
        key = (b, i % self.period)
        call = self.calls.get(key)
        if call is None:
            call = self.calls[key] = self.bind(self.dev_in[b], self.outs[b], i)
        h2d, d2h, stream = self.h2d_stream, self.d2h_stream, self.stream
        if self.used[b]:
            h2d.wait_event(self.done[b])            # step i-2 has read these inputs
        with torch.cuda.stream(h2d):
            self.dev_in[b]["buf"].copy_(self.host["buf"], non_blocking=True)
        self.in_ready[b].record(h2d)
        stream.wait_event(self.in_ready[b])
        if self.used[b]:
            stream.wait_event(self.out_read[b])     # step i-2's output was read back
        call()
        self.done[b].record(stream)
        d2h.wait_event(self.done[b])
        with torch.cuda.stream(d2h):
            self.out_host[b].copy_(self.outs[b], non_blocking=True)
        self.out_read[b].record(d2h)
        self.used[b] = True

    def run(self, warmup, steps):
        """ms per step of `steps` steps (after `warmup`), CUDA events on the
        compute stream around all of them, the last read-back included."""
        for i in range(warmup):
            self.step(i)
        torch.cuda.synchronize()
        torch.cuda._sleep(HOLD_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        self.h2d_stream.wait_event(e0)
        for i in range(steps):
            self.step(warmup + i)
        self.stream.wait_event(self.out_read[(warmup + steps - 1) % 2])
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps


# ------------------------------------------------------------ native decode


def bench_decode(wl, args, world, device, decode_only=True):
    import paged_kv_cache_198_gb300 as tvl

    part = wl.partition_size
    copies = min(4, max(1, math.ceil(3 * L2_BYTES / max(1, wl.kv_bytes())) + 1))
    base = W.to_device(wl, device)
    sets = [base] + [{k: (v.clone() if k in ("k_cache", "v_cache") else v)
                      for k, v in base.items()} for _ in range(copies - 1)]
    s, hq, d = wl.q.shape
    if wl.k_new.shape[0] != s:
        raise SystemExit("the decode step needs a new token for every sequence")
    out = torch.empty(s, hq, d, dtype=torch.float32, device=device)
    ws_bytes = tvl.paged_attention_decode_workspace_size(
        s, hq, wl.num_kv_heads, d, wl.max_blocks_per_seq, wl.block_size, part)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    # one call per step: the new tokens' paged write fused into the decode (+ merge)
    steps = [tvl.bind_paged_decode_step(out, t["q"], t["k_new"], t["v_new"], t["k_cache"],
                                        t["v_cache"], t["block_tables"], t["context_lens"],
                                        wl.scale, partition_size=part, workspace=ws)
             for t in sets]

    def run(i):
        steps[i % copies]()

    args.warmup_run = warm_up(run, args.warmup, 0.0 if args.quick else 0.2)
    torch.cuda.synchronize(device)
    if tvl.get_device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = timed_region(run, args.steps, stream)
    if world > 1:
        torch.distributed.barrier()
    if args.quick:
        return {"elapsed_ms": elapsed_ms, "step_ms": elapsed_ms / args.steps, "copies": copies}
    sus_ms, clocks, sus_n = sustained_region(run, elapsed_ms / args.steps, stream, device)

    res = {"elapsed_ms": elapsed_ms, "step_ms": elapsed_ms / args.steps, "copies": copies,
           "warmup_run": args.warmup_run,
           "sustained_ms": sus_ms, "sustained_steps": sus_n, "clocks": clocks,
           "launches_per_step": 2 if (part == 0 or wl.max_blocks_per_seq * wl.block_size > part)
           else 1}

    if decode_only:
        # the decode alone (tvl_paged_attention_decode over the written
        # caches), back to back, for the decode-only figure
        decs = [tvl.bind_paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"],
                                                t["block_tables"], t["context_lens"], wl.scale,
                                                partition_size=part, workspace=ws)
                for t in sets]
        n_dec = max(20, min(args.steps, 2000))
        res["decode_only_ms"] = timed_region(lambda i: decs[i % copies](), n_dec, stream) / n_dec

    # end to end through the public API (pinned host inputs in, output out)
    def bind(dv, o, i):
        t = sets[i % copies]
        return tvl.bind_paged_decode_step(o, dv["q"], dv["k_new"], dv["v_new"], t["k_cache"],
                                          t["v_cache"], dv["block_tables"], dv["context_lens"],
                                          wl.scale, partition_size=part, workspace=ws)

    e2e = E2E({k: v for k, v in W.to_device(wl, "cpu").items()
               if k in ("q", "k_new", "v_new", "block_tables", "context_lens")},
              (s, hq, d), device, bind, copies)
    res["e2e_ms"] = e2e.run(args.warmup, max(args.steps, 20))
    res["h2d"], res["d2h"] = e2e.h2d_bytes, e2e.d2h_bytes
    if tvl.get_device_status() != 0:
        raise RuntimeError("device status word set during timing")
    return res


def decode_entry(wl, r, hbm_peak, peak_src, profile, steps):
    """Fields of one decode workload's result (headline or extra)."""
    step_bytes = decode_algorithmic_bytes(wl) + write_algorithmic_bytes(wl)
    gbs = step_bytes / (r["step_ms"] / 1e3) / 1e9
    d = {
        "metric": "paged-attn decode achieved HBM GB/s (% of GB300 peak); seq-steps/sec",
        "value": round(gbs, 2), "unit": "GB/s", "steps": steps,
        "ms_per_step": round(r["step_ms"], 5),
        "seq_steps_per_s": round(wl.num_seqs / (r["step_ms"] / 1e3), 1),
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
            "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(gbs / hbm_peak, 4),
            "traffic": recorded_traffic(profile, DECODE_SOURCES),
            "traffic_source": f"profiles/{profile} (dram read + write per launch, when taken "
                              "on the current kernel source)",
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
            "algorithmic_bytes_per_launch": step_bytes,
            "launch_ms_mean": round(r["step_ms"], 5),
            "launch_timing": "calls back to back over the timed region (one call per step), "
                             "CUDA events around it on the launching stream",
        },
        "e2e": {"value": round(step_bytes / (r["e2e_ms"] / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": round(r["e2e_ms"], 5),
                "copies": "pinned host buffers, H2D and D2H streams and two device buffer "
                          "sets: the H2D of step i+1 and the D2H of step i-1 overlap step i"},
        "clocks": r["clocks"],
        "sustained": {"ms_per_step": round(r["sustained_ms"], 5),
                      "value": round(step_bytes / (r["sustained_ms"] / 1e3) / 1e9, 2),
                      "steps": r["sustained_steps"],
                      "frac": round(step_bytes / (r["sustained_ms"] / 1e3) / 1e9 / hbm_peak, 4),
                      "note": "the same step back to back for >= 1 s right after the timed "
                              "steps; `clocks` were sampled over this region"},
        "gpu_launches": r["launches_per_step"] * steps,
        "warmup_run": r.get("warmup_run"),
    }
    if "decode_only_ms" in r:
        dob = decode_algorithmic_bytes(wl)
        d["decode_only"] = {
            "call": "tvl_paged_attention_decode (decode + merge, the write not included)",
            "ms_per_call": round(r["decode_only_ms"], 5),
            "achieved_gbs": round(dob / (r["decode_only_ms"] / 1e3) / 1e9, 1),
            "frac": round(dob / (r["decode_only_ms"] / 1e3) / 1e9 / hbm_peak, 4)}
    return d


# ------------------------------------------------------------ native prefill


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
    writes = [tvl.bind_paged_kv_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                                      t["slot_mapping"]) for t in sets]
    prefills = [tvl.bind_paged_attention_prefill(out, t["q"], t["query_start_loc"],
                                                 t["k_cache"], t["v_cache"], t["block_tables"],
                                                 t["context_lens"], wl.scale, wl.max_q_len)
                for t in sets]

    def step(i):
        writes[i % copies]()
        prefills[i % copies]()

    args.warmup_run = warm_up(step, args.warmup, 0.0 if args.quick else 0.2)
    torch.cuda.synchronize(device)
    elapsed = timed_region(step, args.steps, stream)
    kernel = timed_region(lambda i: prefills[i % copies](), args.steps, stream)
    if args.quick:
        return {"step_ms": elapsed / args.steps, "kernel_ms": kernel / args.steps}
    sus_ms, clocks, sus_n = sustained_region(lambda i: prefills[i % copies](),
                                             kernel / args.steps, stream, device)
    if tvl.get_device_status() != 0:
        raise RuntimeError("device status word set during timing")

    def bind(dv, o, i):
        t = sets[i % copies]
        w = tvl.bind_paged_kv_write(dv["k_new"], dv["v_new"], t["k_cache"], t["v_cache"],
                                    dv["slot_mapping"])
        p = tvl.bind_paged_attention_prefill(o, dv["q"], dv["query_start_loc"], t["k_cache"],
                                             t["v_cache"], dv["block_tables"],
                                             dv["context_lens"], wl.scale, wl.max_q_len)

        def both():
            w()
            p()
        return both

    e2e = E2E({k: base[k].cpu() for k in ("q", "k_new", "v_new", "slot_mapping",
                                          "query_start_loc", "block_tables", "context_lens")},
              tuple(wl.q.shape), device, bind, copies)
    e2e_ms = e2e.run(args.warmup, max(2, min(args.steps, 200)))
    return {"step_ms": elapsed / args.steps, "kernel_ms": kernel / args.steps,
            "sustained_ms": sus_ms, "sustained_steps": sus_n, "clocks": clocks,
            "e2e_ms": e2e_ms, "h2d": e2e.h2d_bytes, "d2h": e2e.d2h_bytes, "copies": copies,
            "warmup_run": args.warmup_run}


def prefill_entry(wl, r, bf16_burst, bf16_sus, peak_src, steps):
    flops = prefill_flops(wl)
    achieved = flops / (r["kernel_ms"] / 1e3) / 1e12
    prof = recorded_profile("prefill_chunked_prefill.txt", PREFILL_SOURCES)
    return {
        "metric": "chunked causal prefill TFLOP/s (causal-visible pairs, % of bf16 tensor peak)",
        "value": round(flops / (r["step_ms"] / 1e3) / 1e12, 2), "unit": "TFLOP/s",
        "steps": steps, "ms_per_step": round(r["step_ms"], 5),
        "config": {"workload": wl.name, "num_seqs": wl.num_seqs,
                   "heads": f"{wl.num_q_heads}/{wl.num_kv_heads}", "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "query_tokens": wl.total_q,
                   "context_tokens": int(wl.context_lens.sum()),
                   "causal_pairs": wl.causal_pairs(), "flops_per_step": flops,
                   "step": "paged KV write of the chunk + causal prefill (two calls)",
                   "l2": f"{r['copies']} rotating copies of q and the caches"},
        "roofline": {"kernel": "prefill_kernel", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": bf16_burst, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16_burst, 4),
                     "traffic": int(float(prof["traffic_bytes_per_launch"])) if prof else None,
                     "tensor_pipe_pct": float(prof["tensor_pipe_pct"]) if prof and
                     "tensor_pipe_pct" in prof else None,
                     "profile": "profiles/prefill_chunked_prefill.txt (ncu, when taken on the "
                                "current kernel source)",
                     "peak_source": f"{peak_src} bf16_tflops (burst: the K launches are a "
                                    f"short region; the sustained region below is set "
                                    f"against bf16_tflops_sustained)",
                     "algorithmic_flops_per_launch": flops,
                     "launch_ms_mean": round(r["kernel_ms"], 5),
                     "launch_timing": "prefill calls back to back over a timed region of "
                                      "their own, CUDA events around it"},
        "e2e": {"value": round(flops / (r["e2e_ms"] / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": round(r["e2e_ms"], 5),
                "note": "copy-bound: 50 MB in and 67 MB out per step over the host link"},
        "clocks": r["clocks"],
        "sustained": {"ms_per_launch": round(r["sustained_ms"], 5),
                      "achieved": round(flops / (r["sustained_ms"] / 1e3) / 1e12, 1),
                      "peak": bf16_sus,
                      "frac": round(flops / (r["sustained_ms"] / 1e3) / 1e12 / bf16_sus, 4),
                      "launches": r["sustained_steps"],
                      "note": "prefill calls back to back for >= 1 s; `clocks` were sampled "
                              "over this region"},
        "gpu_launches": 2 * steps,
        "warmup_run": r.get("warmup_run"),
    }


# ------------------------------------------------------------ CPU baselines


def cpu_baseline_decode(wl, budget_s=10.0, seqs=None):
    """The oracle on the host cores, repeated until about budget_s seconds
    have passed: the paged write + decode of the whole batch, or (seqs given)
    the decode of only those sequences on the drawn cache.  Returns
    (seconds per repetition, bytes per repetition, threads, repetitions)."""
    import numpy as np
    import oracle

    oracle.build()
    cores = oracle.max_threads()
    if seqs is None:
        nbytes = decode_algorithmic_bytes(wl) + write_algorithmic_bytes(wl)
    else:
        mask = np.zeros(wl.num_seqs, dtype=np.uint8)
        mask[list(seqs)] = 1
        ctx = wl.context_lens.tolist()
        nbytes = sum(ctx[i] for i in seqs) * wl.num_kv_heads * wl.head_dim * 4
    reps, t0 = 0, time.perf_counter()
    while True:
        if seqs is None:
            kc, vc = oracle.kv_write(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new,
                                     wl.slot_mapping)
            oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        else:
            oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                          wl.scale, seq_mask=mask)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return (time.perf_counter() - t0) / reps, nbytes, cores, reps


def cpu_baseline_prefill(wl, every=32):
    """The oracle prefill of every `every`-th query row (all heads) on the
    host cores: (seconds, flops of those rows, threads)."""
    import numpy as np
    import oracle

    oracle.build()
    mask = np.zeros(wl.total_q, dtype=np.uint8)
    mask[::every] = 1
    qsl = wl.query_start_loc.tolist()
    ctx = wl.context_lens.tolist()
    pairs = 0
    for s in range(wl.num_seqs):
        lq = qsl[s + 1] - qsl[s]
        for i in range(lq):
            if mask[qsl[s] + i]:
                pairs += ctx[s] - lq + i + 1
    flops = 4.0 * wl.head_dim * wl.num_q_heads * pairs
    t0 = time.perf_counter()
    oracle.prefill(wl.q, wl.query_start_loc, wl.k_cache, wl.v_cache, wl.block_tables,
                   wl.context_lens, wl.scale, row_mask=mask)
    return time.perf_counter() - t0, flops, oracle.max_threads()


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


def reference_arm(args, metric):
    """The oracle on the host cores as the reference arm, on the same
    workload, metric and unit as the native line."""
    wl = W.named(args.config, 0)
    import oracle

    oracle.build()
    if args.config == "chunked_prefill":
        times = []
        for i in range(args.warmup + args.steps):
            sec, flops, cores = cpu_baseline_prefill(wl, every=64)
            if i >= args.warmup:
                times.append(sec)
        per = sum(times) / len(times)
        val = flops / per / 1e12
        line = {"impl": "reference", "metric": "chunked causal prefill TFLOP/s (causal-visible "
                "pairs, % of bf16 tensor peak)", "value": round(val, 6), "unit": "TFLOP/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(per * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name}}
        sample = "every 64th query row of the batch (all heads) per step; " + cpu_model()
    else:
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
                       "partition_size": wl.partition_size}}
        sample = ("the whole workload (paged write + decode of every sequence) per step; "
                  + cpu_model())
    line["cpu_baseline"] = {"value": line["value"], "unit": line["unit"],
                            "cores": oracle.max_threads(), "kind": "oracle", "sample": sample}
    line["e2e"] = {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="llama1b_decode",
                    choices=["llama1b_decode", "continuous_batch", "long_splitk", "tiny",
                             "chunked_prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="print the selected workload only")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: the W warm-up and K timed steps only (no sustained, "
                         "decode-only or end-to-end regions, no CPU baseline, no extras); "
                         "prints ms per step")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.steps = max(1, args.steps)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()
    metric = "paged-attn decode achieved HBM GB/s (% of GB300 peak); seq-steps/sec"

    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, metric)
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

    common = {"n_gpus": world, "warmup": args.warmup, "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}

    wl = rank_workload(args.config, rank)
    if args.quick:
        if args.config == "chunked_prefill":
            r = bench_prefill(wl, args, device)
        else:
            r = bench_decode(wl, args, world, device, decode_only=False)
        print(json.dumps({"quick": True, "workload": wl.name,
                          **{k: round(v, 5) for k, v in r.items() if k.endswith("_ms")}}))
        return
    if args.config == "chunked_prefill":
        if world > 1:
            raise SystemExit("the prefill line is measured on one GPU")
        e = prefill_entry(wl, bench_prefill(wl, args, device), bf16_peak, bf16_sus, peak_src,
                          args.steps)
        line = {**{k: e[k] for k in ("metric", "value", "unit")}, **common, **e}
        print(json.dumps(line))
        return

    r = bench_decode(wl, args, world, device, decode_only=True)
    step_bytes = decode_algorithmic_bytes(wl) + write_algorithmic_bytes(wl)
    (t_ms, e2e_ms), (total_bytes, total_seqs) = combine_ranks(
        [r["elapsed_ms"], r["e2e_ms"] * args.steps], [float(step_bytes), float(wl.num_seqs)],
        world, device)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    e = decode_entry(wl, r, hbm_peak, peak_src, f"decode_{wl.name}.txt", args.steps)
    line = {"metric": metric, "value": round(total_bytes * args.steps / (t_ms / 1e3) / 1e9, 2),
            "unit": "GB/s", **common, "steps": args.steps,
            "ms_per_step": round(t_ms / args.steps, 5),
            "seq_steps_per_s": round(total_seqs * args.steps / (t_ms / 1e3), 1)}
    for k in ("config", "roofline", "e2e", "gpu_launches", "clocks", "sustained", "decode_only",
              "warmup_run"):
        if k in e:
            line[k] = e[k]
    line["e2e"]["value"] = round(total_bytes * args.steps / (e2e_ms / 1e3) / 1e9, 2)
    line["timing"] = ("W warm-up steps (more until 0.2 s have passed: warmup_run); "
                      "synchronize; a ~0.2 ms GPU hold kernel (not timed) so "
                      "the host has queued the first steps; then exactly K steps back to back "
                      "between CUDA events on the launching stream; inputs larger than L2")
    # Every GPU measurement first, the CPU-oracle samples last: the oracle's
    # threads busy every host core, which must not overlap a timed region.
    extras = {}
    if world == 1 and args.config == "llama1b_decode" and not args.no_extras:
        del r
        torch.cuda.empty_cache()
        for name in ("continuous_batch", "long_splitk"):
            xw = W.named(name, 0)
            xr = bench_decode(xw, args, 1, device, decode_only=False)
            line[name] = decode_entry(xw, xr, hbm_peak, peak_src, f"decode_{name}.txt",
                                      args.steps)
            extras[name] = xw
            del xr
            torch.cuda.empty_cache()
        pw = W.named("chunked_prefill", 0)
        line["chunked_prefill"] = prefill_entry(pw, bench_prefill(pw, args, device), bf16_peak,
                                                bf16_sus, peak_src, args.steps)
        extras["chunked_prefill"] = pw

    if not args.no_cpu_baseline and world == 1:
        per, nbytes, cores, reps = cpu_baseline_decode(wl, budget_s=8.0)
        line["cpu_baseline"] = {
            "value": round(nbytes / per / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} full steps (paged write + fp64 decode of all {wl.num_seqs} "
                      f"sequences), {per:.3f} s each; {cpu_model()}"}
        for name in ("continuous_batch", "long_splitk"):
            if name not in extras:
                continue
            xw = extras[name]
            seqs = None if name == "continuous_batch" else [0]
            per, nbytes, cores, reps = cpu_baseline_decode(xw, budget_s=3.0, seqs=seqs)
            what = (f"{reps} full steps (paged write + fp64 decode of all "
                    f"{xw.num_seqs} sequences)" if seqs is None else
                    f"{reps} fp64 decodes of sequence 0 alone "
                    f"({int(xw.context_lens[0])} tokens; the write excluded)")
            line[name]["cpu_baseline"] = {"value": round(nbytes / per / 1e9, 3), "unit": "GB/s",
                                          "cores": cores, "kind": "oracle",
                                          "sample": f"{what}, {per:.3f} s each; {cpu_model()}"}
        if "chunked_prefill" in extras:
            sec, flops, cores = cpu_baseline_prefill(extras["chunked_prefill"], every=32)
            line["chunked_prefill"]["cpu_baseline"] = {
                "value": round(flops / sec / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"fp64 prefill of every 32nd query row (all heads), {sec:.2f} s; "
                          f"{cpu_model()}"}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
