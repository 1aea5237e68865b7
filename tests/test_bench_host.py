"""Host-side pieces of bench.py that need no GPU: the clock record of a
timed region (including one shorter than the sampling period) and the
algorithmic byte / FLOP counts the roofline divides by."""
import bench
from paged_kv_cache_198_gb300 import workloads as W


def _sampler(samples):
    c = bench.ClockSampler(0)
    c.samples = list(samples)
    return c


def test_clock_summary_inside_window():
    c = _sampler([(1.0, 1900.0, 2070.0, 900.0, []), (1.05, 2000.0, 2070.0, 950.0, []),
                  (1.10, 2070.0, 2070.0, 1000.0, ["sw_power_cap"]),
                  (1.15, 1500.0, 2070.0, 500.0, [])])
    s = c.summary(1.01, 1.12)
    assert s["samples"] == 2 and s["window"] == "timed region"
    assert s["sm_mhz"] == 2035.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_short_window_uses_nearest_samples():
    c = _sampler([(1.0, 1980.0, 2070.0, 900.0, []), (1.05, 2060.0, 2070.0, 950.0, []),
                  (1.10, 2070.0, 2070.0, 1000.0, [])])
    s = c.summary(1.051, 1.052)          # a 1 ms region between two samples
    assert s["samples"] == 2 and s["window"] == "nearest"
    assert s["sm_mhz"] == 2065.0


def test_clock_summary_without_samples():
    assert _sampler([]).summary(0.0, 1.0)["samples"] == 0


def test_decode_bytes_count_each_cached_token_once():
    wl = W.named("tiny")
    s, hq, d = wl.q.shape
    kv = int(wl.context_lens.sum()) * wl.num_kv_heads * d * 2 * 2
    nblk = sum((int(c) + 15) // 16 for c in wl.context_lens.tolist())
    assert bench.decode_algorithmic_bytes(wl) == kv + s * hq * d * 6 + 4 * nblk + 4 * s
    assert bench.write_algorithmic_bytes(wl) == 2 * 2 * s * wl.num_kv_heads * d + 4 * s


def test_prefill_flops_count_causal_pairs():
    pw = W.make_prefill(1, [3, 0], [2, 4], num_q_heads=4, num_kv_heads=2)
    # rows of sequence 0 see 4 and 5 keys, rows of sequence 1 see 1..4 keys
    assert pw.causal_pairs() == 4 + 5 + 1 + 2 + 3 + 4
    assert bench.prefill_flops(pw) == 4.0 * 64 * 4 * 19
