"""Host-side pieces of bench.py's JSON line, checked without a GPU."""
import math
import os

import bench
from workload import configs, gen


def test_roofline_entry_fields_and_arithmetic():
    r = bench.roofline_entry(135_368_704, 29.56, 6795.5, "measured", stage_us=34.88)
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert math.isclose(r["achieved"], 135_368_704 / 29.56e-6 / 1e9, rel_tol=1e-4)
    assert math.isclose(r["frac"], r["achieved"] / 6795.5, rel_tol=1e-3)
    st = r["stage_events"]
    assert st["achieved"] < r["achieved"] and math.isclose(st["frac"], st["achieved"] / 6795.5,
                                                           rel_tol=1e-3)
    assert "stage_events" not in bench.roofline_entry(1e8, 10.0, 6795.5, "measured")


def test_traffic_is_null_or_the_recorded_capture():
    """Reported only while the kernel sources hash to the digest of the capture,
    and then close to the algorithmic bytes (no wasted re-reads)."""
    t = bench.verify_traffic_bytes()
    assert t is None or t == bench.VERIFY_TRAFFIC["bytes"]
    w = configs.QWEN3_8B_B1_32K
    lens = gen.ctx_lens(w)
    alg = bench.algorithmic_bytes(w, lens, gen.k_per_seq(w, lens))["verify"]
    assert abs(bench.VERIFY_TRAFFIC["bytes"] / alg - 1.0) < 0.02


def test_algorithmic_bytes_of_the_bench_workload():
    """K and V of every prefix and window position, once, plus queries, outputs and
    scores: the per-launch figure the roofline divides by."""
    w = configs.QWEN3_8B_B1_32K
    lens = gen.ctx_lens(w)
    kps = gen.k_per_seq(w, lens)
    nb = bench.algorithmic_bytes(w, lens, kps)
    L = int(lens[0])
    kv = 2 * w.hkv * (L + w.gamma + 1) * w.head_dim * 2
    assert kv <= nb["verify"] <= kv + 2 * 1024 * 1024
    assert nb["total"] > nb["verify"]


def test_cpu_baseline_fields_on_the_tiny_workload():
    """The cpu_baseline object: full oracle iterations timed on host processes
    (one per unit, up to the core count), with the sample and CPU stated."""
    w = configs.TINY
    lens = gen.ctx_lens(w)
    nb = bench.algorithmic_bytes(w, lens, gen.k_per_seq(w, lens))
    r = bench.time_oracle(w, nb, budget_s=30.0, warmup=1, steps=2)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s"
    assert r["cores"] == min(w.batch * w.hkv, os.cpu_count())
    assert r["value"] > 0 and r["steps"] == 2 and r["warmup"] == 1
    assert "full iterations" in r["sample"] and r["cpu_model"]


def test_percentiles_and_stage_free_helpers():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(xs, 50) == 3.0
    assert bench.percentile(xs, 10) == 1.4 and bench.percentile(xs, 90) == 4.6
    assert bench.verify_kernel_name(configs.QWEN3_8B_B1_32K) == "verify_tc_kernel"


def test_draft_roofline_entry_takes_the_mean_step_bytes():
    r = bench.draft_roofline_entry([100_000_000, 100_000_256, 100_000_512], 10.0, 12.5, 6795.5)
    assert r["bound"] == "hbm" and r["bytes_per_launch"] == 100_000_256
    assert math.isclose(r["frac"], 100_000_256 / 10e-6 / 1e9 / 6795.5, rel_tol=1e-3)
    assert math.isclose(r["stage_events"]["frac"], r["frac"] * 10.0 / 12.5, rel_tol=1e-3)


def test_stack_sweep_bytes_follow_the_closed_form():
    """Per iteration of the 36-layer stack the path reads every prefix K/V row once
    for verify and a fraction gamma * r of them again over the draft steps, and
    writes then reads one fp32 score per (position, KV head):
    layers * (Hkv * 4d * sum L_b * (1 + gamma * r) + 8 * Hkv * sum L_b).  The
    accounting adds only queries, outputs, indices and the dense tails (< 1%)."""
    for gamma, k_pct in bench.STACK_SWEEP:
        w = configs.QWEN3_8B_36L_B4_96K_120K.with_(gamma=gamma, k_pct=k_pct)
        lens = gen.ctx_lens(w)
        nb = bench.algorithmic_bytes(w, lens, gen.k_per_seq(w, lens))
        s = int(lens.sum())
        closed = w.layers * (w.hkv * 4 * w.head_dim * s * (1 + gamma * k_pct / 100)
                             + 8 * w.hkv * s)
        assert 1.0 <= nb["total"] * w.layers / closed < 1.01, (gamma, k_pct)
