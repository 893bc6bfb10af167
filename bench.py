"""Benchmark of the Vegas hot path on GB300: one step = one iteration
(verify + Collect-2-Query capture, top-k select, gamma sparse draft steps) of
the Qwen3-8B-shaped layer at batch 1, context 32768, gamma 4, k = 5%.

Prints one JSON line.  `value` is algorithmic HBM GB/s of the whole iteration
(K/V rows the method must read, captured scores written and read, queries,
outputs and indices) divided by the device time per iteration; `ms_per_step`
is that time.  Inputs are resident in HBM; successive steps rotate over four
copies of the paged cache (>4x the 129 MB L2) so no step finds its K/V in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only other implementation:
the source pages publish no code) on the host cores, on a bounded sample.
Under torchrun each rank runs its own replica of the workload (weak scaling).
"""
from __future__ import annotations

import os

# The CPU oracle legs run single-threaded BLAS so that `cores` is exact.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workload import configs, gen  # noqa: E402

METRIC = ("µs and HBM GB/s (% of 8 TB/s) per verify+select+γ-draft iteration at "
          "32K–128K")
WORKLOAD = configs.QWEN3_8B_B1_32K
ROOFLINE_TBS = 8.0
REPLICAS = 4


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM traffic of one verify launch (dram__bytes_read.sum + dram__bytes_write.sum)
# on this workload, from a one-pass ncu capture of five consecutive verify
# launches of `python bench.py --profile --steps 8 --warmup 3` (134.41 MB read,
# 0.45-0.59 MB written per launch after the first); reported only while
# the kernel sources still hash to the digest they had when the counters were
# taken.
VERIFY_TRAFFIC = {
    "bytes": 134_900_000,
    "sources": ["verify_tc.cu", "split_merge.cuh", "attn_core.cuh", "vegas_common.cuh",
                "kernels.h"],
    "sha256": "524ac9623fb81b6890c125b27ae58a67d58ddc1b80bbd7dd890f37d338483a8c",
}


def verify_traffic_bytes():
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "self_speculative_sparse_paged_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for f in VERIFY_TRAFFIC["sources"]:
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return VERIFY_TRAFFIC["bytes"] if h.hexdigest() == VERIFY_TRAFFIC["sha256"] else None


def max_over_ranks(value, dist, device=None):
    """The largest value over the ranks (the slowest rank's time); value itself
    when there is no process group."""
    if not dist:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step, ms_per_step, world):
    """Whole-job throughput: every rank moves bytes_per_step per step (replicas)."""
    return bytes_per_step * world / (ms_per_step * 1e-3) / 1e9


def algorithmic_bytes(w, lens, kps):
    """Bytes one iteration must move, by stage."""
    d, hkv, hq, T = w.head_dim, w.hkv, w.hq, w.gamma + 1
    row = 4 * d                                   # K + V bf16 per (position, KV head)
    L = np.asarray(lens, dtype=np.int64)
    k = np.asarray(kps, dtype=np.int64)
    verify = int(hkv * row * (L + T).sum() + 2 * 2 * d * hq * T * len(L) + 4 * hkv * L.sum())
    select = int(4 * hkv * L.sum() + 4 * hkv * k.sum())
    draft = [int(hkv * row * (k + w.gamma + 2 + j).sum() + 4 * hkv * k.sum() + 2 * 2 * d * hq * len(L))
             for j in range(w.gamma)]
    return {"verify": verify, "select": select, "draft": draft,
            "total": verify + select + sum(draft)}


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class GpuIteration:
    """The workload resident in HBM: REPLICAS copies of the paged cache in one
    pool (replica r uses physical pages [r * P, (r + 1) * P)), shared queries,
    outputs and workspaces."""

    def __init__(self, w, replicas, dev):
        import torch
        import self_speculative_sparse_paged_gb300 as vg
        self.torch, self.vg, self.w, self.dev, self.R = torch, vg, w, dev, replicas
        self.lens = gen.ctx_lens(w)
        self.kps = gen.k_per_seq(w, self.lens)
        pm = gen.page_map(w, self.lens)
        self.pm = pm
        P = pm.num_pages
        shape = (replicas * P, w.hkv, 16, w.head_dim)
        self.k = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        self.v = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        lens_t = t(self.lens)
        need = t(gen.positions_needed(w, self.lens).astype(np.int32))
        u = t(gen.unit_direction(w))
        owner = t(pm.owner)
        for which, buf in ((0, self.k), (1, self.v)):
            vg.vegas_synth_paged_kv(buf, which, w.seed, 0, owner, P, w.hkv, w.head_dim,
                                    pm.max_pages, lens_t, need, gen.heavy_threshold(w),
                                    w.heavy_last, u)
        for r in range(1, replicas):
            self.k[r * P:(r + 1) * P].copy_(self.k[:P])
            self.v[r * P:(r + 1) * P].copy_(self.v[:P])
        bt = pm.block_table
        self.bt = t(np.stack([np.where(bt >= 0, bt + r * P, -1).astype(np.int32)
                              for r in range(replicas)]))
        self.kv = [vg.paged_kv(self.k, self.v, self.bt[r], w.hq) for r in range(replicas)]
        bf = lambda a: t(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731

        def packed(specs):
            """One device allocation holding tensors of the given (shape, dtype),
            each at a 256-byte boundary, so a step's inputs (and its outputs)
            move between host and device in one copy."""
            sizes = [int(np.prod(sh)) * torch.empty(0, dtype=dt).element_size() for sh, dt in specs]
            offs = [0]
            for n in sizes:
                offs.append(offs[-1] + (n + 255) // 256 * 256)
            buf = torch.empty(offs[-1], dtype=torch.uint8, device=dev)
            return buf, [buf[offs[i]:offs[i] + sizes[i]].view(dt).view(sh)
                         for i, (sh, dt) in enumerate(specs)]

        qv0 = bf(gen.f32_to_bf16_bits(gen.verify_queries_f32(w)))
        qd0 = bf(gen.f32_to_bf16_bits(gen.draft_queries_f32(w)))
        self.io_in, (self.qv, self.qd) = packed([(tuple(qv0.shape), torch.bfloat16),
                                                 (tuple(qd0.shape), torch.bfloat16)])
        self.qv.copy_(qv0)
        self.qd.copy_(qd0)
        self.lens_t, self.kps_t = lens_t, t(self.kps)
        self.stride = int(self.lens.max())
        self.k_max = int(self.kps.max())
        self.tails = [gen.tail_len(w, j) for j in range(w.gamma)]
        self.tl_t = [torch.full((w.batch,), tl, dtype=torch.int32, device=dev) for tl in self.tails]
        self.io_out, (self.out_v, self.out_d, self.idx) = packed(
            [(tuple(self.qv.shape), torch.bfloat16), (tuple(self.qd.shape), torch.bfloat16),
             ((w.batch, w.hkv, self.k_max), torch.int32)])
        self.scores = torch.empty((w.batch, w.hkv, self.stride), dtype=torch.float32, device=dev)
        self.kw_t = torch.zeros((w.batch,), dtype=torch.int32, device=dev)
        # the pages' capture: raw logits of rows {0, gamma} of every query head
        self.raw_rows = len({0, w.gamma})
        self.raw = torch.empty((w.batch, self.raw_rows, w.hq, self.stride), dtype=torch.float32,
                               device=dev)
        nv = vg.vegas_verify_workspace_size(self.kv[0], w.batch, w.gamma)
        self.ws_v = torch.zeros(max(nv, 256), dtype=torch.uint8, device=dev)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.launches_per_step = 2 + w.gamma

    def verify(self, r, capture=True):
        w = self.w
        self.vg.vegas_verify_attn_capture(
            self.kv[r], self.qv, self.out_v, self.scores if capture else None, self.stride,
            self.lens_t, w.batch, w.gamma, 0, w.gamma, self.scale, self.ws_v, self.ws_v.numel())

    def select(self):
        w = self.w
        self.vg.vegas_select_topk(self.scores, self.stride, self.lens_t, self.kps_t, self.idx,
                                  w.batch, w.hkv, self.k_max)

    # -- the "next" variants: collect-all capture, one T for all heads, window selector
    def verify_rows(self, r, mask):
        w = self.w
        self.vg.vegas_verify_attn_capture_rows(
            self.kv[r], self.qv, self.out_v, self.scores, self.stride, self.lens_t, w.batch,
            w.gamma, mask, self.scale, self.ws_v, self.ws_v.numel())

    def verify_raw(self, r):
        w = self.w
        self.vg.vegas_verify_attn_raw_logits(
            self.kv[r], self.qv, self.out_v, self.raw, self.stride, self.lens_t, w.batch,
            w.gamma, (1 << 0) | (1 << w.gamma), self.scale, self.ws_v, self.ws_v.numel())

    def aggregate_raw(self):
        w = self.w
        self.vg.vegas_aggregate_raw_logits(self.raw, self.stride, self.lens_t, w.batch,
                                           self.raw_rows, w.hq, w.hkv, self.stride, self.scores,
                                           self.stride)

    def select_shared(self):
        w = self.w
        self.vg.vegas_select_topk_shared(self.scores, self.stride, self.lens_t, self.kps_t,
                                         self.idx, w.batch, w.hkv, self.k_max)

    def select_outliers(self):
        """The select on a copy of the captured scores in which eight positions
        of every (sequence, KV head) row carry a logit a thousand times the
        row's largest magnitude: a few outliers stretch the row's [min, max]
        (real logits are not bounded like the synthetic ones)."""
        w, torch = self.w, self.torch
        if getattr(self, "scores_out", None) is None:
            rng = np.random.default_rng(w.seed + 11)
            self.scores_out = self.scores.clone()
            for b in range(w.batch):
                L = int(self.lens[b])
                for g in range(w.hkv):
                    row = self.scores_out[b, g, :L]
                    pos = torch.from_numpy(rng.choice(L, size=min(8, L), replace=False)).to(self.dev)
                    row[pos] = 1000.0 * float(row.abs().max().item()) * (1.0 + torch.arange(
                        len(pos), device=self.dev, dtype=torch.float32) / 16)
        self.vg.vegas_select_topk(self.scores_out, self.stride, self.lens_t, self.kps_t, self.idx,
                                  w.batch, w.hkv, self.k_max)

    def select_window(self):
        w = self.w
        # as many positions as the verification-guided selector keeps: sinks + window
        sinks = min(64, self.k_max // 2)
        self.vg.vegas_select_window(self.lens_t, sinks, self.k_max - sinks, self.kw_t, self.idx,
                                    w.batch, w.hkv, self.k_max)

    def window_step(self, r):
        w = self.w
        self.verify(r, capture=False)
        self.select_window()
        for j in range(w.gamma):
            self.vg.vegas_sparse_decode_attn(
                self.kv[r], self.qd[j], self.out_d[j], self.idx, self.k_max, self.kw_t,
                self.lens_t, self.tl_t[j], self.tails[j], w.batch, self.scale)

    def draft(self, r, j):
        w = self.w
        self.vg.vegas_sparse_decode_attn(
            self.kv[r], self.qd[j], self.out_d[j], self.idx, self.k_max, self.kps_t, self.lens_t,
            self.tl_t[j], self.tails[j], w.batch, self.scale)

    def step(self, r, ev=None, capture=True):
        if ev:
            ev[0].record()
        self.verify(r, capture)
        if ev:
            ev[1].record()
        self.select()
        if ev:
            ev[2].record()
        for j in range(self.w.gamma):
            self.draft(r, j)
        if ev:
            ev[3].record()


class LayerStack:
    """`layers` attention layers of one workload shape resident in HBM, each
    with its own paged cache and queries (the layer's generator streams) under
    one block table, run as one decode iteration by vegas_decode_iteration:
    verify(l) then select(l) for every layer, then every draft step over every
    layer; pipelined, select(l) overlaps verify(l + 1) on a second stream."""

    def __init__(self, w, layers, dev):
        import torch
        import self_speculative_sparse_paged_gb300 as vg
        self.torch, self.vg, self.w, self.dev, self.layers = torch, vg, w, dev, layers
        self.lens = gen.ctx_lens(w)
        self.kps = gen.k_per_seq(w, self.lens)
        pm = gen.page_map(w, self.lens)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        bf = lambda a: t(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
        self.lens_t, self.kps_t, self.bt = t(self.lens), t(self.kps), t(pm.block_table)
        need = t(gen.positions_needed(w, self.lens).astype(np.int32))
        u, owner = t(gen.unit_direction(w)), t(pm.owner)
        shape = (pm.num_pages, w.hkv, 16, w.head_dim)
        self.stride = max(int(self.lens.max()), 1)
        self.k_max = max(int(self.kps.max()), 1)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.tails = [gen.tail_len(w, j) for j in range(w.gamma)]
        self.tl_t = [torch.full((w.batch,), tl, dtype=torch.int32, device=dev) for tl in self.tails]
        self.kv, self.qv, self.qd, self.out_v, self.out_d, self.scores, self.idx = ([] for _ in range(7))
        self._keep = []
        for layer in range(layers):
            k = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            v = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            for which, buf in ((0, k), (1, v)):
                vg.vegas_synth_paged_kv(buf, which, w.seed, layer, owner, pm.num_pages, w.hkv,
                                        w.head_dim, pm.max_pages, self.lens_t, need,
                                        gen.heavy_threshold(w), w.heavy_last, u)
            self._keep += [k, v]
            self.kv.append(vg.paged_kv(k, v, self.bt, w.hq))
            self.qv.append(bf(gen.f32_to_bf16_bits(gen.verify_queries_f32(w, layer))))
            self.qd.append(bf(gen.f32_to_bf16_bits(gen.draft_queries_f32(w, layer))))
            self.out_v.append(torch.empty_like(self.qv[-1]))
            self.out_d.append(torch.empty_like(self.qd[-1]))
            self.scores.append(torch.empty((w.batch, w.hkv, self.stride), dtype=torch.float32,
                                           device=dev))
            self.idx.append(torch.empty((w.batch, w.hkv, self.k_max), dtype=torch.int32,
                                        device=dev))
        nv = vg.vegas_verify_workspace_size(self.kv[0], w.batch, w.gamma)
        self.ws = torch.zeros(max(nv, 256), dtype=torch.uint8, device=dev)
        self.kw_t = torch.zeros((w.batch,), dtype=torch.int32, device=dev)
        self.side = torch.cuda.Stream(device=dev)
        self.tails_t = t(np.array([[tl] * w.batch for tl in self.tails], dtype=np.int32))
        self.layer_descs = [vg.layer(self.kv[i], self.qv[i], self.out_v[i], self.qd[i],
                                     self.out_d[i], self.scores[i], self.idx[i])
                            for i in range(layers)]

    def step_without_capture(self):
        """The same iteration with verify's capture off and the query-agnostic
        window selector (up to 64 sinks + a window, as many positions as k): the
        denominator of the capture-plus-select overhead."""
        torch, vg, w = self.torch, self.vg, self.w
        main = torch.cuda.current_stream()
        for layer in range(self.layers):
            vg.vegas_verify_attn_capture(
                self.kv[layer], self.qv[layer], self.out_v[layer], None, self.stride,
                self.lens_t, w.batch, w.gamma, 0, w.gamma, self.scale, self.ws, self.ws.numel(),
                stream=main)
            sinks = min(64, self.k_max // 2)
            vg.vegas_select_window(self.lens_t, sinks, self.k_max - sinks, self.kw_t,
                                   self.idx[layer], w.batch, w.hkv, self.k_max, stream=main)
        for j in range(w.gamma):
            for layer in range(self.layers):
                vg.vegas_sparse_decode_attn(
                    self.kv[layer], self.qd[layer][j], self.out_d[layer][j], self.idx[layer],
                    self.k_max, self.kw_t, self.lens_t, self.tl_t[j], self.tails[j], w.batch,
                    self.scale, stream=main)

    def step(self, pipelined):
        """One iteration through the library's layer-stack call (select(l) on the
        side stream, overlapping verify(l + 1), when pipelined)."""
        torch, vg, w = self.torch, self.vg, self.w
        vg.vegas_decode_iteration(self.layer_descs, self.lens_t, self.kps_t, self.tails_t,
                                  max(self.tails), w.batch, w.gamma, self.stride, self.k_max,
                                  self.scale, self.ws, self.ws.numel(),
                                  stream=torch.cuda.current_stream(),
                                  select_stream=self.side if pipelined else None)


def time_stack(w, layers, dev, stream, verify_plain_us, reps=10):
    """us per iteration of a `layers`-layer stack, serial and with select(l)
    overlapping verify(l + 1) on a second stream (each as a replayed graph)."""
    import torch
    st = LayerStack(w, layers, dev)
    out = {}
    runs = (("serial_us", lambda: st.step(False)), ("pipelined_us", lambda: st.step(True)),
            ("no_capture_window_select_us", st.step_without_capture))
    for name, fn in runs:
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record()
            g.replay()
            e1.record()
        stream.synchronize()
        out[name] = round(1000.0 * e0.elapsed_time(e1) / reps, 2)
    st.vg.vegas_read_device_status(stream)
    out["layers"] = layers
    out["select_hidden_us_per_layer"] = round((out["serial_us"] - out["pipelined_us"]) / layers, 3)
    # capture + verification-guided select over plain verify, pipelined: the
    # iteration's extra time over the capture-free window-selector iteration,
    # per plain verify
    out["capture_plus_select_overhead_pipelined"] = round(
        (out["pipelined_us"] - out["no_capture_window_select_us"]) / (layers * verify_plain_us), 4)
    out["overhead_formula"] = ("(pipelined - no-capture window-selector iteration) / "
                               "(layers x plain verify, back to back)")
    del st
    torch.cuda.empty_cache()
    return out


def time_variants(it, stream, reps=100):
    """us per call of each stage variant, each timed as a graph of `reps` calls
    (rotating the KV replicas) replayed once after a warm replay."""
    import torch
    w = it.w
    all_rows = (1 << (w.gamma + 1)) - 1
    fns = {
        "verify_capture2_us": lambda i: it.verify(i % it.R),
        "verify_collect_all_us": lambda i: it.verify_rows(i % it.R, all_rows),
        "verify_no_capture_us": lambda i: it.verify(i % it.R, capture=False),
        "verify_raw_logits_us": lambda i: it.verify_raw(i % it.R),
        "aggregate_raw_logits_us": lambda i: it.aggregate_raw(),
        "paper_style_capture_us": lambda i: (it.verify_raw(i % it.R), it.aggregate_raw()),
        "select_us": lambda i: it.select(),
        "select_with_outliers_us": lambda i: it.select_outliers(),
        "draft_step_us": lambda i: it.draft(i % it.R, i % w.gamma),
        "select_shared_us": lambda i: it.select_shared(),
        "select_window_us": lambda i: it.select_window(),
        "iteration_window_selector_us": lambda i: it.window_step(i % it.R),
    }
    out = {}
    for name, fn in fns.items():
        with torch.cuda.stream(stream):
            for i in range(it.R):
                fn(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                fn(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record()
            g.replay()
            e1.record()
        stream.synchronize()
        out[name] = round(1000.0 * e0.elapsed_time(e1) / reps, 3)
    it.vg.vegas_read_device_status(stream)
    out["source"] = ("each variant alone in a graph of 100 calls (kernels of consecutive calls "
                     "overlap through programmatic dependent launch)")
    return out


def make_events(torch, n, external):
    if external:
        return [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
                for _ in range(n)]
    return None


def graph_of(torch, stream, fn, n):
    """A CUDA graph of fn(0) .. fn(n - 1) captured on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i)
    return g


def replay_ms(torch, stream, graph, repeats, reps=1):
    """Device ms of `repeats` timed regions, each `reps` replays of `graph`,
    bracketed by CUDA events on the launching stream."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(repeats)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            a.record()
            for _ in range(reps):
                graph.replay()
            b.record()
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def percentile(xs, q):
    xs = sorted(xs)
    if len(xs) == 1:
        return xs[0]
    pos = q / 100.0 * (len(xs) - 1)
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(xs) - 1)
    return xs[lo] + (xs[hi] - xs[lo]) * (pos - lo)


def stage_times(torch, it, stream, n):
    """Mean us of verify, select and one draft step from external events at the
    stage boundaries of a graph of n iterations (the events serialise the stages)."""
    evs = make_events(torch, n, True)
    g = graph_of(torch, stream, lambda i: it.step(i % it.R, evs[i]), n)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    v = [evs[i][0].elapsed_time(evs[i][1]) for i in range(n)]
    s = [evs[i][1].elapsed_time(evs[i][2]) for i in range(n)]
    d = [evs[i][2].elapsed_time(evs[i][3]) for i in range(n)]
    return {"verify_us": 1000 * statistics.mean(v), "select_us": 1000 * statistics.mean(s),
            "draft_us_per_step": 1000 * statistics.mean(d) / max(1, it.w.gamma)}


def per_call_us(torch, stream, fn, n=50):
    """us per call of fn(i) in a graph of n calls replayed after a warm replay
    (consecutive calls overlap through programmatic dependent launch)."""
    g = graph_of(torch, stream, fn, n)
    with torch.cuda.stream(stream):
        g.replay()
    return 1000.0 * replay_ms(torch, stream, g, 1)[0] / n


def verify_kernel_name(w):
    """Kernel vegas_verify_attn_capture runs for this shape (with capture): the
    tcgen05 kernel up to 40 query columns at head_dim 128 and 64 at head_dim 64."""
    cols = ((w.group * (w.gamma + 1) + 1) & ~1) + 2
    limit = 40 if w.head_dim == 128 else 64
    return "verify_tc_kernel" if cols <= limit else "verify_attn_kernel"


def measure_workload(w, dev, stream, peak, peak_kind, iters=8, repeats=5):
    """One extra workload: us and GB/s per iteration (graph of `iters`
    iterations, median of `repeats` timed replays), the stage breakdown, and the
    roofline fractions of the verify and draft kernels (bytes per launch over
    the per-launch time of a graph of back-to-back launches, and over the stage
    events)."""
    import torch
    kv_bytes = w.hkv * 4 * w.head_dim * int(gen.ctx_lens(w).sum())
    replicas = REPLICAS if kv_bytes < 4 * 129e6 else 1
    it = GpuIteration(w, replicas, dev)
    nb = algorithmic_bytes(w, it.lens, it.kps)
    with torch.cuda.stream(stream):
        for i in range(2):
            it.step(i % it.R)
    stream.synchronize()
    n = max(iters // replicas, 1) * replicas
    g = graph_of(torch, stream, lambda i: it.step(i % it.R), n)
    with torch.cuda.stream(stream):
        g.replay()
    ms = [t / n for t in replay_ms(torch, stream, g, repeats)]
    st = stage_times(torch, it, stream, n)
    v_b2b = per_call_us(torch, stream, lambda i: it.verify(i % it.R), 4 * replicas)
    v_plain = per_call_us(torch, stream, lambda i: it.verify(i % it.R, capture=False),
                          4 * replicas)
    sel = per_call_us(torch, stream, lambda i: it.select(), 20)
    d_b2b = per_call_us(torch, stream, lambda i: it.draft(i % it.R, 0), 8 * replicas)
    it.vg.vegas_read_device_status(stream)
    med = statistics.median(ms)
    draft_bytes = nb["draft"][0]
    out = {
        "workload": w.name, "description": w.description,
        "us_per_iteration": round(med * 1000, 2),
        "us_p10_p90": [round(percentile(ms, 10) * 1000, 2), round(percentile(ms, 90) * 1000, 2)],
        "value": round(nb["total"] / (med * 1e-3) / 1e9, 1), "unit": "GB/s",
        "pct_of_8tbs": round(100 * nb["total"] / (med * 1e-3) / 8e12, 2),
        "bytes_per_iteration": nb["total"],
        "stages_us": {k: round(v, 3) for k, v in st.items()},
        "back_to_back_us": {"verify_capture": round(v_b2b, 3), "verify_plain": round(v_plain, 3),
                            "select": round(sel, 3), "draft_step": round(d_b2b, 3)},
        "capture_plus_select_overhead": round((v_b2b + sel) / v_plain - 1.0, 4),
        "roofline_verify": {
            "kernel": verify_kernel_name(w), "bytes_per_launch": nb["verify"],
            "frac_back_to_back": round(nb["verify"] / (v_b2b * 1e-6) / 1e9 / peak, 4),
            "frac_stage_events": round(nb["verify"] / (st["verify_us"] * 1e-6) / 1e9 / peak, 4),
            "peak": peak, "peak_kind": peak_kind},
        "roofline_draft": {
            "kernel": "sparse_decode_kernel", "bytes_per_launch": draft_bytes,
            "frac_back_to_back": round(draft_bytes / (d_b2b * 1e-6) / 1e9 / peak, 4),
            "frac_stage_events": round(statistics.mean(nb["draft"])
                                       / (st["draft_us_per_step"] * 1e-6) / 1e9 / peak, 4)},
        "l2": (f"iterations rotate over {replicas} copies of the paged cache" if replicas > 1
               else "one copy of the paged cache, several times the 129 MB L2"),
    }
    del it, g
    torch.cuda.empty_cache()
    return out


def measure_stack(w, dev, stream, peak, peak_kind, repeats=3):
    """The full-depth layer stack at one (gamma, k) point: us and GB/s per
    pipelined iteration through vegas_decode_iteration, the capture-free
    window-selector baseline, and the verify and draft kernels' roofline
    fractions (one launch per layer, back to back)."""
    import torch
    st = LayerStack(w, w.layers, dev)
    nb = algorithmic_bytes(w, st.lens, st.kps)
    total = nb["total"] * w.layers
    res = {}
    for name, fn in (("pipelined", lambda i: st.step(True)), ("serial", lambda i: st.step(False)),
                     ("no_capture_window_select", lambda i: st.step_without_capture())):
        with torch.cuda.stream(stream):
            fn(0)
        stream.synchronize()
        g = graph_of(torch, stream, fn, 1)
        with torch.cuda.stream(stream):
            g.replay()
        res[name] = statistics.median(replay_ms(torch, stream, g, repeats))
        del g
    vg, L = st.vg, w.layers

    def verify_l(i, capture=True):
        l = i % L
        vg.vegas_verify_attn_capture(st.kv[l], st.qv[l], st.out_v[l],
                                     st.scores[l] if capture else None, st.stride, st.lens_t,
                                     w.batch, w.gamma, 0, w.gamma, st.scale, st.ws, st.ws.numel())

    def draft_l(i):
        l = i % L
        vg.vegas_sparse_decode_attn(st.kv[l], st.qd[l][0], st.out_d[l][0], st.idx[l], st.k_max,
                                    st.kps_t, st.lens_t, st.tl_t[0], st.tails[0], w.batch,
                                    st.scale)
    v_us = per_call_us(torch, stream, verify_l, L)
    vp_us = per_call_us(torch, stream, lambda i: verify_l(i, False), L)
    d_us = per_call_us(torch, stream, draft_l, L)
    vg.vegas_read_device_status(stream)
    med = res["pipelined"]
    out = {
        "workload": f"{w.name}_gamma{w.gamma}_k{w.k_pct}pct", "description": w.description,
        "layers": L, "gamma": w.gamma, "k_pct": w.k_pct,
        "us_per_iteration": round(med * 1000, 1),
        "serial_us": round(res["serial"] * 1000, 1),
        "no_capture_window_select_us": round(res["no_capture_window_select"] * 1000, 1),
        "value": round(total / (med * 1e-3) / 1e9, 1), "unit": "GB/s",
        "pct_of_8tbs": round(100 * total / (med * 1e-3) / 8e12, 2),
        "bytes_per_iteration": total,
        "capture_plus_select_overhead_pipelined": round(
            (res["pipelined"] - res["no_capture_window_select"]) * 1000 / (L * vp_us), 4),
        "overhead_formula": "(pipelined - no-capture window-selector iteration) / "
                            "(layers x plain verify, back to back)",
        "roofline_verify": {"kernel": verify_kernel_name(w), "us": round(v_us, 2),
                            "frac_back_to_back": round(nb["verify"] / (v_us * 1e-6) / 1e9 / peak, 4)},
        "roofline_draft": {"kernel": "sparse_decode_kernel", "us": round(d_us, 2),
                           "frac_back_to_back": round(nb["draft"][0] / (d_us * 1e-6) / 1e9 / peak,
                                                      4)},
        "peak": peak, "peak_kind": peak_kind,
        "l2": "36 layers of KV cache (tens of GB): nothing survives in L2 between layers",
    }
    del st
    torch.cuda.empty_cache()
    return out


# The metric's range at full depth: (gamma, k%) from the lightest to the
# heaviest draft phase, and the point the bench line reports.
STACK_SWEEP = ((2, 3), (2, 10), (4, 5), (8, 3), (8, 10))


def stack_sweep(peak, peak_kind):
    """The 36-layer Qwen3-8B stack (batch 4, 96K-120K) at each STACK_SWEEP point:
    one measure_stack result a point, with the clocks sampled while it ran."""
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    for gamma, k_pct in STACK_SWEEP:
        w = configs.QWEN3_8B_36L_B4_96K_120K.with_(gamma=gamma, k_pct=k_pct)
        sampler = ClockSampler(dev.index)
        sampler.start()
        out = measure_stack(w, dev, stream, peak, peak_kind)
        out["clocks"] = sampler.stop()
        yield out


def run_gpu(args, rank, world, dist, peak, peak_kind):
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = configs.BY_NAME[args.workload]
    kv_bytes = w.hkv * 4 * w.head_dim * int(gen.ctx_lens(w).sum())
    replicas = REPLICAS if kv_bytes < 4 * 129e6 else 1
    it = GpuIteration(w, replicas, dev)
    vg = it.vg
    nbytes = algorithmic_bytes(w, it.lens, it.kps)
    stream = torch.cuda.Stream(device=dev)
    K, W = args.steps, args.warmup

    # warm-up: every path once eagerly (configures kernels), then W steps
    with torch.cuda.stream(stream):
        for i in range(max(W, 1)):
            it.step(i % it.R)
            it.verify(i % it.R, capture=False)
    stream.synchronize()
    vg.vegas_read_device_status(stream)

    # The timed region is K iterations: `reps` replays of a graph of `chunk`
    # iterations (no event nodes between the kernels, so each may launch while
    # its predecessor drains).  It is repeated `repeats` times, each timed on
    # its own; the line reports the median and the 10th/90th percentiles.
    chunk = max(it.R, min(K, 100) // it.R * it.R)
    reps = max(1, math.ceil(K / chunk))
    K_eff = reps * chunk
    graph = graph_of(torch, stream, lambda i: it.step(i % it.R), chunk)
    plain = graph_of(torch, stream, lambda i: it.step(i % it.R, capture=False), chunk)
    with torch.cuda.stream(stream):
        graph.replay()
        plain.replay()
    stream.synchronize()
    est_ms = replay_ms(torch, stream, graph, 1, reps)[0]
    repeats = int(max(50, min(200, 10000.0 / max(est_ms, 1e-3))))

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    region_ms = replay_ms(torch, stream, graph, repeats, reps)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    plain_ms = replay_ms(torch, stream, plain, max(5, repeats // 10), reps)
    clocks = sampler.stop()
    vg.vegas_read_device_status(stream)

    step_ms = [t / K_eff for t in region_ms]
    ms_step = max_over_ranks(statistics.median(step_ms), dist, dev)
    timing = {"repeats": repeats, "steps_per_repeat": K_eff,
              "ms_per_step_p10": round(percentile(step_ms, 10), 5),
              "ms_per_step_median": round(statistics.median(step_ms), 5),
              "ms_per_step_p90": round(percentile(step_ms, 90), 5),
              "plain_iteration_ms_median": round(statistics.median(plain_ms) / K_eff, 5)}
    stages = stage_times(torch, it, stream, chunk)
    stages["source"] = ("external CUDA events at the stage boundaries of a separately "
                        "replayed graph (events there serialise the stages)")
    if args.profile:
        # the timed region and the stages only: every other leg is left out so
        # that a profiler run holds just this workload's memory and launches
        vb = per_call_us(torch, stream, lambda i: it.verify(i % it.R), 4 * it.R)
        vp = per_call_us(torch, stream, lambda i: it.verify(i % it.R, capture=False), 4 * it.R)
        sl = per_call_us(torch, stream, lambda i: it.select(), 8)
        dr = per_call_us(torch, stream, lambda i: it.draft(i % it.R, i % w.gamma), 8)
        variants = {"verify_capture2_us": round(vb, 3), "verify_no_capture_us": round(vp, 3),
                    "select_us": round(sl, 3), "draft_step_us": round(dr, 3)}
        e2e = None
        return (it, nbytes, ms_step, K_eff, stages, timing, clocks, e2e, variants, {})
    e2e = run_e2e(it, stream, min(K_eff, 500), nbytes)
    variants = time_variants(it, stream)
    variants["layer_stack_8"] = time_stack(w, 8, dev, stream, variants["verify_no_capture_us"])
    extra = {}
    if world == 1 and not args.quick:
        del it
        torch.cuda.empty_cache()
        for ew in (configs.QWEN3_8B_B1_32K, configs.QWEN3_8B_B8_48K_64K,
                   configs.GPTOSS_20B_B4_128K):
            if ew.name != w.name:
                extra[ew.name] = measure_workload(ew, dev, stream, peak, peak_kind)
        sw = configs.QWEN3_8B_36L_B4_96K_120K.with_(gamma=4, k_pct=5)
        extra[sw.name + "_gamma4_k5pct"] = measure_stack(sw, dev, stream, peak, peak_kind)
        it = None
    return (it, nbytes, ms_step, K_eff, stages, timing, clocks, e2e, variants, extra)


def run_e2e(it, stream, steps, nbytes):
    """Same metric through the public API with host buffers: every step copies
    its queries from pinned host memory, runs the iteration, and reads back the
    verify outputs, the draft outputs and the selected indices."""
    torch = it.torch
    # the step's queries (verify and draft) and its outputs (verify and draft
    # outputs, selected indices) each sit in one packed device buffer
    in_h = torch.empty(it.io_in.shape, dtype=torch.uint8, pin_memory=True)
    in_h.copy_(it.io_in.cpu())
    out_h = torch.empty(it.io_out.shape, dtype=torch.uint8, pin_memory=True)
    # One graph per KV replica holds the whole step: the host-to-device copy
    # of the step's queries, the iteration, and the device-to-host copy of its
    # outputs (pinned host memory), so a step costs the host one launch and
    # one synchronisation.
    graphs = []
    for r in range(it.R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            it.io_in.copy_(in_h, non_blocking=True)
            it.step(r)
            out_h.copy_(it.io_out, non_blocking=True)
        graphs.append(g)
    bi = in_h.numel()
    bo = out_h.numel()

    def one(i):
        with torch.cuda.stream(stream):
            graphs[i % it.R].replay()
        stream.synchronize()

    for i in range(3):
        one(i)
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    dt = (time.perf_counter() - t0) / steps
    return {"value": round(nbytes["total"] / dt / 1e9, 2), "unit": "GB/s",
            "us_per_iteration": round(dt * 1e6, 2), "steps": steps,
            "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
            "timing": "host wall clock, stream synchronised every step; the copies "
                      "are nodes of the step's graph"}


# ---------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------
def oracle_unit_inputs(w, b, g):
    """fp64 inputs of the iteration restricted to (sequence b, KV head g): the
    unit's K/V rows (every position the iteration touches) in a one-head paged
    cache with an identity block table, its G heads' verify and draft queries."""
    lens = gen.ctx_lens(w)
    L = int(lens[b])
    n = int(gen.positions_needed(w, lens)[b])
    pos = np.arange(n, dtype=np.int64)
    pages = (n + 15) // 16
    kc = np.zeros((pages, 1, 16, w.head_dim), dtype=np.float64)
    vc = np.zeros_like(kc)
    kc[pos // 16, 0, pos % 16] = gen.bf16_bits_to_f64(gen.kv_rows_bf16(w, 0, "k", b, g, pos, L))
    vc[pos // 16, 0, pos % 16] = gen.bf16_bits_to_f64(gen.kv_rows_bf16(w, 0, "v", b, g, pos, L))
    heads = slice(g * w.group, (g + 1) * w.group)
    qv = gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(gen.verify_queries_f32(w)))[b:b + 1, :, heads]
    qd = gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(gen.draft_queries_f32(w)))[:, b:b + 1, heads]
    bt = np.arange(pages, dtype=np.int32)[None, :]
    k = gen.k_per_seq(w, lens)[b:b + 1]
    return (qv, qd, kc, vc, bt, lens[b:b + 1], k, 1.0 / math.sqrt(w.head_dim))


def _oracle_worker(conn, w, units):
    """One host process of the oracle pool: builds its units' inputs once, then
    runs oracle.iteration over them whenever the parent asks."""
    import oracle
    inputs = [oracle_unit_inputs(w, b, g) for b, g in units]
    conn.send("ready")
    while conn.recv() == "run":
        for x in inputs:
            oracle.iteration(*x)
        conn.send("done")


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


class OraclePool:
    """The oracle iteration over every (sequence, KV head) unit of a workload, in
    parallel on the host cores: one spawned process per core (BLAS single-threaded
    in each), units dealt round-robin and kept by their process, so a step is
    one full iteration of the workload."""

    def __init__(self, w, cores=None):
        import multiprocessing as mp
        units = [(b, g) for b in range(w.batch) for g in range(w.hkv)]
        n = max(1, min(len(units), cores or os.cpu_count() or 1))
        ctx = mp.get_context("spawn")        # safe after CUDA was initialised
        self.procs, self.conns = [], []
        for i in range(n):
            a, bconn = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(bconn, w, units[i::n]), daemon=True)
            p.start()
            self.procs.append(p)
            self.conns.append(a)
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")
        self.cores = n
        self.units = len(units)

    def step(self) -> float:
        """Wall seconds of one full iteration (every unit) over the pool."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send("run")
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            try:
                c.send("stop")
            except Exception:
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()


def time_oracle(w, nbytes, budget_s, warmup=1, steps=None, cores=None):
    """Times full oracle iterations of the workload on the host cores: `warmup`
    untimed, then `steps` timed (or as many as budget_s allows when steps is None,
    at least one; a given `steps` is also cut at budget_s)."""
    pool = OraclePool(w, cores)
    try:
        for _ in range(max(0, warmup)):
            pool.step()
        times = []
        t_start = time.perf_counter()
        while True:
            times.append(pool.step())
            if steps is not None and len(times) >= steps:
                break
            if time.perf_counter() - t_start >= budget_s:
                break
    finally:
        pool.close()
    dt = statistics.median(times)
    return {"value": round(nbytes["total"] / dt / 1e9, 4), "unit": "GB/s", "cores": pool.cores,
            "kind": "oracle", "steps": len(times), "warmup": max(0, warmup),
            "s_per_step": round(dt, 4), "cpu_model": cpu_model(),
            "sample": (f"{len(times)} full iterations of the workload (all {pool.units} "
                       f"(sequence, KV head) units, fp64 numpy), units spread over "
                       f"{pool.cores} host processes, one BLAS thread each; median wall time")}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def roofline_entry(bytes_per_launch, launch_us, peak, peak_kind, stage_us=None,
                   kernel="verify_tc_kernel"):
    """The bench line's roofline object for the verify kernel: algorithmic bytes
    per launch over its average launch duration (CUDA events on the launching
    stream around a graph of back-to-back launches, divided by their count)
    against the HBM peak, the ncu traffic while the sources match, and (context)
    the same bytes over the duration between stage events placed around the
    launch inside an iteration graph (those events cut the programmatic-launch
    overlap with the previous kernel, so they add its launch latency)."""
    achieved = bytes_per_launch / (launch_us * 1e-6) / 1e9
    out = {"kernel": kernel, "bound": "hbm", "achieved": round(achieved, 1),
           "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
           "peak_kind": peak_kind, "traffic": verify_traffic_bytes(),
           "bytes_per_launch": bytes_per_launch, "duration_us": round(launch_us, 3),
           "duration_source": "CUDA events around a graph of back-to-back launches (rotating "
                              "the KV replicas) on the launching stream, per launch"}
    if stage_us:
        a2 = bytes_per_launch / (stage_us * 1e-6) / 1e9
        out["stage_events"] = {"duration_us": round(stage_us, 3), "achieved": round(a2, 1),
                               "frac": round(a2 / peak, 4)}
    return out


def draft_roofline_entry(step_bytes, step_us, stage_us, peak):
    """The draft kernel's roofline object: the mean algorithmic bytes of one
    draft step (the steps' tails differ by one position each) over the per-step
    duration of a graph of back-to-back steps, against the HBM peak; the same
    bytes over the stage-event duration as context."""
    d_bytes = int(round(statistics.mean(step_bytes)))
    return {"kernel": "sparse_decode_kernel", "bound": "hbm", "bytes_per_launch": d_bytes,
            "duration_us": round(step_us, 3),
            "frac": round(d_bytes / (step_us * 1e-6) / 1e9 / peak, 4),
            "duration_source": "CUDA events around a graph of back-to-back draft steps "
                               "(rotating the KV replicas and the step index) on the "
                               "launching stream, per step",
            "stage_events": {"duration_us": round(stage_us, 3),
                             "frac": round(d_bytes / (stage_us * 1e-6) / 1e9 / peak, 4)}}


def base_config(w, lens, kps):
    kv = w.hkv * 4 * w.head_dim * int(lens.sum())
    reps = REPLICAS if kv < 4 * 129e6 else 1
    l2 = (f"steps rotate over {reps} copies of the paged KV cache ({reps}x {kv / 1e6:.0f} MB)"
          if reps > 1 else f"one copy of the paged KV cache ({kv / 1e6:.0f} MB, >4x the 129 MB L2)")
    return {"workload": w.name, "description": w.description, "batch": w.batch,
            "ctx_len": int(lens.max()), "gamma": w.gamma, "k": int(kps.max()),
            "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim, "page_size": 16,
            "l2": l2, "parallelism": "replicas"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="only the headline workload (no extra workloads)")
    ap.add_argument("--profile", action="store_true",
                    help="timed region, stages and back-to-back verify/select only (profiler runs)")
    ap.add_argument("--stack-sweep", action="store_true",
                    help="only the 36-layer stack at the corners of the (gamma, k) range, "
                         "one JSON line per point")
    ap.add_argument("--workload", default=WORKLOAD.name, choices=sorted(configs.BY_NAME),
                    help="the headline workload (default: the Qwen3-8B layer, batch 1, 32K)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = configs.BY_NAME[args.workload]
    lens, kps = gen.ctx_lens(w), gen.k_per_seq(w, gen.ctx_lens(w))
    nbytes = algorithmic_bytes(w, lens, kps)
    peak, peak_kind = read_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        # Each step is one full oracle iteration of the workload (all its
        # (sequence, KV head) units on the host cores); --warmup untimed steps
        # first, then --steps timed ones, cut at 240 s so the arm ends in minutes.
        ref = time_oracle(w, nbytes, budget_s=240.0, warmup=args.warmup, steps=args.steps)
        line = {"impl": "reference", "metric": METRIC, "value": ref["value"], "unit": "GB/s",
                "n_gpus": args.gpus, "steps": ref["steps"], "warmup": ref["warmup"],
                "ms_per_step": round(ref["s_per_step"] * 1000, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": base_config(w, lens, kps),
                "cpu_baseline": {k: ref[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                     "cpu_model")},
                "e2e": {"value": ref["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "note": "fp64 CPU oracle (the pages publish no implementation to install); "
                        "ms_per_step is the median wall time of one full iteration"}
        print(json.dumps(line))
        return

    if args.stack_sweep:
        if rank == 0:
            for line in stack_sweep(peak, peak_kind):
                print(json.dumps(line), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    (it, nbytes, ms_step, K_eff, stages, timing, clocks, e2e, variants, extra) = run_gpu(
        args, rank, world, dist, peak, peak_kind)
    us_step = ms_step * 1000.0
    gbs = job_gbs(nbytes["total"], ms_step, 1)
    line = {"metric": METRIC, "value": round(job_gbs(nbytes["total"], ms_step, world), 2),
            "unit": "GB/s",
            "n_gpus": world, "steps": K_eff, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "us_per_iteration": round(us_step, 2),
            "timing": timing,
            "pct_of_8tbs": round(100 * gbs / (ROOFLINE_TBS * 1000), 2),
            "pct_of_measured_hbm": round(100 * gbs / peak, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": base_config(w, lens, kps),
            "bytes_per_iteration": nbytes["total"],
            "gpu_launches": K_eff * (2 + w.gamma) * timing["repeats"], "clocks": clocks,
            "e2e": e2e}
    v_us = stages["verify_us"]
    line["stages"] = {k: (round(v, 3) if isinstance(v, float) else v) for k, v in stages.items()}
    # the capture-plus-top-k overhead over plain verify, back to back (each kernel in a
    # graph of its own launches), and over the stage events
    vb2b, vplain = variants["verify_capture2_us"], variants["verify_no_capture_us"]
    line["capture_plus_select_overhead"] = round((vb2b + variants["select_us"]) / vplain - 1.0, 4)
    line["capture_overhead"] = round(vb2b / vplain - 1.0, 4)
    line["overhead_formula"] = ("(verify with capture + select) / plain verify - 1, each "
                                "timed back to back in a graph of its own launches")
    line["roofline"] = roofline_entry(nbytes["verify"], vb2b, peak, peak_kind, v_us,
                                      kernel=verify_kernel_name(w))
    # the draft kernel, the same way: per launch back to back, stage events as context
    line["roofline_draft"] = draft_roofline_entry(nbytes["draft"], variants["draft_step_us"],
                                                  stages["draft_us_per_step"], peak)
    # the "next" rows, measured the same way on the same workload: collect-all
    # capture, one T shared by all heads, the query-agnostic window selector
    line["variants"] = variants
    if extra:
        line["workloads"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        ref = time_oracle(w, nbytes, budget_s=15.0, warmup=1)
        line["cpu_baseline"] = {k: ref[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                    "cpu_model")}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
