#!/usr/bin/env python
"""Benchmark of the block-sparse attention hot path on one GB300 (or N ranks).

A step is one pass of the whole hot path over one batch of the synthetic
workload: BlockMask build (fa_block_mask_build) + fused forward (fa_fwd).
Default workload: packed grouped attention at scale (bf16, B=1, H=4, D=128,
4096 groups x 17 variates = 69632 tokens, block-diagonal group mask).

Printed on rank 0: one JSON line with
  value        forward TFLOP/s on visited 128x128 tiles (4 r c D per tile,
               r x c the tile's in-range rows x columns), whole job, per step
  windows_per_s  groups (independent windows) processed per second
  roofline     the forward kernel against the measured HBM (memory-bound
               shapes) or bf16 tensor peak (compute-bound shapes)
  e2e          the same metric through the public API with pinned host
               buffers, host<->device copies inside the timed region
  cpu_baseline the fp64 oracle on a bounded sample, on the host cores
  workloads    the other workloads (document, causal soft-cap, window+ALiBi
               GQA, grouped fp32) measured the same way
Each timed step is one replay of a CUDA graph holding the two launches, with
CUDA events around it on the launching stream; L2 is flushed (256 MiB write)
before every step, outside the events.  ``--impl reference`` times the oracle
instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from block_sparse_attention_fa_gb300 import synth  # noqa: E402

METRIC = "fwd TFLOP/s on visited blocks & % of GB300 bf16 tensor peak; windows/s grouped"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEADLINE = "grouped_bf16"
SECONDARY = ["document_bf16", "causal_softcap_bf16", "window_alibi_gqa_bf16", "window_alibi_softcap_bf16",
             "grouped_fp32"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- accounting

def tile_sizes(n, T):
    return np.minimum(128, T - 128 * np.arange(n))


def visited_flops(w, bm_np):
    """Sum over (b, hq) of 4 r c D over the visited tiles."""
    nq = bm_np["kv_num_blocks"].shape[-1]
    r = tile_sizes(nq, w.T).astype(np.float64)
    c = tile_sizes(bm_np["kv_indices"].shape[-1], w.kv_len).astype(np.float64)
    total = 0.0
    Bm, Hm = bm_np["kv_num_blocks"].shape[:2]
    for b in range(Bm):
        for h in range(Hm):
            for qb in range(nq):
                n1 = bm_np["kv_num_blocks"][b, h, qb]
                n2 = bm_np["full_kv_num_blocks"][b, h, qb]
                idx = np.concatenate([bm_np["kv_indices"][b, h, qb, :n1], bm_np["full_kv_indices"][b, h, qb, :n2]])
                total += r[qb] * c[idx].sum()
    reps = (w.B // Bm) * (w.Hq // Hm)
    return 4.0 * w.D * total * reps


def build_bytes(Bm, Hm, nq, nkv, T, mask, table_bytes=0):
    """Bytes the BlockMask builder must move at least: the four arrays
    written (two [Bm, Hm, nq, nkv] index arrays and two [Bm, Hm, nq] counts,
    int32) and the mask's own data read once (segment ids or the table)."""
    written = 2 * 4 * Bm * Hm * nq * nkv + 2 * 4 * Bm * Hm * nq
    read = 4 * Bm * T if mask == "document" else table_bytes
    return written + read


def build_roofline(build_ms, nbytes, peaks, peak_src):
    gbs = nbytes / (build_ms * 1e-3) / 1e9
    return {"bound": "hbm", "build_ms": round(build_ms, 4), "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes,
            "peak_source": peak_src, "kernel": "block_mask_kernel"}


def tcgen05_peak_tflops(device, sm_mhz):
    """The tensor pipe's issue rate: 8192 dense bf16 FLOP per clock per SM
    (128 x 256 x 16 MMA in 128 cycles, measured by a tcgen05 probe) at the SM
    clock sampled during the timed region."""
    import torch
    if not sm_mhz:
        return None
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return sms * 8192 * sm_mhz * 1e6 / 1e12


def algorithmic_bytes(w):
    """Bytes the forward must move at least: Q, K, V read, O and lse written."""
    el = 2 if w.dtype == "bf16" else 4
    return (w.B * w.T * w.D * el * (2 * w.Hq + 2 * w.Hkv)) + w.B * w.Hq * w.T * 4


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons, busy = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                s, m, pw = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            sm.append(s)
            smax.append(m)
            busy.append((pw, s))
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed"]}
        # samples under load: the upper half by power draw
        busy.sort()
        loaded = [s for _, s in busy[len(busy) // 2:]] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU timing

class Runner:
    """Holds device inputs for one workload and runs build + forward."""

    def __init__(self, w, device):
        import torch
        from block_sparse_attention_fa_gb300 import fa
        self.torch, self.fa, self.w, self.device = torch, fa, w, device
        t0 = time.time()
        q, k, v = w.qkv()
        self.host = (q, k, v)
        self.seg = w.segments()
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.dt = dt
        self.q, self.k, self.v = (torch.from_numpy(x).to(device).to(dt) for x in (q, k, v))
        self.seg_d = torch.from_numpy(self.seg).to(device) if self.seg is not None else None
        self.score_kw = {"score": w.score}
        if w.score in ("softcap", "alibi_softcap"):
            self.score_kw["softcap"] = w.softcap
        if w.score in ("alibi", "alibi_softcap"):
            self.score_kw["alibi_slopes"] = torch.from_numpy(w.slopes()).to(device)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=device)
        self.ws = fa.Workspace(device)
        self.bm = self.build()
        self.ws.check()
        self.bm_np = self.bm.numpy()
        self.flops = visited_flops(w, self.bm_np)
        self.setup_s = time.time() - t0

    def build(self):
        w = self.w
        Bm = self.seg.shape[0] if self.seg is not None else 1
        return self.fa.block_mask(w.mask, Bm, 1, w.T, w.T, window=w.window, prefix_len=w.prefix_len,
                                  seg_ids=self.seg_d, workspace=self.ws)

    def fwd(self, bm=None):
        return self.fa.fwd(self.q, self.k, self.v, bm or self.bm, out=self.out, lse=self.lse,
                           workspace=self.ws, **self.score_kw)

    def graph(self, fn):
        """Capture fn (our C-ABI launches only, no allocation) in a CUDA graph,
        so a timed step costs one graph launch of host time."""
        torch = self.torch
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.ws.check()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def time_graph(self, g, steps, warmup, flush):
        """Per-step CUDA-event times (ms) of graph replays, L2 flushed before each."""
        torch = self.torch
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, c in evs:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            g.replay()
            c.record(stream)
        torch.cuda.synchronize()
        self.ws.check()
        return [a.elapsed_time(c) for a, c in evs]

    def time_build(self, steps, warmup, flush):
        """fa_block_mask_build alone (one CUDA graph replay per step, L2
        flushed before each): per-step times in ms."""
        g = self.graph(lambda: self.bm.rebuild(workspace=self.ws))
        return self.time_graph(g, steps, warmup, flush)

    def time_steps(self, steps, warmup, flush):
        """(step times, forward-kernel times) in ms: a step is BlockMask build
        + forward; the forward is also timed alone (the dominant kernel)."""
        step_g = self.graph(lambda: (self.bm.rebuild(workspace=self.ws), self.fwd()))
        fwd_g = self.graph(lambda: self.fwd())
        return self.time_graph(step_g, steps, warmup, flush), self.time_graph(fwd_g, steps, warmup, flush)

    def e2e(self, steps, warmup):
        """Metric through the public API with pinned host buffers: every step
        copies its inputs host -> device, builds the BlockMask, runs the
        forward and copies O and lse device -> host.  Steps are pipelined over
        three streams with two buffer sets: step i+1's inputs go up while step
        i computes and step i-1's result comes down (the two copy directions
        of the host link run at once)."""
        torch, w = self.torch, self.w
        hq, hk, hv = (torch.from_numpy(x).to(self.dt).pin_memory() for x in self.host)
        hseg = torch.from_numpy(self.seg).pin_memory() if self.seg is not None else None
        ho = [torch.empty(self.q.shape, dtype=self.dt).pin_memory() for _ in range(2)]
        hl = [torch.empty(self.lse.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
        slopes = self.score_kw.get("alibi_slopes")
        hsl = slopes.cpu().pin_memory() if slopes is not None else None
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv) + ((hseg,) if hseg is not None else ())
                  + ((hsl,) if hsl is not None else ()))
        d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
        dev = self.device
        up, comp, down = (torch.cuda.Stream(device=dev) for _ in range(3))
        bufs = []
        for _ in range(2):
            d = {"q": torch.empty_like(self.q), "k": torch.empty_like(self.k), "v": torch.empty_like(self.v),
                 "o": torch.empty_like(self.q), "lse": torch.empty_like(self.lse),
                 "seg": torch.empty_like(self.seg_d) if self.seg_d is not None else None,
                 "slopes": torch.empty_like(slopes) if slopes is not None else None,
                 "ws": self.fa.Workspace(dev)}
            bufs.append(d)
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]
        Bm = self.seg.shape[0] if self.seg is not None else 1

        def step(i):
            d, j = bufs[i % 2], i % 2
            with torch.cuda.stream(up):
                up.wait_event(ev_comp[j])          # the compute of step i-2 is done with these inputs
                d["q"].copy_(hq, non_blocking=True)
                d["k"].copy_(hk, non_blocking=True)
                d["v"].copy_(hv, non_blocking=True)
                if hseg is not None:
                    d["seg"].copy_(hseg, non_blocking=True)
                if hsl is not None:
                    d["slopes"].copy_(hsl, non_blocking=True)
                ev_up[j].record(up)
            with torch.cuda.stream(comp):
                comp.wait_event(ev_up[j])
                comp.wait_event(ev_down[j])        # step i-2's output has left this buffer
                kw = dict(self.score_kw)
                if hsl is not None:
                    kw["alibi_slopes"] = d["slopes"]
                bm = self.fa.block_mask(w.mask, Bm, 1, w.T, w.T, window=w.window, prefix_len=w.prefix_len,
                                        seg_ids=d["seg"], workspace=d["ws"], stream=comp)
                self.fa.fwd(d["q"], d["k"], d["v"], bm, out=d["o"], lse=d["lse"], workspace=d["ws"],
                            stream=comp, **kw)
                ev_comp[j].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(ev_comp[j])
                ho[j].copy_(d["o"], non_blocking=True)
                hl[j].copy_(d["lse"], non_blocking=True)
                ev_down[j].record(down)

        for i in range(warmup):
            step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            step(warmup + i)
        torch.cuda.synchronize()
        sec = (time.perf_counter() - t0) / steps
        for d in bufs:
            d["ws"].check()
        return sec, h2d, d2h


KERNEL_SOURCES = ["fwd_bf16.cu", "fa_api.cu", "ptx.cuh", "fa_internal.h", "tanh_poly.h", "tanh2_poly.h"]


def kernel_source_digest():
    """sha256 (first 16 hex digits) of the bf16 forward's sources, in order."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_attention_fa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload):
    """DRAM bytes (read + write) of one forward launch from the committed ncu
    capture of this workload, or None when there is none or the kernel's
    sources have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    t = d.get("workloads", {}).get(workload)
    if t is None or d.get("source_digest") != kernel_source_digest():
        return None
    return int(t["read"]) + int(t["write"])


def summarize(w, r, step_ms, fwd_ms, peaks, peak_src, build_ms=None, floor_ms=None):
    ms = statistics.median(step_ms)
    fms = statistics.mean(fwd_ms)
    tflops = r.flops / (ms * 1e-3) / 1e12
    fwd_tflops = r.flops / (fms * 1e-3) / 1e12
    bytes_ = algorithmic_bytes(w)
    gbs = bytes_ / (fms * 1e-3) / 1e9
    # which roofline bounds the forward: arithmetic intensity vs ridge point
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    intensity = r.flops / bytes_
    if w.dtype == "fp32":
        # a latency-bound launch: its floor is the time of one graph-launched
        # kernel that does nothing measurable, taken in the same run
        fl = floor_ms if floor_ms else None
        roof = {"bound": "latency", "achieved": round(fms * 1e3, 2),
                "peak": round(fl * 1e3, 2) if fl else None, "unit": "us",
                "frac": round(fl / fms, 4) if fl else None, "traffic": None,
                "floor": "one-element add kernel replayed from a CUDA graph, same run"}
    elif intensity < ridge:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None}
    else:
        roof = {"bound": "tensor", "achieved": round(fwd_tflops, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(fwd_tflops / peaks["bf16_tflops"], 4), "traffic": None}
    if w.dtype == "bf16":
        roof["traffic"] = measured_traffic(w.name)
    roof["peak_source"] = peak_src
    roof["kernel"] = "fwd_bf16_kernel" if w.dtype == "bf16" else "fwd_fp32_kernel"
    roof["kernel_ms"] = round(fms, 4)
    roof["algorithmic_bytes"] = bytes_
    roof["visited_flops"] = r.flops
    out = {
        "ms_per_step": round(ms, 4),
        "tflops": round(tflops, 2),
        "pct_bf16_peak": round(100 * tflops / peaks["bf16_tflops"], 2),
        "fwd_ms": round(fms, 4),
        "fwd_tflops": round(fwd_tflops, 2),
        "fwd_gbs": round(gbs, 1),
        "tokens_per_s": round(w.B * w.T / (ms * 1e-3), 1),
        "visited_tiles": int(r.bm_np["kv_num_blocks"].sum() + r.bm_np["full_kv_num_blocks"].sum()),
        "roofline": roof,
    }
    if w.groups:
        out["windows_per_s"] = round(w.groups * w.B / (ms * 1e-3), 1)
    if build_ms is not None:
        bmn = r.bm_np
        Bm, Hm, nq = bmn["kv_num_blocks"].shape
        nkv = bmn["kv_indices"].shape[-1]
        out["build"] = build_roofline(statistics.mean(build_ms), build_bytes(Bm, Hm, nq, nkv, w.T, w.mask),
                                      peaks, peak_src)
    return out


def compact(entry, tc_peak):
    """The few numbers of a workload the last lines of the output keep:
    kernel ms, the roofline fraction keyed by its bound ("tensor" of the
    cuBLAS peak, "tc05" of the tcgen05 issue rate, "hbm" of the copy
    bandwidth, "floor" the launch floor over the time), and the builder's
    HBM fraction ("build")."""
    roof = entry["roofline"]
    key = {"tensor": "tensor", "hbm": "hbm", "latency": "floor"}.get(roof["bound"], roof["bound"])
    c = {"ms": entry["fwd_ms"], key: roof["frac"] if roof["frac"] is None else round(roof["frac"], 3)}
    if roof["bound"] == "tensor" and tc_peak:
        c["tc05"] = round(roof["achieved"] / tc_peak, 3)
    if "build" in entry:
        c["build"] = round(entry["build"]["frac"], 3)
    return c


def launch_floor_ms(device, steps, warmup, flush):
    """CUDA-event time of one graph replay holding one trivial kernel: the
    launch floor of any single-kernel step on this GPU."""
    import torch
    x = torch.zeros(1, device=device)
    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        x.add_(1.0)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        x.add_(1.0)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, c in evs:
        flush.zero_()
        a.record(stream)
        g.replay()
        c.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(c) for a, c in evs)


# ---------------------------------------------------- the builder at scale

# A BlockMask large enough that its writes leave L2 (129 MB): document masks
# over 16 packed rows of 131072 tokens (documents of 256-2048 tokens, the
# document workload's recipe), nq = nkv = 1024, 134 MB of index arrays.
BUILD_SCALE = {"B": 16, "T": 131072, "seed": 41}


def build_scale_section(device, flush, steps, warmup, peaks, peak_src):
    import torch
    from block_sparse_attention_fa_gb300 import fa
    B, T = BUILD_SCALE["B"], BUILD_SCALE["T"]
    seg = torch.from_numpy(synth.document_segments(BUILD_SCALE["seed"], B, T)).to(device)
    ws = fa.Workspace(device)
    bm = fa.block_mask("document", B, 1, T, T, seg_ids=seg, workspace=ws)
    ws.check()

    def fn():
        bm.rebuild(workspace=ws)

    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, c in evs:
        flush.zero_()
        a.record(stream)
        g.replay()
        c.record(stream)
    torch.cuda.synchronize()
    ws.check()
    ms = statistics.mean(a.elapsed_time(c) for a, c in evs)
    out = build_roofline(ms, build_bytes(B, 1, bm.nq, bm.nkv, T, "document"), peaks, peak_src)
    out["config"] = {"mask": "document", "B": B, "T": T, "nq": bm.nq, "nkv": bm.nkv}
    del bm, seg
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------- split-KV decoding path

def decode_bytes(w):
    """Algorithmic HBM bytes of one decoding forward with every key visible:
    K and V once per (b, kv head), Q and O (bf16) and lse once."""
    kv = 2 * w.B * w.Hkv * w.T * w.D * 2
    qo = 2 * w.B * w.Hq * w.Tq * w.D * 2
    return kv + qo + w.B * w.Hq * w.Tq * 4


def decode_section(device, flush, steps, warmup, peaks, peak_src):
    """Time fa_fwd_decode (split kernel + combine kernel, one CUDA graph
    replay, L2 flushed before each) on each decoding workload."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    out = {}
    for name, w in synth.DECODE_WORKLOADS.items():
        q, k, v = (torch.from_numpy(x).to(device).to(torch.bfloat16) for x in w.qkv())
        table = w.table()
        tab = torch.from_numpy(synth.pack_table(table)).to(device) if table is not None else None
        bm = fa.block_mask(w.mask, tab.shape[0] if tab is not None else 1, 1, w.Tq, w.T, window=w.window,
                           prefix_len=w.prefix_len, table=tab)
        splits = fa.decode_splits(q, k, bm)
        parts = fa.decode_partials(q, splits)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device=device)
        ws = fa.Workspace(device)

        def fn():
            fa.fwd_decode(q, k, v, bm, num_splits=splits, out=o, lse=lse, partials=parts, workspace=ws)

        side = torch.cuda.Stream(device=device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        ws.check()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, c in evs:
            flush.zero_()
            a.record(stream)
            g.replay()
            c.record(stream)
        torch.cuda.synchronize()
        ws.check()
        ms = statistics.mean(a.elapsed_time(c) for a, c in evs)
        nbytes = decode_bytes(w)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {
            "config": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "q_len": w.Tq, "kv_len": w.T, "D": w.D,
                       "mask": w.mask, "score": w.score, "splits": splits,
                       "rows_per_group": (w.Hq // w.Hkv) * w.Tq},
            "ms": round(ms, 4),
            "tokens_per_s": round(w.B * w.Tq / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peak_src,
                         "kernels": ["decode_split_kernel", "decode_combine_kernel"],
                         "algorithmic_bytes": nbytes},
        }
        del q, k, v, parts, o, lse
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------- backward

BACKWARD_WORKLOADS = ["causal_softcap_bf16", "window_alibi_softcap_bf16"]


def backward_section(device, flush, steps, warmup, peaks, peak_src):
    """Time fa_bwd (row statistics, dK/dV and dQ kernels, one CUDA graph replay, L2
    flushed) after a forward on the same inputs.  Algorithmic FLOPs: 5
    products per visited tile (S, dP, dV, dK, dQ) = 2.5 x the forward's."""
    import torch
    from block_sparse_attention_fa_gb300 import fa
    out = {}
    for name in BACKWARD_WORKLOADS:
        w = synth.WORKLOADS[name]
        r = Runner(w, device)
        o, lse = r.fwd()
        dout = torch.from_numpy(synth.round_to_bf16(synth.standard_normal(w.seed + 500, tuple(r.q.shape)))).to(
            device).to(torch.bfloat16)
        f32 = dict(dtype=torch.float32, device=device)
        dq, dk, dv = torch.empty(r.q.shape, **f32), torch.empty(r.k.shape, **f32), torch.empty(r.v.shape, **f32)
        rowstats = fa.bwd_rowstats(r.q)
        r.bm.cols(workspace=r.ws)
        g = r.graph(lambda: fa.bwd(r.q, r.k, r.v, o, lse, dout, r.bm, dq=dq, dk=dk, dv=dv, rowstats=rowstats,
                                   workspace=r.ws, **r.score_kw))
        ms = statistics.mean(r.time_graph(g, steps, warmup, flush))
        flops = 2.5 * r.flops
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "tflops": round(tf, 2),
                     "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                                  "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                                  "peak_source": peak_src, "algorithmic_flops": flops,
                                  "kernels": ["bwd_rowstats_kernel", "bwd_tc_kernel<dK/dV>", "bwd_tc_kernel<dQ>"]}}
        del r, dq, dk, dv, dout
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------- CPU (oracle) side

def oracle_rate(w, seconds, threads, seed=0, max_rows=None):
    """Rows/s of the oracle on seeded random rows of the workload, sized to
    take about `seconds` (one calibration batch first)."""
    import oracle
    q, k, v = w.qkv()
    seg = w.segments()
    kw = {"mask": w.mask, "window": w.window, "prefix_len": w.prefix_len, "seg": seg, "score": w.score,
          "softcap": w.softcap, "slopes": w.slopes()}
    rng = np.random.default_rng(seed)
    total = w.B * w.Hq * w.T
    n0 = min(total, max(threads * 4, 64))
    rows = rng.choice(total, size=n0, replace=False).astype(np.int64)
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, rows=rows, threads=threads, **kw)
    dt0 = time.perf_counter() - t0
    n = int(min(total, max(n0, n0 * seconds / max(dt0, 1e-6))))
    if max_rows:
        n = min(n, max_rows)
    rows = rng.choice(total, size=n, replace=False).astype(np.int64)
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, rows=rows, threads=threads, **kw)
    dt = time.perf_counter() - t0
    return n, dt, total


def cpu_baseline(w, flops, seconds):
    import oracle
    threads = oracle.default_threads()
    n, dt, total = oracle_rate(w, seconds, threads)
    rows_per_s = n / dt
    value = rows_per_s * (flops / total) / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} seeded random query rows of {total} ({w.name}), full fp64 rows, "
                      f"{dt:.1f} s; value = rows/s x visited FLOPs per row",
            "rows_per_s": round(rows_per_s, 2)}


# ----------------------------------------------------------------------- main

def max_over_ranks(x: float) -> float:
    """Max of a per-rank scalar over all ranks (identity on one rank).  The
    only cross-rank traffic of the benchmark: the data path has none."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    threads = oracle.default_threads()
    # visited FLOPs from the oracle's own tile scan (no GPU involved)
    seg = w.segments()
    bm = oracle.block_mask(mask=w.mask, B=seg.shape[0] if seg is not None else 1, H=1, q_len=w.T, kv_len=w.T,
                           window=w.window, prefix_len=w.prefix_len, seg=seg, threads=threads)
    flops = visited_flops(w, bm)
    per_step = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    q, k, v = w.qkv()
    kw = {"mask": w.mask, "window": w.window, "prefix_len": w.prefix_len, "seg": seg, "score": w.score,
          "softcap": w.softcap, "slopes": w.slopes()}
    total = w.B * w.Hq * w.T
    n, dt0, _ = oracle_rate(w, min(per_step, 5.0), threads)
    rows_per_step = min(total, max(threads, int(n * per_step / max(dt0, 1e-6))))
    rng = np.random.default_rng(1)
    times = []
    for s in range(args.warmup + args.steps):
        rows = rng.choice(total, size=min(rows_per_step, total), replace=False).astype(np.int64)
        t0 = time.perf_counter()
        oracle.fwd(q, k, v, rows=rows, threads=threads, **kw)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec_per_row = sum(times) / (len(times) * rows_per_step)
    value = (flops / total) / sec_per_row / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T,
                                        "D": w.D, "mask": w.mask, "score": w.score, "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} seeded random query rows per step of {total}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if w.groups:
        line["windows_per_s"] = w.groups * w.B * (1.0 / (sec_per_row * total))
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=list(synth.WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the split-KV decoding workloads and print their section")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the backward workloads and print their section")
    ap.add_argument("--build-only", action="store_true",
                    help="time only the BlockMask builder at scale and print its section")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_src = load_peaks()
    from block_sparse_attention_fa_gb300 import fa
    fa.load_library()

    if args.decode_only or args.backward_only or args.build_only:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        if args.decode_only:
            out = {"decode": decode_section(device, flush, args.steps, args.warmup, peaks, peak_src)}
        elif args.backward_only:
            out = {"backward": backward_section(device, flush, args.steps, args.warmup, peaks, peak_src)}
        else:
            out = {"build_at_scale": build_scale_section(device, flush, args.steps, args.warmup, peaks, peak_src)}
        print(json.dumps(out), flush=True)
        return

    r = Runner(w, device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device.index) as clk:
        step_ms, fwd_ms = r.time_steps(args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if world > 1:
        worst = max_over_ranks(statistics.median(step_ms))
        dist.barrier()
        step_ms = [worst] * len(step_ms)
    build_ms = r.time_build(args.steps, args.warmup, flush)
    floor_ms = launch_floor_ms(device, args.steps, args.warmup, flush)
    head = summarize(w, r, step_ms, fwd_ms, peaks, peak_src, build_ms=build_ms, floor_ms=floor_ms)
    clocks = clk.summary()
    tc_peak = tcgen05_peak_tflops(device, clocks.get("sm_mhz"))
    if head["roofline"]["bound"] == "tensor" and tc_peak:
        head["roofline"]["frac_tcgen05"] = round(head["roofline"]["achieved"] / tc_peak, 4)

    extra = {}
    if rank == 0 and w.name == "grouped_bf16":
        # the dense-masked pass over the same inputs: every tile partial
        nq = r.bm.nq
        dense = fa.BlockMask(1, 1, w.T, w.T, "document", 0, 0, r.seg_d, device)
        dense.kv_num_blocks.fill_(nq)
        dense.kv_indices.copy_(torch.arange(nq, dtype=torch.int32, device=device).expand(1, 1, nq, nq))
        dense.full_kv_num_blocks.zero_()
        dense.full_kv_indices.fill_(-1)
        dsteps = max(3, args.steps // 4)
        dg = r.graph(lambda: r.fwd(dense))
        dms = statistics.mean(r.time_graph(dg, dsteps, 2, flush))
        dflops = 4.0 * w.D * w.T * w.T * w.B * w.Hq
        extra["dense_masked_pass"] = {"fwd_ms": round(dms, 3), "tflops": round(dflops / (dms * 1e-3) / 1e12, 1),
                                      "windows_per_s": round(w.groups / (dms * 1e-3), 1),
                                      "speedup_block_sparse": round(dms / head["fwd_ms"], 1)}

    e2e = None
    if not args.no_e2e:
        sec, h2d, d2h = r.e2e(max(3, args.steps // 4), 2)
        e2e = {"value": round(r.flops / sec / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(sec * 1e3, 3)}
        if w.groups:
            e2e["windows_per_s"] = round(w.groups * w.B / sec, 1)

    secondary = {}
    if rank == 0 and not args.no_secondary:
        for name in SECONDARY:
            if name == w.name:
                continue
            w2 = synth.WORKLOADS[name]
            r2 = Runner(w2, device)
            s2, f2 = r2.time_steps(args.steps, args.warmup, flush)
            b2 = r2.time_build(args.steps, args.warmup, flush)
            secondary[name] = summarize(w2, r2, s2, f2, peaks, peak_src, build_ms=b2, floor_ms=floor_ms)
            if secondary[name]["roofline"]["bound"] == "tensor" and tc_peak:
                roof = secondary[name]["roofline"]
                roof["frac_tcgen05"] = round(roof["achieved"] / tc_peak, 4)
            del r2
            torch.cuda.empty_cache()

    decode = None
    if rank == 0 and not args.no_decode:
        decode = decode_section(device, flush, args.steps, args.warmup, peaks, peak_src)
    backward = None
    if rank == 0 and not args.no_backward:
        backward = backward_section(device, flush, max(3, args.steps // 4), args.warmup, peaks, peak_src)

    build_scale = None
    if rank == 0 and not args.no_secondary:
        build_scale = build_scale_section(device, flush, args.steps, args.warmup, peaks, peak_src)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(w, r.flops, args.cpu_seconds)

    if rank == 0:
        n = world
        # The last keys are the compact per-workload summary, so that the
        # tail of the line holds every configuration's roofline fraction.
        summary = {w.name: compact(head, tc_peak)}
        for name, entry in secondary.items():
            summary[name] = compact(entry, tc_peak)
        if build_scale:
            summary["build_16x131072"] = {"ms": build_scale["build_ms"], "hbm": round(build_scale["frac"], 3)}
        for name, entry in (backward or {}).items():
            summary["bwd_" + name] = {"ms": entry["ms"], "tensor": round(entry["roofline"]["frac"], 3)}
        for name, entry in (decode or {}).items():
            summary[name] = {"ms": entry["ms"], "hbm": round(entry["roofline"]["frac"], 3)}
        line = {
            "metric": METRIC,
            "value": round(head["tflops"] * n, 3),
            "unit": "TFLOP/s",
            "n_gpus": n,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1) inputs, shapes of the workload)",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "D": w.D,
                       "mask": w.mask, "score": w.score, "groups": w.groups,
                       "step": "fa_block_mask_build + fa_fwd (one CUDA graph replay)",
                       "l2": "flushed between steps (256 MiB write, outside the per-step events)", "parallelism": f"replicas x{n}"},
            "pct_bf16_peak": head["pct_bf16_peak"],
            "windows_per_s": head.get("windows_per_s", None) and round(head["windows_per_s"] * n, 1),
            "tokens_per_s": round(head["tokens_per_s"] * n, 1),
            "fwd_ms": head["fwd_ms"],
            "fwd_tflops": head["fwd_tflops"],
            "roofline": head["roofline"],
            "build": head.get("build"),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
            "peaks": {"source": peak_src, **peaks, "tcgen05_issue_tflops": tc_peak and round(tc_peak, 1),
                      "note": "frac: of the measured peaks (cuBLAS bf16 burst, HBM copy); "
                              "frac_tcgen05: of SMs x 8192 FLOP/clk x the sampled SM clock"},
            **extra,
            "decode": decode,
            "backward": backward,
            "build_at_scale": build_scale,
            "workloads": secondary,
            "summary": summary,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
