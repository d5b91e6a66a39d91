#!/usr/bin/env python
"""Benchmark of the W4A16 INT4-weight MoE layer (sigmoid+bias routing) on GB300.

A step is one pass of the whole layer over one batch: route, align, gate/up
GEMM with fused SiLU*mul, down GEMM, top-k weighted sum.  Default workload:
the Kimi-K2 EP8 decode shard (64 tokens, hidden 7168, intermediate 2048, 48
of 384 experts local, top-8).  Inputs are seeded synthetic data of that shape;
weights are random INT4 with BF16 group-32 scales.

Timing: L2 is never warm across steps: the loop rotates over R independent
layer replicas (distinct weights and inputs, like consecutive layers of a
model), and every step's own weight working set already exceeds the 129 MB
L2.  A step is one replay of a CUDA graph holding one chord_moe_layer call
(the call a user makes, with its kernels chained by programmatic launches);
the region of K steps is bracketed by a barrier and torch.cuda.synchronize(),
and the max over ranks is reported.  Kernel durations (for the roofline)
come from a second CUDA-event-timed region of K steps that runs the same
layer as four graph replays (route+align, gate/up, down, combine: the
layer's C-ABI calls one by one) with events between them.  Clocks:
nvidia-smi polls every 200 ms from before the timed regions to after them,
and the same step keeps replaying untimed around them (about a second in
all), so the samples are taken under the timed load.

The JSON line's headline (`value`, `roofline`, ...) is the selected workload
(default EP8 decode); unless --only is given, `workloads` carries the same
fields for the metric's other layer shards, measured the same way in the same
run: the TP8 decode shard (HBM-bound, GB/s) and the EP8 prefill shard
(tensor-bound, TFLOP/s against the measured BF16 peak: the burst figure when
the timed region lasts under a second, else the sustained one).

`e2e` repeats the measurement through the public single call
(chord_moe_layer) with pinned HOST inputs and outputs: each step copies x
and the router logits host->device and the layer output device->host, on
two copy streams, so the copies of neighbouring steps overlap a step's
kernels.

`--impl reference` times the CPU oracle (numpy, FP64) on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 MoE layer tokens/s; decode HBM GB/s, prefill TFLOPS vs GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_SOURCES = {
    "small": ["w4a16_int4_weight_sigmoid_gb300/csrc/gemm_small.cu",
              "w4a16_int4_weight_sigmoid_gb300/csrc/common.cuh"],
    "large": ["w4a16_int4_weight_sigmoid_gb300/csrc/gemm_large.cu",
              "w4a16_int4_weight_sigmoid_gb300/csrc/tc5.cuh",
              "w4a16_int4_weight_sigmoid_gb300/csrc/common.cuh"],
}


def parse_args():
    from w4a16_int4_weight_sigmoid_gb300 import workload as wl
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(wl.WORKLOADS), default=wl.EP8_DECODE.name)
    p.add_argument("--replicas", type=int, default=4)
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-budget-s", type=float, default=20.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", action="store_true",
                   help="measure the selected workload only (by default the line also carries the "
                        "metric's other layer workloads under 'workloads')")
    p.add_argument("--report", choices=["route_align", "m_sweep", "grouped"], default=None,
                   help="report-only measurements instead of the headline line: router+align "
                        "microseconds per (M, BLOCK_M), the layer over M = 1..8192 at EP8 shapes, "
                        "or the grouped-layout GEMMs at EP8 expert shapes")
    return p.parse_args()


# ----------------------------------------------------------------- helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str, gemm_path: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since the capture; else None."""
    record = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(record):
        return None
    with open(record) as f:
        entries = json.load(f)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("path", "small") == gemm_path:
            if e.get("source_sha") == source_sha(KERNEL_SOURCES[gemm_path]):
                return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.out = ""

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.out, _ = self.proc.communicate()
        return self.summary()

    def summary(self):
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# --------------------------------------------------------------- workloads
class Replica:
    """One layer's weights, inputs and buffers on the device."""

    def __init__(self, shape, seed, device, keep_host=False):
        import torch
        from w4a16_int4_weight_sigmoid_gb300 import chord
        from w4a16_int4_weight_sigmoid_gb300 import workload as wl
        from w4a16_int4_weight_sigmoid_gb300.layer import W4A16MoELayer, to_device
        self.shape = shape
        d = wl.layer_inputs(shape, seed)
        self.host = d if keep_host else None
        self.layer = W4A16MoELayer(d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"], shape.E_total,
                                   shape.expert_begin, shape.topk, device=device)
        self.x = to_device(d["x"], device)
        self.logits = to_device(d["logits"], device)
        self.bias = to_device(d["bias"], device)
        self.x_pinned = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
        self.logits_pinned = torch.from_numpy(d["logits"]).pin_memory()
        del d
        M, k, E, H, I = shape.M, shape.topk, shape.E_local, shape.H, shape.I
        self.plan = chord.chord_moe_layer_plan(M, shape.E_total, k)
        self.large = self.plan.path == chord.CHORD_PATH_LARGE_M
        self.bm = 16 if self.large else self.plan.rows_per_pass   # the layer's own choice
        self.cap = chord.chord_moe_align_capacity(M, k, E, self.bm)
        i32, dev = torch.int32, device
        self.tw = torch.empty((M, k), dtype=torch.float32, device=dev)
        self.ti = torch.empty((M, k), dtype=torch.int32, device=dev)
        self.sorted = torch.empty(self.cap, dtype=i32, device=dev)
        self.eids = torch.empty(self.cap // self.bm, dtype=i32, device=dev)
        self.ntpp = torch.empty(1, dtype=i32, device=dev)
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.pos = torch.empty(M * k, dtype=i32, device=dev)
        wsb = chord.chord_moe_align_workspace_bytes(M, k, E)
        self.aws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
        self.h = torch.empty((self.cap, I), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((self.cap, H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.ws_gu = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(self.cap, H, True),
                                 dtype=torch.uint8, device=dev)
        self.ws_dn = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(self.cap, I, False),
                                 dtype=torch.uint8, device=dev)
        self.align_launches = 1 if wsb == 0 else 2
        self.gemm_launches = 3 if self.large else 2     # + the row gather on the tcgen05 path
        # chord_moe_layer routes and aligns in one launch for small batches (the
        # library's rule: one align chunk, and up to 4 tokens at top-k <= 8,
        # else up to 16 tokens or 32 assignments)
        n = M * k
        fused = n <= 4096 and E <= 1024 and (M <= 4 if k <= 8 else (M <= 16 or n <= 32))
        self.layer_launches = (1 if fused else 1 + self.align_launches) + self.gemm_launches + 1

    # the layer's steps, each one C-ABI call (the calls chord_moe_layer makes)
    def route_align(self):
        from w4a16_int4_weight_sigmoid_gb300 import chord
        s = self.shape
        chord.chord_moe_route(self.logits, self.bias, s.topk, self.tw, self.ti)
        chord.chord_moe_align(self.ti, s.expert_begin, s.E_local, self.bm, self.sorted, self.eids,
                              self.ntpp, self.counts, self.offsets, self.pos, self.aws)

    def gate_up(self):
        from w4a16_int4_weight_sigmoid_gb300 import chord
        s = self.shape
        chord.chord_w4a16_moe_gemm(self.x, True, self.layer.w13, s.E_local, 2 * s.I, s.H, s.M, s.topk,
                                   self.sorted, self.eids, self.ntpp, self.counts, self.offsets, self.bm,
                                   chord.CHORD_EPI_SILU_MUL, self.h, self.ws_gu, tuning=self.plan,
                                   dev_status=self.status)

    def down(self):
        from w4a16_int4_weight_sigmoid_gb300 import chord
        s = self.shape
        chord.chord_w4a16_moe_gemm(self.h, False, self.layer.w2, s.E_local, s.H, s.I, s.M, s.topk,
                                   self.sorted, self.eids, self.ntpp, self.counts, self.offsets, self.bm,
                                   chord.CHORD_EPI_STORE, self.y, self.ws_dn, tuning=self.plan,
                                   dev_status=self.status)

    def combine(self):
        from w4a16_int4_weight_sigmoid_gb300 import chord
        chord.chord_moe_sum(self.y, self.tw, self.pos, self.out)

    def layer_call(self):
        self.layer.forward(self.x, self.logits, self.bias, out=self.out)

    def capture(self):
        import torch
        self.graphs = []
        for fn in (self.route_align, self.gate_up, self.down, self.combine):
            fn()                      # eager run first: sets kernel attributes
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            self.graphs.append(g)
        self.layer_call()             # eager run first: workspace, kernel attributes
        torch.cuda.synchronize()
        self.layer_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.layer_graph):
            self.layer_call()
        torch.cuda.synchronize()

    def stats(self):
        """Touched experts and local rows of this replica's routing."""
        c = self.counts.cpu().numpy()
        return int((c > 0).sum()), int(c.sum())


def algorithmic(shape, touched, rows):
    """Bytes and FLOPs one launch of each GEMM must move / do (padding rows
    not counted): touched experts' INT4 weights + BF16 scales, activation rows
    in, rows out."""
    H, I = shape.H, shape.I
    w13 = 2 * I * H // 2 + 2 * I * (H // 32) * 2
    w2 = H * I // 2 + H * (I // 32) * 2
    return {
        "gate_up": {"bytes": touched * w13 + rows * H * 2 + rows * I * 2, "flops": 2 * rows * 2 * I * H},
        "down": {"bytes": touched * w2 + rows * I * 2 + rows * H * 2, "flops": 2 * rows * H * I},
    }


# ---------------------------------------------------------------- our arm
def peak_for(peaks, region_s):
    """BF16 peak for a tensor-bound kernel: the burst figure for a region
    shorter than a second (the kernel runs at its unthrottled clock), the
    sustained one for a longer region."""
    if region_s < 1.0:
        return peaks["bf16_tflops"], "burst"
    return peaks["bf16_tflops_sustained"], "sustained"


def soak(reps, seconds):
    """Replay the replicas' layer graphs, untimed, for about `seconds`."""
    import torch
    end = time.perf_counter() + seconds
    i = 0
    while time.perf_counter() < end:
        for _ in range(16):
            reps[i % len(reps)].layer_graph.replay()
            i += 1
        torch.cuda.synchronize()


def measure_workload(shape, steps, warmup, R, world, rank, local, seed_base, e2e_steps, sampler_uuid):
    """Time one layer workload: K layer-graph replays (the step), then the
    same K steps as the layer's C-ABI calls one by one for kernel durations,
    then the public call with host copies (e2e).  Returns the fields of its
    JSON entry (and replica 0 for the CPU baseline)."""
    import torch
    device = f"cuda:{local}"
    reps = [Replica(shape, seed_base + 1000 * r + 7919 * rank, device, keep_host=(r == 0))
            for r in range(R)]
    for r in reps:
        r.capture()
    for i in range(warmup):
        reps[i % R].layer_graph.replay()
        for g in reps[i % R].graphs:
            g.replay()
    torch.cuda.synchronize()
    for r in reps:
        assert r.status.item() == 0, f"device status {r.status.item()}"
        assert r.layer.dev_status.item() == 0, f"layer device status {r.layer.dev_status.item()}"
    st = [r.stats() for r in reps]

    nev = 5
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(sampler_uuid)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_sampled = time.perf_counter()
    # nvidia-smi polls every 200 ms, longer than the timed region of a short
    # run: the same step keeps the GPU under the same load before and after
    # the timed regions, so that every sample is taken under load
    soak(reps, 0.3)
    t0.record()
    for i in range(steps):
        reps[i % R].layer_graph.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = allreduce_max(t0.elapsed_time(t1), world)
    # kernel durations: the same steps as the layer's calls one by one
    torch.cuda.synchronize()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record()
    for i in range(steps):
        e = evs[i]
        gs = reps[i % R].graphs
        e[0].record()
        gs[0].replay()
        e[1].record()
        gs[1].replay()
        e[2].record()
        gs[2].replay()
        e[3].record()
        gs[3].replay()
        e[4].record()
    k1.record()
    torch.cuda.synchronize()
    barrier(world)
    soak(reps, 1.0 - (time.perf_counter() - t_sampled))
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = ("the timed regions plus untimed replays of the same step before and after them, "
                            f"{time.perf_counter() - t_sampled:.2f} s in all")
    staged_ms = allreduce_max(k0.elapsed_time(k1), world)
    names = ["route_align", "gate_up", "down", "combine"]
    per = {n: [] for n in names}
    for e in evs:
        for j, n in enumerate(names):
            per[n].append(e[j].elapsed_time(e[j + 1]))
    kern_us = {n: 1000.0 * statistics.fmean(v) for n, v in per.items()}

    # algorithmic work per launch, averaged over the replica rotation
    alg = {"gate_up": {"bytes": 0.0, "flops": 0.0}, "down": {"bytes": 0.0, "flops": 0.0}}
    for i in range(steps):
        a = algorithmic(shape, *st[i % R])
        for k in alg:
            for q in ("bytes", "flops"):
                alg[k][q] += a[k][q] / steps

    peaks, peak_src = load_peaks()
    bf16_peak, peak_kind = peak_for(peaks, staged_ms / 1e3)
    src = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    dom = max(("gate_up", "down"), key=lambda n: kern_us[n])
    roofs = {}
    for kname in ("gate_up", "down"):
        t_s = kern_us[kname] * 1e-6
        t_hbm = alg[kname]["bytes"] / (peaks["hbm_gbs"] * 1e9)
        t_tc = alg[kname]["flops"] / (bf16_peak * 1e12)
        if t_hbm >= t_tc:
            ach = alg[kname]["bytes"] / t_s / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "peak_source": f"{src}, hbm_gbs"}
        else:
            ach = alg[kname]["flops"] / t_s / 1e12
            roof = {"bound": "tensor", "achieved": ach, "peak": bf16_peak, "unit": "TFLOP/s",
                    "peak_source": f"{src}, bf16 {peak_kind} (timed region {staged_ms / 1e3:.3f} s)"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["traffic"] = committed_traffic(kname, shape.name, "large" if reps[0].large else "small")
        roof["kernel"] = f"{'gemm_large (tcgen05)' if reps[0].large else 'gemm_small'} ({kname})"
        roof["algorithmic_bytes_per_launch"] = alg[kname]["bytes"]
        roof["algorithmic_flops_per_launch"] = alg[kname]["flops"]
        roofs[kname] = roof

    # whole-layer roofline: slower of bytes at HBM peak and FLOPs at the BF16 peak
    lay_bytes = alg["gate_up"]["bytes"] + alg["down"]["bytes"]
    lay_flops = alg["gate_up"]["flops"] + alg["down"]["flops"]
    t_lay_min = max(lay_bytes / (peaks["hbm_gbs"] * 1e9), lay_flops / (bf16_peak * 1e12))
    ms_per_step = elapsed_ms / steps
    value = shape.M * steps * world / (elapsed_ms / 1e3)

    # ----------------------------------------------------------- e2e
    outs_pinned = [torch.empty((shape.M, shape.H), dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    for i in range(max(3, R)):   # warm the whole path, copies included, on every replica
        r = reps[i % R]
        r.x.copy_(r.x_pinned, non_blocking=True)
        r.logits.copy_(r.logits_pinned, non_blocking=True)
        r.layer.forward(r.x, r.logits, r.bias, out=r.out)
        outs_pinned[i % R].copy_(r.out, non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    # Every step copies its inputs host->device and its output device->host
    # inside the timed region.  The copies run on two side streams, so step
    # i+1's inputs and step i-1's output move while step i computes (the
    # replicas' buffers rotate, and events order each copy against the steps
    # that use the same buffers), as a serving loop would pipeline them.
    main = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(R)]
    computed = [torch.cuda.Event() for _ in range(R)]
    out_read = [torch.cuda.Event() for _ in range(R)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    h2d_s.wait_stream(main)
    d2h_s.wait_stream(main)
    for i in range(e2e_steps):
        k = i % R
        r = reps[k]
        with torch.cuda.stream(h2d_s):
            if i >= R:
                h2d_s.wait_event(computed[k])   # the step that last read these buffers is done
            r.x.copy_(r.x_pinned, non_blocking=True)
            r.logits.copy_(r.logits_pinned, non_blocking=True)
            in_ready[k].record(h2d_s)
        main.wait_event(in_ready[k])
        if i >= R:
            main.wait_event(out_read[k])        # the output buffer's last read is done
        r.layer.forward(r.x, r.logits, r.bias, out=r.out)
        computed[k].record(main)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(computed[k])
            outs_pinned[k].copy_(r.out, non_blocking=True)
            out_read[k].record(d2h_s)
    main.wait_stream(d2h_s)
    main.wait_stream(h2d_s)
    e1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = allreduce_max(e0.elapsed_time(e1), world)
    h2d = shape.M * shape.H * 2 + shape.M * shape.E_total * 4
    d2h = shape.M * shape.H * 2
    e2e = {"value": shape.M * e2e_steps * world / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "api": "chord_moe_layer",
           "copies": "every step's inputs in and output out, on two copy streams overlapping the "
                     "neighbouring steps' kernels"}
    for r in reps:
        assert r.status.item() == 0 and r.layer.dev_status.item() == 0, "device status after timing"

    launches_per_step = reps[0].layer_launches
    staged_launches = reps[0].align_launches + reps[0].gemm_launches + 2   # + route, combine
    fields = {
        "value": value, "unit": "tokens/s", "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
        "config": {"workload": shape.name, "M": shape.M, "H": shape.H, "I": shape.I,
                   "E_total": shape.E_total, "E_local": shape.E_local, "topk": shape.topk,
                   "weights": "INT4 group-32 symmetric, BF16 scales; BF16 activations",
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {R} rotating layer replica(s), each step's touched "
                         f"weights ~{alg['gate_up']['bytes'] / 1e6 + alg['down']['bytes'] / 1e6:.0f} MB "
                         f"> 129 MB L2",
                   "touched_experts_per_replica": [x[0] for x in st],
                   "local_rows_per_replica": [x[1] for x in st]},
        "e2e": e2e,
        "gpu_launches": launches_per_step * steps,
        "kernel_timing": {"how": "second timed region of the same steps as the layer's C-ABI calls one "
                                 "by one (four graph replays, CUDA events between them)",
                          "steps": steps, "ms_per_step": staged_ms / steps,
                          "gpu_launches": staged_launches * steps},
        "roofline": roofs[dom],
        "roofline_per_gemm": roofs,
        "layer_roofline": {"bytes": lay_bytes, "flops": lay_flops, "t_min_us": t_lay_min * 1e6,
                           "t_us": ms_per_step * 1e3, "frac": t_lay_min / (ms_per_step * 1e-3),
                           "bf16_peak": f"{peak_kind} {bf16_peak} TFLOP/s"},
        "kernels_us": kern_us,
        "clocks": clocks,
    }
    host = reps[0].host
    del reps
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return fields, host


def run_ours(args, world, rank, local):
    import torch
    from w4a16_int4_weight_sigmoid_gb300 import build as B
    from w4a16_int4_weight_sigmoid_gb300 import chord
    from w4a16_int4_weight_sigmoid_gb300 import workload as wl

    B.build()
    chord.lib()
    torch.cuda.set_device(local)
    shape = wl.WORKLOADS[args.workload]
    decode = shape.M * shape.topk / shape.E_total < 64
    steps = args.steps if args.steps is not None else (20000 if decode else 300)
    warmup = max(3, args.warmup if args.warmup is not None else (200 if decode else 10))
    R = max(1, args.replicas)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        if uuid and not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else max(10, min(steps, 200))
    head, host = measure_workload(shape, steps, warmup, R, world, rank, local, shape.seed, e2e_steps, uuid)
    line = {"metric": METRIC, "value": head.pop("value"), "unit": head.pop("unit"), "n_gpus": world,
            "steps": head.pop("steps"), "warmup": head.pop("warmup"), "ms_per_step": head.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", **head,
            "step": "one chord_moe_layer call (CUDA graph replay; kernels chained by programmatic launches)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, host, args.cpu_budget_s)
    del host
    # the metric's other layer workloads, same steps, in the same line: the
    # TP8 decode shard (HBM GB/s) and the EP8 prefill shard (TFLOPS)
    if not args.only:
        extra = {}
        for other in wl.LAYER_WORKLOADS:
            if other.name == shape.name:
                continue
            o_decode = other.M * other.topk / other.E_total < 64
            o_R = 2 if o_decode else 1
            o_steps = max(steps, 20)
            o_e2e = max(10, min(o_steps, 50))
            fields, h = measure_workload(other, o_steps, warmup, o_R, world, rank, local, other.seed, o_e2e, uuid)
            del h
            fields["tokens_per_s"] = fields.pop("value")
            fields.pop("unit")
            extra[other.name] = fields
        line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------- oracle timing
def oracle_tokens_per_s(shape, host, budget_s, max_tokens=None):
    """Time the oracle on a bounded sample of tokens that have local experts."""
    import oracle
    w, ids, _ = oracle.route(host["logits"], host["bias"], shape.topk)
    local = np.any((ids >= shape.expert_begin) & (ids < shape.expert_begin + shape.E_local), axis=1)
    cand = np.nonzero(local)[0]
    n, t_total, cpu_total, done = 0, 0.0, 0.0, []
    for tok in cand:
        t = time.perf_counter()
        c = time.process_time()
        oracle.moe_layer_tokens(np.array([tok]), host["x"], host["logits"], host["bias"], host["w13_q"],
                                host["w13_s"], host["w2_q"], host["w2_s"], shape.topk, shape.expert_begin)
        cpu_total += time.process_time() - c
        t_total += time.perf_counter() - t
        n += 1
        done.append(int(tok))
        if t_total >= budget_s or (max_tokens and n >= max_tokens):
            break
    # threads the oracle kept busy on average: process CPU time over wall time
    return n / t_total, n, t_total, cpu_total / t_total


def cpu_baseline(shape, host, budget_s):
    v, n, t, cores = oracle_tokens_per_s(shape, host, budget_s)
    return {"value": v, "unit": "tokens/s", "cores": round(cores, 1), "cores_available": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} tokens (each with >= 1 local expert) of {shape.name}, one at a time "
                      f"through the FP64 numpy oracle, {t:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    from w4a16_int4_weight_sigmoid_gb300 import workload as wl
    shape = wl.WORKLOADS[args.workload]
    host = wl.layer_inputs(shape)
    steps = args.steps if args.steps is not None else 8
    warmup = args.warmup if args.warmup is not None else 1
    # each step is one token; stop early when the time budget runs out
    budget = 150.0
    oracle_tokens_per_s(shape, host, 1e9, max_tokens=max(1, min(warmup, 2)))
    v, n, t, cores = oracle_tokens_per_s(shape, host, budget, max_tokens=steps)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": n, "warmup": warmup, "ms_per_step": 1e3 * t / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": shape.name, "M": shape.M, "H": shape.H, "I": shape.I,
                       "E_total": shape.E_total, "E_local": shape.E_local, "topk": shape.topk},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": round(cores, 1),
                             "cores_available": os.cpu_count(), "kind": "oracle",
                             "sample": f"{n} tokens of {shape.name} (one per step), FP64 numpy oracle"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def graph_us(fns, reps_in_graph=20, replays=30):
    """Median microseconds of one pass of fns, from a CUDA graph holding
    reps_in_graph passes, replayed between CUDA events on the launching stream."""
    import torch
    for f in fns:
        f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps_in_graph):
            for f in fns:
                f()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1000.0 / reps_in_graph)
    ts.sort()
    return ts[len(ts) // 2]


def run_report(args):
    """Report-only curves (one JSON line): router+align latency per (M,
    BLOCK_M) over 384 experts, or the whole layer over M at EP8 shapes."""
    import torch
    from w4a16_int4_weight_sigmoid_gb300 import build as B
    from w4a16_int4_weight_sigmoid_gb300 import chord
    from w4a16_int4_weight_sigmoid_gb300 import workload as wl
    from w4a16_int4_weight_sigmoid_gb300.layer import W4A16MoELayer, to_device
    B.build()
    chord.lib()
    dev = "cuda:0"
    rows = []
    if args.report == "route_align":
        E, k = wl.ROUTER_ALIGN_E, wl.ROUTER_ALIGN_TOPK
        for M in wl.ROUTER_ALIGN_M:
            logits, bias = wl.router_inputs(M, E, wl.ROUTER_ALIGN_SEED)
            lg, bs = to_device(logits, dev), to_device(bias, dev)
            tw = torch.empty((M, k), dtype=torch.float32, device=dev)
            ti = torch.empty((M, k), dtype=torch.int32, device=dev)
            route = lambda: chord.chord_moe_route(lg, bs, k, tw, ti)
            t_route = graph_us([route])
            for bm in wl.ROUTER_ALIGN_BM:
                cap = chord.chord_moe_align_capacity(M, k, E, bm)
                i32 = torch.int32
                st = torch.empty(cap, dtype=i32, device=dev)
                eid = torch.empty(cap // bm, dtype=i32, device=dev)
                ntpp = torch.empty(1, dtype=i32, device=dev)
                cnt = torch.empty(E, dtype=i32, device=dev)
                off = torch.empty(E + 1, dtype=i32, device=dev)
                pos = torch.empty(M * k, dtype=i32, device=dev)
                wsb = chord.chord_moe_align_workspace_bytes(M, k, E)
                aws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
                align = lambda: chord.chord_moe_align(ti, 0, E, bm, st, eid, ntpp, cnt, off, pos, aws)
                fused = lambda: chord.chord_moe_route_align(lg, bs, k, 0, E, bm, tw, ti, st, eid, ntpp, cnt,
                                                            off, pos, aws)
                rows.append({"M": M, "block_m": bm, "route_us": round(t_route, 2),
                             "align_us": round(graph_us([align]), 2),
                             "route_then_align_us": round(graph_us([route, align]), 2),
                             "chord_moe_route_align_us": round(graph_us([fused]), 2)})
        note = "CUDA graph of 20 back-to-back passes, median of 30 replays; 384 experts, top-8, all local"
    elif args.report == "grouped":
        # the grouped layouts at the pages' scenarios, Kimi EP8 expert shapes:
        # masked decode with 32 tokens per expert, contiguous prefill with 128
        base = wl.EP8_DECODE
        E, H, I = base.E_local, base.H, base.I
        d = wl.layer_inputs(wl.LayerShape("grouped", 64, H, I, base.E_total, E, 0, base.topk, base.seed))
        layer = W4A16MoELayer(d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"], base.E_total, 0, base.topk,
                              device=dev)
        del d
        peaks, _ = load_peaks()
        wbytes = {"gate_up": E * (2 * I * H // 2 + 2 * I * (H // 32) * 2), "down": E * (H * I // 2 + H * (I // 32) * 2)}
        for layout, per_e in (("masked", 32), ("contiguous", 128)):
            rows_n = E * per_e
            g = torch.full((E,), per_e, dtype=torch.int32, device=dev)
            x = to_device(wl.activations(rows_n, H, 81), dev)
            h = torch.empty((rows_n, I), dtype=torch.bfloat16, device=dev)
            y = torch.empty((rows_n, H), dtype=torch.bfloat16, device=dev)
            ws = torch.zeros(chord.chord_w4a16_grouped_workspace_bytes(E, rows_n), dtype=torch.uint8, device=dev)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            for (name, A, W, N, K, epi, C), path in [
                    (gm, p) for gm in (("gate_up", x, layer.w13, 2 * I, H, chord.CHORD_EPI_SILU_MUL, h),
                                       ("down", h, layer.w2, H, I, chord.CHORD_EPI_STORE, y))
                    for p in (chord.CHORD_PATH_SMALL_M, chord.CHORD_PATH_LARGE_M, chord.CHORD_PATH_AUTO)]:
                tun = chord.chord_tuning(path, 0, 0, 0)
                if layout == "masked":
                    f = lambda A=A, W=W, N=N, K=K, epi=epi, C=C, tun=tun: chord.chord_w4a16_grouped_gemm_masked(
                        A.view(E, per_e, K), g, W, N, K, epi, C.view(E, per_e, -1), ws, per_e, tuning=tun,
                        dev_status=st)
                else:
                    f = lambda A=A, W=W, N=N, K=K, epi=epi, C=C, tun=tun: chord.chord_w4a16_grouped_gemm_contiguous(
                        A, g, W, N, K, epi, C, ws, per_e, tuning=tun, dev_status=st)
                us = graph_us([f], reps_in_graph=10, replays=20)
                byts = wbytes[name] + rows_n * K * 2 + rows_n * (N // 2 if epi == chord.CHORD_EPI_SILU_MUL else N) * 2
                flops = 2.0 * rows_n * N * K
                t_hbm, t_tc = byts / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops_sustained"] * 1e12)
                bound = "hbm" if t_hbm >= t_tc else "tensor"
                rows.append({"layout": layout, "rows_per_expert": per_e, "gemm": name, "us": round(us, 2),
                             "path": {chord.CHORD_PATH_SMALL_M: "register-mma", chord.CHORD_PATH_LARGE_M: "tcgen05",
                                      chord.CHORD_PATH_AUTO: "auto"}[path],
                             "bound": bound, "frac": round(max(t_hbm, t_tc) / (us * 1e-6), 4),
                             "achieved": round(byts / (us * 1e-6) / 1e9, 1) if bound == "hbm"
                             else round(flops / (us * 1e-6) / 1e12, 1),
                             "unit": "GB/s" if bound == "hbm" else "TFLOP/s"})
            torch.cuda.synchronize()
            assert st.item() == 0, f"device status {st.item()}"
        note = ("grouped-layout GEMMs, 48 experts of Kimi EP8 shapes (H 7168, I 2048), every expert's weights "
                "touched; CUDA graph of 10 back-to-back calls, median of 20 replays; frac against the measured "
                "HBM rate or sustained BF16 rate, whichever bounds")
    else:
        base = wl.EP8_DECODE
        d = wl.layer_inputs(wl.LayerShape("m_sweep", 8192, base.H, base.I, base.E_total, base.E_local,
                                          0, base.topk, base.seed))
        layer = W4A16MoELayer(d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"], base.E_total, 0, base.topk,
                              device=dev)
        x, lg, bs = to_device(d["x"], dev), to_device(d["logits"], dev), to_device(d["bias"], dev)
        del d
        M = 1
        while M <= 8192:
            xm, lm = x[:M].contiguous(), lg[:M].contiguous()
            out = torch.empty((M, base.H), dtype=torch.bfloat16, device=dev)
            layer.workspace(M)
            n_in = 5 if M >= 1024 else 20
            fwd = lambda: layer.forward(xm, lm, bs, out=out)
            us = graph_us([fwd], reps_in_graph=n_in, replays=10)
            plan = chord.chord_moe_layer_plan(M, base.E_total, base.topk)
            row = {"M": M, "us": round(us, 2), "tokens_per_s": round(M / (us * 1e-6), 1),
                   "path": "tcgen05" if plan.path == chord.CHORD_PATH_LARGE_M else "register-mma",
                   "rows_per_pass": plan.rows_per_pass}
            for name, pth in (("us_register_mma", chord.CHORD_PATH_SMALL_M),
                              ("us_tcgen05", chord.CHORD_PATH_LARGE_M)):
                tun = chord.chord_tuning(pth, 0, 0, 0)
                f2 = lambda: layer.forward(xm, lm, bs, out=out, tuning=tun)
                row[name] = round(graph_us([f2], reps_in_graph=n_in, replays=10), 2)
            rows.append(row)
            M *= 2
        note = ("one layer, chord_moe_layer, EP8 shapes (H 7168, I 2048, 48 of 384 experts, top-8), "
                "the first M tokens of one seeded 8192-token draw; CUDA graph of back-to-back calls")
    if torch.cuda.is_available() and args.report == "m_sweep":
        assert int(layer.dev_status.item()) == 0
    print(json.dumps({"report": args.report, "unit": "us", "note": note, "rows": rows}))


def main():
    args = parse_args()
    if args.report:
        run_report(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
