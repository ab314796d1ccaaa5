"""Benchmark: cold-L2 microseconds per MoE-layer call and achieved HBM GB/s.

Workload (default): the Ling-shaped verify step -- hidden 2560, 512 routed
experts, top-8 softmax + renormalisation, SwiGLU inter 512, M = 6 tokens, bf16,
weights N(0, 0.02) drawn per layer from seed 1000 + layer, tokens N(0, 1)
redrawn per call from seed 1_000_000 + call.  Distinct layer weight sets are
cycled (and each call reads a different x) so every call's weights come from
HBM, not L2: between two calls of the same layer the other layers stream
several times the L2 size.  One step = one layer call (router + top-k +
compaction + gate/up + SwiGLU + down + combine).

Timing: K calls are captured (PDL chains intact) into CUDA graphs of G calls
and replayed; CUDA events on the launching stream bracket exactly K calls,
with a barrier and a device synchronize on both sides; max over ranks.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--M 6] [--zipf]
    python bench.py --shape ling_tp4      # the per-GPU slice of a 4-way TP split (inter 128)
    python bench.py --impl reference     # the CPU oracle on the same workload
    python bench.py --sweep               # M x routing sweep (writes JSON lines)
    python bench.py --lm-head [--M 1]     # the bf16 vocabulary projection
    python bench.py --crossover           # the contraction on CUDA cores vs tensor cores, M_e = 1..16
    torchrun ... bench.py --gpus N --tp   # the layer split N ways (tensor parallel): every rank streams
                                          # 1/N of each expert, an all-gather of the fp32 partials and
                                          # their ordered sum end each call
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cold-L2 µs/MoE-layer call and achieved HBM GB/s (% of GB300 peak) at M=1/6/16"
UNIT = "µs/call"
L2_BYTES = 126 * 1024 * 1024      # replaced by the device's value when a GPU is present
NOMINAL_HBM_GBS = 8000.0          # the GB300's nominal HBM3e bandwidth (~8 TB/s)


# --------------------------------------------------------------- helpers --

def algorithmic_bytes(hidden, n_experts, topk, inter, M, n_active, fp8=False):
    """Bytes the layer must move per call: each distinct activated expert's
    gate/up and down weights once, the router weight once, x in, out out and
    the routing indices out.  Weights of experts nobody chose are not counted
    (that is the work the routing avoids).  fp8: one byte per expert weight
    plus the fp32 row scales ((2I + H) per expert); the router stays bf16."""
    expert = 3 * hidden * inter + (2 * inter + hidden) * 4 if fp8 else 3 * hidden * inter * 2
    return (n_active * expert + n_experts * hidden * 2 + 2 * M * hidden * 2 + M * topk * 4)


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


LAYER_SOURCES = [os.path.join(ROOT, "weight_streaming_expert_gb300", "csrc", f)
                 for f in ("layer_kernel.cuh", "routing.cuh", "common.cuh", "kernels.cuh",
                           "layer_kernel_a.cu", "layer_kernel_b.cu", "layer_kernel_c.cu", "layer_kernel_d.cu",
                           "layer_kernel_e.cu", "layer_kernel_f.cu", "layer_kernel_g.cu", "layer_kernel_h.cu",
                           "layer_kernel_i.cu", "layer_kernel_j.cu", "layer_kernel_k.cu", "layer_kernel_l.cu")]
# DRAM traffic records of one ncu capture each: bf16 and fp8 expert weights
TRAFFIC_FILES = {False: os.path.join(ROOT, "profiles", "layer_traffic.json"),
                 True: os.path.join(ROOT, "profiles", "layer_traffic_fp8.json")}


def measured_peaks():
    """HBM copy bandwidth measured on the GB300s (MEASURED_PEAKS.json),
    else the earlier measurement of 6.8 TB/s, with a warning on stderr."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    print("bench: MEASURED_PEAKS.json not found; fractions use the fallback peak of 6800 GB/s",
          file=sys.stderr, flush=True)
    return 6800.0, "fallback"


def fractions(gbs, peak):
    """Achieved bandwidth as a fraction of the measured copy peak and of the
    nominal ~8 TB/s."""
    return {"frac_of_peak": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, period_ms=50):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- setup --

def dist_setup(n_gpus):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, ws, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v):
    if pg is None:
        return v
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


class Workload:
    """Distinct layers on the device plus pools of token batches."""

    def __init__(self, shape, n_layers, M, pool, zipf, device, layer_seed0=1000, variant=False, fp8=False):
        import torch
        from weight_streaming_expert_gb300 import MoELayer
        from weight_streaming_expert_gb300 import workloads as wl
        self.shape, self.M, self.device = shape, M, device
        self.layers = []
        for l in range(n_layers):
            if fp8:  # E4M3 expert codes with fp32 row scales
                w_r, q_gu, s_gu, q_d, s_d = wl.fp8_expert_weights(shape, seed=layer_seed0 + l, device=device)
                self.layers.append(MoELayer.fp8(w_r, q_gu, s_gu, q_d, s_d, topk=shape.topk))
                del w_r, q_gu, s_gu, q_d, s_d
                torch.cuda.empty_cache()
                continue
            w_r, w_gu, w_d = wl.layer_weights(shape, seed=layer_seed0 + l, device=device)
            kw = {}
            if variant:  # a shared expert, routed scale 2.5, the bias for selection only
                g = torch.Generator(device=device).manual_seed(layer_seed0 + 500 + l)
                H, I = shape.hidden, shape.inter
                kw = dict(shared_gate_up=(torch.randn(2 * I, H, generator=g, device=device) * wl.WEIGHT_STD)
                          .to(torch.bfloat16),
                          shared_down=(torch.randn(H, I, generator=g, device=device) * wl.WEIGHT_STD)
                          .to(torch.bfloat16),
                          routed_scale=2.5, bias_selection_only=True)
            self.layers.append(MoELayer(w_r, w_gu, w_d, topk=shape.topk, **kw))
            del w_r, w_gu, w_d, kw
            torch.cuda.empty_cache()
        self.n_use = len(self.layers)
        self.set_routing(zipf)
        self.new_pool(M, pool)

    def use_layers(self, n):
        """Cycle the first n layers (at most all of them)."""
        self.n_use = max(1, min(n, len(self.layers)))

    def set_routing(self, zipf):
        from weight_streaming_expert_gb300 import workloads as wl
        bias = wl.zipf_router_bias(self.shape.n_experts) if zipf else None
        for layer in self.layers:
            layer.set_router_bias(bias)
        self.zipf = zipf

    def new_pool(self, M, pool):
        import torch
        from weight_streaming_expert_gb300 import workloads as wl
        self.M = M
        H, k = self.shape.hidden, self.shape.topk
        self.xs = [wl.tokens(M, H, seed=1_000_000 + i, device=self.device) for i in range(pool)]
        self.outs = [torch.empty((M, H), dtype=torch.bfloat16, device=self.device) for _ in range(pool)]
        self.idxs = [torch.empty((M, k), dtype=torch.int32, device=self.device) for _ in range(pool)]

    def layer(self, c):
        return self.layers[c % self.n_use]

    def call(self, c, stream=None):
        i = c % len(self.xs)
        self.layer(c)(self.xs[i], out=self.outs[i], topk_idx=self.idxs[i], stream=stream)

    def close(self):
        for layer in self.layers:
            layer.close()
        self.layers = []


def n_layers_for(M, shape, l2_bytes, requested, fp8=False):
    if requested:
        return requested
    # distinct layers so that >= 3 x L2 of other layers' weights stream
    # between two calls of the same layer (at least 4)
    est_active = min(M * shape.topk, shape.n_experts) * 0.85 + 1
    per_call = algorithmic_bytes(shape.hidden, shape.n_experts, shape.topk, shape.inter, M, est_active, fp8)
    return max(4, int(math.ceil(3 * l2_bytes / per_call)) + 1)


# ----------------------------------------------------------------- timing --

def time_graph(wkl, steps, warmup, pg, graph_len=64, sample_clocks=False, gpu_index=0):
    """Returns (ms_per_step, per-call distinct-expert counts of one graph)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in range(warmup):
            wkl.call(c, stream=s)
    s.synchronize()
    G = min(graph_len, steps)
    graphs = []
    # one graph per distinct remainder so that EXACTLY `steps` calls are timed
    full, rem = divmod(steps, G)
    lens = ([G] if full else []) + ([rem] if rem else [])
    for n in lens:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for c in range(n):
                    wkl.call(c, stream=s)
        graphs.append(g)
    # untimed replay of each graph (first-launch upload)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    active = []
    for c in range(G):
        i = c % len(wkl.xs)
        active.append(int(torch.unique(wkl.idxs[i]).numel()))
    sampler = ClockSampler(gpu_index) if sample_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        # pre-roll: one untimed replay of the last graph right before the first
        # event, so that the stream is busy when the timed graph is launched and
        # the first timed call does not pay the graph's launch latency (a layer
        # call in a model step is one of many kernels of a larger graph)
        graphs[-1].replay()
        torch.cuda.nvtx.range_push("bench_timed")
        e0.record(s)
        for _ in range(full):
            graphs[0].replay()
        if rem:
            graphs[-1].replay()
        e1.record(s)
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(pg)
    clocks = sampler.stop() if sampler else None
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(pg, ms), active, clocks


def time_kernel_alone(wkl, calls):
    """Layer-kernel durations (ms) without PDL overlap: each call is launched
    without PDL between two events, all captured into one CUDA graph and
    replayed, so no host gap sits between the events."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(calls)]
    with torch.cuda.stream(s):
        for ev in evs:
            for e in ev:
                e.record(s)      # create the events before capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for c in range(calls):
                i = c % len(wkl.xs)
                wkl.layer(c).forward_timed(wkl.xs[i], wkl.outs[i], wkl.idxs[i], evs[c], stream=s)
    g.replay()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return np.array([ev[0].elapsed_time(ev[1]) for ev in evs])


# trace slots (moe_read_trace): 0 wait passed, 1 matvec done, 12 top-k done,
# 3 groups counted (producer; its first copies follow), 13 compaction done,
# 4 first gate/up tile, 5 gate/up left, 6 h rows of all CTAs, 7 down left,
# 8 combine done, 9 last gate/up issue, 10 down prefetch issued
def phase_breakdown(wkl, reps=2):
    """Phase timeline of the layer kernel inside a PDL-chained graph: every
    layer's last call of a traced graph, times relative to that call's first
    CTA passing its dependency wait (us; median over the calls read)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    n = reps * wkl.n_use
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for c in range(n):
                i = c % len(wkl.xs)
                wkl.layer(c)(wkl.xs[i], out=wkl.outs[i], topk_idx=wkl.idxs[i], stream=s, trace=True)
    g.replay()
    torch.cuda.synchronize()
    rows = []
    for layer in wkl.layers[:wkl.n_use]:
        t = layer.read_trace().astype(np.float64)
        t0 = t[:, 0].min()
        r = (t - t0) / 1000.0
        rows.append({
            "matvec_done": r[:, 1].max(), "topk_done": r[:, 12].max(), "groups_counted": r[:, 3].max(),
            "compaction_done": r[:, 13].max(),
            "first_gateup_tile_median": float(np.median(r[:, 4])), "gateup_end_min": r[:, 5].min(),
            "gateup_end_max": r[:, 5].max(), "h_ready": r[:, 6].max(), "down_end_min": r[:, 7].min(),
            "down_end_max": r[:, 7].max(), "combine_end": r[:, 8].max(),
            "gateup_tiles_per_cta_min": float(t[:, 11].min()), "gateup_tiles_per_cta_max": float(t[:, 11].max())})
    return {k: round(float(np.median([r[k] for r in rows])), 3) for k in rows[0]}


def time_e2e(wkl, steps):
    """Through the public API with host buffers: per call, the H2D copy of that
    call's tokens from pinned memory, the layer, and the D2H copies of its
    output and routing indices; events bracket all of it."""
    import torch
    M, H, k = wkl.M, wkl.shape.hidden, wkl.shape.topk
    P = len(wkl.xs)
    hx = [x.cpu().pin_memory() for x in wkl.xs]
    ho = [torch.empty((M, H), dtype=torch.bfloat16).pin_memory() for _ in range(P)]
    hi = [torch.empty((M, k), dtype=torch.int32).pin_memory() for _ in range(P)]
    dx = [torch.empty((M, H), dtype=torch.bfloat16, device=wkl.device) for _ in range(P)]
    s = torch.cuda.Stream()

    def one(c):
        i = c % P
        dx[i].copy_(hx[i], non_blocking=True)
        wkl.layer(c)(dx[i], out=wkl.outs[i], topk_idx=wkl.idxs[i], stream=s)
        ho[i].copy_(wkl.outs[i], non_blocking=True)
        hi[i].copy_(wkl.idxs[i], non_blocking=True)

    with torch.cuda.stream(s):
        for c in range(min(8, steps)):
            one(c)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for c in range(steps):
            one(c)
        e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / steps
    return us, M * H * 2, M * H * 2 + M * k * 4


ORACLE_FN = {"plain": "moe_forward", "variant": "moe_forward (shared expert, routed scale 2.5, selection-only bias)",
             "fp8": "moe_forward_fp8"}


def oracle_layer(shape, kind):
    """The oracle call of one token on the timed workload's first layer
    (weight seed 1000; the variant's shared expert from seed 1500, as the
    Workload builds it): kind "plain", "variant" or "fp8"."""
    import torch
    from oracle.oracle import Oracle
    from weight_streaming_expert_gb300 import workloads as wl
    orc = Oracle()
    dev = "cuda" if _has_cuda() else "cpu"
    if kind == "fp8":
        w_r, q_gu, s_gu, q_d, s_d = wl.fp8_expert_weights(shape, seed=1000, device=dev)
        h = (wl.bf16_bits(w_r), q_gu.cpu().numpy(), s_gu.cpu().numpy(), q_d.cpu().numpy(), s_d.cpu().numpy())
        return lambda x, bias: orc.moe_forward_fp8(x, *h, shape.topk, bias=bias)
    w_r, w_gu, w_d = wl.layer_weights(shape, seed=1000, device=dev)
    h = (wl.bf16_bits(w_r), wl.bf16_bits(w_gu), wl.bf16_bits(w_d))
    kw = {}
    if kind == "variant":
        g = torch.Generator(device=dev).manual_seed(1500)
        H, I = shape.hidden, shape.inter
        kw = dict(shared_gate_up=wl.bf16_bits((torch.randn(2 * I, H, generator=g, device=dev) * wl.WEIGHT_STD)
                                              .to(torch.bfloat16)),
                  shared_down=wl.bf16_bits((torch.randn(H, I, generator=g, device=dev) * wl.WEIGHT_STD)
                                           .to(torch.bfloat16)),
                  routed_scale=2.5, bias_selection_only=True)
    return lambda x, bias: orc.moe_forward(x, *h, shape.topk, bias=bias, **kw)


def oracle_call_us(shape, M, zipf, budget_s, call=None, max_calls=None, kind="plain"):
    """Mean wall time of the CPU oracle on one layer call, timed on samples of
    ONE token each (the oracle's work is linear in M, so a call costs M of
    them).  Returns (us_per_call, n_samples, call)."""
    from weight_streaming_expert_gb300 import workloads as wl
    if call is None:
        call = oracle_layer(shape, kind)
    bias = wl.zipf_router_bias(shape.n_experts).numpy() if zipf else None
    xs = [wl.bf16_bits(wl.tokens(1, shape.hidden, seed=1_000_000 + i)) for i in range(64)]
    call(xs[0], bias)     # warm caches
    times = []
    t_start = time.perf_counter()
    i = 0
    while True:
        t0 = time.perf_counter()
        call(xs[i % len(xs)], bias)
        times.append(time.perf_counter() - t0)
        i += 1
        if max_calls is not None and i >= max_calls:
            break
        if time.perf_counter() - t_start > budget_s and i >= 3:
            break
    per_token = statistics.mean(times)
    return per_token * M * 1e6, len(times), call


def workload_name(args, shape, M):
    """The timed workload, named by what it is (both arms)."""
    return (f"Ling-shaped MoE {'block-verify' if M >= 16 else 'verify' if M > 1 else 'decode'} step"
            f"{' (per-GPU slice of a 4-way TP split)' if args.shape == 'ling_tp4' else ''}: "
            f"hidden {shape.hidden}, {shape.n_experts} experts, top-{shape.topk} softmax+renorm, "
            f"SwiGLU inter {shape.inter}, "
            f"{'+ shared expert, routed scale 2.5, bias for selection only, ' if args.variant else ''}"
            f"{'fp8 E4M3 expert weights with fp32 row scales, ' if args.fp8 else ''}"
            f"M={M}, {'Zipf(1.1) router bias' if args.zipf else 'uniform routing'}")


def oracle_kind(args):
    return "fp8" if args.fp8 else "variant" if args.variant else "plain"


def _has_cuda():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# ------------------------------------------------------------------ arms --

def run_ours(args):
    import torch
    from weight_streaming_expert_gb300 import workloads as wl
    rank, ws, local, pg = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    prop = torch.cuda.get_device_properties(dev)
    l2 = getattr(prop, "L2_cache_size", L2_BYTES) or L2_BYTES
    shape = wl.SHAPES[args.shape]
    M = args.M
    n_layers = n_layers_for(M, shape, l2, args.layers, args.fp8)
    # the side measurements (M = 1, M = 16 Zipf) cycle as many layers as
    # their own per-call bytes need to keep L2 cold: build them all once
    side = ((1, False), (16, True)) if (args.all_m and rank == 0) else ()
    n_side = {m2: n_layers_for(m2, shape, l2, args.layers, args.fp8) for m2, _ in side}
    wkl = Workload(shape, max([n_layers] + list(n_side.values())), M, args.pool, args.zipf, dev,
                   variant=args.variant, fp8=args.fp8)
    wkl.use_layers(n_layers)
    ms, active, clocks = time_graph(wkl, args.steps, args.warmup, pg, sample_clocks=(rank == 0),
                                    gpu_index=local)
    mean_active = float(np.mean(active)) + (1.0 if args.variant else 0.0)  # + the shared expert
    bytes_call = algorithmic_bytes(shape.hidden, shape.n_experts, shape.topk, shape.inter, M, mean_active, args.fp8)
    us = ms * 1000.0
    gbs = bytes_call / (us * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()
    # the layer kernel alone (no PDL overlap with its neighbours) and its phases
    alone_us = float(time_kernel_alone(wkl, min(256, max(16, args.steps))).mean() * 1000.0)
    phases = phase_breakdown(wkl)
    traffic = None
    traffic_file = TRAFFIC_FILES[bool(args.fp8)]
    if os.path.exists(traffic_file):
        with open(traffic_file) as f:
            tr = json.load(f)
        if (tr.get("source_hash") == source_hash(LAYER_SOURCES) and tr.get("M") == M
                and args.shape == tr.get("shape", "ling") and not args.variant
                and bool(tr.get("fp8", False)) == bool(args.fp8)):
            # measured on a smaller run (one layer, 8 calls): DRAM traffic
            # follows the algorithmic bytes, so scale it to this run's launches
            traffic = int(round(tr["bytes_per_launch"] * bytes_call / tr["algorithmic_bytes_per_launch"]))
    e2e_us, h2d, d2h = (None, 0, 0)
    if not args.no_e2e:
        e2e_us, h2d, d2h = time_e2e(wkl, min(args.steps, 4000))
        e2e_us = max_over_ranks(pg, e2e_us)
    by_m = {}
    for m2, z2 in side:
        wkl.set_routing(z2)
        wkl.new_pool(m2, args.pool)
        wkl.use_layers(n_side[m2])
        by_m[f"M={m2}" + ("_zipf" if z2 else "")] = side_measurement(wkl, args, shape, m2, peak)
    wkl.set_routing(args.zipf)
    fp8_by_m = {}
    if side and not args.fp8 and not args.variant and args.fp8_side:
        # the same layer shape with fp8 (E4M3) expert weights: half the bytes
        wkl.close()
        torch.cuda.empty_cache()
        n8 = {m2: n_layers_for(m2, shape, l2, args.layers, True) for m2 in (6, 1)}
        w8 = Workload(shape, max(n8.values()), 6, args.pool, False, dev, fp8=True)
        for m2 in (6, 1):
            w8.new_pool(m2, args.pool)
            w8.use_layers(n8[m2])
            fp8_by_m[f"M={m2}"] = side_measurement(w8, args, shape, m2, peak, fp8=True)
        w8.close()
        torch.cuda.empty_cache()
    cpu = None
    if not args.no_cpu_baseline and rank == 0:
        wkl.close()
        torch.cuda.empty_cache()
        kind = oracle_kind(args)
        us_cpu, n, _ = oracle_call_us(shape, M, args.zipf, args.cpu_budget, kind=kind)
        cpu = {"value": round(us_cpu, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n} single-token calls of the CPU oracle's {ORACLE_FN[kind]} on layer seed 1000 "
                         f"(x seeds 1e6+i), mean x M={M}; single-threaded C++"}
    else:
        wkl.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8 weights, bf16 tokens" if args.fp8 else "bf16",
            "data": "synthetic: seeded N(0,0.02) bf16 weights, N(0,1) bf16 tokens (random init, no checkpoint)",
            "config": {"workload": workload_name(args, shape, M),
                       "M": M, "layers_cycled": n_layers, "x_pool": args.pool,
                       "l2_policy": f"inputs larger than L2: {n_layers} distinct layer weight sets cycled, "
                                    f"fresh x per call; L2 {l2 // (1024 * 1024)} MiB",
                       "graph_calls": min(64, args.steps), "parallelism": f"replicas x{ws}",
                       "pre_roll": "one untimed replay of the same graph right before the first event"},
            "achieved_gbs": round(gbs, 1), **fractions(gbs, peak),
            "peak_gbs": peak, "peak_kind": peak_kind, "nominal_peak_gbs": NOMINAL_HBM_GBS,
            "mean_active_experts": round(mean_active, 2), "algorithmic_bytes_per_call": int(bytes_call),
            "kernel_us": {"moe_layer_kernel_in_chain": round(us, 3), "moe_layer_kernel_alone": round(alone_us, 3),
                          "alone_timing": "graph replay, no PDL, events around each launch"},
            "phases_us": phases,
            "roofline": {"bound": "hbm", "kernel": "moe_layer_kernel", "achieved": round(gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": traffic,
                         "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                         "algorithmic_bytes_per_launch": int(bytes_call), "peak_kind": peak_kind,
                         "launch_duration": "timed-region mean per launch (one launch per call, PDL-chained)"},
            "cpu_baseline": cpu,
            "e2e": None if e2e_us is None else {"value": round(e2e_us, 3), "unit": UNIT,
                                                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        if by_m:
            line["by_M"] = by_m
        if fp8_by_m:
            line["fp8_experts_by_M"] = fp8_by_m
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def side_measurement(wkl, args, shape, M, peak, fp8=False):
    """One side configuration, timed like the headline (graph replay of
    exactly min(steps, 4000) calls, cold L2)."""
    ms2, act2, _ = time_graph(wkl, min(args.steps, 4000), args.warmup, None)
    act2 = [a + (1 if args.variant else 0) for a in act2]
    b2 = algorithmic_bytes(shape.hidden, shape.n_experts, shape.topk, shape.inter, M, float(np.mean(act2)), fp8)
    gbs = b2 / (ms2 * 1e-3) / 1e9
    return {"us_per_call": round(ms2 * 1000, 3), "achieved_gbs": round(gbs, 1), **fractions(gbs, peak),
            "mean_active_experts": round(float(np.mean(act2)), 2), "layers_cycled": wkl.n_use,
            "calls_timed": min(args.steps, 4000)}


def run_reference(args):
    """The CPU oracle as the reference arm: same metric, unit and workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from weight_streaming_expert_gb300 import workloads as wl
    shape = wl.SHAPES[args.shape]
    budget = args.cpu_budget
    # warmup samples (untimed), then timed samples bounded by the budget
    kind = oracle_kind(args)
    us_w, _, call = oracle_call_us(shape, args.M, args.zipf, budget_s=0.0,
                                   max_calls=max(1, min(args.warmup, 3)), kind=kind)
    us, n, _ = oracle_call_us(shape, args.M, args.zipf, budget_s=budget, call=call,
                              max_calls=max(1, args.steps))
    cores = 1
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": 0,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 accumulate over E4M3 x row scale" if args.fp8 else "f32 accumulate over bf16",
        "data": "synthetic: seeded N(0,0.02) bf16 weights, N(0,1) bf16 tokens",
        "config": {"workload": workload_name(args, shape, args.M), "M": args.M},
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} single-token calls of the oracle's {ORACLE_FN[kind]} (of {args.steps} "
                                   f"requested steps, bounded to {budget:.0f} s), mean x M={args.M}"},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def tp_exchange(part, pg, world):
    """The exchange step of a tensor-parallel split: every rank's fp32
    partial output [M, H] gathered side by side into [world, M, H], the same
    on every rank (an all-gather; the ordered sum that follows makes it an
    all-reduce whose order is fixed)."""
    import torch
    if pg is None or world == 1:
        return part.unsqueeze(0)
    M, H = part.shape
    out = torch.empty((world * M, H), dtype=part.dtype, device=part.device)
    pg.all_gather_into_tensor(out, part.contiguous())
    return out.view(world, M, H)


def run_tp(args):
    """The Ling-shaped layer split over the ranks (the post's TP4 when run on
    4 GPUs): rank r holds gate/up rows and down columns [r I/N, (r+1) I/N)
    of every expert and routes every token.  One step = the layer call with
    its unrounded fp32 output, the all-gather of the N partials (NCCL), and
    their ordered sum with one bf16 rounding (moe_combine_partials).  Launched
    call by call (no graph: the collective is enqueued by the host)."""
    import torch
    from weight_streaming_expert_gb300 import MoELayer, combine_partials, tp_slice
    from weight_streaming_expert_gb300 import workloads as wl
    rank, ws, local, pg = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    prop = torch.cuda.get_device_properties(dev)
    l2 = getattr(prop, "L2_cache_size", L2_BYTES) or L2_BYTES
    shape = wl.SHAPES["ling"]
    M = args.M
    if shape.inter % ws or shape.inter // ws not in (128, 256, 512):
        raise SystemExit(f"--tp: inter {shape.inter} cannot be split {ws} ways")
    sl = wl.LayerShape(hidden=shape.hidden, n_experts=shape.n_experts, topk=shape.topk, inter=shape.inter // ws)
    n_layers = n_layers_for(M, sl, l2, args.layers)
    layers = []
    for l in range(n_layers):
        w_r, w_gu, w_d = wl.layer_weights(shape, seed=1000 + l, device=dev)
        gu, d = tp_slice(w_gu, w_d, rank, ws)
        del w_gu, w_d
        layers.append(MoELayer(w_r, gu, d, topk=shape.topk))
        del w_r, gu, d
        torch.cuda.empty_cache()
    xs = [wl.tokens(M, shape.hidden, seed=1_000_000 + i, device=dev) for i in range(args.pool)]
    parts = [torch.empty((M, shape.hidden), dtype=torch.float32, device=dev) for _ in range(2)]
    outs = [torch.empty((M, shape.hidden), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    idxs = [torch.empty((M, shape.topk), dtype=torch.int32, device=dev) for _ in range(args.pool)]
    s = torch.cuda.current_stream()

    def step(c):
        i = c % args.pool
        layers[c % n_layers](xs[i], out=parts[c % 2], topk_idx=idxs[i], out_f32=True, stream=s)
        combine_partials(tp_exchange(parts[c % 2], pg, ws), out=outs[c % 2], stream=s)

    for c in range(args.warmup):
        step(c)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    e0.record(s)
    for c in range(args.steps):
        step(c)
    e1.record(s)
    torch.cuda.synchronize()
    barrier(pg)
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / args.steps)
    active = [int(torch.unique(idxs[c % args.pool]).numel()) for c in range(min(args.steps, args.pool))]
    status = max(layer.status() for layer in layers)
    for layer in layers:
        layer.close()
    peak, peak_kind = measured_peaks()
    per_gpu = algorithmic_bytes(sl.hidden, sl.n_experts, sl.topk, sl.inter, M, float(np.mean(active)))
    us = ms * 1000.0
    gbs = per_gpu / (us * 1e-6) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": False, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,0.02) bf16 weights, N(0,1) bf16 tokens (random init, no checkpoint)",
            "config": {"workload": f"Ling-shaped MoE step split {ws} ways (tensor parallel): hidden {shape.hidden}, "
                                   f"{shape.n_experts} experts, top-{shape.topk}, inter {shape.inter} "
                                   f"({sl.inter} per rank), M={M}, uniform routing",
                       "M": M, "layers_cycled": n_layers, "x_pool": args.pool,
                       "l2_policy": f"inputs larger than L2: {n_layers} distinct layer slices cycled, fresh x per call",
                       "parallelism": f"tp{ws}", "exchange": "all-gather of fp32 partials + ordered sum, one rounding"},
            "achieved_gbs_per_gpu": round(gbs, 1), **fractions(gbs, peak), "peak_kind": peak_kind,
            "algorithmic_bytes_per_call_per_gpu": int(per_gpu), "mean_active_experts": round(float(np.mean(active)), 2),
            "device_status": status, "gpu_launches": 2 * args.steps}), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_sweep(args):
    import torch
    from weight_streaming_expert_gb300 import workloads as wl
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    shape = wl.SHAPES[args.shape]
    peak, peak_kind = measured_peaks()
    wkl = Workload(shape, args.layers or 8, 1, args.pool, False, dev)
    for zipf in (False, True):
        wkl.set_routing(zipf)
        for M in (1, 2, 4, 6, 8, 16, 32, 64):
            wkl.new_pool(M, args.pool)
            ms, active, _ = time_graph(wkl, args.steps, args.warmup, None)
            b = algorithmic_bytes(shape.hidden, shape.n_experts, shape.topk, shape.inter, M, float(np.mean(active)))
            gb = b / (ms * 1e-3) / 1e9
            print(json.dumps({"sweep": True, "M": M, "routing": "zipf" if zipf else "uniform",
                              "us_per_call": round(ms * 1000, 3), "achieved_gbs": round(gb, 1),
                              **fractions(gb, peak), "peak_kind": peak_kind,
                              "mean_active_experts": round(float(np.mean(active)), 2),
                              "phases_us": phase_breakdown(wkl, reps=1)}), flush=True)
    wkl.close()


def crossover_summary(res, Ms, margin=0.03):
    """res[(M_e, engine)] = us per call.  The smallest M_e from which the
    tensor cores are faster by more than `margin` at every larger M_e too
    (None if never), the M_e at which the CUDA cores are faster by more than
    `margin`, and the time ratio CUDA / tensor per M_e."""
    Ms = sorted(Ms)
    tc = [M for M in Ms if res[(M, "tensor_cores")] < (1.0 - margin) * res[(M, "cuda_cores")]]
    cross = None
    for i, M in enumerate(Ms):
        if all(m in tc for m in Ms[i:]):
            cross = M
            break
    return {"tensor_cores_faster_from_M_e": cross,
            "cuda_cores_faster_at_M_e": [M for M in Ms if res[(M, "cuda_cores")] < (1.0 - margin) * res[(M, "tensor_cores")]],
            "ratio_cuda_over_tensor": {str(M): round(res[(M, "cuda_cores")] / res[(M, "tensor_cores")], 3) for M in Ms}}


def run_crossover(args):
    """The expert contraction on the CUDA cores and on the tensor cores
    (include/gemv.h) over the layer's packed tiles: one launch streams the
    gate/up rows (k = hidden) or the down rows (k = inter) of 46 experts --
    the distinct experts of an M = 6 call -- for M_e tokens; 4 distinct
    weight sets (about 1 GB) are cycled so every call reads from HBM.  One
    JSON line per (shape, M_e, engine), then one per shape with the
    crossover: the smallest M_e from which the tensor cores are faster."""
    import torch
    from weight_streaming_expert_gb300 import gemv as G
    from weight_streaming_expert_gb300 import workloads as wl
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    shape = wl.SHAPES[args.shape]
    H, I, A, n_sets = shape.hidden, shape.inter, 46, 4
    peak, peak_kind = measured_peaks()
    Ms = tuple(args.crossover_m) if args.crossover_m else (1, 2, 3, 4, 6, 8, 12, 16)
    shapes = (("gate_up", A * 2 * I, H), ("down", A * H, I))
    for name, rows, k in (s_ for s_ in shapes if args.crossover_shape in ("both", s_[0])):
        gen = torch.Generator(device=dev).manual_seed(4242 + rows)
        packs = []
        for _ in range(n_sets):
            w = (torch.randn(rows, k, generator=gen, device=dev) * wl.WEIGHT_STD).to(torch.bfloat16)
            packs.append(G.pack(w))
            del w
        torch.cuda.empty_cache()
        res = {}
        for M in Ms:
            xs = [wl.tokens(M, k, seed=7_000_000 + i, device=dev) for i in range(n_sets)]
            ys = [torch.empty((M, rows), dtype=torch.float32, device=dev) for _ in range(n_sets)]
            for eng_name, eng in (("cuda_cores", G.CUDA_CORES), ("tensor_cores", G.TENSOR_CORES)):
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                n = max(n_sets, min(args.steps, 256) // n_sets * n_sets)
                with torch.cuda.stream(s):
                    for c in range(max(args.warmup, n_sets)):
                        G.gemv(packs[c % n_sets], xs[c % n_sets], eng, ys[c % n_sets], stream=s)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=s):
                        for c in range(n):
                            G.gemv(packs[c % n_sets], xs[c % n_sets], eng, ys[c % n_sets], stream=s)
                    g.replay()
                s.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                with torch.cuda.stream(s):
                    e0.record(s)
                    g.replay()
                    e1.record(s)
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) * 1000.0 / n
                b = rows * k * 2 + M * k * 2 + M * rows * 4
                gbs = b / (us * 1e-6) / 1e9
                res[(M, eng_name)] = us
                print(json.dumps({"crossover": True, "shape": f"{name} ({A} experts: {rows} x {k} bf16)", "M_e": M,
                                  "engine": eng_name, "us_per_call": round(us, 3), "achieved_gbs": round(gbs, 1),
                                  "frac_of_peak": round(gbs / peak, 4), "peak_kind": peak_kind,
                                  "weight_sets_cycled": n_sets, "calls": n}), flush=True)
        print(json.dumps(dict(crossover_summary=True, shape=name, **crossover_summary(res, Ms))), flush=True)
        del packs
        torch.cuda.empty_cache()


def run_lm_head(args):
    """The vocabulary projection (include/lm_head.h), timed like the layer:
    calls captured into CUDA graphs (PDL intact), two distinct weight copies
    cycled (together far above L2) and a fresh x per call.  One JSON line."""
    import torch
    from weight_streaming_expert_gb300 import LmHead
    from weight_streaming_expert_gb300 import workloads as wl
    rank, ws, local, pg = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    H = wl.LING.hidden
    V = wl.LM_HEAD_VOCAB // (4 if args.shape == "ling_tp4" else 1)
    M = min(args.M, 16)
    heads = [LmHead(wl.lm_head_weight(V, H, seed=5000 + i, device=dev)) for i in range(2)]
    torch.cuda.empty_cache()
    xs = [wl.tokens(M, H, seed=1_000_000 + i, device=dev) for i in range(args.pool)]
    outs = [torch.empty((M, V), dtype=torch.float32, device=dev) for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    call = lambda c: heads[c % 2](xs[c % len(xs)], outs[c % 2], stream=s)
    with torch.cuda.stream(s):
        for c in range(args.warmup):
            call(c)
    s.synchronize()
    G = min(64, args.steps)
    full, rem = divmod(args.steps, G)
    graphs = []
    for n in ([G] if full else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for c in range(n):
                    call(c)
        graphs.append(g)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(full):
            graphs[0].replay()
        if rem:
            graphs[-1].replay()
        e1.record(s)
    torch.cuda.synchronize()
    barrier(pg)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / args.steps)
    status = max(h.status() for h in heads)
    for h in heads:
        h.close()
    bytes_call = V * H * 2 + M * H * 2 + M * V * 4
    us = ms * 1000.0
    gbs = bytes_call / (us * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()
    if rank == 0:
        print(json.dumps({
            "metric": "cold-L2 \u00b5s per lm_head call and achieved HBM GB/s (% of GB300 peak)",
            "value": round(us, 3), "unit": "\u00b5s/call", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic: seeded N(0,0.02) bf16 weight, N(0,1) bf16 tokens",
            "config": {"workload": f"bf16 lm_head GEMV: hidden {H}, vocab {V}"
                                   f"{' (vocab-parallel quarter)' if args.shape == 'ling_tp4' else ''}, M={M}, fp32 logits",
                       "M": M, "weights_cycled": 2,
                       "l2_policy": f"inputs larger than L2: 2 weight copies of {V * H * 2 / 1e6:.0f} MB cycled, fresh x per call",
                       "graph_calls": G, "parallelism": f"replicas x{ws}"},
            "achieved_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "peak_gbs": peak, "peak_kind": peak_kind,
            "algorithmic_bytes_per_call": int(bytes_call), "device_status": status,
            "roofline": {"bound": "hbm", "kernel": "lm_head_kernel", "achieved": round(gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None,
                         "algorithmic_bytes_per_launch": int(bytes_call), "peak_kind": peak_kind},
            "gpu_launches": args.steps, "clocks": clocks}), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8192)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--M", type=int, default=6)
    ap.add_argument("--shape", choices=["ling", "ling_tp4"], default="ling",
                    help="ling: hidden 2560, 512 experts, top-8, inter 512; ling_tp4: its 4-way TP slice, inter 128")
    ap.add_argument("--zipf", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="distinct layer weight sets (0 = auto)")
    ap.add_argument("--pool", type=int, default=64, help="distinct token batches cycled")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-m", dest="all_m", action="store_false",
                    help="skip the M=1 and M=16 (Zipf) side measurements")
    ap.add_argument("--no-fp8-side", dest="fp8_side", action="store_false",
                    help="skip the fp8-expert M=6 and M=1 side measurements")
    ap.add_argument("--tp", action="store_true",
                    help="split every layer over the ranks (tensor parallel): 1/N of each expert per rank, "
                         "fp32 partial outputs all-gathered and summed in rank order")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle timing")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--fp8", action="store_true", help="layers with fp8 (E4M3) expert weights and row scales")
    ap.add_argument("--variant", action="store_true",
                    help="layers with a shared expert, routed scale 2.5 and the router bias for selection only")
    ap.add_argument("--crossover", action="store_true",
                    help="the expert contraction on CUDA cores vs tensor cores over M_e = 1..16 (JSON lines)")
    ap.add_argument("--crossover-m", dest="crossover_m", type=int, nargs="+", default=None,
                    help="--crossover: the token counts M_e to time (default 1 2 3 4 6 8 12 16)")
    ap.add_argument("--crossover-shape", dest="crossover_shape", choices=["both", "gate_up", "down"], default="both")
    ap.add_argument("--lm-head", dest="lm_head", action="store_true",
                    help="time the bf16 vocabulary projection (hidden 2560, vocab 157,184; M <= 16) instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.lm_head:
        run_lm_head(args)
    elif args.sweep:
        run_sweep(args)
    elif args.crossover:
        run_crossover(args)
    elif args.tp:
        run_tp(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
