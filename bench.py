#!/usr/bin/env python
"""Benchmark of the GB300 routed-MoE layer (GLM-5.2 sigmoid router, int4 experts).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one pass of the whole layer (router, activation quantiser, expert
union, fused gate/up, down + ordered reduction) over one batch of synthetic
input.  The default workload is the GLM-5.2-shaped layer at decode batch 1
(hidden 6144, 256 experts top-8, intermediate 2048, 1 shared expert, int4
per-row weights).  Eight independently seeded layer weight sets (4.86 GB each)
stay resident and the steps cycle through them, so every step streams weights
that are not in L2 (1.2 GB of other weights pass between two uses of a set).

`value` is tokens/s with inputs already in HBM, timed with CUDA events over
exactly K steps (CUDA-graph replays), max over ranks.  `e2e` is the same
metric through the C ABI with x copied in from pinned host memory and the
output copied back every step.  `roofline` reports the dominant kernel: the
fused gate/up weight stream against the measured HBM copy bandwidth at decode
sizes, the gate/up grouped GEMM against the measured dense tensor rate at
prefill sizes.  `cpu_baseline` is
the plain CPU oracle timed on a bounded sample of the same workload.

--impl reference times that oracle as the reference arm (rank 0 only).
Multi-GPU (torchrun): independent replicas, one per GPU, no collective on the
data path; weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and achieved HBM GB/s vs ~8 TB/s (decode), int8 TOPS (prefill)"
UNIT = "tokens/s"
WORKLOADS = {
    # name: (synth config, residual block stack?)
    "glm_moe_layer_decode_b1": ("glm_decode_b1", False),
    "glm_moe_layer_verify_b8": ("glm_verify_b8", False),
    "glm_moe_layer_prefill_2048": ("glm_prefill_2048", False),
    "glm_moe_stack8_decode_b1": ("glm_stack8_b1", True),
    "glm_moe_stack8_decode_b8": ("glm_stack8_b8", True),
    # the checkpoint converter step (not a layer forward): GB/s, not tokens/s
    "glm_fp8_to_int4": (None, False),
}
DEFAULT_WORKLOAD = "glm_moe_layer_decode_b1"
# Dominant kernel per path: decode batches (<= 16 tokens) stream the weights
# (HBM-bound); larger batches run the grouped GEMM (tensor-pipe bound).
HOT_KERNEL_DECODE = "stream_kernel<0> (fused int4 gate/up, SiLU*up, max abs h)"
HOT_KERNEL_SINGLE = "decode_layer_kernel (the whole layer as one persistent kernel)"
HOT_KERNEL_DECODE8 = "gateup_kernel<12,1,8> (int8 gate/up rows, SiLU*up, max abs h)"
HOT_KERNEL_PREFILL = ("umma_gemm_kernel<0, 1> (tcgen05 f16-exact gate/up GEMM, tokens x 256 weight rows per MMA, "
                      "packed weights by TMA, SiLU*up, max abs h)")
# DRAM bytes (read + write) per launch of the dominant kernel from one ncu
# capture of the current kernel source, or None.  Keyed by workload; a
# capture covers the workload's plain configuration only (int4 experts, plain
# top-K, one layer per step), so the variants report None.
TRAFFIC = {
    # decode_layer_kernel at decode batch 1 (DRAM byte counters of 3 launches,
    # one resident GLM-shaped layer set, caches flushed before each):
    # 176.72 MB read + 0.37 MB written per launch
    "glm_moe_layer_decode_b1": 177.09e6,
    # umma_gemm_kernel<0, 1> (gate/up, packed weights by TMA) at prefill 2048,
    # full capture of the profiling layout (16 physical experts aliased over
    # the 257 table entries; the routing, tiles and bytes per tile are the
    # full layer's): 2.550 GB read + 0.134 GB written per launch
    "glm_moe_layer_prefill_2048": 2.684e9,
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--layers", type=int, default=8, help="resident layer weight sets cycled by the steps")
    p.add_argument("--light", action="store_true",
                   help="profiling only: 17 physical experts aliased over the 257 table entries")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--weight-bits", type=int, choices=[4, 8], default=4,
                   help="expert weight width (4: packed int4, the headline; 8: per-row int8)")
    p.add_argument("--top-p", type=float, default=0.0,
                   help="adaptive expert top-p in (0, 1) (0: plain top-K, the headline)")
    p.add_argument("--fp8-experts", type=int, default=64,
                   help="glm_fp8_to_int4: stacked gate matrices converted per launch")
    p.add_argument("--no-secondary", action="store_true",
                   help="default workload only: skip the verify-8 and prefill-2048 lines timed after it")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle sample budget")
    p.add_argument("--ref-seconds", type=float, default=150.0, help="reference arm time box")
    p.add_argument("--four-kernel", action="store_true",
                   help="decode batches: run the four-kernel launch plan instead of the single persistent kernel")
    p.add_argument("--probe", choices=["gateup", "down", "router"], default="gateup",
                   help="kernel timed live by the roofline probe (the roofline figure is the gate/up kernel's)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value, world, device="cpu"):
    """The largest of every rank's `value` (the job's time is its slowest
    rank's); the process group must be up when world > 1."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def layer_bytes_per_expert(cfg, wbits=4):
    """Weight bytes of one expert: int4 packed (two per byte) or int8 rows, plus fp32 row scales."""
    if wbits == 8:
        return 2 * (cfg.I * cfg.D + cfg.I * 4) + cfg.D * cfg.I + cfg.D * 4
    import synth
    return synth.expert_bytes(cfg)


def gateup_bytes_per_expert(cfg, wbits=4):
    return 2 * (cfg.I * (cfg.D if wbits == 8 else cfg.D // 2) + cfg.I * 4)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.proc = None
        self.path = None
        self.t_on = self.t_off = None
        self.bus = None
        try:
            import torch
            props = torch.cuda.get_device_properties(dev_index)
            bus, dv = getattr(props, "pci_bus_id", None), getattr(props, "pci_device_id", None)
            if bus is not None and dv is not None:
                self.bus = f"{bus:02x}:{dv:02x}.0"
        except Exception:
            self.bus = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu=pci.bus_id,{self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50", "-f", self.path]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9 and (self.bus is None or parts[0].lower().endswith(self.bus)):
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "samples_loaded": len(loaded)}


def traffic_for(workload, top_p, wbits, stack, light):
    """The captured DRAM bytes of the workload's dominant kernel when the run
    is the configuration the capture covered, else None."""
    if stack or light or wbits != 4 or 0.0 < top_p < 1.0:
        return None
    return TRAFFIC.get(workload)


def measured_peak(kind="hbm_gbs"):
    """A peak from MEASURED_PEAKS.json, else the profiling fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j[kind]), "measured"
    except Exception:
        return fallback[kind], "fallback"


# ------------------------------------------------------------ layer set-up

def build_layers(cfg, n_layers, light, dev, rank_seed=0, top_p=0.0, wbits=4):
    """n_layers resident GLM-shaped layers, weights drawn on the GPU from the
    seeded generator and packed by the library's own int4 packer."""
    import torch
    import serving_router_sigmoid_gb300 as moe
    import synth
    layers, keep = [], []
    for l in range(n_layers):
        lid = l + 1000 * rank_seed
        Wr = synth.router_weight(cfg, lid).to(dev)
        bias = synth.router_bias(cfg, lid).to(dev)
        phys = {}
        n_phys = 16 if light else cfg.E
        pack = moe.pack_int8 if wbits == 8 else moe.pack_int4
        for e in list(range(n_phys)) + [cfg.E]:
            g, u, d = synth.expert_fp32(cfg, e, lid, dev)
            gq, gs = pack(g)
            uq, us = pack(u)
            dq, ds = pack(d)
            phys[e] = (gq, gs, uq, us, dq, ds)
            del g, u, d
        table = [phys[e if e < n_phys or e == cfg.E else e % n_phys] for e in range(cfg.E)] + [phys[cfg.E]]
        layers.append(moe.MoeLayer(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale, max(cfg.T, 1),
                                   Wr, bias, table, top_p, wbits))
        keep.append((Wr, bias, phys))
    torch.cuda.synchronize()
    return layers, keep


def union_sizes(layers, xs):
    """(distinct routed experts + shared) per layer for its input, via the debug entry."""
    import torch
    sizes = []
    for layer, x in zip(layers, xs):
        d = layer.moe_layer_debug(x, union=True)
        torch.cuda.synchronize()
        sizes.append(int(d["n_union"].item()))
    return sizes


# ----------------------------------------------------------------- our arm

def run_ours(args, workload, rank, world, local, n_layers=None, steps=None, warmup=None, with_e2e=True,
             with_cpu=True, top_p=None, wbits=None):
    """One workload on this rank's GPU; returns rank 0's JSON object (None on
    the other ranks).  The process group, if any, is already up."""
    import torch
    import serving_router_sigmoid_gb300 as moe
    import synth

    cfg = synth.CONFIGS[WORKLOADS[workload][0]]
    stack = WORKLOADS[workload][1]
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if n_layers is None:
        n_layers = 8 if stack else max(1, args.layers)
    t_setup = time.time()
    top_p = args.top_p if top_p is None else top_p
    wbits = args.weight_bits if wbits is None else wbits
    layers, keep = build_layers(cfg, n_layers, args.light, dev, rank_seed=rank, top_p=top_p, wbits=wbits)
    T = cfg.T
    for lyr in layers:
        if args.four_kernel:
            lyr.set_option(moe.MOE_OPT_DECODE_SINGLE_KERNEL, 0)
    single = (T <= 16 and not args.four_kernel
              and layers[0].get_option(moe.MOE_OPT_DECODE_SINGLE_KERNEL_AVAILABLE) == 1)
    s = torch.cuda.Stream(device=dev)
    norm_w = synth.norm_weight(cfg, dev)
    # inputs: one token batch per layer set (single layer), or a pool of batches (stack)
    xs = [synth.x_rows(cfg, T, "cpu", "bench-x", l + 100 * rank).to(dev) for l in range(n_layers)]
    outs = [torch.empty_like(x) for x in xs]
    xwork = torch.empty((T, cfg.D), device=dev)

    def step_fn(i):
        if stack:
            xwork.copy_(xs[i % n_layers])
            for layer in layers:
                layer.moe_block_forward(xwork, norm_w, cfg.eps)
        else:
            layers[i % n_layers].moe_layer_forward(xs[i % n_layers], outs[i % n_layers])

    # one graph per layer set (single layer) or two alternating graphs (stack),
    # each with its own probe events so a step's probe is read while the next
    # step runs
    n_graph = 2 if stack else n_layers
    probes = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_graph)]
    use_graph = not args.no_graph
    graphs = []
    with torch.cuda.stream(s):
        for i in range(n_graph):  # eager warm-up of every code path
            step_fn(i)
        torch.cuda.synchronize()
        probe_id = {"gateup": moe.MOE_PROBE_GATE_UP, "down": moe.MOE_PROBE_DOWN,
                    "router": moe.MOE_PROBE_ROUTER}[args.probe]
        # the single-kernel layer is the whole step: the step time is its
        # launch time, and no probe events sit between its launches
        use_probe = stack or not single
        if not stack and use_probe:
            for l, layer in enumerate(layers):
                layer.set_probe(probe_id, *probes[l])
        if use_graph:
            for i in range(n_graph):
                if stack:
                    layers[0].set_probe(probe_id, *probes[i])
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    step_fn(i)
                graphs.append(g)
        elif stack:
            layers[0].set_probe(probe_id, *probes[0])
            n_graph = 1
        # without probes, runs of n_layers consecutive steps are also captured
        # in one graph, as a serving engine captures a model's layers: the
        # steps then follow each other without a graph launch in between
        run_graph = None
        if use_graph and not use_probe and n_layers > 1:
            run_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(run_graph, stream=s):
                for i in range(n_layers):
                    step_fn(i)
        torch.cuda.synchronize()

    def launch(i, left=1):
        """Issues step i (and, through the run graph, the steps after it
        when a whole run starts at i and fits in `left`); returns the number
        of steps issued."""
        if run_graph is not None and i % n_layers == 0 and left >= n_layers:
            run_graph.replay()
            return n_layers
        if use_graph:
            graphs[i % n_graph].replay()
        else:
            step_fn(i)
        return 1

    # single kernel; else router + gate/up + down + reduce (int8 rows: the down
    # kernel reduces, three); above 16 tokens quantiser, logits, select,
    # permute, gate/up, requant, down, reduce (+ the f16 operand rows for the
    # tcgen05 GEMMs; int8 rows: no requant and no operand rows)
    if single:
        kernels_per_forward = 1
    elif T <= 16:
        kernels_per_forward = 3 if wbits == 8 else 4
    else:
        kernels_per_forward = 7 if wbits == 8 else 9
    kernels_per_forward += 1 if stack else 0
    launches_per_step = kernels_per_forward * (len(layers) if stack else 1)
    setup_s = time.time() - t_setup

    clocks = ClockSampler(local)
    clocks.start()
    # warm-up: at least W steps and at least ~0.5 s of work so clocks ramp up
    w_done = 0
    t0 = time.time()
    with torch.cuda.stream(s):
        n_sync = 0
        while w_done < warmup or time.time() - t0 < 0.5:
            w_done += launch(w_done, 1 << 30)
            if w_done >= n_sync + 64:
                n_sync = w_done
                s.synchronize()
        s.synchronize()

    K = steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    probe_ms = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    with torch.cuda.stream(s):
        ev0.record(s)
        i = 0
        while i < K:
            i += launch(w_done + i, K - i)
            if i >= 2 and use_probe:
                b, e = probes[(w_done + i - 2) % n_graph]
                e.synchronize()
                probe_ms.append(b.elapsed_time(e))
        ev1.record(s)
    torch.cuda.synchronize()
    if use_probe:
        b, e = probes[(w_done + K - 1) % n_graph]
        probe_ms.append(b.elapsed_time(e))
    clocks.mark_off()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    tokens = T * K * world
    value = tokens / (elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / K

    # algorithmic bytes of the dominant kernel and of a whole step
    u1 = union_sizes(layers, xs if not stack else [xs[0]] * len(layers))
    u1_mean = sum(u1) / len(u1)
    gu_bytes = u1_mean * gateup_bytes_per_expert(cfg, wbits) + T * cfg.D + T * cfg.S * cfg.I * 4
    step_bytes_layer = (u1_mean * layer_bytes_per_expert(cfg, wbits) + cfg.E * cfg.D * 4 + cfg.E * 4 +
                        2 * T * cfg.D * 4)
    step_bytes = step_bytes_layer * (len(layers) if stack else 1)
    if use_probe:
        probe_avg_ms, launches_timed = sum(probe_ms) / len(probe_ms), len(probe_ms)
    else:  # back-to-back launches of the one kernel: the gaps between them count
        probe_avg_ms, launches_timed = ms_per_step, K
    grouped = T > 16
    traffic = traffic_for(workload, top_p, wbits, stack, args.light)
    if single:
        # one kernel is the whole layer: its algorithmic bytes are the step's
        peak, peak_kind = measured_peak("hbm_gbs")
        achieved = step_bytes_layer / (probe_avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": HOT_KERNEL_SINGLE, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind + " HBM copy bandwidth",
                "traffic": traffic, "algorithmic_bytes_per_launch": step_bytes_layer,
                "avg_launch_ms": probe_avg_ms, "launches_timed": launches_timed}
    elif args.probe != "gateup":
        roof = {"bound": "hbm", "kernel": args.probe, "achieved": None, "peak": None, "unit": "GB/s",
                "frac": None, "traffic": None, "avg_launch_ms": probe_avg_ms, "launches_timed": launches_timed}
    elif not grouped:
        peak, peak_kind = measured_peak("hbm_gbs")
        achieved = gu_bytes / (probe_avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": HOT_KERNEL_DECODE if wbits == 4 else HOT_KERNEL_DECODE8,
                "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind + " HBM copy bandwidth",
                "traffic": traffic, "algorithmic_bytes_per_launch": gu_bytes,
                "avg_launch_ms": probe_avg_ms, "launches_timed": launches_timed}
    else:
        # int8 ops of the gate/up GEMM: every routed (token, expert) pair and
        # every token through the shared expert, 2 ops per multiply-add
        rows = T * cfg.K + T * cfg.n_shared
        ops = 2.0 * rows * (2 * cfg.I) * cfg.D
        # the burst peak: the GEMM runs for ~2 ms at a time at full clocks,
        # not for seconds under the power cap
        peak, peak_kind = measured_peak("bf16_tflops")
        achieved = ops / (probe_avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": HOT_KERNEL_PREFILL, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": peak_kind + " dense bf16 (burst); sm_103a has no int8 tcgen05 kind, so the "
                             "densest tensor rate for these operands is the 16-bit one",
                "traffic": traffic, "algorithmic_ops_per_launch": ops,
                "avg_launch_ms": probe_avg_ms, "launches_timed": launches_timed}

    # end to end through the C ABI: pinned host x -> device, forward, out -> pinned host
    e2e = None
    if with_e2e and not args.no_e2e:
        Ke = max(16, min(K, 2000))
        xh = [x.cpu().pin_memory() for x in xs]
        oh = torch.empty((T, cfg.D), dtype=torch.float32).pin_memory()
        xd = torch.empty((T, cfg.D), device=dev)
        od = torch.empty((T, cfg.D), device=dev)
        for lyr in layers:
            lyr.set_probe(moe.MOE_PROBE_NONE)

        def e2e_step(i):
            if stack:
                xd.copy_(xh[i % n_layers], non_blocking=True)
                for lyr in layers:
                    lyr.moe_block_forward(xd, norm_w, cfg.eps)
                oh.copy_(xd, non_blocking=True)
            else:
                # one C-ABI call: the copy in, the forward and the copy out
                layers[i % n_layers].forward_host(xh[i % n_layers], oh, s)

        with torch.cuda.stream(s):
            for i in range(min(64, Ke)):
                e2e_step(i)
            s.synchronize()
            if world > 1:
                torch.distributed.barrier()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(s)
            for i in range(Ke):
                e2e_step(i)
            a1.record(s)
            s.synchronize()
        e_ms = a0.elapsed_time(a1)
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": T * Ke * world / (e_ms / 1e3), "unit": UNIT, "steps": Ke,
               "h2d_bytes_per_step": T * cfg.D * 4, "d2h_bytes_per_step": T * cfg.D * 4,
               "api": "moe_block_forward" if stack else "moe_layer_forward_host", "graph": False,
               "d2h": ("copy" if stack or T > 16 else
                       "the kernel's stores into the page-locked output (no copy after the forward)")}

    cpu = None
    if rank == 0 and with_cpu and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, stack, args.cpu_seconds, dev)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": warmup,
        "warmup_steps_run": w_done,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"int{wbits} weights x int8 activations -> int32, fp32 scales", "data": "synthetic",
        "config": {"workload": workload, "hidden": cfg.D, "moe_intermediate": cfg.I, "experts": cfg.E,
                   "top_k": cfg.K, "shared_experts": cfg.n_shared, "tokens_per_step": T,
                   "layers_per_step": len(layers) if stack else 1, "layer_sets_cycled": n_layers,
                   "routed_scale": cfg.routed_scale, "zipf_skew": cfg.skew, "top_p": top_p,
                   "weight_bits": wbits,
                   "experts_streamed_per_layer": u1_mean, "cuda_graph": use_graph,
                   "steps_per_graph": n_layers if run_graph is not None else 1, "light": args.light,
                   "decode_plan": ("single persistent kernel" if single else "four kernels") if T <= 16 else None,
                   "l2": ("inputs larger than L2: the steps cycle %d resident layer weight sets "
                          "(%.2f GB between reuses of a set)" % (n_layers, (n_layers - 1) * step_bytes_layer / 1e9))
                   if n_layers > 1 or T > 1 else "single set",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs_step": step_bytes / (ms_per_step / 1e3) / 1e9,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "setup_s": round(setup_s, 1),
    }
    for lyr in layers:
        lyr.close()
    del keep, layers, xs, outs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line if rank == 0 else None


# ------------------------------------------------------------ CPU oracle

def _oracle_layer_for(cfg, x_np, layer_id, dev):
    import oracle
    import synth
    Wr = synth.router_weight(cfg, layer_id).numpy()
    b = synth.router_bias(cfg, layer_id).numpy()
    idx, _, _ = oracle.router(x_np, Wr, b, cfg.K, cfg.routed_scale)
    need = sorted(set(idx.reshape(-1).tolist()) | {cfg.E})
    ex = {}
    for e in need:
        g, u, d = synth.expert_fp32(cfg, e, layer_id, dev)
        ex[e] = oracle.pack_expert(g.cpu().numpy(), u.cpu().numpy(), d.cpu().numpy())
    return oracle.Layer(cfg.D, cfg.I, cfg.E, cfg.K, cfg.n_shared, cfg.routed_scale, Wr, b, ex)


def host_cpu():
    """(CPU model, uname -m) of this host, as far as the system reports them."""
    import platform
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                model = ln.split(":", 1)[1].strip()
                if not model.isdigit():
                    break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return model or "unknown", platform.machine()


def _time_oracle(fn, budget_s, max_reps=None):
    reps, t0 = 0, time.time()
    while True:
        fn()
        reps += 1
        el = time.time() - t0
        if el >= budget_s or (max_reps and reps >= max_reps):
            return reps, el


def cpu_baseline(cfg, stack, budget_s, dev="cpu", max_reps=None):
    """The oracle as it stands on this host's cores, on a bounded sample: one
    token of the workload (through all 8 layers for the stack) repeated until
    the budget is used, with all cores (OpenMP over output rows) and then with
    one thread.  Returns the cpu_baseline object."""
    import synth
    import oracle
    x = synth.x_rows(cfg, 1, "cpu", "cpu-sample").numpy()
    n_l = 8 if stack else 1
    Ls = [_oracle_layer_for(cfg, x, l, dev) for l in range(n_l)]
    w = synth.norm_weight(cfg).numpy()

    def one():
        if stack:
            y = x.copy()
            for L in Ls:
                y = L.block_forward(y, w, cfg.eps)
        else:
            Ls[0].forward(x)

    cores = oracle.max_threads()
    reps, el = _time_oracle(one, budget_s, max_reps)
    oracle.set_threads(1)
    try:
        reps1, el1 = _time_oracle(one, budget_s / 3, max_reps)
    finally:
        oracle.set_threads(cores)
    model, machine = host_cpu()
    return {"value": reps * x.shape[0] / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_1thread": reps1 * x.shape[0] / el1, "cpu_model": model, "machine": machine,
            "sample": f"{reps} forward(s) of {x.shape[0]} token through {n_l} GLM-shaped layer(s) "
                      f"({'residual block stack' if stack else 'one MoE layer'}), plain C oracle, "
                      f"{el:.1f} s wall on {cores} threads; {reps1} forward(s) in {el1:.1f} s on 1 thread"}


def run_reference(args, cfg, stack, rank):
    if rank != 0:
        return None
    import oracle
    import synth
    dev = "cuda" if _has_cuda() else "cpu"
    x = synth.x_rows(cfg, 1, "cpu", "cpu-sample").numpy()
    n_l = 8 if stack else 1
    Ls = [_oracle_layer_for(cfg, x, l, dev) for l in range(n_l)]
    w = synth.norm_weight(cfg).numpy()

    def one():
        if stack:
            y = x.copy()
            for L in Ls:
                y = L.block_forward(y, w, cfg.eps)
        else:
            Ls[0].forward(x)

    for _ in range(min(args.warmup, 3)):
        one()
    t0 = time.time()
    done = 0
    while done < args.steps and time.time() - t0 < args.ref_seconds:
        one()
        done += 1
    el = time.time() - t0
    value = done / el
    sample = (f"{done} of {args.steps} steps timed (time box {args.ref_seconds:.0f} s); each step 1 token "
              f"through {n_l} GLM-shaped layer(s) of the plain C oracle; warm-up {min(args.warmup, 3)}")
    model, machine = host_cpu()
    cpu = {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle", "sample": sample,
           "cpu_model": model, "machine": machine}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / max(done, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 weights x int8 activations -> int32, fp32 scales",
            "data": "synthetic",
            "config": {"workload": args.workload, "hidden": cfg.D, "moe_intermediate": cfg.I, "experts": cfg.E,
                       "top_k": cfg.K, "shared_experts": cfg.n_shared, "tokens_per_step": 1,
                       "layers_per_step": n_l},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _has_cuda():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def run_fp8_converter(args, local, n_experts=64, steps=20, warmup=5):
    """The checkpoint converter step (FP8 E4M3 with 128 x 128 block scales ->
    packed int4 + row scales) on the stacked gate matrices of n_experts
    GLM-shaped experts: [n_experts * 2048, 6144] codes (805 MB at 64, far
    larger than L2).  HBM-bound: algorithmic bytes = codes read + packed bytes
    written + scales, per launch."""
    import torch
    import serving_router_sigmoid_gb300 as moe
    import synth
    dev = torch.device("cuda", local)
    O, I = n_experts * 2048, 6144
    codes, si = synth.fp8_checkpoint_matrix(O, I, seed=77, device=dev)
    torch.cuda.empty_cache()  # the generator's fp32 temporaries
    q4 = torch.empty((O, I // 2), dtype=torch.uint8, device=dev)
    sc = torch.empty(O, dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(warmup):
            moe.moe_fp8_block_to_int4(codes, si, q4, sc, stream=s)
        s.synchronize()
        clocks = ClockSampler(local)
        clocks.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            moe.moe_fp8_block_to_int4(codes, si, q4, sc, stream=s)
        e1.record(s)
        s.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    nbytes = O * I + O * (I // 2) + 4 * O + 4 * si.numel()
    peak, peak_kind = measured_peak("hbm_gbs")
    achieved = nbytes / (ms / 1e3) / 1e9
    del codes, si, q4, sc
    torch.cuda.empty_cache()
    return {"metric": "FP8 E4M3 block-scaled -> int4 converter throughput", "value": achieved, "unit": "GB/s",
            "ms_per_step": ms, "steps": steps, "warmup": warmup,
            "config": {"rows": O, "cols": I, "matrices": f"{n_experts} stacked GLM gate matrices",
                       "l2": "inputs larger than L2 (%.0f MB of codes per launch)" % (O * I / 1e6)},
            "roofline": {"bound": "hbm", "kernel": "fp8_to_int4_kernel<12>", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind + " HBM copy bandwidth",
                         "traffic": TRAFFIC.get("glm_fp8_to_int4"), "algorithmic_bytes_per_launch": nbytes,
                         "avg_launch_ms": ms, "launches_timed": steps},
            "gpu_launches": steps, "clocks": clk}


SECONDARY = ("glm_moe_layer_verify_b8", "glm_moe_layer_prefill_2048")
SECONDARY_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "roofline", "e2e", "clocks", "gpu_launches")


def secondary_lines(args, rank, world, local):
    """The other two single-layer workloads of the metric (verify batch 8 and
    prefill 2048), timed in the same process after the headline with two
    resident layer weight sets each (9.7 GB, inputs larger than L2); the
    headline workload again with adaptive expert top-p 0.7 and with int8
    experts (four resident sets, 2x the weight bytes); and the FP8 -> int4
    converter step."""
    out = {}
    runs = [(wl, 0.0, 4, 2, wl) for wl in SECONDARY] + [
        (DEFAULT_WORKLOAD, 0.7, 4, 8, DEFAULT_WORKLOAD + "_topp0.7"),
        (DEFAULT_WORKLOAD, 0.0, 8, 4, DEFAULT_WORKLOAD + "_int8")]
    for wl, tp, wb, nl, key in runs:
        line = run_ours(args, wl, rank, world, local, n_layers=nl, steps=max(args.steps, 10),
                        warmup=max(3, min(args.warmup, 20)), with_cpu=False, top_p=tp, wbits=wb)
        if line is None:
            continue
        sub = {k: line[k] for k in SECONDARY_KEYS}
        sub["config"] = {k: line["config"][k] for k in ("tokens_per_step", "zipf_skew", "experts_streamed_per_layer",
                                                        "layer_sets_cycled", "l2", "cuda_graph", "top_p",
                                                        "weight_bits", "decode_plan")}
        out[key] = sub
    if rank == 0:
        out["glm_fp8_to_int4"] = run_fp8_converter(args, local)
    return out


def main():
    args = parse_args()
    rank, world, local = env_rank()
    import synth
    if args.workload == "glm_fp8_to_int4":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the layer forward only"}))
            return
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(run_fp8_converter(args, local, n_experts=args.fp8_experts, steps=args.steps,
                                           warmup=max(3, args.warmup))), flush=True)
        return
    cfg = synth.CONFIGS[WORKLOADS[args.workload][0]]
    stack = WORKLOADS[args.workload][1]
    if args.impl == "reference":
        line = run_reference(args, cfg, stack, rank)
    else:
        if world != args.gpus:
            print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        import torch
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=dev)
        line = run_ours(args, args.workload, rank, world, local)
        if world == 1 and not args.no_secondary and args.workload == DEFAULT_WORKLOAD:
            sec = secondary_lines(args, rank, world, local)
            if line is not None:
                line["secondary"] = sec
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
