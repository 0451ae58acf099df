#!/usr/bin/env python3
"""Benchmark of the group-quantized MoE decode path on GB300.

Default workload: batch-1 decode through a stack of 24 resident MoE layers
(d_model 4096, d_ff 1024, 512 routed experts + 1 shared expert, top-4,
4-bit codes with a bf16 scale and bias per group of 64; 87 GB of weights,
far larger than L2). One step = one token through all 24 layers (RMSNorm,
router, softmax/top-4, SwiGLU experts, shared expert, combine, residual).
Seeded synthetic weights and activations (no trained model exists here).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload stack4|stack2|layer|expert|gemv|gemv8|host] [--layers L] [--batch B]
                  [--rows R --cols C --per-row]   (gemv8: the int8 MLP / QKV GEMV)

Prints one JSON line. With N > 1 (torchrun) every rank runs its own decode
stream on its own GPU (replicas; no data-path collective); the slowest
rank's time is reported and `value` counts all ranks' tokens.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode µs/layer and tokens/s; q4 GEMV HBM GB/s vs ~8 TB/s peak"
D_MODEL, D_FF, N_EXPERTS, TOP_K = 4096, 1024, 512, 4
EPS = 1e-6


# ------------------------------------------------------------------ helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def layer_weight_bytes(bits: int) -> int:
    from bit_group_quantized_gb300 import synth

    shape = synth.PoolShape(D_MODEL, D_FF, N_EXPERTS, bits)
    # router + shared-gate vector + 4 routed experts + 1 shared expert
    return N_EXPERTS * D_MODEL * 2 + D_MODEL * 2 + (TOP_K + 1) * shape.expert_bytes


def layer_algorithmic_bytes(bits: int) -> int:
    # weights + RMSNorm weight + normalised input (bf16) + residual read/write (fp32)
    return layer_weight_bytes(bits) + D_MODEL * 2 + D_MODEL * 2 + D_MODEL * 4 * 2


KERNEL_SOURCES = ("fused.cu", "common.cuh", "topk.cuh", "fused.h")  # what k_fused_decode is built from
TRAFFIC_RECORD = os.path.join("profiles", "k_fused_decode_traffic.json")


def kernel_sources_hash() -> str:
    import hashlib

    csrc = os.path.join(ROOT, "bit_group_quantized_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(n_layers: int, bits: int):
    """DRAM bytes of one k_fused_decode launch: the committed record of a
    1-layer ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) scaled
    by the number of layers (each layer reads the same bytes); None if there is
    no record for this width or the kernel sources changed since the capture."""
    path = os.path.join(ROOT, TRAFFIC_RECORD)
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(f"{bits}bit")
    if not rec or rec.get("kernel_sources_sha256_16") != kernel_sources_hash():
        return None
    return int(rec["traffic_bytes_per_layer"]) * n_layers


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_sample(bits: int, n_layers: int, seed: int = 0):
    """Time the fp64 oracle on one token through `n_layers` layers of the stack.

    Runs in this process on the host cores (numpy/BLAS threads). Expert
    regeneration on the host is excluded from the timed part.
    """
    import numpy as np
    import torch

    from bit_group_quantized_gb300 import synth
    from oracle import bgq_oracle as O

    shape = synth.PoolShape(D_MODEL, D_FF, N_EXPERTS, bits)

    def b16(t):
        return t.contiguous().view(torch.int16).numpy().astype(np.uint16)

    h = O.bf16_to_f64(b16(synth.activations(seed, 0, 1, D_MODEL)[0]))
    total = 0.0
    for l in range(n_layers):
        R = b16(synth.router(seed, l, N_EXPERTS, D_MODEL))
        G = b16(synth.shared_gate(seed, l, D_MODEL))
        rho = b16(synth.rho(seed, l, D_MODEL))
        t0 = time.perf_counter()
        a = O.round_bf16(O.rmsnorm(h, rho, EPS))
        idx = O.route(R, a, TOP_K, G)[2]
        total += time.perf_counter() - t0
        cache = {}
        for e in list(idx) + [N_EXPERTS]:
            q, sb = synth.expert_pool_range(seed, l, shape, int(e), 1)
            cache[int(e)] = [(m[0].numpy(), b16(m[1])) for m in synth.expert_matrices(q[0], sb[0], shape)]
        t0 = time.perf_counter()
        out, _, _, _ = O.moe_layer(R, G, lambda e: cache[e], cache[N_EXPERTS], bits, a, TOP_K)
        h = h + out
        total += time.perf_counter() - t0
    return total / n_layers  # seconds per layer-token


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    """The oracle as the reference arm: fp64 on the host cores. Each timed step
    is a bounded sample of the workload: one of its layers for one token
    (router, top-4, four routed experts, shared expert, RMSNorm, residual);
    tokens/s is that layer time extrapolated to the whole stack."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    bits = 2 if args.workload == "stack2" else 4
    n_layers = args.layers
    for _ in range(args.warmup):
        oracle_sample(bits, 1)
    times = [oracle_sample(bits, 1, seed=s + 1) for s in range(args.steps)]
    s_layer = statistics.mean(times)
    tok_s = 1.0 / (s_layer * n_layers)
    cores = cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tok_s, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s_layer * 1000, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": stack_config(args, bits, world),
        "detail": {"step": "one layer of the stack for one token (the bounded sample that was timed)",
                   "us_per_layer": round(s_layer * 1e6, 1),
                   "extrapolated_ms_per_token": round(s_layer * n_layers * 1000, 3)},
        "cpu_baseline": {"value": round(tok_s, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: 1 of {n_layers} layers for one token (router + 4 experts + shared),"
                                   " extrapolated to the full stack"},
        "e2e": {"value": round(tok_s, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def stack_config(args, bits: int, world: int) -> dict:
    """The workload of the decode-stack lines (identical in both arms)."""
    from bit_group_quantized_gb300 import synth

    shape = synth.PoolShape(D_MODEL, D_FF, N_EXPERTS, bits)
    return {"workload": workload_name(args, bits), "layers": args.layers, "batch": 1,
            "bytes_per_layer": layer_algorithmic_bytes(bits),
            "l2": "inputs larger than L2 (the stack holds %.1f GB of weights)" % (
                args.layers * shape.expert_bytes * (N_EXPERTS + 1) / 1e9),
            "parallelism": f"replicas x{world}"}


def workload_name(args, bits=None) -> str:
    if args.workload in ("stack4", "stack2"):
        if bits is None:
            bits = 4 if args.workload == "stack4" else 2
        return (f"moe_decode_stack: {args.layers} layers x (512 routed + 1 shared SwiGLU experts, d_model 4096, "
                f"d_ff 1024, top-4), {bits}-bit codes, group 64 bf16 scale+bias, batch 1")
    if args.workload == "layer":
        return (f"moe_layer: 512 routed + 1 shared experts, d_model 4096, d_ff 1024, top-4, 4-bit, batch {args.batch}"
                f", ring of {args.ring} distinct layers")
    if args.workload == "host":
        return (f"moe_layer with the 512 routed experts in pinned host memory (router and shared expert in HBM), "
                f"d_model 4096, d_ff 1024, top-4, 4-bit, batch {args.batch}, ring of 16 inputs, "
                + ("selected experts copied into HBM slots, then computed" if args.fetch == "copy"
                   else "selected experts read directly while computing"))
    if args.workload == "expert":
        return (f"moe_expert_swiglu: one SwiGLU expert (gate/up 1024x4096, down 4096x1024), 4-bit, group 64, "
                f"batch {args.batch}, ring of {args.ring} experts")
    if args.workload == "chain":
        return (f"bgq_gemv_chain: rmsnorm (bf16 weight), then 4-bit 4096x4096 projection, then 4-bit 4096x4096 "
                f"o_proj + residual, group 64, batch {args.batch}, dependent launches, ring of {args.ring} chains")
    if args.workload == "gemv8":
        return (f"q8_gemv: {args.rows}x{args.cols} 8-bit codes, " +
                ("one bf16 scale+bias per row" if args.per_row else "group 64 bf16 scale+bias") +
                f", batch {args.batch}, ring of {args.ring} matrices")
    return f"q4_gemv: 1024x4096 4-bit, group 64, batch 1, variant {args.variant}, ring of {args.ring} matrices"


# ------------------------------------------------------------------ ranks
def slowest_rank(value: float, world: int, device) -> float:
    """The largest of every rank's value (a time): the job is as slow as its
    slowest replica. Identity for one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world: int, ms_per_step: float) -> float:
    """Every rank decodes one token per step (replicas, weak scaling)."""
    return world * 1000.0 / ms_per_step


# ------------------------------------------------------------------ GPU arm
class DecodeStack:
    """A resident stack of synthetic layers, its workspace and a decode step
    (one token through every layer) captured in a CUDA graph."""

    def __init__(self, bits, n_layers, seed, dev, use_graph=True):
        import torch

        from bit_group_quantized_gb300 import lib, synth

        self.lib, self.torch, self.dev, self.bits, self.n_layers = lib, torch, dev, bits, n_layers
        shape = synth.PoolShape(D_MODEL, D_FF, N_EXPERTS, bits)
        layers, rhos, self.keep = [], [], []
        for l in range(n_layers):
            t = synth.layer_tensors(seed, l, shape, device=dev)
            self.keep.append(t)
            layers.append(lib.MoELayer(D_MODEL, D_FF, N_EXPERTS, TOP_K, bits, t["router"], t["shared_gate"],
                                       t["pool_q"][:N_EXPERTS], t["pool_sb"][:N_EXPERTS], t["pool_q"][N_EXPERTS],
                                       t["pool_sb"][N_EXPERTS]))
            rhos.append(synth.rho(seed, l, D_MODEL, device=dev))
        self.rhos = rhos
        self.stack = lib.Stack(layers, rhos)
        self.ws = lib.workspace(self.stack.ws_bytes, dev)
        self.x_in = synth.activations(seed, 0, 1, D_MODEL, device=dev)[0].clone()
        self.x_out = torch.empty_like(self.x_in)
        self.stream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()
        self.graph = None
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                self.step()
            self.stream.synchronize()
            if use_graph:
                self.graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(self.graph, stream=self.stream):
                    self.step()
        self.fused = lib.load().moe_stack_trace_entries(self.stack.c_layers, n_layers) > 0

    def step(self):
        self.lib.moe_stack_decode(self.stack, self.x_in, EPS, ws=self.ws, x_next=self.x_out, stream=self.stream)
        self.x_in.copy_(self.x_out)

    def run(self, n):
        with self.torch.cuda.stream(self.stream):
            for _ in range(n):
                if self.graph is not None:
                    self.graph.replay()
                else:
                    self.step()

    def check_status(self, when):
        self.stream.synchronize()
        status = self.lib.read_device_status(self.ws, self.stream)
        if status != self.lib.OK:
            raise RuntimeError(f"device status {when}: {self.lib.status_string(status)}")

    def timed(self, steps):
        """ms per step over `steps` graph replays (CUDA events on the stream)."""
        torch = self.torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        self.run(steps)
        e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / steps

    def free(self):
        del self.graph, self.stack, self.keep, self.ws, self.rhos
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def stack_roofline(bits, n_layers, ms, fused, traffic_n_layers=None):
    peak, peak_kind = peaks()
    achieved = n_layers * layer_algorithmic_bytes(bits) / (ms * 1e-3) / 1e9
    return {"bound": "hbm",
            "kernel": ("k_fused_decode (one launch per token, all %d layers)" % n_layers) if fused
            else "moe_stack_decode step (multi-kernel path)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_kind": f"{peak_kind} copy bandwidth (burst)", "frac_of_8tbs": round(achieved / 8000.0, 4),
            "traffic": profiled_traffic(n_layers, bits) if fused else None,
            "traffic_source": "ncu dram__bytes_read+write of a 1-layer capture x layers (%s)" % TRAFFIC_RECORD}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from bit_group_quantized_gb300 import lib

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    lib.load()

    bits = 2 if args.workload == "stack2" else 4
    n_layers = args.layers
    ds = DecodeStack(bits, n_layers, args.seed + rank, dev, use_graph=not args.no_graph)
    ds.run(args.warmup)
    ds.check_status("after warm-up")

    # ---- timed region (device time, CUDA events on the launching stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    ms = ds.timed(args.steps)
    torch.cuda.synchronize()
    clock = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = slowest_rank(ms, world, dev)
    ds.check_status("after the timed steps")

    # ---- end to end through the public API with host buffers: every step
    # copies the token in from pinned host memory, runs moe_stack_decode and
    # reads the result back into pinned host memory, where the host takes it
    # as the next token; the three are captured once in a CUDA graph (the
    # way a decode loop on this GPU issues them), replayed and waited for
    # every step
    xh = torch.empty(D_MODEL, dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(ds.x_in.cpu())
    oh = torch.empty(D_MODEL, dtype=torch.bfloat16, pin_memory=True)
    e2e_steps = max(1, min(args.steps, 500))

    def e2e_step():
        ds.x_in.copy_(xh, non_blocking=True)
        lib.moe_stack_decode(ds.stack, ds.x_in, EPS, ws=ds.ws, x_next=ds.x_out, stream=ds.stream)
        oh.copy_(ds.x_out, non_blocking=True)

    e2e_graph = None
    with torch.cuda.stream(ds.stream):
        e2e_step()
        ds.stream.synchronize()
        if not args.no_graph:
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph, stream=ds.stream):
                e2e_step()
            for _ in range(3):
                e2e_graph.replay()
                ds.stream.synchronize()
                xh.copy_(oh)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(ds.stream):
        for _ in range(e2e_steps):
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_step()
            ds.stream.synchronize()
            xh.copy_(oh)
    e2e_s = slowest_rank((time.perf_counter() - t0) / e2e_steps, world, dev)
    del e2e_graph
    fused = ds.fused
    ds.free()

    # ---- the same stack at 2 bits (the workload's second width), same run
    other = None
    if args.workload == "stack4" and not args.no_stack2:
        d2 = DecodeStack(2, n_layers, args.seed + rank, dev, use_graph=not args.no_graph)
        d2.run(args.warmup)
        d2.check_status("after the 2-bit warm-up")
        if world > 1:
            dist.barrier()
        clocks2 = ClockSampler(local)
        time.sleep(0.3)
        ms2 = slowest_rank(d2.timed(args.steps), world, dev)
        clock2 = clocks2.stop()
        d2.check_status("after the 2-bit timed steps")
        other = {"workload": workload_name(args, 2), "value": round(whole_job_tokens_per_s(world, ms2), 2),
                 "unit": "tokens/s", "ms_per_step": round(ms2, 5), "us_per_layer": round(ms2 * 1000 / n_layers, 3),
                 "steps": args.steps, "dtype": "u2 codes x s24 fixed-point x (dp4a), f32 accumulate",
                 "roofline": stack_roofline(2, n_layers, ms2, d2.fused), "clocks": clock2,
                 "gpu_launches": (1 if d2.fused else 1 + 6 * n_layers + 1) * args.steps}
        d2.free()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n_s = 2
        s_layer = oracle_sample(bits, n_s, seed=args.seed)
        cpu = {"value": round(1.0 / (s_layer * n_layers), 5), "unit": "tokens/s", "cores": cpu_cores(),
               "kind": "oracle",
               "sample": f"one token through {n_s} of the {n_layers} layers (fp64 numpy/BLAS), "
                         "extrapolated to the stack"}

    if rank == 0:
        layer_bytes = layer_algorithmic_bytes(bits)
        us_layer = ms * 1000 / n_layers
        # the persistent kernel runs a whole token in one launch; the multi-kernel
        # fallback launches widen + 6 per layer + the final norm
        launches = 1 if fused else 1 + 6 * n_layers + 1
        line = {
            "metric": METRIC, "value": round(whole_job_tokens_per_s(world, ms), 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": f"u{bits} codes x s24 fixed-point x (dp4a), f32 accumulate",
            "data": "synthetic (seeded counter-based generator; no trained weights)",
            "config": stack_config(args, bits, world),
            "detail": {"us_per_layer": round(us_layer, 3),
                       "gbs_per_layer": round(layer_bytes / (us_layer * 1e-6) / 1e9, 1),
                       "graph": not args.no_graph},
            "roofline": stack_roofline(bits, n_layers, ms, fused),
            "e2e": {"value": round(world / e2e_s, 2), "unit": "tokens/s", "h2d_bytes_per_step": D_MODEL * 2,
                    "d2h_bytes_per_step": D_MODEL * 2,
                    "how": ("per step: copy of the token from pinned host memory, moe_stack_decode, copy of the "
                            "result to pinned host memory (" + ("one CUDA graph replay" if not args.no_graph
                                                                 else "eager calls") +
                            "), wait, the host takes the result as the next token; host wall clock")},
            "gpu_launches": launches * args.steps,
            "clocks": clock,
            "cpu_baseline": cpu,
        }
        if other is not None:
            line["stack2"] = other
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _timed_graph(torch, stream, body, n_replays, warmup):
    """Capture body() once in a CUDA graph, warm up, then time n_replays
    replays with CUDA events on `stream`; returns ms per replay."""
    with torch.cuda.stream(stream):
        body()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        for _ in range(warmup):
            g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_replays):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) / n_replays


def run_layer(args):
    """One MoE layer at batch B per step, cycling through `ring` distinct
    resident layers and inputs (so router and shared weights are not L2 hits)."""
    import torch

    from bit_group_quantized_gb300 import lib, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib.load()
    B, R = args.batch, args.ring
    shape = synth.PoolShape(D_MODEL, D_FF, N_EXPERTS, 4)
    layers, keep, xs, outs = [], [], [], []
    for r in range(R):
        t = synth.layer_tensors(args.seed + 100, r, shape, device=dev)
        keep.append(t)
        layers.append(lib.MoELayer(D_MODEL, D_FF, N_EXPERTS, TOP_K, 4, t["router"], t["shared_gate"],
                                   t["pool_q"][:N_EXPERTS], t["pool_sb"][:N_EXPERTS], t["pool_q"][N_EXPERTS],
                                   t["pool_sb"][N_EXPERTS]))
        xs.append(synth.activations(args.seed + 100, r, B, D_MODEL, device=dev))
        outs.append(torch.empty((B, D_MODEL), dtype=torch.bfloat16, device=dev))
    ws = lib.workspace(lib.moe_layer_workspace_bytes(layers[0], B), dev)
    distinct = []
    for r in range(R):
        idx = lib.moe_layer_forward(layers[r], xs[r], ws=ws, want_route=True)[2]
        distinct.append(len(set(idx.flatten().tolist())))
    stream = torch.cuda.Stream(device=dev)

    def body():
        for r in range(R):
            lib.moe_layer_forward(layers[r], xs[r], ws=ws, out=outs[r], stream=stream)

    n_rep = max(1, args.steps // R)
    clocks = ClockSampler(0)
    ms = _timed_graph(torch, stream, body, n_rep, args.warmup) / R
    clock = clocks.stop()
    dmean = sum(distinct) / len(distinct)
    layer_bytes = N_EXPERTS * D_MODEL * 2 + D_MODEL * 2 + (dmean + 1) * shape.expert_bytes + B * D_MODEL * 4
    achieved = layer_bytes / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": METRIC, "value": round(B * 1000.0 / ms, 2), "unit": "tokens/s", "n_gpus": 1,
        "steps": n_rep * R, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u4 codes; dp4a / tcgen05 f16, f32 accumulate",
        "data": "synthetic", "config": {"workload": workload_name(args), "us_per_layer": round(ms * 1000, 3),
                                        "distinct_experts_mean": dmean, "bytes_per_layer": int(layer_bytes)},
        "roofline": {"bound": "hbm", "kernel": "moe_layer_forward (all launches)", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": None},
        "clocks": clock}), flush=True)
    return 0


def run_host(args):
    """One MoE layer whose routed-expert pool (3.6 GB) lives in pinned host
    memory (NVLink-C2C on a GB300 node); router and shared expert stay in HBM.
    --fetch direct: the grouped kernels read the selected experts straight from
    host memory while computing (fetch overlapped with compute); --fetch copy:
    moe_layer_forward_streamed copies them into HBM slots first, then computes
    (serial fetch, as the pages do). A ring of 16 inputs selects different
    experts per call (16 x ~28 MB exceeds L2)."""
    import torch

    from bit_group_quantized_gb300 import lib, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib.load()
    B, R = args.batch, 16
    shape = synth.PoolShape(D_MODEL, D_FF, N_EXPERTS, 4)
    t = synth.layer_tensors(args.seed + 300, 0, shape, device=dev)
    pool_q = t["pool_q"][:N_EXPERTS].to("cpu").pin_memory()
    pool_sb = t["pool_sb"][:N_EXPERTS].to("cpu").pin_memory()
    shared_q, shared_sb = t["pool_q"][N_EXPERTS].clone(), t["pool_sb"][N_EXPERTS].clone()
    router, gate = t["router"], t["shared_gate"]
    del t
    torch.cuda.empty_cache()
    layer = lib.MoELayer(D_MODEL, D_FF, N_EXPERTS, TOP_K, 4, router, gate, pool_q, pool_sb, shared_q, shared_sb)
    xs = [synth.activations(args.seed + 300, r, B, D_MODEL, device=dev) for r in range(R)]
    outs = [torch.empty((B, D_MODEL), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    ws = lib.workspace(lib.moe_layer_workspace_bytes(layer, B), dev)
    copy = args.fetch == "copy"
    slots = torch.empty(lib.moe_stream_slots_bytes(layer, B), dtype=torch.uint8, device=dev) if copy else None
    distinct = [len(set(lib.moe_layer_forward(layer, xs[r], ws=ws, want_route=True)[2].flatten().tolist()))
                for r in range(R)]
    stream = torch.cuda.Stream(device=dev)

    def body():
        for r in range(R):
            if copy:
                lib.moe_layer_forward_streamed(layer, xs[r], slots=slots, ws=ws, out=outs[r], stream=stream)
            else:
                lib.moe_layer_forward(layer, xs[r], ws=ws, out=outs[r], stream=stream)

    n_rep = max(1, args.steps // R)
    clocks = ClockSampler(0)
    ms = _timed_graph(torch, stream, body, n_rep, args.warmup) / R
    clock = clocks.stop()
    dmean = sum(distinct) / len(distinct)
    host_bytes = dmean * shape.expert_bytes
    print(json.dumps({
        "metric": METRIC, "value": round(B * 1000.0 / ms, 2), "unit": "tokens/s", "n_gpus": 1,
        "steps": n_rep * R, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u4 codes; dp4a, f32 accumulate", "data": "synthetic",
        "config": {"workload": workload_name(args), "us_per_layer": round(ms * 1000, 3),
                   "fetch": args.fetch, "distinct_experts_mean": dmean, "host_bytes_per_layer": int(host_bytes),
                   "host_read_gbs": round(host_bytes / (ms * 1e-3) / 1e9, 1)},
        "roofline": None, "clocks": clock}), flush=True)
    return 0


def run_gemv(args):
    """q4_gemv (1024x4096, batch 1) per step, cycling through `ring` distinct matrices."""
    import torch

    from bit_group_quantized_gb300 import lib, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib.load()
    R = args.ring = max(args.ring, 64)  # 64 x 2.2 MB: the ring exceeds L2
    rows, cols = 1024, 4096
    mats = []
    for r in range(R):
        q, sb = synth.qmatrix(args.seed + r, rows, cols, 4, device=dev)
        mats.append(lib.QMatrix(q, sb, rows, cols, 4))
    xs = [synth.activations(args.seed, 1000 + r, 1, cols, device=dev) for r in range(R)]
    ys = [torch.empty((1, rows), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.Stream(device=dev)

    def body():
        for r in range(R):
            if args.variant == 0:
                lib.q4_gemv(mats[r], xs[r], y=ys[r], stream=stream)
            else:
                lib.qgemv_variant(mats[r], xs[r], args.variant, y=ys[r], stream=stream)

    n_rep = max(1, args.steps // R)
    ms = _timed_graph(torch, stream, body, n_rep, args.warmup) / R
    nbytes = rows * cols // 2 + rows * cols // 64 * 4 + cols * 2 + rows * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": n_rep * R,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4 codes", "data": "synthetic",
        "config": {"workload": workload_name(args), "us_per_gemv": round(ms * 1000, 3), "bytes": nbytes},
        "roofline": {"bound": "hbm", "kernel": "k_qgemv", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_kind": peak_kind, "traffic": None}}), flush=True)
    return 0


def run_expert(args):
    """moe_expert_swiglu (one SwiGLU expert: gate/up 1024x4096, down 4096x1024,
    4-bit) on B tokens per step, cycling through a ring of distinct experts
    larger than L2."""
    import torch

    from bit_group_quantized_gb300 import lib, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib.load()
    shape = synth.PoolShape(4096, 1024, 1, 4)
    R = args.ring = max(args.ring, -(-600_000_000 // shape.expert_bytes))
    q, sb = synth.expert_pool_range(args.seed, 0, shape, 0, R, device=dev)
    experts = []
    for r in range(R):
        m = synth.expert_matrices(q[r], sb[r], shape)
        experts.append(lib.Expert(*[lib.QMatrix(mq, ms, mq.shape[0], ms.shape[1] * 64, 4) for mq, ms in m]))
    B = args.batch
    xs = [synth.activations(args.seed, 3000 + r, B, shape.d, device=dev) for r in range(R)]
    ws = lib.workspace(lib.expert_workspace_bytes(experts[0], B), dev)
    stream = torch.cuda.Stream(device=dev)

    def body():
        for r in range(R):
            lib.moe_expert_swiglu(experts[r], xs[r], ws=ws, stream=stream)

    n_rep = max(1, args.steps // R)
    ms = _timed_graph(torch, stream, body, n_rep, args.warmup) / R
    nbytes = shape.expert_bytes + B * shape.d * 2 * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    # the library takes an explicit expert to the tensor cores from 16 tokens
    tc = B >= 16
    dtype = ("u4 codes -> f16 x scaled f16 tokens (tcgen05 kind::f16), f32 accumulate" if tc
             else "u4 codes x s24 fixed-point x (dp4a), f32 accumulate")
    kernel = ("k_tc_act + k_tc_gemm gate/up + k_tc_act + k_tc_gemm down (one expert)" if tc
              else "k_gateup + k_down (one expert)")
    print(json.dumps({
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": n_rep * R,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {"workload": workload_name(args), "us_per_expert": round(ms * 1000, 3), "bytes": nbytes,
                   "tokens_per_s": round(B / (ms * 1e-3), 1),
                   "l2": f"ring of {R} experts ({R * shape.expert_bytes / 1e6:.0f} MB) cycled, larger than L2"},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": None}}), flush=True)
    return 0


def run_chain(args):
    """bgq_gemv_chain (rmsnorm, a 4096x4096 4-bit projection, a 4096x4096 4-bit
    o_proj + residual, as dependent launches) per step, cycling through a ring
    of distinct chains larger than L2."""
    import torch

    from bit_group_quantized_gb300 import lib, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib.load()
    d, B = 4096, max(1, min(args.batch, 8))
    mat_bytes = d * d // 2 + d * d // 64 * 4
    R = args.ring = max(args.ring, -(-400_000_000 // (2 * mat_bytes)))
    chains, xs, outs = [], [], []
    for r in range(R):
        mats = []
        for i in range(2):
            q, sb = synth.qmatrix(args.seed + 7 * r + i, d, d, 4, device=dev)
            mats.append(lib.QMatrix(q, sb, d, d, 4))
        chains.append(mats)
        xs.append(synth.activations(args.seed, 2000 + r, B, d, device=dev))
        outs.append(torch.empty((B, d), dtype=torch.bfloat16, device=dev))
    rho = synth.rho(args.seed, 0, d, device=dev)
    ws = lib.workspace(lib.gemv_chain_workspace_bytes(chains[0], B), dev)
    stream = torch.cuda.Stream(device=dev)

    def body():
        for r in range(R):
            lib.gemv_chain(chains[r], xs[r], norm=True, rho=rho, residual=True, ws=ws, out=outs[r], stream=stream)

    n_rep = max(1, args.steps // R)
    clocks = ClockSampler(0)
    ms = _timed_graph(torch, stream, body, n_rep, args.warmup) / R
    clock = clocks.stop()
    nbytes = 2 * mat_bytes + d * 2 + 2 * B * d * 2  # weights, rho, x in, out
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": n_rep * R,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4 codes x s24 fixed-point x (dp4a), f32 accumulate", "data": "synthetic",
        "config": {"workload": workload_name(args), "us_per_chain": round(ms * 1000, 3), "bytes": nbytes,
                   "batch": B, "l2": f"ring of {R} chains ({R * 2 * mat_bytes / 1e6:.0f} MB) cycled, larger than L2"},
        "roofline": {"bound": "hbm", "kernel": "k_rmsnorm + 2 x k_qgemv_int (dependent launches, whole chain)",
                     "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": None},
        "clocks": clock}), flush=True)
    return 0


def run_gemv8(args):
    """q8_gemv (int8 weights, rows x cols, batch B) per step, cycling through a
    ring of distinct matrices larger than L2 (4 x 129 MB at least)."""
    import torch

    from bit_group_quantized_gb300 import lib, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    lib.load()
    rows, cols, B = args.rows, args.cols, args.batch
    group = cols if args.per_row else 64
    gpr = cols // group
    mat_bytes = rows * cols + rows * gpr * 4
    R = args.ring = max(args.ring, -(-600_000_000 // mat_bytes))
    mats = []
    for r in range(R):
        q, sb = synth.qmatrix(args.seed + r, rows, cols, 8, device=dev, group=group)
        mats.append(lib.QMatrix(q, sb, rows, cols, 8, group))
    xs = [synth.activations(args.seed, 2000 + r, B, cols, device=dev) for r in range(R)]
    ys = [torch.empty((B, rows), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.Stream(device=dev)

    def body():
        for r in range(R):
            lib.q8_gemv(mats[r], xs[r], y=ys[r], stream=stream)

    n_rep = max(1, args.steps // R)
    ms = _timed_graph(torch, stream, body, n_rep, args.warmup) / R
    nbytes = mat_bytes + B * cols * 2 + B * rows * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": n_rep * R,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8 codes x s24 fixed-point x (dp4a), f32 accumulate", "data": "synthetic",
        "config": {"workload": workload_name(args), "us_per_gemv": round(ms * 1000, 3), "bytes": nbytes,
                   "l2": f"ring of {R} matrices ({R * mat_bytes / 1e6:.0f} MB) cycled, larger than L2"},
        "roofline": {"bound": "hbm", "kernel": "k_q8gemv", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_kind": peak_kind, "traffic": None}}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="stack4", choices=["stack4", "stack2", "layer", "expert", "gemv", "gemv8", "host",
                                                             "chain"])
    ap.add_argument("--variant", type=int, default=0, help="gemv: 0 integer (production), 1 standard, "
                                                            "2 reordered (the page's fma form), 3 hoisted fp32")
    ap.add_argument("--ring", type=int, default=8, help="layer/gemv: distinct weight copies cycled through")
    ap.add_argument("--layers", type=int, default=24)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--fetch", default="direct", choices=["direct", "copy"],
                    help="host: read host-resident experts directly (direct) or copy them into HBM first (copy)")
    ap.add_argument("--rows", type=int, default=4096, help="gemv8: output rows")
    ap.add_argument("--cols", type=int, default=4096, help="gemv8: input columns")
    ap.add_argument("--per-row", action="store_true", help="gemv8: one (scale, bias) per row (the FC2 format)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack2", action="store_true", help="stack4: skip the 2-bit stack measured after it")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "layer":
        return run_layer(args)
    if args.workload == "gemv":
        return run_gemv(args)
    if args.workload == "gemv8":
        return run_gemv8(args)
    if args.workload == "expert":
        return run_expert(args)
    if args.workload == "host":
        return run_host(args)
    if args.workload == "chain":
        return run_chain(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
