#!/usr/bin/env python
"""Benchmark of the QMoE layer forward on GB300.

Default workload: the decode stack -- 48 independent QMoE layers of shape
H=2048, inter=768, E=128, top-k=8, INT4 block 32, BF16, run back to back on
T=8 packed tokens, layer l+1 consuming layer l's output. One step is 12 passes
through the 48 layers (576 layer calls, each with its own router logits; every
step of the method: routing, grouping, fc1 + SwiGLU, fc2, combine), about
28 ms, so the default 20 steps time more than half a second. Weights total
16.3 GB, far larger than L2, so no flush is needed between steps. The calls are
captured once in a CUDA graph through the public C ABI and replayed.

The same line carries the prefill half of the metric (`prefill`): the same 48
layers' weights on T=8192 packed tokens (16 sequences of lengths
~U[128,1024]), the grouped tcgen05 path, one step = one pass through the 48
layers, with its own roofline (grouped fc1 and the whole layer against the
measured dense BF16 peak), e2e and CPU baseline.

--workload prefill / int3 / int2: one layer of the named shape.

Prints one JSON line (rank 0). --impl reference times the CPU oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

LAYERS = 48
METRIC = "QMoE layer tokens/s (decode T<=8, prefill 8K) + % HBM / tensor roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "prefill", "int3", "int2", "router"], default="decode",
                    help="decode: 48-layer stack; prefill: one 8K layer; int3: one INT3 Zipf layer "
                         "(--T, --block); int2: one INT2 32K layer; router: the router-logit GEMM "
                         "alone (qmoe_router_logits, --T tokens, default 8192)")
    ap.add_argument("--block", type=int, default=64, help="INT3 block size (64 or 128)")
    ap.add_argument("--T", type=int, default=None, help="tokens per step (decode default 8)")
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--passes", type=int, default=12,
                    help="decode: passes through the layer stack per step (a step of about 28 ms, so "
                         "that the default 20 steps time more than 0.5 s)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode: leave out the prefill half of the line")
    ap.add_argument("--prefill-steps", type=int, default=None, help="prefill steps (default: --steps)")
    ap.add_argument("--cpu-sample-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--options", action="store_true",
                    help="run qmoe_forward_ex with FC1/FC2 biases and full-softmax routing weights")
    ap.add_argument("--decode-layer-kernel", action="store_true",
                    help="decode: qmoe_forward_ex with the decode layer kernel (fc1 and fc2 in one "
                         "persistent kernel) instead of one kernel per stage")
    ap.add_argument("--format", choices=["int", "mxfp4", "nvfp4"], default="int",
                    help="decode / prefill: expert weight format (the FP4 formats: E2M1 codes with E8M0 block-32 "
                         "or E4M3 block-16 scales; NVFP4 with per-expert global scales)")
    ap.add_argument("--path", choices=["auto", "decode", "grouped", "tiles", "ws"], default="auto",
                    help="kernel path of every call (auto: decode for T <= 8 and for mid-size batches "
                         "with few routes per expert, grouped otherwise; grouped: its kernel by the route "
                         "count; tiles / ws: the grouped path's route-tile / weights-stationary kernel)")
    ap.add_argument("--clock-log", default=None,
                    help="CSV file for the nvidia-smi clock samples (default: a file in the temp directory)")
    return ap.parse_args()


# --------------------------------------------------------------------------- common

def pass_count(args):
    return args.passes if args.workload == "decode" else 1


def workload_config(args, shape, layers, world):
    """The `config` object of the bench line (the same for both arms)."""
    passes = pass_count(args)
    step = (f"one step = {passes} passes through the {layers} layers (call c runs layer c mod {layers} "
            f"on call c-1's output, with its own router logits)" if passes > 1 else
            f"one step = one pass through the {layers} layer(s)")
    return {"workload": (f"{args.workload}: {layers} QMoE layers H={shape.H} inter={shape.inter} "
                         f"E={shape.E} k={shape.k} {['INT%d' % shape.bits, 'MXFP4', 'NVFP4'][shape.format]} "
                         f"b{shape.block} "
                         f"{'BF16' if shape.dtype == 0 else 'FP16'} T={shape.T} per rank"),
            "T": shape.T, "layers": layers, "passes": passes, "step": step, "parallelism": f"replicas x{world}",
            "l2": "weights 16.3 GB >> L2, no flush" if args.workload == "decode" else "inputs > L2 per step",
            **({"options": "fc1/fc2 biases N(0, 0.5), full-softmax routing weights"}
               if getattr(args, "options", False) else {}),
            **({"decode_layer_kernel": 1} if getattr(args, "decode_layer_kernel", False) else {}),
            **({"path": args.path} if getattr(args, "path", "auto") != "auto" else {}),
            **({"format": args.format} if getattr(args, "format", "int") != "int" else {})}


def reduce_max(v, device):
    """Largest value of v over the ranks of the default process group (the job's
    time is its slowest rank's); v itself without a process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens_per_rank_step, world, seconds_per_step):
    """Whole-job throughput: the tokens of every rank over the slowest rank's step."""
    return tokens_per_rank_step * world / seconds_per_step


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_shape(args):
    if args.workload == "decode":
        T = args.T or 8
        shape, recipe, _ = synthetic.decode_layer(T)
        fmt = {"int": 0, "mxfp4": 1, "nvfp4": 2}[getattr(args, "format", "int")]
        if fmt:
            shape.format, shape.block = fmt, 32 if fmt == 1 else 16
        return shape, recipe
    if args.workload == "int3":
        shape, recipe, _ = synthetic.int3_zipf(args.T or 512, args.block)
        return shape, recipe
    if args.workload == "int2":
        shape, recipe, _ = synthetic.int2_prefill_32k()
        if args.T:
            shape.T = args.T
        return shape, recipe
    shape, recipe, _ = synthetic.prefill_8k()
    if args.T:
        shape.T = args.T
    fmt = {"int": 0, "mxfp4": 1, "nvfp4": 2}[getattr(args, "format", "int")]
    if fmt:
        shape.format, shape.block = fmt, 32 if fmt == 1 else 16
    return shape, recipe


def layer_count(args):
    return args.layers if args.workload == "decode" else 1


def host_inputs(shape, recipe, layers, rank):
    """x for layer 0 and the router logits of every layer (seeded per rank and layer)."""
    x = synthetic.make_activations(shape, recipe, 5000 + rank)["x"]
    logits = np.stack([synthetic.make_activations(shape, recipe, 1000 + l + 7919 * rank)["logits"]
                       for l in range(layers)])
    return x, logits


def distinct_experts(logits_bits, dtype, k):
    """Number of distinct experts each layer selects (top-k of the raw logits)."""
    out = []
    for lb in logits_bits:
        if dtype == synthetic.FP16:
            v = lb.view(np.float16).astype(np.float64)
        else:
            v = (lb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        order = np.argsort(-v, axis=1, kind="stable")[:, :k]
        out.append(len(np.unique(order)))
    return out


def expert_bytes(shape):
    """Packed codes + scales of one expert: (fc1, fc2)."""
    H, I, b, B = shape.H, shape.inter, shape.bits, shape.block
    sb = 1 if shape.format else 2      # FP4 formats: 8-bit block scales
    fc1 = 2 * I * (H * b // 8 + (H // B) * sb)
    fc2 = H * (I * b // 8 + (I // B) * sb)
    return fc1, fc2


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str | None, path: str | None = None):
        import tempfile

        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(), f"qmoe_clocks_{os.getpid()}.csv")
        self.uuid = device_uuid

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle

def oracle_rate(shape, recipe, args, rank, budget_s):
    """Tokens/s of the CPU oracle on a bounded sample of the workload: consecutive
    layers of the stack (decode) or a subset of the tokens (prefill)."""
    import oracle

    cores = oracle.num_cores()
    layers = layer_count(args)
    x, logits = host_inputs(shape, recipe, layers, rank)
    weights_cache = {}

    def weights(l):
        if l not in weights_cache:
            full = synthetic.make_numpy(shape, recipe, 1000 + l)
            weights_cache.clear()
            weights_cache[l] = full
        return weights_cache[l]

    def op_of(w):
        return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                              shape.dtype, 0, shape.format, w.get("g1"), w.get("g2"))

    done_tokens = 0
    spent = 0.0
    if args.workload == "decode":
        cur = x
        l = 0
        while l < layers and spent < budget_s:
            w = weights(l)
            inp = dict(w, x=cur, logits=logits[l])
            t0 = time.perf_counter()
            cur, _ = oracle.forward(op_of(w), inp, nthreads=cores)
            spent += time.perf_counter() - t0
            done_tokens += shape.T
            l += 1
        sample = f"{l} consecutive decode layers x {shape.T} tokens (layer-tokens {done_tokens})"
    else:
        w = weights(0)
        inp = dict(w, x=x, logits=logits[0])
        batch = max(cores, 16)
        start = 0
        while spent < budget_s and start < shape.T:
            toks = np.arange(start, min(start + batch, shape.T))
            t0 = time.perf_counter()
            oracle.forward(op_of(w), inp, tokens=toks, nthreads=cores)
            spent += time.perf_counter() - t0
            done_tokens += len(toks)
            start += batch
        sample = f"{done_tokens} of the {shape.T} prefill tokens of one layer"
    # the same oracle on one thread, on a small sample: one layer (decode) or 16 tokens
    if args.workload == "decode":
        inp1 = dict(weights(0), x=x, logits=logits[0])
        t0 = time.perf_counter()
        oracle.forward(op_of(inp1), inp1, nthreads=1)
        one = shape.T / (time.perf_counter() - t0)
        one_sample = f"one decode layer x {shape.T} tokens"
    else:
        inp1 = dict(weights(0), x=x, logits=logits[0])
        toks = np.arange(0, min(16, shape.T))
        t0 = time.perf_counter()
        oracle.forward(op_of(inp1), inp1, tokens=toks, nthreads=1)
        one = len(toks) / (time.perf_counter() - t0)
        one_sample = f"{len(toks)} tokens of one layer"
    return {"value": done_tokens / spent, "unit": "layer-tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample, "seconds": round(spent, 2),
            "single_thread": {"value": one, "sample": one_sample}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    shape, recipe = workload_shape(args)
    per_step = []
    budget = max(2.0, args.cpu_sample_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state
    res = None
    for _ in range(args.steps):
        res = oracle_rate(shape, recipe, args, 0, budget)
        per_step.append(res["value"])
    value = statistics.median(per_step)
    prefill = None
    if args.workload == "decode" and not args.no_prefill:
        pshape, precipe, _ = synthetic.prefill_8k()
        pargs = argparse.Namespace(**{**vars(args), "workload": "prefill"})
        pres = oracle_rate(pshape, precipe, pargs, 0, args.cpu_sample_seconds)
        prefill = {"value": pres["value"], "unit": "layer-tokens/s", "cpu_baseline": pres,
                   "e2e": {"value": pres["value"], "unit": "layer-tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "layer-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, shape, layer_count(args), world),
        "cpu_baseline": {**res, "value": value},
        "e2e": {"value": value, "unit": "layer-tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        **({"prefill": prefill} if prefill else {}),
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU

def kernel_traffic(key):
    """DRAM bytes per launch of a roofline kernel from the committed ncu summary,
    or None when the kernel's sources changed since that capture."""
    import hashlib
    try:
        data = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        ent = data[key]
        h = hashlib.sha256()
        for f in ent["sources"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
    except (OSError, ValueError, KeyError):
        return None
    return int(ent["dram_bytes_per_launch"]) if h.hexdigest() == ent["source_sha256"] else None


def p_path(shape, forced="auto"):
    """The kernel path of a call (csrc/api.cu, resolve_path): "decode" or "grouped"."""
    if forced in ("grouped", "tiles", "ws"):
        return "grouped"
    if forced != "auto":
        return forced
    R = shape.T * shape.k
    if shape.T <= 8:
        return "decode"
    few = R < 64 or R < 4 * shape.E
    return "decode" if few and shape.T <= 64 and R <= 512 else "grouped"


def launches_per_layer(path, shape, layer_kernel=False):
    """Kernels one qmoe_forward call launches (csrc/api.cu and csrc/route.cu)."""
    small = shape.T * shape.k <= 512
    route = 1 if small else 4            # fused route+group, or route, count, scan, scatter
    if path == "decode":
        return route + (2 if layer_kernel else 3)   # (layer kernel or fc1, fc2), combine
    return route + 1 + 3                 # gather, fc1, fc2, combine


class Stack:
    """`passes` passes through `layers` QMoE layers (weights W[l]) on T tokens, through
    the public C ABI: call c runs layer c mod layers on the previous call's output
    (call 0 on x) with its own router logits. Inputs are copied from pinned host
    memory; the calls are captured in CUDA graphs."""

    def __init__(self, qm, shape, W, x_h, logits_h, passes, device, options=None, path=0):
        import torch

        self.qm, self.shape, self.W, self.options = qm, shape, W, options
        self.layers, self.passes = len(W), passes
        self.calls = passes * self.layers
        assert logits_h.shape[0] == self.calls
        self.p = qm.problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                            shape.dtype, path, shape.format)
        self.x_pin = torch.from_numpy(x_h.view(np.int16)).pin_memory()
        self.lg_pin = torch.from_numpy(logits_h.view(np.int16)).pin_memory()
        self.x_d = self.x_pin.to(device)
        self.lg_d = self.lg_pin.to(device)
        self.bufs = [torch.empty((shape.T, shape.H), dtype=torch.int16, device=device) for _ in range(2)]
        self.ws = torch.empty(qm.qmoe_workspace_bytes(self.p), dtype=torch.uint8, device=device)
        self.out_pin = torch.empty((shape.T, shape.H), dtype=torch.int16).pin_memory()
        self.final = self.bufs[(self.calls - 1) % 2]

    def args(self, c):
        src = self.x_d if c == 0 else self.bufs[(c - 1) % 2]
        w = self.W[c % self.layers]
        return (src, self.lg_d[c], w["fc1_q"], w["fc1_s"], None, w["fc2_q"], w["fc2_s"], None,
                self.bufs[c % 2], self.ws)

    def step(self):
        o = self.options
        for c in range(self.calls):
            if self.shape.format:
                w = self.W[c % self.layers]
                self.qm.qmoe_forward_ex(self.p, 0, None, None, *self.args(c), fc1_global_scale=w.get("g1"),
                                        fc2_global_scale=w.get("g2"))
            elif o is not None:
                l = c % self.layers
                self.qm.qmoe_forward_ex(self.p, o["full_softmax"], o["b1"][l] if o["b1"] else None,
                                        o["b2"][l] if o["b2"] else None, *self.args(c),
                                        decode_layer_kernel=o["layer_kernel"])
            else:
                self.qm.qmoe_forward(self.p, *self.args(c))

    def capture(self, stream):
        import torch

        with torch.cuda.stream(stream):
            self.step()                   # eager warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.step()
        return g

    def stage_graphs(self, stream):
        """Per stage, one graph of that stage alone for the last pass's calls (the
        workspace holds a valid previous state): the stage kernels' own durations."""
        import torch

        out = []
        for st in range(4):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in range(self.calls - self.layers, self.calls):
                    self.qm.qmoe_forward_stages(self.p, st, st, *self.args(c))
            out.append(g)
        return out

    def h2d_bytes(self):
        return int(self.x_pin.numel() * 2 + self.lg_pin.numel() * 2)

    def d2h_bytes(self):
        return int(self.out_pin.numel() * 2)


def device_uuid(device):
    import torch

    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        return None


def time_graph(g, stream, steps, warmup, device, clock_path, world):
    """Warm-up replays, then exactly `steps` replays between events on the launching
    stream, with a barrier and a synchronize on both sides: (per-step ms list,
    mean ms per step over the slowest rank, clock summary)."""
    import torch
    import torch.distributed as dist

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(device_uuid(device), clock_path) as clocks:
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            marks[0].record()
            for i in range(steps):
                g.replay()
                marks[i + 1].record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    ms = reduce_max(marks[0].elapsed_time(marks[-1]) / steps, device)
    return step_ms, ms, clocks.summary()


def replay_synchronised(g, stream):
    """One replay on `stream` (the stage graphs read the workspace state it leaves),
    finished before anything else is timed."""
    import torch

    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()


def time_stages(graphs, stream, steps, launches):
    """ms per launch of each stage: events around `steps` replays of its graph."""
    import torch

    out = np.zeros(len(graphs))
    for st, gst in enumerate(graphs):
        with torch.cuda.stream(stream):
            gst.replay()   # warm, on the timed stream, finished before the timed region
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            for _ in range(steps):
                gst.replay()
            b.record()
        torch.cuda.synchronize()
        out[st] = a.elapsed_time(b) / (steps * launches)
    return out


def time_e2e(stack, g, stream, steps, device):
    """Seconds per step, end to end: pinned host inputs -> device, the step's calls,
    the result -> pinned host memory, every step."""
    import torch

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        with torch.cuda.stream(stream):
            stack.x_d.copy_(stack.x_pin, non_blocking=True)
            stack.lg_d.copy_(stack.lg_pin, non_blocking=True)
            g.replay()
            stack.out_pin.copy_(stack.final, non_blocking=True)
        stream.synchronize()
    return reduce_max((time.perf_counter() - t0) / steps, device)


def stage_us(stage_ms):
    return {"route_group": round(stage_ms[0] * 1e3, 2), "fc1": round(stage_ms[1] * 1e3, 2),
            "fc2": round(stage_ms[2] * 1e3, 2), "combine": round(stage_ms[3] * 1e3, 2)}


def tensor_roofline(shape, fc1_ms, peaks, traffic):
    """The grouped fc1 launch against the measured dense BF16 peak (FP16 operands run
    at the same rate): 2 x routes x 2I x H FLOPs per launch."""
    flops = 2.0 * shape.T * shape.k * (2 * shape.inter * shape.H)
    tf = peaks.get("bf16_tflops")
    peak = tf if tf else 1900.0
    achieved = flops / (fc1_ms / 1e3) / 1e12
    out = {"bound": "tensor", "kernel": "grouped fc1 dequant-GEMM + SwiGLU (tcgen05, FP16 operands)",
           "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
           "peak_source": "measured burst" if tf else "fallback", "algorithmic_flops_per_launch": flops,
           "traffic": traffic, "traffic_unit": "bytes per launch (ncu)"}
    if peaks.get("bf16_tflops_sustained"):
        out["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    return out


def layer_flops(shape):
    return 2.0 * shape.T * shape.k * (2 * shape.inter * shape.H + shape.H * shape.inter)


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    from quantized_mixture_experts_route_gb300 import build as qbuild

    if rank == 0:
        qbuild.build()
    if world > 1:
        dist.barrier()
    import quantized_mixture_experts_route_gb300 as qm

    shape, recipe = workload_shape(args)
    layers = layer_count(args)
    passes = pass_count(args)
    W = [synthetic.make_torch_weights(shape, recipe, 1000 + l, device) for l in range(layers)]
    x_h, logits_h = host_inputs(shape, recipe, layers * passes, rank)
    options = None
    if args.options:
        gb = torch.Generator(device=device)
        gb.manual_seed(7)
        tdt = torch.bfloat16 if shape.dtype == synthetic.BF16 else torch.float16
        B1 = [(torch.randn((shape.E, 2 * shape.inter), generator=gb, device=device) * 0.5).to(tdt)
              .view(torch.int16) for _ in range(layers)]
        B2 = [(torch.randn((shape.E, shape.H), generator=gb, device=device) * 0.5).to(tdt)
              .view(torch.int16) for _ in range(layers)]
        options = dict(full_softmax=1, b1=B1, b2=B2, layer_kernel=0)
    if args.decode_layer_kernel:
        options = dict(options or dict(full_softmax=0, b1=None, b2=None), layer_kernel=1)
    path = {"auto": qm.QMOE_PATH_AUTO, "decode": qm.QMOE_PATH_DECODE, "grouped": qm.QMOE_PATH_GROUPED,
            "tiles": qm.QMOE_PATH_GROUPED_ROUTE_TILES, "ws": qm.QMOE_PATH_GROUPED_WS}[args.path]
    stack = Stack(qm, shape, W, x_h, logits_h, passes, device, options, path)
    s = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    g = stack.capture(s)
    gs = stack.stage_graphs(s)
    torch.cuda.synchronize()

    step_ms, ms, clocks = time_graph(g, s, args.steps, args.warmup, device, args.clock_log, world)
    replay_synchronised(g, s)
    stage_ms = time_stages(gs, s, args.steps, layers)
    e2e_s = time_e2e(stack, g, s, args.steps, device)

    # the prefill half of the metric: the same 48 layers' weights on 8192 packed tokens
    prefill = None
    if (args.workload == "decode" and not args.options and not args.decode_layer_kernel and not args.no_prefill
            and args.format == "int"):
        pshape, precipe, _ = synthetic.prefill_8k()
        px_h, plg_h = host_inputs(pshape, precipe, layers, rank)
        pstack = Stack(qm, pshape, W, px_h, plg_h, 1, device)
        pg = pstack.capture(s)
        pgs = pstack.stage_graphs(s)
        psteps = args.prefill_steps or args.steps
        pclock = (args.clock_log + ".prefill") if args.clock_log else None
        pstep_ms, pms, pclocks = time_graph(pg, s, psteps, args.warmup, device, pclock, world)
        replay_synchronised(pg, s)
        pstage_ms = time_stages(pgs, s, psteps, layers)
        pe2e_s = time_e2e(pstack, pg, s, psteps, device)
        prefill = dict(shape=pshape, recipe=precipe, stack=pstack, step_ms=pstep_ms, ms=pms, clocks=pclocks,
                       stage_ms=pstage_ms, e2e_s=pe2e_s, steps=psteps, logits=plg_h)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    value = job_rate(shape.T * layers * passes, world, ms / 1e3)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    fc1_b, fc2_b = expert_bytes(shape)
    # the captured kernels' workloads (traffic figures hold for the plain call only)
    default_kernel = (args.workload in ("decode", "prefill") and not args.options and not args.decode_layer_kernel
                      and args.format == "int")
    nact = distinct_experts(logits_h, shape.dtype, shape.k)
    if p_path(shape, args.path) == "decode":
        # the single-stage graphs run on the routing of the last call
        bytes_fc1 = float(nact[-1]) * fc1_b
        hbm = peaks.get("hbm_gbs")
        peak = hbm if hbm else 6800.0
        achieved = bytes_fc1 / (stage_ms[1] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "decode fc1 dequant-GEMV + SwiGLU",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": "measured" if hbm else "fallback",
                "algorithmic_bytes_per_launch": int(bytes_fc1),
                "traffic": kernel_traffic("decode_fc1") if default_kernel else None,
                "traffic_unit": "bytes per launch (ncu)"}
        per_call_ms = ms / (layers * passes)
        if args.decode_layer_kernel:
            # the stage calls run the separate kernels: the layer kernel is read through the whole call
            lb = float(np.mean(nact)) * (fc1_b + fc2_b)
            achieved = lb / (per_call_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "kernel": "decode layer kernel (whole call: routing, layer kernel, combine)",
                    "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "peak_source": "measured" if hbm else "fallback",
                    "algorithmic_bytes_per_launch": int(lb), "traffic": None,
                    "traffic_unit": "bytes per launch (ncu)"}
        extra = {"distinct_experts_per_layer_mean": float(np.mean(nact)),
                 "fc2_GBps": round(float(nact[-1]) * fc2_b / (stage_ms[2] / 1e3) / 1e9, 1),
                 "layer_GBps": round(float(np.mean(nact)) * (fc1_b + fc2_b) / (per_call_ms / 1e3) / 1e9, 1),
                 "layer_frac_of_hbm": round(float(np.mean(nact)) * (fc1_b + fc2_b) / (per_call_ms / 1e3) / 1e9
                                            / peak, 4)}
    else:
        roof = tensor_roofline(shape, stage_ms[1], peaks,
                               kernel_traffic("prefill_fc1") if default_kernel else None)
        lt = layer_flops(shape) / (ms / layers / 1e3) / 1e12
        extra = {"fc1_GBps": round(float(nact[-1]) * fc1_b / (stage_ms[1] / 1e3) / 1e9, 1),
                 "distinct_experts_per_layer_mean": float(np.mean(nact)),
                 "layer_tflops": round(lt, 1), "layer_frac": round(lt / roof["peak"], 4)}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "layer-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "ms_per_step_stats": {"median": round(float(np.median(step_ms)), 4),
                              "min": round(float(np.min(step_ms)), 4), "max": round(float(np.max(step_ms)), 4)},
        "timed_region_s": round(ms * args.steps / 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16-mma/fp32-acc",
        "data": "synthetic",
        "config": workload_config(args, shape, layers, world),
        "roofline": roof,
        "stage_us": stage_us(stage_ms),
        "e2e": {"value": round(shape.T * layers * passes * world / e2e_s, 1), "unit": "layer-tokens/s",
                "h2d_bytes_per_step": stack.h2d_bytes(), "d2h_bytes_per_step": stack.d2h_bytes()},
        "gpu_launches": int(launches_per_layer(p_path(shape, args.path), shape, args.decode_layer_kernel) * layers * passes
                            * args.steps),
        "clocks": clocks,
        **extra,
    }
    if prefill is not None:
        ps = prefill["shape"]
        pms = prefill["ms"]
        proof = tensor_roofline(ps, prefill["stage_ms"][1], peaks, kernel_traffic("prefill_fc1"))
        lt = layer_flops(ps) / (pms / layers / 1e3) / 1e12
        pn = distinct_experts(prefill["logits"], ps.dtype, ps.k)
        line["prefill"] = {
            "workload": (f"prefill: {layers} QMoE layers (the decode stack's weights) on T={ps.T} packed "
                         f"tokens from {len(prefill['recipe'].seq_lens)} sequences ~U[128,1024]; "
                         f"one step = one pass through the {layers} layers"),
            "value": round(job_rate(ps.T * layers, world, pms / 1e3), 1), "unit": "layer-tokens/s",
            "steps": prefill["steps"], "ms_per_step": round(pms, 4),
            "ms_per_layer": round(pms / layers, 4),
            "ms_per_step_stats": {"median": round(float(np.median(prefill["step_ms"])), 4),
                                  "min": round(float(np.min(prefill["step_ms"])), 4),
                                  "max": round(float(np.max(prefill["step_ms"])), 4)},
            "timed_region_s": round(pms * prefill["steps"] / 1e3, 3),
            "roofline": proof,
            "layer_roofline": {"bound": "tensor", "algorithmic_flops_per_layer": layer_flops(ps),
                               "achieved": round(lt, 1), "peak": proof["peak"], "unit": "TFLOP/s",
                               "frac": round(lt / proof["peak"], 4)},
            "stage_us": stage_us(prefill["stage_ms"]),
            "distinct_experts_per_layer_mean": float(np.mean(pn)),
            "e2e": {"value": round(ps.T * layers * world / prefill["e2e_s"], 1), "unit": "layer-tokens/s",
                    "h2d_bytes_per_step": prefill["stack"].h2d_bytes(),
                    "d2h_bytes_per_step": prefill["stack"].d2h_bytes()},
            "gpu_launches": int(launches_per_layer("grouped", ps) * layers * prefill["steps"]),
            "clocks": prefill["clocks"],
            "l2": "weights 16.3 GB and activations > L2, no flush",
        }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_rate(shape, recipe, args, 0, args.cpu_sample_seconds)
        if prefill is not None:
            line["prefill"]["cpu_baseline"] = oracle_rate(prefill["shape"], prefill["recipe"],
                                                          argparse.Namespace(**{**vars(args), "workload": "prefill"}),
                                                          0, args.cpu_sample_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_router(args):
    """qmoe_router_logits alone: logits [T][128] = x [T][2048] . W_router^T, BF16, timed
    with CUDA events over `steps` calls on one stream (inputs resident in HBM)."""
    import torch

    from quantized_mixture_experts_route_gb300 import build as qbuild

    qbuild.build()
    import quantized_mixture_experts_route_gb300 as qm

    T, H, E = args.T or 8192, 2048, 128
    dev = torch.device("cuda", 0)
    p = qm.problem(T, H, 768, E, 8, 4, 32, synthetic.BF16)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    x = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16).view(torch.int16)
    w = (torch.randn((E, H), generator=gen, device=dev) * 0.05).to(torch.bfloat16).view(torch.int16)
    out = torch.empty((T, E), dtype=torch.int16, device=dev)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            qm.qmoe_router_logits(p, x, w, out, stream=s)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record()
        for _ in range(args.steps):
            qm.qmoe_router_logits(p, x, w, out, stream=s)
        b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    flops = 2.0 * T * H * E
    peak = peaks.get("bf16_tflops") or 1900.0
    tf = flops / (ms / 1e3) / 1e12
    print(json.dumps({
        "metric": "router-logit GEMM tokens/s", "value": round(T / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "dtype": "bf16-mma/fp32-acc", "data": "synthetic",
        "config": {"workload": f"router: logits [{T}][{E}] = x [{T}][{H}] . W_router [{E}][{H}]^T, BF16"},
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tf / peak, 4), "algorithmic_flops_per_launch": flops,
                     "peak_source": "measured burst" if peaks.get("bf16_tflops") else "fallback"},
        "gpu_launches": args.steps}), flush=True)


def main():
    args = parse()
    if args.options and args.impl == "reference":
        raise SystemExit("--options applies to the CUDA arm only")
    if args.workload == "router":
        if args.impl == "reference":
            raise SystemExit("--workload router applies to the CUDA arm only")
        run_router(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
