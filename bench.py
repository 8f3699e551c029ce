#!/usr/bin/env python
"""Benchmark of the QMoE layer forward on GB300.

Default workload: the decode stack -- 48 independent QMoE layers of shape
H=2048, inter=768, E=128, top-k=8, INT4 block 32, BF16, run back to back on
T=8 packed tokens, layer l+1 consuming layer l's output. One step is one pass
through the 48 layers (every step of the method: routing, grouping, fc1 +
SwiGLU, fc2, combine). Weights total 16.3 GB, far larger than L2, so no flush
is needed between steps. The 48 layer calls are captured once in a CUDA graph
through the public C ABI and replayed.

--workload prefill: one layer of the same shape on T=8192 packed tokens
(16 sequences of lengths ~U[128,1024]), the grouped tcgen05 path.

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
    ap.add_argument("--workload", choices=["decode", "prefill", "int3", "int2"], default="decode",
                    help="decode: 48-layer stack; prefill: one 8K layer; int3: one INT3 Zipf layer "
                         "(--T, --block); int2: one INT2 32K layer")
    ap.add_argument("--block", type=int, default=64, help="INT3 block size (64 or 128)")
    ap.add_argument("--T", type=int, default=None, help="tokens per step (decode default 8)")
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--cpu-sample-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--options", action="store_true",
                    help="run qmoe_forward_ex with FC1/FC2 biases and full-softmax routing weights")
    ap.add_argument("--clock-log", default=None,
                    help="CSV file for the nvidia-smi clock samples (default: a file in the temp directory)")
    return ap.parse_args()


# --------------------------------------------------------------------------- common

def workload_config(args, shape, layers, world):
    """The `config` object of the bench line (the same for both arms)."""
    return {"workload": (f"{args.workload}: {layers} QMoE layers H={shape.H} inter={shape.inter} "
                         f"E={shape.E} k={shape.k} INT{shape.bits} b{shape.block} "
                         f"{'BF16' if shape.dtype == 0 else 'FP16'} T={shape.T} per rank"),
            "T": shape.T, "layers": layers, "parallelism": f"replicas x{world}",
            "l2": "weights 16.3 GB >> L2, no flush" if args.workload == "decode" else "inputs > L2 per step",
            **({"options": "fc1/fc2 biases N(0, 0.5), full-softmax routing weights"}
               if getattr(args, "options", False) else {})}


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
    fc1 = 2 * I * (H * b // 8 + (H // B) * 2)
    fc2 = H * (I * b // 8 + (I // B) * 2)
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

    op = oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                        shape.dtype)
    done_tokens = 0
    spent = 0.0
    if args.workload == "decode":
        cur = x
        l = 0
        while l < layers and spent < budget_s:
            w = weights(l)
            inp = dict(w, x=cur, logits=logits[l])
            t0 = time.perf_counter()
            cur, _ = oracle.forward(op, inp, nthreads=cores)
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
            oracle.forward(op, inp, tokens=toks, nthreads=cores)
            spent += time.perf_counter() - t0
            done_tokens += len(toks)
            start += batch
        sample = f"{done_tokens} of the {shape.T} prefill tokens of one layer"
    # the same oracle on one thread, on a small sample: one layer (decode) or 16 tokens
    if args.workload == "decode":
        inp1 = dict(weights(0), x=x, logits=logits[0])
        t0 = time.perf_counter()
        oracle.forward(op, inp1, nthreads=1)
        one = shape.T / (time.perf_counter() - t0)
        one_sample = f"one decode layer x {shape.T} tokens"
    else:
        inp1 = dict(weights(0), x=x, logits=logits[0])
        toks = np.arange(0, min(16, shape.T))
        t0 = time.perf_counter()
        oracle.forward(op, inp1, tokens=toks, nthreads=1)
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
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "layer-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, shape, layer_count(args), world),
        "cpu_baseline": {**res, "value": value},
        "e2e": {"value": value, "unit": "layer-tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
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


def p_path(shape):
    return "decode" if shape.T <= 8 else "grouped"


def launches_per_layer(path, shape):
    """Kernels one qmoe_forward call launches (see csrc/api.cu and csrc/route.cu)."""
    small = shape.T * shape.k <= 512
    route = 1 if small else 4            # fused route+group, or route, count, scan, scatter
    if path == "decode":
        return route + 3                 # fc1, fc2, combine
    return route + 1 + 3                 # gather, fc1, fc2, combine

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
    path = qm.QMOE_PATH_AUTO
    p = qm.problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                   shape.dtype, path)
    W = [synthetic.make_torch_weights(shape, recipe, 1000 + l, device) for l in range(layers)]
    x_h, logits_h = host_inputs(shape, recipe, layers, rank)
    x_pin = torch.from_numpy(x_h.view(np.int16)).pin_memory()
    lg_pin = torch.from_numpy(logits_h.view(np.int16)).pin_memory()
    x_d = x_pin.to(device)
    lg_d = lg_pin.to(device)
    bufs = [torch.empty((shape.T, shape.H), dtype=torch.int16, device=device) for _ in range(2)]
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device=device)
    out_pin = torch.empty((shape.T, shape.H), dtype=torch.int16).pin_memory()

    def layer_io(l):
        src = x_d if l == 0 else bufs[(l - 1) % 2]
        return src, bufs[l % 2]

    def layer_args(l):
        src, dst = layer_io(l)
        w = W[l]
        return (src, lg_d[l], w["fc1_q"], w["fc1_s"], None, w["fc2_q"], w["fc2_s"], None, dst, ws)

    B1 = B2 = None
    if args.options:
        gb = torch.Generator(device=device)
        gb.manual_seed(7)
        tdt = torch.bfloat16 if shape.dtype == synthetic.BF16 else torch.float16
        B1 = [(torch.randn((shape.E, 2 * shape.inter), generator=gb, device=device) * 0.5).to(tdt)
              .view(torch.int16) for _ in range(layers)]
        B2 = [(torch.randn((shape.E, shape.H), generator=gb, device=device) * 0.5).to(tdt)
              .view(torch.int16) for _ in range(layers)]

    def step():
        for l in range(layers):
            if args.options:
                qm.qmoe_forward_ex(p, 1, B1[l], B2[l], *layer_args(l))
            else:
                qm.qmoe_forward(p, *layer_args(l))

    def stage_only(st):
        # one stage of every layer, back to back: its kernels' own durations, with no
        # timing nodes between them (the workspace holds a valid previous state)
        for l in range(layers):
            qm.qmoe_forward_stages(p, st, st, *layer_args(l))

    final = bufs[(layers - 1) % 2]
    s = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()  # eager warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    gs = []
    for st in range(4):
        gst = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gst, stream=s):
            stage_only(st)
        gs.append(gst)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        uuid = None
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(uuid, args.clock_log) as clocks:
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            marks[0].record()
            for i in range(args.steps):
                g.replay()
                marks[i + 1].record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    ms = reduce_max(marks[0].elapsed_time(marks[-1]) / args.steps, device)

    # stage durations: CUDA events on the launching stream around `steps` replays of
    # each single-stage graph (every layer's launch of that stage)
    stage_ms = np.zeros(4)
    g.replay()
    for st in range(4):
        gs[st].replay()   # warm
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record()
            for _ in range(args.steps):
                gs[st].replay()
            b.record()
        torch.cuda.synchronize()
        stage_ms[st] = a.elapsed_time(b) / (args.steps * layers)  # ms per launch of each stage

    # end to end: pinned host inputs -> device, 48 layers, result -> host, every step
    torch.cuda.synchronize()
    e2e_t0 = time.perf_counter()
    for _ in range(args.steps):
        with torch.cuda.stream(s):
            x_d.copy_(x_pin, non_blocking=True)
            lg_d.copy_(lg_pin, non_blocking=True)
            g.replay()
            out_pin.copy_(final, non_blocking=True)
        s.synchronize()
    e2e_s = reduce_max((time.perf_counter() - e2e_t0) / args.steps, device)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    tokens_per_step = shape.T * layers * world
    value = job_rate(shape.T * layers, world, ms / 1e3)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    fc1_b, fc2_b = expert_bytes(shape)
    # the captured kernels' workloads (traffic figures hold for the plain call only)
    default_kernel = args.workload in ("decode", "prefill") and not args.options
    if shape.T <= 8:
        nact = distinct_experts(logits_h, shape.dtype, shape.k)
        # the single-stage graphs run on the routing of the last layer
        bytes_fc1 = float(nact[-1]) * fc1_b
        hbm = peaks.get("hbm_gbs")
        achieved = bytes_fc1 / (stage_ms[1] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "decode fc1 dequant-GEMV + SwiGLU",
                "achieved": round(achieved, 1), "peak": hbm if hbm else 6800.0, "unit": "GB/s",
                "frac": round(achieved / (hbm if hbm else 6800.0), 4),
                "peak_source": "measured" if hbm else "fallback",
                "algorithmic_bytes_per_launch": int(bytes_fc1),
                "traffic": kernel_traffic("decode_fc1") if default_kernel else None,
                "traffic_unit": "bytes per launch (ncu)"}
        extra = {"distinct_experts_per_layer_mean": float(np.mean(nact)),
                 "fc2_GBps": round(float(nact[-1]) * fc2_b / (stage_ms[2] / 1e3) / 1e9, 1),
                 "layer_GBps": round(float(np.mean(nact)) * (fc1_b + fc2_b) / (ms / layers / 1e3) / 1e9, 1)}
    else:
        flops = 2.0 * shape.T * shape.k * (2 * shape.inter * shape.H)
        tf = peaks.get("bf16_tflops")
        achieved = flops / (stage_ms[1] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "grouped fc1 dequant-GEMM + SwiGLU (tcgen05, FP16 operands)",
                "achieved": round(achieved, 1), "peak": tf if tf else 1900.0, "unit": "TFLOP/s",
                "frac": round(achieved / (tf if tf else 1900.0), 4),
                "peak_source": "measured" if tf else "fallback", "algorithmic_flops_per_launch": flops,
                "traffic": kernel_traffic("prefill_fc1") if default_kernel else None,
                "traffic_unit": "bytes per launch (ncu)"}
        # the same launch read as a byte stream: the selected experts' fc1 codes + scales
        nact = distinct_experts(logits_h, shape.dtype, shape.k)
        extra = {"fc1_GBps": round(float(nact[-1]) * fc1_b / (stage_ms[1] / 1e3) / 1e9, 1),
                 "distinct_experts_per_layer_mean": float(np.mean(nact))}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "layer-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "ms_per_step_stats": {"median": round(float(np.median(step_ms)), 4),
                              "min": round(float(np.min(step_ms)), 4), "max": round(float(np.max(step_ms)), 4)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16-mma/fp32-acc",
        "data": "synthetic",
        "config": workload_config(args, shape, layers, world),
        "roofline": roof,
        "stage_us": {"route_group": round(stage_ms[0] * 1e3, 2), "fc1": round(stage_ms[1] * 1e3, 2),
                     "fc2": round(stage_ms[2] * 1e3, 2), "combine": round(stage_ms[3] * 1e3, 2)},
        "e2e": {"value": round(tokens_per_step / e2e_s, 1), "unit": "layer-tokens/s",
                "h2d_bytes_per_step": int(x_pin.numel() * 2 + lg_pin.numel() * 2),
                "d2h_bytes_per_step": int(out_pin.numel() * 2)},
        "gpu_launches": int(launches_per_layer(p_path(shape), shape) * layers * args.steps),
        "clocks": clocks.summary(),
        **extra,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_rate(shape, recipe, args, 0, args.cpu_sample_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    if args.options and args.impl == "reference":
        raise SystemExit("--options applies to the CUDA arm only")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
