#!/usr/bin/env python
"""Throughput of the routed-expert Q4_K MoE FFN layer on GB300.

One step is one pass of the layer (router -> permutation -> gate/up+SwiGLU
-> down -> slot-ordered combine) over every layer of a rotation of
independently seeded layers, i.e. `layers` calls of moe_layer with T tokens
each.  The rotation's weights (48 x 340 MB for the Qwen3-30B-A3B shape) are
far larger than L2, and consecutive uses of one layer are separated by every
other layer's traffic, so no L2 flush is needed.

Prints one JSON line (rank 0).  `value` is MoE-FFN tokens per second through
one layer (T * layers_per_step * steps / time, summed over ranks); the
roofline object compares the achieved algorithmic bytes per call (unique
selected experts' Q4_K bytes + x + y + idx + w) with the measured HBM copy
bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from quantized_routed_expert_02_gb300 import synth  # noqa: E402

DEFAULT_CONFIG = "a3b_decode"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.SHAPES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the rotation length")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="bound on the oracle's CPU-baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------- ranks

def max_over_ranks(value, dist=None, device="cpu"):
    """The largest `value` over all ranks (every rank receives it); the value
    itself without a process group."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Units per second of the whole job: each of `world` replicas processed
    `units_per_rank`, and the job took the slowest rank's `seconds`."""
    return units_per_rank * world / seconds


# ---------------------------------------------------------------- inputs

def _gen_layer(job):
    name, layer, rank = job
    shape = synth.SHAPES[name]
    blobs = synth.expert_blobs(shape, layer)
    Wr = synth.router_weights(shape, layer)
    x = synth.activations_fast(shape, layer + 7919 * rank)
    return layer, x, Wr, blobs


def generate(name, n_layers, rank, workers):
    import multiprocessing as mp
    jobs = [(name, layer, rank) for layer in range(n_layers)]
    if workers <= 1 or n_layers == 1:
        for j in jobs:
            yield _gen_layer(j)
        return
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        for r in pool.imap(_gen_layer, jobs):
            yield r


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 20 ms, each tagged with the host clock when
    read, so the ones inside the timed region can be picked out."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.rows = []
        self.thread = None

    def _reader(self):
        for line in self.proc.stdout:
            self.rows.append((time.perf_counter(), line.strip().split(",")))

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        # a region shorter than the sampling period: take the samples nearest to it
        near = inside or [r for t, r in self.rows if t0 - 0.1 <= t <= t1 + 0.1]
        sm, smax, reasons = [], None, set()
        for r in near:
            try:
                sm.append(float(r[0]))
                smax = float(r[1])
                for nm, v in zip(self.NAMES, r[4:8]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_inside_timed_region": len(inside)}


def profiled_traffic(kernel_src, profile):
    """DRAM bytes per launch recorded by the ncu summary in profiles/, if that
    summary was taken of the kernel source as it is now (hash match)."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, kernel_src), "rb").read()
        text = open(os.path.join(ROOT, "profiles", profile)).read()
    except OSError:
        return None
    h = hashlib.sha256(src).hexdigest()[:16]
    fields = dict(ln.split(":", 1) for ln in text.splitlines() if ":" in ln and not ln.startswith(" "))
    if fields.get("source-sha256-16", "").strip() != h:
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


def measured_peaks():
    """(HBM GB/s, sustained dense bf16 TFLOP/s, kind) from MEASURED_PEAKS.json,
    else the recipe's fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1700.0, "fallback"


# ---------------------------------------------------------------- oracle (CPU) timing

def oracle_sample(name, seconds, layers_available, rank=0):
    """Time the fp64 oracle on whole layer calls of the workload until
    `seconds` of CPU time have been spent (at least one call)."""
    from oracle.oracle import Oracle
    shape = synth.SHAPES[name]
    o = Oracle()
    calls, t_total, layer = 0, 0.0, 0
    T = shape.T
    tokens = None
    if T > 64:
        # prefill: a bounded token subset of one layer per call
        tokens = np.arange(0, T, max(1, T // 64), dtype=np.int32)[:64]
    while True:
        _, x, Wr, blobs = _gen_layer((name, layer % max(1, layers_available), rank))
        bias = synth.router_bias(shape)
        t0 = time.perf_counter()
        r = o.router(x, Wr, bias, shape.k)
        o.ffn(x, r["idx"], r["w"], blobs["gate"], blobs["up"], blobs["down"], shape.E, shape.I,
              tokens=tokens)
        t_total += time.perf_counter() - t0
        calls += 1
        layer += 1
        if t_total >= seconds:
            break
    ntok = T if tokens is None else len(tokens)
    threads = min(o.max_threads(), ntok)
    return {
        "value": ntok * calls / t_total,
        "unit": "tokens/s",
        "cores": threads,
        "kind": "oracle",
        "sample": (f"{calls} layer call(s) of {name} (T={T}"
                   + (f", FFN on {ntok} of {T} tokens, router on all" if tokens is not None else "")
                   + f"), fp64 C oracle, {t_total:.1f} s"),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return
    shape = synth.SHAPES[args.config]
    times = []
    last = None
    for step in range(args.warmup + args.steps):
        last = oracle_sample(args.config, 0.0, 1, 0)
        if step >= args.warmup:
            times.append(last["value"])
    value = statistics.median(times)
    line = {
        "impl": "reference", "metric": "MoE FFN tokens/s (one layer)", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.config, "T": shape.T, "H": shape.H, "E": shape.E,
                   "k": shape.k, "I": shape.I},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": last["cores"],
                         "kind": "oracle", "sample": "each step: " + last["sample"]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    shape = synth.SHAPES[args.config]
    n_layers = args.layers or shape.layers
    workers = max(1, min(16, (os.cpu_count() or 2) // max(1, world)))

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from quantized_routed_expert_02_gb300 import moeq4k as m

    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    layers = []
    t_gen = time.perf_counter()
    for layer, x, Wr, blobs in generate(args.config, n_layers, rank, workers):
        L = dict(
            x=torch.from_numpy(x).to(dev),
            x_host=torch.from_numpy(x).pin_memory(),
            Wr=torch.from_numpy(Wr).to(dev),
            gate=torch.from_numpy(blobs["gate"]).to(dev),
            up=torch.from_numpy(blobs["up"]).to(dev),
            down=torch.from_numpy(blobs["down"]).to(dev),
            idx=torch.empty(T, k, dtype=torch.int32, device=dev),
            w=torch.empty(T, k, dtype=torch.float32, device=dev),
            y=torch.empty(T, H, dtype=torch.float32, device=dev),
        )
        layers.append(L)
        del blobs
    t_gen = time.perf_counter() - t_gen
    b = synth.router_bias(shape)
    bias = None if b is None else torch.from_numpy(b).to(dev)
    ws = m.alloc_workspace(T, H, E, k, I, device=dev)
    ws_host = m.alloc_workspace(T, H, E, k, I, device=dev, host_staging=True)
    y_host = torch.empty(T, H, dtype=torch.float32).pin_memory()

    stream = torch.cuda.Stream(device=dev)

    def one_step(s):
        for L in layers:
            m.moe_layer(L["x"], L["Wr"], bias, L["gate"], L["up"], L["down"], k, I,
                        L["idx"], L["w"], L["y"], ws, stream=s)

    # eager warm-up, then capture one step (the whole rotation) as a CUDA graph
    with torch.cuda.stream(stream):
        one_step(stream)
    stream.synchronize()
    code, detail = m.moe_read_device_status(ws, stream)
    if code != 0:
        raise RuntimeError(f"device status {m.status_str(code)} ({detail})")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        one_step(stream)

    # CUDAGraph.replay() launches on the current stream: make it `stream`
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            graph.replay()
    torch.cuda.synchronize()

    # algorithmic bytes of one step, from the routing each call made
    per_expert = 2 * shape.gate_bytes + shape.down_bytes
    act_bytes = T * H * 4 * 2 + T * k * 8
    step_bytes = 0
    uniques = []
    for L in layers:
        u = int(torch.unique(L["idx"]).numel())
        uniques.append(u)
        step_bytes += u * per_expert + act_bytes
    wr_bytes = n_layers * E * H * 4

    gpu_id = 0
    try:
        props = torch.cuda.get_device_properties(dev)
        gpu_id = str(props.uuid)
        if not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = str(local_rank)
    clocks = ClockSampler(gpu_id)

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_region0 = time.perf_counter()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t_region1 = time.perf_counter()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop(t_region0, t_region1)
    code, detail = m.moe_read_device_status(ws, stream)
    if code != 0:  # a device-side error or time-out inside the timed region voids the number
        raise RuntimeError(f"device status after the timed region: {m.status_str(code)} ({detail})")
    ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    ms_per_step = ms / args.steps
    tokens_per_step = T * n_layers
    value = whole_job_rate(tokens_per_step * args.steps, world, ms / 1e3)

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(1, min(args.steps, 10))
        for L in layers[:2]:
            m.moe_layer_host(L["x_host"], L["Wr"], bias, L["gate"], L["up"], L["down"], k, I,
                             L["idx"], L["w"], y_host, ws_host, stream=stream)
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            for L in layers:
                m.moe_layer_host(L["x_host"], L["Wr"], bias, L["gate"], L["up"], L["down"], k, I,
                                 L["idx"], L["w"], y_host, ws_host, stream=stream)
        dt = max_over_ranks(time.perf_counter() - t0, dist, dev)
        e2e = {"value": whole_job_rate(T * n_layers * e2e_steps, world, dt), "unit": "tokens/s",
               "h2d_bytes_per_step": n_layers * T * H * 4,
               "d2h_bytes_per_step": n_layers * T * H * 4}

    peak, tflops_peak, peak_kind = measured_peaks()
    call_us = ms_per_step * 1e3 / n_layers
    achieved = (step_bytes / n_layers) / (call_us * 1e-6) / 1e9
    single = m.moe_layer_launch_count(T, H, E, k, I) == 1
    traffic = profiled_traffic("quantized_routed_expert_02_gb300/csrc/decode_fused.cu",
                               "decode_fused_a3b_decode.md") if (single and args.config == "a3b_decode") else None
    # The tensor-core path (T*k >= 256 routed slots) is a dense contraction: its roofline is
    # the slower of the bytes at HBM peak and the FLOPs at the tensor peak
    # (fp16 operands; the dense fp16 and bf16 peaks are equal on this part).
    flops_per_call = 6.0 * T * k * H * I
    tensor_path = T * k >= 256
    hbm_floor_us = (step_bytes / n_layers) / (peak * 1e9) * 1e6
    tensor_floor_us = flops_per_call / (tflops_peak * 1e12) * 1e6
    if tensor_path and tensor_floor_us > hbm_floor_us:
        tf = flops_per_call / (call_us * 1e-6) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tf, 1), "peak": tflops_peak,
                    "unit": "TFLOP/s", "frac": round(tf / tflops_peak, 4), "traffic": None,
                    "hbm_frac": round(achieved / peak, 4)}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": traffic}
    roofline.update({
        "kernel": ("decode_fused_kernel (the only launch of a call; duration = timed region / calls)"
                   if single else "moe_layer call (all launches of one call)"),
        "peak_kind": peak_kind + (" (sustained bf16 GEMM)" if roofline["bound"] == "tensor" else ""),
        "algorithmic_bytes_per_call": step_bytes / n_layers,
        "flops_per_call": flops_per_call,
        "achieved_incl_router_weight": round(
            ((step_bytes + wr_bytes) / n_layers) / (call_us * 1e-6) / 1e9, 1),
    })

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_sample(args.config, args.cpu_seconds, n_layers, rank)

    launches = m.moe_layer_launch_count(T, H, E, k, I) * n_layers * args.steps
    if rank == 0:
        line = {
            "metric": "MoE FFN tokens/s (one layer)",
            "value": round(value, 1),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "us_per_layer_call": round(call_us, 3),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16xf16->f32" if tensor_path else "f32",
            "data": "synthetic",
            "config": {
                "workload": args.config, "T": T, "H": H, "E": E, "k": k, "I": I,
                "layers_per_step": n_layers, "weights": "Q4_K",
                "unique_experts_per_call": round(sum(uniques) / len(uniques), 2),
                "l2": "inputs larger than L2 (layer rotation, no flush)",
                "parallelism": f"replicas x{world}",
                "graph": "one CUDA graph per step",
                "input_gen_s": round(t_gen, 1),
            },
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
