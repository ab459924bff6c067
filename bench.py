#!/usr/bin/env python3
"""Benchmark: Q4_K decode GEMV weight-stream GB/s at 4096×4096, one token.

One step is one decode pass over `--layers` (default 64) distinct
4096×4096 Q4_K weights, each a one-token GEMV through the C ABI
(q4k_matmul): 64 × 9.44 MB = 604 MB of weights per step, 4.7× the 129 MB L2,
so no step finds its weights in L2 and no flush is needed.  The timed region
replays the step as a CUDA graph (the launches are the library's own kernels,
captured once).  `value` is whole-job weight bytes per second.

Also reported: `roofline` (the GEMV kernel against the measured HBM copy
bandwidth), `e2e` (the same step through the raw-pointer C ABI with the
activations copied in from pinned host memory and the outputs copied back,
every step, no graph), `cpu_baseline` (the CPU oracle on a bounded sample of
the same workload), `clocks` (nvidia-smi sampled during the timed region).

`--impl reference` times the CPU oracle itself on the same workload, metric
and unit (the reference arm for this build).

Multi-GPU (torchrun, one process per GPU): every rank runs its own copy of
the workload (weak scaling, no data-path collective); elapsed time is the
maximum over ranks, value = bytes of all ranks ÷ that time.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "Q4_K GEMV weight-stream GB/s and % of GB300 HBM peak at 4096×4096, batch 1"
K_DIM, N_DIM, TOKENS = 4096, 4096, 1
Q4K_ROW_BYTES = K_DIM // 256 * 144
WEIGHT_BYTES = N_DIM * Q4K_ROW_BYTES                      # 9,437,184 per GEMV
ALG_BYTES = WEIGHT_BYTES + 4 * K_DIM * TOKENS + 4 * N_DIM * TOKENS  # weights + x + y
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "q4k_gemv_t1_4096x4096.md")
KERNEL_SOURCES = [os.path.join(ROOT, "quantized_matmul_q4_gb300", "csrc", f)
                  for f in ("q4k_gemv.cu", "common.cuh", "sync.cuh")]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=64, help="distinct weights per step")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    return a


# ----------------------------------------------------------------------------
# ranks
# ----------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world: int, use_cuda: bool):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Largest `value` over all ranks (the job's elapsed time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is None:
        return
    if device is not None and device.type == "cuda":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

CLOCK_FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
                "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                "clocks_event_reasons.sw_power_cap"]
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampled every 50 ms in a background process."""

    def __init__(self, gpu_id: str):
        self.samples = []  # (host_time, sm_mhz, max_mhz, {reason: active})
        self.proc = None
        self.error = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError) as e:
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            flags = {r: parts[5 + i].lower() in ("active", "1", "yes") for i, r in enumerate(REASONS)}
            self.samples.append((time.time(), sm, mx, flags))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": f"nvidia-smi unavailable: {self.error}"}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "samples inside the timed region"
        if not inside:
            # The timed region was shorter than the sampling period: take the
            # samples nearest to it (taken while the warm-up and timed steps ran).
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            note = "timed region shorter than the sampling period: nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi samples"}
        reasons = sorted({r for s in inside for r, on in s[3].items() if on})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured (MEASURED_PEAKS.json hbm_gbs)"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback 6.8 TB/s"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources have not changed since it was captured."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None, "no ncu summary committed"
    fields = {}
    with open(PROFILE_SUMMARY) as f:
        for line in f:
            if ":" in line and not line.lstrip().startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip().strip("-* `")] = v.strip().strip("` ")
    try:
        traffic = int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None, "ncu summary has no dram_bytes_per_launch"
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return traffic, "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch"


def make_workload(layers: int, seed: int = 0):
    import synth
    g = synth.rng(seed)
    W = synth.q4k_weights(g, N_DIM * layers, K_DIM)       # layer l = rows [l·N, (l+1)·N)
    x = synth.activations(g, layers, K_DIM)               # layer l reads row l
    return W, x


def workload_config(layers: int) -> dict:
    return {"workload": f"Q4_K decode GEMV K=4096 N=4096 T=1, {layers} distinct weights per step",
            "inputDim": K_DIM, "outputDim": N_DIM, "tokens": TOKENS, "layers_per_step": layers,
            "weight_bytes_per_gemv": WEIGHT_BYTES,
            "l2": f"inputs larger than L2: {layers * WEIGHT_BYTES / 1e6:.0f} MB of weights per step",
            "weights": "random Q4_K blocks, seed 0 (synth.q4k_weights)",
            "activations": "fp32 N(0,1), seed 0"}


def cpu_baseline(W, x, layers: int, budget_s: float, rows_per_sample: int | None = None) -> dict:
    import oracle
    threads = oracle.max_threads()
    n_done, elapsed, l = 0, 0.0, 0
    rows = rows_per_sample or N_DIM
    t0 = time.perf_counter()
    while elapsed < budget_s or n_done == 0:
        Wl = W[l * N_DIM:l * N_DIM + rows]
        oracle.q4k_matmul(x[l:l + 1], Wl, K_DIM, rows)
        n_done += 1
        l = (l + 1) % layers
        elapsed = time.perf_counter() - t0
    gbs = n_done * rows * Q4K_ROW_BYTES / elapsed / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_done} one-token GEMVs of {rows}x4096 rows of the step's weights "
                      f"({elapsed:.1f} s), C oracle: fp64 dequantize-then-matmul, OpenMP over rows"}


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle
# ----------------------------------------------------------------------------

def run_reference(a) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    rows = 512  # each step: 512 output rows of one 4096×4096 layer (1.18 MB of weights)
    layers = min(a.layers, 4)
    W, x = make_workload(layers)
    oracle.build()
    threads = oracle.max_threads()

    def step(i):
        l = i % layers
        r0 = (i // layers * rows) % N_DIM
        oracle.q4k_matmul(x[l:l + 1], W[l * N_DIM + r0:l * N_DIM + r0 + rows], K_DIM, rows)

    for i in range(a.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(a.steps):
        step(a.warmup + i)
    elapsed = time.perf_counter() - t0
    gbs = a.steps * rows * Q4K_ROW_BYTES / elapsed / 1e9
    sample = (f"each step: one-token GEMV over {rows} of the 4096 rows of a 4096x4096 Q4_K weight "
              f"(C oracle, fp64, OpenMP over rows)")
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": elapsed / a.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(a.layers) | {"reference_sample": f"{rows} output rows of one "
                                                   f"of {layers} host weights per step"},
            "impl": "reference",
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(a) -> None:
    import torch
    rank, world, local = dist_env()
    if world != a.gpus:
        a.gpus = world if world > 1 else a.gpus
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, True)

    import quantized_matmul_q4_gb300 as q
    lib = q.library()

    layers = a.layers
    W_host, x_host = make_workload(layers, seed=0)
    W = torch.from_numpy(W_host.reshape(-1)).to(device)
    x = torch.from_numpy(x_host).to(device)
    y = torch.empty((layers, N_DIM), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream
    wp, xp, yp = W.data_ptr(), x.data_ptr(), y.data_ptr()

    def step_direct():
        for l in range(layers):
            rc = lib.q4k_matmul(xp + 4 * K_DIM * l, wp + WEIGHT_BYTES * l, yp + 4 * N_DIM * l,
                                K_DIM, N_DIM, TOKENS, sp)
            if rc != 0:
                raise q.Q4mmError(rc, q.last_error())

    # Warm the library (device query, kernel attributes) outside capture.
    with torch.cuda.stream(stream):
        step_direct()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        step_direct()
    stream.synchronize()

    props = torch.cuda.get_device_properties(device)
    gpu_id = str(getattr(props, "uuid", "") or local)
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            graph.replay()
    stream.synchronize()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(a.steps):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    t_host1 = time.time()
    torch.cuda.synchronize(device)
    barrier(dist, device)
    local_ms = e0.elapsed_time(e1)
    time.sleep(0.12)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    q.device_status(stream)

    elapsed_ms = max_over_ranks(local_ms, dist, device)
    ms_per_step = elapsed_ms / a.steps
    n_ranks = max(world, 1)
    value = n_ranks * layers * WEIGHT_BYTES / (ms_per_step * 1e-3) / 1e9

    peaks = measured_peaks()
    launch_s = local_ms * 1e-3 / (a.steps * layers)
    achieved = ALG_BYTES / launch_s / 1e9
    traffic, traffic_note = profiled_traffic()
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": "q4k_gemv_t1_kernel", "alg_bytes_per_launch": ALG_BYTES,
                "avg_launch_us": launch_s * 1e6, "peak_source": peaks["source"],
                "traffic_source": traffic_note}

    e2e = None
    if not a.no_e2e:
        x_pin = torch.from_numpy(x_host).pin_memory()
        y_pin = torch.empty((layers, N_DIM), dtype=torch.float32).pin_memory()
        e2e_steps = max(1, min(a.steps, 300))

        def e2e_step():
            x.copy_(x_pin, non_blocking=True)
            step_direct()
            y_pin.copy_(y, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
        stream.synchronize()
        barrier(dist, device)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            f0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            f1.record(stream)
        f1.synchronize()
        e2e_ms = max_over_ranks(f0.elapsed_time(f1), dist, device) / e2e_steps
        e2e = {"value": n_ranks * layers * WEIGHT_BYTES / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": layers * K_DIM * 4, "d2h_bytes_per_step": layers * N_DIM * 4,
               "steps": e2e_steps, "ms_per_step": e2e_ms,
               "path": "q4k_matmul C ABI per layer, activations from pinned host memory, outputs back"}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(W_host, x_host, layers, a.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": n_ranks,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i32+f32",
                "arithmetic": "fp32 activations split exactly (to 2^-21 of each 256-value block's "
                              "maximum) into three int8 planes; 4-bit codes x planes in int32 dp4a; "
                              "scales, mins and combination in fp32",
                "data": "synthetic", "config": workload_config(layers),
                "pct_of_hbm_peak": 100.0 * value / n_ranks / peaks["hbm_gbs"],
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": a.steps * layers, "clocks": clocks,
                "gpu": props.name}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main(argv=None):
    a = parse_args(argv)
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
