#!/usr/bin/env python3
"""Benchmark of the library's kernels through its C ABI, one JSON line.

Default workload (`q4k_gemv_4096x4096_t1`): Q4_K decode GEMV weight-stream
GB/s at 4096×4096, one token.  One step is one decode pass over 64 distinct
4096×4096 Q4_K weights, each a one-token GEMV (q4k_matmul): 64 × 9.44 MB =
604 MB of weights per step, 4.7× the 129 MB L2, so no step finds its weights
in L2 and no flush is needed.  `--workload` selects another of the table
below (prefill on the tensor cores or in FP32, ternary GEMV, a Llama-2-7B
decode sweep, smaller GEMVs); each is sized above L2 the same way.

The timed region replays the step as a CUDA graph (the launches are the
library's own kernels, captured once).  `value` is whole-job weight bytes
per second (GB/s workloads) or 2·K·N·T flops per second (TFLOP/s workloads).

Also reported: `roofline` (the dominant kernel against the measured HBM copy
bandwidth, the measured sustained bf16 tensor rate, or the FP32 FMA rate of
152 SMs at 2.07 GHz), `e2e` (the same step through the raw-pointer C ABI
with the activations copied in from pinned host memory and the outputs
copied back, every step, no graph), `cpu_baseline` (the CPU oracle on a
bounded sample of the same workload), `clocks` (nvidia-smi sampled during
the timed region).

`--impl reference` times the CPU oracle itself on a bounded sample of the
same workload, in the same metric and unit.

Multi-GPU (torchrun, one process per GPU): every rank runs its own copy of
the workload (weak scaling, no data-path collective); elapsed time is the
maximum over ranks, value = work of all ranks ÷ that time.
"""
from __future__ import annotations

import argparse
import dataclasses
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
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1700.0
FALLBACK_BF16_TFLOPS_BURST = 1900.0
# FP32 FMA peak: 152 SMs × 128 FP32 lanes × 2 flop per FMA × 2.07 GHz (maximum SM clock).
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
CSRC = os.path.join(ROOT, "quantized_matmul_q4_gb300", "csrc")
COMMON_SOURCES = ["common.cuh", "sync.cuh"]


@dataclasses.dataclass
class Workload:
    name: str
    kind: str                 # "q4k", "q4_0", "q4k_ffn" (gate + up, fused SwiGLU) or "ternary"
    entry: str                # C-ABI symbol called once per matrix
    mats: list                # (K, N) of each launch in one layer
    tokens: int
    layers: int               # layers per step (distinct device buffers)
    unit: str                 # "GB/s" (weight bytes) or "TFLOP/s" (2·K·N·T)
    bound: str                # roofline of the dominant kernel: "hbm", "tensor" or "alu"
    kernel: str               # dominant kernel
    metric: str
    sources: list             # kernel sources (under csrc/) hashed for the traffic record
    profile: str | None = None  # ncu summary with dram_bytes_per_launch, under profiles/
    distinct: int = 4         # distinct host-generated weights per matrix (the rest are copies)
    kernels_per_call: int = 1  # kernel launches one C-ABI call makes
    arithmetic: str = ""


def _q4k_bytes(K, N):
    return N * (K // 256) * 144


def weight_bytes(kind, K, N):
    if kind == "q4k":
        return _q4k_bytes(K, N)
    if kind == "q4_0":
        return N * (K // 32) * 18
    if kind == "q4k_ffn":
        return 2 * _q4k_bytes(K, N)
    if kind == "q4k_tc":
        return -(-N // 256) * 256 * (K // 64) * 48
    if kind == "q6k":
        return N * (K // 256) * 210
    return N * (K // 4)


T1_ARITH = ("fp32 activations rounded once per 32-value group to a multiple of 2^-23 of the power of two above "
            "the group's maximum / 255 and split into four byte planes; 4-bit codes x planes in int32 dp4a; scales, "
            "mins and combination in fp32")
LLAMA = [(4096, 4096)] * 4 + [(4096, 11008)] * 2 + [(11008, 4096)]
WORKLOADS = {w.name: w for w in [
    Workload("q4k_gemv_4096x4096_t1", "q4k", "q4k_matmul", [(4096, 4096)], 1, 64, "GB/s", "hbm",
             "gemv_t1_kernel", METRIC, ["q4k_gemv.cu", "t1_geometry.h"], "q4k_gemv_t1_4096x4096.md",
             distinct=64, arithmetic=T1_ARITH),
    Workload("q4k_gemv_8192x8192_t1", "q4k", "q4k_matmul", [(8192, 8192)], 1, 16, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K GEMV weight-stream GB/s at 8192x8192, batch 1", ["q4k_gemv.cu", "t1_geometry.h"],
             distinct=4, arithmetic=T1_ARITH),
    Workload("q4k_gemv_16384x16384_t1", "q4k", "q4k_matmul", [(16384, 16384)], 1, 4, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K GEMV weight-stream GB/s at 16384x16384, batch 1", ["q4k_gemv.cu", "t1_geometry.h"],
             distinct=1, arithmetic=T1_ARITH),
    Workload("q4k_gemv_4096x1024_t1", "q4k", "q4k_matmul", [(4096, 1024)], 1, 128, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K GEMV weight-stream GB/s at 4096->1024, batch 1",
             ["q4k_gemv.cu", "t1_geometry.h"], arithmetic=T1_ARITH),
    Workload("q4k_gemv_1024x1024_t1", "q4k", "q4k_matmul", [(1024, 1024)], 1, 512, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K GEMV weight-stream GB/s at 1024x1024, batch 1",
             ["q4k_gemv.cu", "t1_geometry.h"], arithmetic=T1_ARITH),
    Workload("q4k_prefill_tc_4096x11008_t64", "q4k", "q4k_matmul_tc", [(4096, 11008)], 64, 16,
             "TFLOP/s", "tensor", "q4k_mm_tc_kernel",
             "Q4_K prefill TFLOP/s, 64 tokens x 4096 -> 11008, tcgen05 with bf16 operands",
             ["q4k_mm_tc.cu", "cluster.cuh"], "q4k_mm_tc_4096x11008_t64.md", arithmetic="bf16 operands (dequantized in fp32, rounded once), "
                                          "fp32 accumulation in tensor memory"),
    Workload("q4k_prefill_tc_relayout_4096x11008_t64", "q4k_tc", "q4k_matmul_tc_relayouted", [(4096, 11008)],
             64, 16, "TFLOP/s", "tensor", "q4k_mm_tc_kernel",
             "Q4_K prefill TFLOP/s, 64 tokens x 4096 -> 11008, tcgen05 with bf16 operands, weights relayouted "
             "once for the tensor cores", ["q4k_mm_tc.cu", "cluster.cuh"], "q4k_mm_tc_relayout_4096x11008_t64.md",
             arithmetic="bf16 operands (dequantized in fp32 from pre-decoded fp32 sub-block scales, rounded "
                        "once), fp32 accumulation in tensor memory"),
    Workload("q4k_prefill_fp32_4096x11008_t64", "q4k", "q4k_matmul", [(4096, 11008)], 64, 16,
             "TFLOP/s", "alu", "q4k_mm_fp32_kernel",
             "Q4_K prefill TFLOP/s, 64 tokens x 4096 -> 11008, FP32 FMA", ["q4k_mm_fp32.cu", "cluster.cuh"],
             "q4k_mm_fp32_4096x11008_t64.md", arithmetic="fp32 dequantization and fp32 FMA"),
    Workload("q4_0_gemv_4096x4096_t1", "q4_0", "q4_0_gemv", [(4096, 4096)], 1, 64, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_0 GEMV weight-stream GB/s at 4096x4096, batch 1", ["q4k_gemv.cu", "t1_geometry.h"],
             "q4_0_gemv_t1_4096x4096.md", distinct=64, arithmetic=T1_ARITH),
    Workload("q6k_gemv_4096x4096_t1", "q6k", "q6k_gemv", [(4096, 4096)], 1, 48, "GB/s", "hbm",
             "gemv_t1_kernel", "Q6_K GEMV weight-stream GB/s at 4096x4096, batch 1", ["q4k_gemv.cu", "t1_geometry.h"],
             "q6k_gemv_t1_4096x4096.md", distinct=48, arithmetic=T1_ARITH.replace("4-bit", "6-bit")),
    Workload("llama7b_ffn_swiglu_t1", "q4k_ffn", "q4k_ffn_swiglu", [(4096, 11008)], 1, 32, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K fused gate+up SwiGLU weight-stream GB/s, Llama-2-7B FFN (32 layers x "
             "4096 -> 2 x 11008), batch 1", ["q4k_gemv.cu", "t1_geometry.h"], "q4k_ffn_swiglu_llama7b_t1.md", distinct=1,
             arithmetic=T1_ARITH + "; h = silu(g)*u in fp32"),
    Workload("llama7b_ffn_swiglu_t8", "q4k_ffn", "q4k_ffn_swiglu", [(4096, 11008)], 8, 32, "GB/s", "alu",
             "q4k_gemv_multi_kernel", "Q4_K fused gate+up SwiGLU weight-stream GB/s, Llama-2-7B FFN (32 layers x "
             "4096 -> 2 x 11008), 8 tokens", ["q4k_gemv_multi.cu", "multi_geometry.h"], distinct=1,
             arithmetic="fp32 dequantization and fp32 FMA; h = silu(g)*u in fp32"),
    Workload("llama7b_gate_up_t1", "q4k", "q4k_matmul", [(4096, 11008)] * 2, 1, 32, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K gate and up projections as two GEMVs, weight-stream GB/s, Llama-2-7B "
             "FFN (32 layers x 2 x 4096 -> 11008), batch 1", ["q4k_gemv.cu", "t1_geometry.h"], distinct=1, arithmetic=T1_ARITH),
    Workload("ternary_gemv_2560x6912_t1", "ternary", "ternary_gemv", [(2560, 6912)], 1, 64, "GB/s",
             "hbm", "gemv_t1_kernel", "BitNet b1.58 ternary GEMV weight-stream GB/s at 2560->6912, "
             "batch 1", ["ternary_gemv.cu", "q4k_gemv.cu", "t1_geometry.h"], "ternary_t1_2560x6912.md",
             arithmetic="fp32 activations rounded once per 32-value group to a multiple of 2^-23 of the power of "
                        "two above the group's maximum / 255 and split into four byte planes; 2-bit fields x planes "
                        "in int32 dp4a; fp32 combination, scale applied once"),
    Workload("ternary_gemv_2560x6912_t16", "ternary", "ternary_gemv", [(2560, 6912)], 16, 64, "GB/s",
             "alu", "ternary_tile_kernel", "BitNet b1.58 ternary GEMV weight-stream GB/s at 2560->6912, "
             "16 tokens", ["ternary_gemv.cu"], "ternary_tile_2560x6912_t16.md", arithmetic="fp32"),
    Workload("llama7b_decode_t1", "q4k", "q4k_matmul", LLAMA, 1, 32, "GB/s", "hbm",
             "gemv_t1_kernel", "Q4_K decode sweep weight-stream GB/s, Llama-2-7B shapes (32 layers "
             "x q,k,v,o,gate,up,down), batch 1", ["q4k_gemv.cu", "t1_geometry.h"], distinct=1, arithmetic=T1_ARITH),
    Workload("llama7b_decode_t4", "q4k", "q4k_matmul", LLAMA, 4, 32, "GB/s", "alu",
             "q4k_gemv_multi_kernel", "Q4_K decode sweep weight-stream GB/s, Llama-2-7B shapes (32 layers x "
             "q,k,v,o,gate,up,down), 4 tokens", ["q4k_gemv_multi.cu", "multi_geometry.h"], distinct=1,
             arithmetic="fp32 dequantization and fp32 FMA"),
    Workload("llama7b_decode_t16", "q4k", "q4k_matmul", LLAMA, 16, 32, "GB/s", "alu",
             "q4k_gemv_multi_kernel", "Q4_K decode sweep weight-stream GB/s, Llama-2-7B shapes (32 "
             "layers x q,k,v,o,gate,up,down), 16 tokens (two 8-token passes per matrix)",
             ["q4k_gemv_multi.cu", "multi_geometry.h"], distinct=1, arithmetic="fp32 dequantization and fp32 FMA",
             kernels_per_call=2),
    Workload("llama7b_decode_t8", "q4k", "q4k_matmul", LLAMA, 8, 32, "GB/s", "alu",
             "q4k_gemv_multi_kernel", "Q4_K decode sweep weight-stream GB/s, Llama-2-7B shapes (32 "
             "layers x q,k,v,o,gate,up,down), 8 tokens", ["q4k_gemv_multi.cu", "multi_geometry.h"], distinct=1,
             arithmetic="fp32 dequantization and fp32 FMA"),
]}
DEFAULT_WORKLOAD = "q4k_gemv_4096x4096_t1"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--layers", type=int, default=None, help="layers per step (default: the workload's)")
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
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained") or d["bf16_tflops"]),
                "source": "measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS_BURST,
            "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS,
            "source": "fallback (6.8 TB/s, 1.9 PFLOP/s bf16 burst, 1.7 sustained)"}


def kernel_source_hash(w: Workload) -> str:
    h = hashlib.sha256()
    for name in w.sources + COMMON_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_path(w: Workload):
    return os.path.join(ROOT, "profiles", w.profile) if w.profile else None


def profiled_traffic(w: Workload, path: str | None = None):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources have not changed since it was captured."""
    path = path or profile_path(w)
    if not path or not os.path.exists(path):
        return None, "no ncu traffic record committed for this kernel"
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.lstrip().startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip().strip("-* `")] = v.strip().strip("` ")
    try:
        traffic = int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None, "ncu summary has no dram_bytes_per_launch"
    if fields.get("kernel_source_sha256") != kernel_source_hash(w):
        return None, "kernel changed since the ncu capture"
    return traffic, "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch"


class Plan:
    """The launches of one step: per layer, one C-ABI call per matrix, each
    with its own weight, activation and output buffers."""

    def __init__(self, w: Workload, layers: int):
        self.w, self.layers, self.T = w, layers, w.tokens
        self.launches = []  # (K, N, w_off, x_off, y_off, mat index)
        wo = xo = yo = 0
        for _ in range(layers):
            for m, (K, N) in enumerate(w.mats):
                self.launches.append((K, N, wo, xo, yo, m))
                wo += -(-weight_bytes(w.kind, K, N) // 256) * 256
                xo += self.T * K
                yo += self.T * N
        self.w_total, self.x_total, self.y_total = wo, xo, yo
        self.weight_bytes = sum(weight_bytes(w.kind, K, N) for K, N, *_ in self.launches)
        self.alg_bytes = sum(weight_bytes(w.kind, K, N) + 4 * self.T * (K + N)
                             for K, N, *_ in self.launches)
        self.flops = sum(2.0 * K * N * self.T for K, N, *_ in self.launches)

    def per_step(self) -> float:
        """The metric's numerator for one step."""
        return self.weight_bytes / 1e9 if self.w.unit == "GB/s" else self.flops / 1e12


def host_inputs(w: Workload, seed: int = 0):
    """Per matrix: `distinct` host weights, one activation [T, K] and (ternary) a scale."""
    import synth
    g = synth.rng(seed)
    mats = []
    for K, N in w.mats:
        n = max(1, w.distinct)
        if w.kind in ("q4k", "q4k_tc"):
            Ws = [synth.q4k_weights(g, N, K) for _ in range(n)]
        elif w.kind == "q4_0":
            Ws = [synth.q4_0_weights(g, N, K) for _ in range(n)]
        elif w.kind == "q6k":
            Ws = [synth.q6k_weights(g, N, K) for _ in range(n)]
        elif w.kind == "q4k_ffn":
            import numpy as np
            Ws = [np.concatenate([synth.q4k_weights(g, N, K).reshape(-1), synth.q4k_weights(g, N, K).reshape(-1)])
                  for _ in range(n)]
        else:
            Ws = [synth.ternary_weights(g, N, K) for _ in range(n)]
        scale = float(synth.ternary_scale(g)) if w.kind == "ternary" else 1.0
        x = synth.activations(g, w.tokens, K)
        mats.append((Ws, x, scale))
    return mats


def workload_config(w: Workload, plan: Plan) -> dict:
    return {"workload": w.name, "entry": w.entry, "format": w.kind,
            "matrices_per_layer": [{"inputDim": K, "outputDim": N} for K, N in w.mats],
            "tokens": w.tokens, "layers_per_step": plan.layers, "launches_per_step": len(plan.launches),
            "weight_bytes_per_step": plan.weight_bytes,
            "l2": f"inputs larger than L2: {plan.weight_bytes / 1e6:.0f} MB of weights per step "
                  f"(L2 129 MB), no flush",
            "weights": f"random {dict(q4k='Q4_K blocks', q4_0='Q4_0 blocks', q4k_ffn='Q4_K blocks (gate, up)', q6k='Q6_K blocks', q4k_tc='Q4_K blocks relayouted once on the GPU by q4k_relayout_tc (not timed)').get(w.kind, 'ternary codes')}, seed 0 "
                       f"(synth), {w.distinct} distinct host copies per matrix",
            "activations": "fp32 N(0,1), seed 0"}


def oracle_call(w: Workload, K, N, W, x, scale, rows, r0=0):
    import oracle
    if w.kind in ("q4k", "q4k_tc"):
        # The relayouted weight is the same matrix: the oracle takes the
        # canonical blocks it was made from.
        oracle.q4k_matmul(x, W.reshape(N, -1)[r0:r0 + rows], K, rows)
    elif w.kind == "q4_0":
        oracle.q4_0_matmul(x, W.reshape(N, -1)[r0:r0 + rows], K, rows)
    elif w.kind == "q6k":
        oracle.q6k_matmul(x, W.reshape(N, -1)[r0:r0 + rows], K, rows)
    elif w.kind == "q4k_ffn":
        Wg, Wu = W.reshape(2, N, -1)
        oracle.q4k_ffn_swiglu(x, Wg[r0:r0 + rows], Wu[r0:r0 + rows], K, rows)
    else:
        oracle.ternary_gemv(x, W.reshape(N, -1)[r0:r0 + rows], scale, K, rows)


def oracle_rows(w: Workload) -> int:
    """Output rows per oracle call: about 0.1–0.5 s of CPU work each."""
    K, N = w.mats[0]
    return max(8, min(N, int(4e8 // (K * w.tokens))))


def oracle_unit_value(w: Workload, K, rows, calls, elapsed) -> float:
    if w.unit == "GB/s":
        return calls * weight_bytes(w.kind, K, rows) / elapsed / 1e9
    return calls * 2.0 * K * rows * w.tokens / elapsed / 1e12


def cpu_baseline(w: Workload, mats, budget_s: float) -> dict:
    import oracle
    threads = oracle.max_threads()
    K, N = w.mats[0]
    Ws, x, scale = mats[0]
    rows = oracle_rows(w)
    n_done, elapsed = 0, 0.0
    t0 = time.perf_counter()
    while elapsed < budget_s or n_done == 0:
        oracle_call(w, K, N, Ws[n_done % len(Ws)], x, scale, rows, (n_done * rows) % (N - rows + 1))
        n_done += 1
        elapsed = time.perf_counter() - t0
    return {"value": oracle_unit_value(w, K, rows, n_done, elapsed), "unit": w.unit, "cores": threads,
            "kind": "oracle",
            "sample": f"{n_done} calls of {w.tokens} token(s) x {K} -> {rows} rows of the workload's "
                      f"first matrix ({elapsed:.1f} s); C oracle, fp64, OpenMP over rows"}


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle
# ----------------------------------------------------------------------------

def run_reference(a) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = WORKLOADS[a.workload]
    w = dataclasses.replace(w, distinct=min(w.distinct, 2))
    plan = Plan(w, a.layers or w.layers)
    mats = host_inputs(w)
    oracle.build()
    threads = oracle.max_threads()
    K, N = w.mats[0]
    rows = oracle_rows(w)

    def step(i):
        Ws, x, scale = mats[0]
        oracle_call(w, K, N, Ws[i % len(Ws)], x, scale, rows, (i * rows) % (N - rows + 1))

    for i in range(a.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(a.steps):
        step(a.warmup + i)
    elapsed = time.perf_counter() - t0
    value = oracle_unit_value(w, K, rows, a.steps, elapsed)
    sample = (f"each step: {w.tokens} token(s) x {K} -> {rows} of the {N} output rows of the "
              f"workload's first matrix (C oracle, fp64, OpenMP over rows)")
    line = {"metric": w.metric, "value": value, "unit": w.unit, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": elapsed / a.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, plan) | {"reference_sample": sample},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": w.unit, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": w.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
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
    w = WORKLOADS[a.workload]
    fn = getattr(lib, w.entry)
    plan = Plan(w, a.layers or w.layers)
    mats = host_inputs(w, seed=0)
    W = torch.empty(plan.w_total, dtype=torch.uint8, device=device)
    x = torch.empty(plan.x_total, dtype=torch.float32, device=device)
    y = torch.empty(plan.y_total, dtype=torch.float32, device=device)
    x_host = torch.empty(plan.x_total, dtype=torch.float32)
    seen = {}
    for li, (K, N, wo, xo, yo, m) in enumerate(plan.launches):
        Ws, xm, _ = mats[m]
        nb = weight_bytes(w.kind, K, N)
        k = seen.get(m, 0)
        seen[m] = k + 1
        if w.kind == "q4k_tc":
            # The one-time relayout, on the GPU, before anything is timed.
            canon = torch.from_numpy(Ws[k % len(Ws)].reshape(-1)).to(device)
            q.q4k_relayout_tc_ptr(canon.data_ptr(), W.data_ptr() + wo, K, N, 0)
            torch.cuda.synchronize(device)
            del canon
        else:
            W[wo:wo + nb].copy_(torch.from_numpy(Ws[k % len(Ws)].reshape(-1)))
        x_host[xo:xo + w.tokens * K] = torch.from_numpy(xm.reshape(-1))
    x.copy_(x_host)
    torch.cuda.synchronize(device)
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream
    wp, xp, yp = W.data_ptr(), x.data_ptr(), y.data_ptr()
    calls = []
    for K, N, wo, xo, yo, m in plan.launches:
        if w.kind == "q4k_ffn":
            calls.append((xp + 4 * xo, wp + wo, wp + wo + _q4k_bytes(K, N), yp + 4 * yo, K, N, w.tokens, sp))
        elif w.kind != "ternary":
            calls.append((xp + 4 * xo, wp + wo, yp + 4 * yo, K, N, w.tokens, sp))
        else:
            calls.append((xp + 4 * xo, wp + wo, mats[m][2], yp + 4 * yo, K, N, w.tokens, sp))

    def step_direct():
        for c in calls:
            rc = fn(*c)
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
    value = n_ranks * plan.per_step() / (ms_per_step * 1e-3)

    # Roofline of the dominant kernel, from this rank's own device time.
    peaks = measured_peaks()
    step_s = local_ms * 1e-3 / a.steps
    launch_s = step_s / len(plan.launches)
    hbm_achieved = plan.alg_bytes / step_s / 1e9
    traffic, traffic_note = profiled_traffic(w) if (a.layers is None or a.layers == w.layers) \
        else (None, "non-default layer count")
    if w.bound == "hbm":
        roofline = {"bound": "hbm", "achieved": hbm_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": hbm_achieved / peaks["hbm_gbs"], "peak_source": peaks["source"] + " hbm_gbs"}
    else:
        tflops = plan.flops / step_s / 1e12
        # A tensor-core kernel is held to the burst cuBLAS rate (the higher
        # of the two measured figures); the sustained rate is reported beside it.
        peak = peaks["bf16_tflops"] if w.bound == "tensor" else FP32_FMA_TFLOPS
        src = (peaks["source"] + " bf16_tflops (burst)" if w.bound == "tensor" else
               "derived: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz")
        roofline = {"bound": w.bound, "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                    "frac": tflops / peak, "peak_source": src,
                    **({"frac_of_sustained": tflops / peaks["bf16_tflops_sustained"]} if w.bound == "tensor" else {}),
                    "hbm": {"achieved": hbm_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": hbm_achieved / peaks["hbm_gbs"]}}
    roofline.update({"traffic": traffic, "kernel": w.kernel,
                     "alg_bytes_per_launch": plan.alg_bytes / len(plan.launches),
                     "avg_launch_us": launch_s * 1e6, "traffic_source": traffic_note})

    e2e = None
    if not a.no_e2e:
        x_pin = x_host.pin_memory()
        y_pin = torch.empty(plan.y_total, dtype=torch.float32).pin_memory()
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
        e2e = {"value": n_ranks * plan.per_step() / (e2e_ms * 1e-3), "unit": w.unit,
               "h2d_bytes_per_step": plan.x_total * 4, "d2h_bytes_per_step": plan.y_total * 4,
               "steps": e2e_steps, "ms_per_step": e2e_ms,
               "path": f"{w.entry} C ABI per matrix, activations from pinned host memory, outputs back"}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(w, mats, a.cpu_seconds)

    if rank == 0:
        dtype = {"hbm": "i32+f32" if "dp4a" in w.arithmetic else "f32", "tensor": "bf16",
                 "alu": "f32"}[w.bound]
        line = {"metric": w.metric, "value": value, "unit": w.unit, "n_gpus": n_ranks,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
                "arithmetic": w.arithmetic, "data": "synthetic", "config": workload_config(w, plan),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": a.steps * len(plan.launches) * w.kernels_per_call, "clocks": clocks,
                "gpu": props.name}
        if w.unit == "GB/s":
            line["pct_of_hbm_peak"] = 100.0 * value / n_ranks / peaks["hbm_gbs"]
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
