"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random bytes and floats with numpy's PCG64
(``numpy.random.default_rng(seed)``).  It holds none of the matmul's
arithmetic: no dequantization, no decoding, no dot products.  Both the CUDA
path and the CPU oracle consume what it returns, unchanged.

Q4_K weights are drawn as raw block bytes in the canonical field order
(fp16 d, fp16 dmin, 12 scale bytes, 128 qs bytes).  Uniform random scale and
qs bytes give exactly the distribution the workloads call for: the 12-byte
6-bit packing is a bijection between 96 bits and eight 6-bit scales plus eight
6-bit mins, so uniform bytes mean every scale and min is uniform on 0..63 and
independent, and uniform qs bytes mean every 4-bit code is uniform on 0..15.
d ~ U[1e-3, 1e-2] and dmin ~ U[0, 1e-2] are rounded to fp16 by numpy.

Q4_0 weights are 18-byte blocks: fp16 d ~ U[1e-3, 1e-2] and 16 uniform qs
bytes (every 4-bit code uniform on 0..15).

Q6_K blocks are uniform bytes (uniform 6-bit codes and signed 8-bit scales)
with fp16 d ~ U[1e-3, 1e-2] in their last two bytes.

Ternary weights are drawn uniformly from the 81 byte values whose four 2-bit
fields are all 0, 1 or 2 — the same as drawing each code uniformly from
{-1, 0, +1} independently.
"""
from __future__ import annotations

import numpy as np

Q4K_VALUES = 256
Q4K_BYTES = 144


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def q4k_weights(g: np.random.Generator, N: int, K: int,
                d_range=(1e-3, 1e-2), dmin_range=(0.0, 1e-2)) -> np.ndarray:
    """Random Q4_K weight: uint8 [N, K/256·144], rows of contiguous blocks."""
    assert K % Q4K_VALUES == 0 and K > 0 and N > 0
    nb = K // Q4K_VALUES
    d = g.uniform(d_range[0], d_range[1], size=(N, nb)).astype("<f2")
    dmin = g.uniform(dmin_range[0], dmin_range[1], size=(N, nb)).astype("<f2")
    scales = g.integers(0, 256, size=(N, nb, 12), dtype=np.uint8)
    qs = g.integers(0, 256, size=(N, nb, 128), dtype=np.uint8)
    blocks = np.empty((N, nb, Q4K_BYTES), np.uint8)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:4] = dmin.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 4:16] = scales
    blocks[:, :, 16:144] = qs
    return blocks.reshape(N, nb * Q4K_BYTES)


Q40_VALUES = 32
Q40_BYTES = 18


def q4_0_weights(g: np.random.Generator, N: int, K: int, d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Random Q4_0 weight: uint8 [N, K/32·18], rows of contiguous 18-byte
    blocks (fp16 d ~ U[1e-3, 1e-2], then 16 uniform qs bytes)."""
    assert K % Q40_VALUES == 0 and K > 0 and N > 0
    nb = K // Q40_VALUES
    d = g.uniform(d_range[0], d_range[1], size=(N, nb)).astype("<f2")
    qs = g.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    blocks = np.empty((N, nb, Q40_BYTES), np.uint8)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:18] = qs
    return blocks.reshape(N, nb * Q40_BYTES)


Q6K_BYTES = 210


def q6k_weights(g: np.random.Generator, N: int, K: int, d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Random Q6_K weight: uint8 [N, K/256·210]: uniform ql and qh bytes
    (every 6-bit code uniform on 0..63), uniform signed scale bytes, fp16
    d ~ U[1e-3, 1e-2] in the last two bytes of each block."""
    assert K % Q4K_VALUES == 0 and K > 0 and N > 0
    nb = K // Q4K_VALUES
    blocks = g.integers(0, 256, size=(N, nb, Q6K_BYTES), dtype=np.uint8)
    d = g.uniform(d_range[0], d_range[1], size=(N, nb)).astype("<f2")
    blocks[:, :, 208:210] = d.view(np.uint8).reshape(N, nb, 2)
    return blocks.reshape(N, nb * Q6K_BYTES)


def _valid_ternary_bytes() -> np.ndarray:
    """Byte values whose four 2-bit fields each hold 0, 1 or 2 (81 of them)."""
    vals = [b for b in range(256) if all(((b >> (2 * i)) & 3) != 3 for i in range(4))]
    return np.array(vals, np.uint8)


_TERNARY_BYTES = _valid_ternary_bytes()


def ternary_weights(g: np.random.Generator, N: int, K: int) -> np.ndarray:
    """Random BitNet b1.58 weight: uint8 [N, K/4], codes uniform on {-1, 0, +1}."""
    assert K % 4 == 0 and K > 0 and N > 0
    idx = g.integers(0, _TERNARY_BYTES.size, size=(N, K // 4))
    return _TERNARY_BYTES[idx]


def ternary_scale(g: np.random.Generator) -> np.float32:
    return np.float32(g.uniform(0.5, 2.0))


def activations(g: np.random.Generator, T: int, K: int, kind: str = "normal") -> np.ndarray:
    """fp32 activations [T, K]: N(0, 1), or integers uniform on [-8, 8]."""
    if kind == "normal":
        return g.standard_normal((T, K), dtype=np.float32)
    if kind == "int":
        return g.integers(-8, 9, size=(T, K)).astype(np.float32)
    raise ValueError(kind)


# The workloads, by what they are.  Every one is drawn with seed 0, weight
# first, then (ternary) the scale, then activations.
WORKLOADS = {
    "q4k_gemv_1024x1024_t1": dict(kind="q4k", K=1024, N=1024, T=1),
    "q4k_gemv_4096x1024_t1": dict(kind="q4k", K=4096, N=1024, T=1),
    "q4k_gemv_4096x4096_t1": dict(kind="q4k", K=4096, N=4096, T=1),
    "q4k_prefill_4096x11008_t64": dict(kind="q4k", K=4096, N=11008, T=64),
    "q4_0_gemv_4096x4096_t1": dict(kind="q4_0", K=4096, N=4096, T=1),
    "q6k_gemv_4096x4096_t1": dict(kind="q6k", K=4096, N=4096, T=1),
    "ternary_gemv_2560x6912_t1": dict(kind="ternary", K=2560, N=6912, T=1),
    "ternary_gemv_2560x6912_t16": dict(kind="ternary", K=2560, N=6912, T=16),
}

# One Llama-2-7B transformer layer's Q4_K linear weights as (K, N) pairs:
# q, k, v, o are 4096→4096, gate and up 4096→11008, down 11008→4096.
LLAMA7B_LAYER = [(4096, 4096)] * 4 + [(4096, 11008)] * 2 + [(11008, 4096)]
LLAMA7B_LAYERS = 32


def q4k_case(name_or_dims, seed: int = 0, xkind: str = "normal"):
    """(x, W, K, N, T) for a named workload or a (K, N, T) tuple."""
    if isinstance(name_or_dims, str):
        w = WORKLOADS[name_or_dims]
        K, N, T = w["K"], w["N"], w["T"]
    else:
        K, N, T = name_or_dims
    g = rng(seed)
    W = q4k_weights(g, N, K)
    x = activations(g, T, K, xkind)
    return x, W, K, N, T


def ternary_case(name_or_dims, seed: int = 0, xkind: str = "normal"):
    """(x, W, scale, K, N, T) for a named workload or a (K, N, T) tuple."""
    if isinstance(name_or_dims, str):
        w = WORKLOADS[name_or_dims]
        K, N, T = w["K"], w["N"], w["T"]
    else:
        K, N, T = name_or_dims
    g = rng(seed)
    W = ternary_weights(g, N, K)
    scale = ternary_scale(g)
    x = activations(g, T, K, xkind)
    return x, W, scale, K, N, T


def q4_0_case(name_or_dims, seed: int = 0, xkind: str = "normal"):
    """(x, W, K, N, T) with a Q4_0 weight, for a named workload or (K, N, T)."""
    if isinstance(name_or_dims, str):
        w = WORKLOADS[name_or_dims]
        K, N, T = w["K"], w["N"], w["T"]
    else:
        K, N, T = name_or_dims
    g = rng(seed)
    W = q4_0_weights(g, N, K)
    x = activations(g, T, K, xkind)
    return x, W, K, N, T


def q6k_case(name_or_dims, seed: int = 0, xkind: str = "normal"):
    """(x, W, K, N, T) with a Q6_K weight, for a named workload or (K, N, T)."""
    if isinstance(name_or_dims, str):
        w = WORKLOADS[name_or_dims]
        K, N, T = w["K"], w["N"], w["T"]
    else:
        K, N, T = name_or_dims
    g = rng(seed)
    W = q6k_weights(g, N, K)
    x = activations(g, T, K, xkind)
    return x, W, K, N, T
