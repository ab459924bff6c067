"""CPU oracle for the Q4_K and BitNet b1.58 ternary x·Wᵀ products.

TEST INFRASTRUCTURE ONLY.  The oracle is the checker the CUDA path is compared
against; it is not part of the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import it.  It shares no code with ``quantized_matmul_q4_gb300`` and never
imports it.

The arithmetic lives in ``q4mm_oracle.c`` (plain C, double precision, built
with gcc -O2 and no fast-math); this module only builds it, loads it with
ctypes and marshals numpy arrays.  See the C file's header for the passages
of the pages each function follows.

Pins (what checks the oracle against something other than itself) are in
``tests/test_oracle_pins.py``: a hand-worked block, closed forms, special
cases, the lazy-dmin identity, integer counts for the ternary code-dot, an
exact-rational brute force, and planted mistakes that the pins must catch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4mm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None

Q4K_VALUES = 256
Q4K_BYTES = 144


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library and declare its symbols."""
    global _LIB
    if path is None and _LIB is not None:
        return _LIB
    with _LOCK:
        if path is None and _LIB is not None:
            return _LIB
        lib = ctypes.CDLL(path or build())
        i64, i32, dbl, flt = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
        vp = ctypes.c_void_p
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = dbl
        lib.oracle_round_bf16.argtypes = [flt]
        lib.oracle_round_bf16.restype = flt
        lib.oracle_q4k_dequant_block.argtypes = [vp, vp]
        lib.oracle_q4k_dequant_block.restype = None
        lib.oracle_q4k_dequant.argtypes = [vp, i64, i64, vp]
        lib.oracle_q4k_dequant.restype = i32
        lib.oracle_q4k_tc_bytes.argtypes = [i64, i64]
        lib.oracle_q4k_tc_bytes.restype = i64
        lib.oracle_q4k_tc_relayout.argtypes = [vp, i64, i64, vp]
        lib.oracle_q4k_tc_relayout.restype = i32
        lib.oracle_q4k_tc_dequant.argtypes = [vp, i64, i64, vp]
        lib.oracle_q4k_tc_dequant.restype = i32
        for name in ("oracle_q4k_matmul", "oracle_q4k_matmul_bf16", "oracle_q4k_matmul_lazy"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, i64, i64, i64, vp, i32]
            fn.restype = i32
        lib.oracle_q4k_ffn_swiglu.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, i32]
        lib.oracle_q4k_ffn_swiglu.restype = i32
        lib.oracle_q6k_dequant_block.argtypes = [vp, vp]
        lib.oracle_q6k_dequant_block.restype = None
        lib.oracle_q6k_dequant.argtypes = [vp, i64, i64, vp]
        lib.oracle_q6k_dequant.restype = i32
        lib.oracle_q6k_matmul.argtypes = [vp, vp, i64, i64, i64, vp, i32]
        lib.oracle_q6k_matmul.restype = i32
        lib.oracle_q6k_pack_block.argtypes = [ctypes.c_uint16, vp, vp, vp]
        lib.oracle_q6k_pack_block.restype = None
        lib.oracle_q4_0_dequant_block.argtypes = [vp, vp]
        lib.oracle_q4_0_dequant_block.restype = None
        lib.oracle_q4_0_dequant.argtypes = [vp, i64, i64, vp]
        lib.oracle_q4_0_dequant.restype = i32
        lib.oracle_q4_0_matmul.argtypes = [vp, vp, i64, i64, i64, vp, i32]
        lib.oracle_q4_0_matmul.restype = i32
        lib.oracle_q4_0_pack_block.argtypes = [ctypes.c_uint16, vp, vp]
        lib.oracle_q4_0_pack_block.restype = None
        lib.oracle_ternary_gemv.argtypes = [vp, vp, flt, i64, i64, i64, vp, vp, i32]
        lib.oracle_ternary_gemv.restype = i32
        lib.oracle_q4k_pack_block.argtypes = [ctypes.c_uint16, ctypes.c_uint16, vp, vp, vp, vp]
        lib.oracle_q4k_pack_block.restype = None
        lib.oracle_ternary_pack.argtypes = [vp, i64, vp]
        lib.oracle_ternary_pack.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        if path is None:
            _LIB = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_q4k(W: np.ndarray, K: int, N: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if K <= 0 or K % Q4K_VALUES:
        raise ValueError(f"inputDim {K} is not a positive multiple of 256")
    if W.size != N * (K // Q4K_VALUES) * Q4K_BYTES:
        raise ValueError("weight bytes do not match N·K/256·144")
    return W


def _check_x(x: np.ndarray, K: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    if x.shape[1] != K:
        raise ValueError("activation rows must have inputDim elements")
    return x


def fp16_to_double(bits: int, lib=None) -> float:
    return (lib or load()).oracle_fp16_to_double(bits)


def round_bf16(v: float, lib=None) -> float:
    return (lib or load()).oracle_round_bf16(v)


def q4k_dequant(W: np.ndarray, K: int, N: int, lib=None) -> np.ndarray:
    """Dequantized fp32 weight [N, K]."""
    W = _check_q4k(W, K, N)
    out = np.empty((N, K), np.float32)
    if (lib or load()).oracle_q4k_dequant(_ptr(W), K, N, _ptr(out)) != 0:
        raise ValueError("oracle_q4k_dequant rejected its arguments")
    return out


Q4K_TC_CHUNK_BYTES = 48  # bytes per row and 64 values in the tensor-core layout
Q4K_TC_TILE_ROWS = 256   # rows per tile of that layout


def q4k_tc_bytes(K: int, N: int, lib=None) -> int:
    """Size of the relayouted weight (rows rounded up to whole tiles)."""
    n = (lib or load()).oracle_q4k_tc_bytes(K, N)
    if n < 0:
        raise ValueError("bad relayout sizes")
    return n


def q4k_tc_relayout(W: np.ndarray, K: int, N: int, lib=None) -> np.ndarray:
    """The one-time relayout of a Q4_K weight for the tensor cores: tiles of
    256 rows, each 64-value chunk of a tile one contiguous run of 256 rows x
    48 bytes (fp32 d·sc, dmin·m of both sub-blocks of the slab, then its 32
    code bytes); zero rows pad the last tile."""
    W = _check_q4k(W, K, N)
    lib = lib or load()
    R = np.empty(q4k_tc_bytes(K, N, lib), np.uint8)
    if lib.oracle_q4k_tc_relayout(_ptr(W), K, N, _ptr(R)) != 0:
        raise ValueError("oracle_q4k_tc_relayout rejected its arguments")
    return R


def q4k_tc_dequant(R: np.ndarray, K: int, N: int, lib=None) -> np.ndarray:
    """Dequantized fp32 weight [N, K] of a relayouted Q4_K weight."""
    R = np.ascontiguousarray(R, dtype=np.uint8)
    lib = lib or load()
    if R.size != q4k_tc_bytes(K, N, lib):
        raise ValueError("relayouted weight bytes do not match the tiled size")
    out = np.empty((N, K), np.float32)
    if lib.oracle_q4k_tc_dequant(_ptr(R), K, N, _ptr(out)) != 0:
        raise ValueError("oracle_q4k_tc_dequant rejected its arguments")
    return out


def _matmul(fn_name: str, x, W, K, N, threads, lib):
    W = _check_q4k(W, K, N)
    x = _check_x(x, K)
    T = x.shape[0]
    y = np.empty((T, N), np.float64)
    rc = getattr(lib or load(), fn_name)(_ptr(x), _ptr(W), K, N, T, _ptr(y), threads)
    if rc != 0:
        raise RuntimeError(f"{fn_name} failed with {rc}")
    return y


def q4k_matmul(x, W, K, N, threads=0, lib=None) -> np.ndarray:
    """y = x · dequant(W)ᵀ, double accumulation; returns float64 [T, N]."""
    return _matmul("oracle_q4k_matmul", x, W, K, N, threads, lib)


def q4k_matmul_bf16(x, W, K, N, threads=0, lib=None) -> np.ndarray:
    """As q4k_matmul with x and the fp32 dequantized w rounded to bfloat16."""
    return _matmul("oracle_q4k_matmul_bf16", x, W, K, N, threads, lib)


def q4k_matmul_lazy(x, W, K, N, threads=0, lib=None) -> np.ndarray:
    """The lazy-dmin form (scale·Σxq − offset·Σx per sub-block), double."""
    return _matmul("oracle_q4k_matmul_lazy", x, W, K, N, threads, lib)


def q4k_ffn_swiglu(x, Wg, Wu, K, N, threads=0, lib=None):
    """(g, u, h) float64 [T, N]: g = x·dequant(Wg)ᵀ, u = x·dequant(Wu)ᵀ, h = silu(g)·u."""
    Wg = _check_q4k(Wg, K, N)
    Wu = _check_q4k(Wu, K, N)
    x = _check_x(x, K)
    T = x.shape[0]
    g = np.empty((T, N), np.float64)
    u = np.empty((T, N), np.float64)
    h = np.empty((T, N), np.float64)
    rc = (lib or load()).oracle_q4k_ffn_swiglu(_ptr(x), _ptr(Wg), _ptr(Wu), K, N, T, _ptr(g), _ptr(u),
                                                _ptr(h), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_q4k_ffn_swiglu failed with {rc}")
    return g, u, h


Q40_VALUES, Q40_BYTES = 32, 18


def _check_q4_0(W: np.ndarray, K: int, N: int) -> np.ndarray:
    if K <= 0 or K % Q40_VALUES:
        raise ValueError(f"inputDim {K} is not a positive multiple of {Q40_VALUES}")
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if W.size != N * (K // Q40_VALUES) * Q40_BYTES:
        raise ValueError("weight bytes do not match N·K/32·18")
    return W


def q4_0_dequant(W: np.ndarray, K: int, N: int, lib=None) -> np.ndarray:
    """Dequantized fp32 Q4_0 weight [N, K]."""
    W = _check_q4_0(W, K, N)
    out = np.empty((N, K), np.float32)
    if (lib or load()).oracle_q4_0_dequant(_ptr(W), K, N, _ptr(out)) != 0:
        raise ValueError("oracle_q4_0_dequant rejected its arguments")
    return out


def q4_0_matmul(x, W, K, N, threads=0, lib=None) -> np.ndarray:
    """y = x · dequant_q4_0(W)ᵀ, double accumulation; returns float64 [T, N]."""
    W = _check_q4_0(W, K, N)
    x = _check_x(x, K)
    T = x.shape[0]
    y = np.empty((T, N), np.float64)
    rc = (lib or load()).oracle_q4_0_matmul(_ptr(x), _ptr(W), K, N, T, _ptr(y), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_q4_0_matmul failed with {rc}")
    return y


def q4_0_pack_block(d_bits: int, q, lib=None) -> np.ndarray:
    """Encode one 18-byte Q4_0 block from d (fp16 bits) and 32 codes (0..15)."""
    q = np.ascontiguousarray(q, dtype=np.int32)
    assert q.size == Q40_VALUES
    out = np.zeros(Q40_BYTES, np.uint8)
    (lib or load()).oracle_q4_0_pack_block(d_bits, _ptr(q), _ptr(out))
    return out


def ternary_gemv(x, W, scale, K, N, threads=0, lib=None):
    """Returns (dot float64 [T, N] without scale, y float32 [T, N] with scale)."""
    if K <= 0 or K % 4:
        raise ValueError(f"inputDim {K} is not a positive multiple of 4")
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if W.size != N * (K // 4):
        raise ValueError("weight bytes do not match N·K/4")
    x = _check_x(x, K)
    T = x.shape[0]
    dot = np.empty((T, N), np.float64)
    y = np.empty((T, N), np.float32)
    rc = (lib or load()).oracle_ternary_gemv(_ptr(x), _ptr(W), float(scale), K, N, T,
                                              _ptr(dot), _ptr(y), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_ternary_gemv failed with {rc}")
    return dot, y


def q4k_pack_block(d_bits: int, dmin_bits: int, sc, m, q, lib=None) -> np.ndarray:
    """Encode one 144-byte Q4_K block from d, dmin (fp16 bits), 8 scales, 8 mins, 256 codes."""
    sc = np.ascontiguousarray(sc, dtype=np.int32)
    m = np.ascontiguousarray(m, dtype=np.int32)
    q = np.ascontiguousarray(q, dtype=np.int32)
    assert sc.size == 8 and m.size == 8 and q.size == Q4K_VALUES
    out = np.zeros(Q4K_BYTES, np.uint8)
    (lib or load()).oracle_q4k_pack_block(d_bits, dmin_bits, _ptr(sc), _ptr(m), _ptr(q), _ptr(out))
    return out


def ternary_pack(codes, lib=None) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    assert codes.size % 4 == 0
    out = np.zeros(codes.size // 4, np.uint8)
    (lib or load()).oracle_ternary_pack(_ptr(codes), codes.size, _ptr(out))
    return out


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()


Q6K_VALUES, Q6K_BYTES = 256, 210


def _check_q6k(W: np.ndarray, K: int, N: int) -> np.ndarray:
    if K <= 0 or K % Q6K_VALUES:
        raise ValueError(f"inputDim {K} is not a positive multiple of {Q6K_VALUES}")
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if W.size != N * (K // Q6K_VALUES) * Q6K_BYTES:
        raise ValueError("weight bytes do not match N·K/256·210")
    return W


def q6k_dequant(W: np.ndarray, K: int, N: int, lib=None) -> np.ndarray:
    """Dequantized fp32 Q6_K weight [N, K]."""
    W = _check_q6k(W, K, N)
    out = np.empty((N, K), np.float32)
    if (lib or load()).oracle_q6k_dequant(_ptr(W), K, N, _ptr(out)) != 0:
        raise ValueError("oracle_q6k_dequant rejected its arguments")
    return out


def q6k_matmul(x, W, K, N, threads=0, lib=None) -> np.ndarray:
    """y = x · dequant_q6k(W)ᵀ, double accumulation; returns float64 [T, N]."""
    W = _check_q6k(W, K, N)
    x = _check_x(x, K)
    T = x.shape[0]
    y = np.empty((T, N), np.float64)
    rc = (lib or load()).oracle_q6k_matmul(_ptr(x), _ptr(W), K, N, T, _ptr(y), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_q6k_matmul failed with {rc}")
    return y


def q6k_pack_block(d_bits: int, sc, q, lib=None) -> np.ndarray:
    """Encode one 210-byte Q6_K block from d (fp16 bits), 16 scales and 256 codes (0..63)."""
    sc = np.ascontiguousarray(sc, dtype=np.int32)
    q = np.ascontiguousarray(q, dtype=np.int32)
    assert sc.size == 16 and q.size == Q6K_VALUES
    out = np.zeros(Q6K_BYTES, np.uint8)
    (lib or load()).oracle_q6k_pack_block(d_bits, _ptr(sc), _ptr(q), _ptr(out))
    return out
