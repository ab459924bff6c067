"""ctypes binding of libq4mm.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
Q4K_VALUES = 256
Q4K_BYTES = 144

_SYMBOLS = ("q4k_matmul", "q4k_matmul_tc", "q4k_matmul_tc_noalloc", "q4k_relayout_tc", "q4k_matmul_tc_relayouted",
            "q4_0_gemv", "q6k_gemv", "q4k_ffn_swiglu", "ternary_gemv",
            "q4mm_last_error", "q4mm_device_status", "q4mm_version", "q4mm_test_fail_next_wait")


class Q4mmError(RuntimeError):
    """A q4mm entry point returned a negative status."""

    def __init__(self, code: int, message: str):
        super().__init__(f"q4mm status {code}: {message}")
        self.code = code


def library_path() -> str:
    return os.environ.get("Q4MM_LIB", os.path.join(PKG, "libq4mm.so"))


def _load() -> ctypes.CDLL:
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"libq4mm.so not found at {path}: build it with `python quantized_matmul_q4_gb300/_build.py` "
            "(needs nvcc); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    for name in ("q4k_matmul", "q4k_matmul_tc", "q4k_matmul_tc_noalloc", "q4k_matmul_tc_relayouted", "q4_0_gemv",
                 "q6k_gemv"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        fn.restype = i32
    lib.q4k_relayout_tc.argtypes = [vp, vp, i32, i32, vp]
    lib.q4k_relayout_tc.restype = i32
    lib.q4k_ffn_swiglu.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
    lib.q4k_ffn_swiglu.restype = i32
    lib.ternary_gemv.argtypes = [vp, vp, f32, vp, i32, i32, i32, vp]
    lib.ternary_gemv.restype = i32
    lib.q4mm_last_error.argtypes = []
    lib.q4mm_last_error.restype = ctypes.c_char_p
    lib.q4mm_device_status.argtypes = [vp, i32]
    lib.q4mm_device_status.restype = i32
    lib.q4mm_version.argtypes = []
    lib.q4mm_version.restype = i32
    lib.q4mm_test_fail_next_wait.argtypes = [i32, ctypes.c_longlong]
    lib.q4mm_test_fail_next_wait.restype = i32
    return lib


_LIB = _load()


def library() -> ctypes.CDLL:
    return _LIB


def last_error() -> str:
    return _LIB.q4mm_last_error().decode()


def version() -> int:
    return _LIB.q4mm_version()


def _check(rc: int) -> None:
    if rc != 0:
        raise Q4mmError(rc, last_error())


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


# Raw-pointer entry points (device pointers, sizes, stream handle).

def q4k_matmul_ptr(x: int, w: int, y: int, K: int, N: int, T: int, stream: int = 0) -> None:
    _check(_LIB.q4k_matmul(x, w, y, K, N, T, stream))


def q4k_matmul_tc_ptr(x: int, w: int, y: int, K: int, N: int, T: int, stream: int = 0) -> None:
    _check(_LIB.q4k_matmul_tc(x, w, y, K, N, T, stream))


def q4k_matmul_tc_noalloc_ptr(x: int, w: int, y: int, K: int, N: int, T: int, stream: int = 0) -> None:
    _check(_LIB.q4k_matmul_tc_noalloc(x, w, y, K, N, T, stream))


def q4k_relayout_tc_ptr(w: int, w_tc: int, K: int, N: int, stream: int = 0) -> None:
    _check(_LIB.q4k_relayout_tc(w, w_tc, K, N, stream))


def q4k_matmul_tc_relayouted_ptr(x: int, w_tc: int, y: int, K: int, N: int, T: int, stream: int = 0) -> None:
    _check(_LIB.q4k_matmul_tc_relayouted(x, w_tc, y, K, N, T, stream))


def q4_0_gemv_ptr(x: int, w: int, y: int, K: int, N: int, T: int, stream: int = 0) -> None:
    _check(_LIB.q4_0_gemv(x, w, y, K, N, T, stream))


def q6k_gemv_ptr(x: int, w: int, y: int, K: int, N: int, T: int, stream: int = 0) -> None:
    _check(_LIB.q6k_gemv(x, w, y, K, N, T, stream))


def q4k_ffn_swiglu_ptr(x: int, w_gate: int, w_up: int, h: int, K: int, N: int, T: int,
                       stream: int = 0) -> None:
    _check(_LIB.q4k_ffn_swiglu(x, w_gate, w_up, h, K, N, T, stream))


def ternary_gemv_ptr(x: int, w: int, scale: float, y: int, K: int, N: int, T: int,
                     stream: int = 0) -> None:
    _check(_LIB.ternary_gemv(x, w, ctypes.c_float(scale), y, K, N, T, stream))


def arm_wait_failure(stage: int, limit_cycles: int) -> None:
    """Test hook: the calling thread's next call withholds weight stage `stage`
    and bounds its in-kernel waits by `limit_cycles` (see include/q4mm.h)."""
    _check(_LIB.q4mm_test_fail_next_wait(int(stage), int(limit_cycles)))


def device_status(stream=None, clear: bool = True) -> None:
    """Raise Q4mmError if a bounded in-kernel wait ran out on this device."""
    _check(_LIB.q4mm_device_status(_stream_ptr(stream), int(clear)))


# Tensor entry points (torch CUDA tensors; y allocated unless `out` is given).

def _prep(x, w, K, bytes_per_row, out, N):
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    if w.dtype != torch.uint8 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("the packed weight must be a contiguous uint8 CUDA tensor")
    x2 = x.reshape(-1, x.shape[-1])
    T, K_ = x2.shape
    if K is not None and K != K_:
        raise ValueError("x's last dimension must equal inputDim")
    if N is None:
        if bytes_per_row(K_) <= 0 or w.numel() % bytes_per_row(K_):
            raise ValueError("weight size is not a whole number of rows")
        N = w.numel() // bytes_per_row(K_)
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or not out.is_cuda or not out.is_contiguous() or out.numel() != T * N:
        raise ValueError("out must be a contiguous float32 CUDA tensor with tokens·outputDim elements")
    return x2, T, K_, N, out


def q4k_matmul(x, w, N: int | None = None, out=None, stream=None):
    """y[T, N] = x[T, K] · dequant(W)ᵀ in FP32 (decode GEMV up to 8 tokens)."""
    x2, T, K, N, out = _prep(x, w, None, lambda k: (k // Q4K_VALUES) * Q4K_BYTES, out, N)
    q4k_matmul_ptr(x2.data_ptr(), w.data_ptr(), out.data_ptr(), K, N, T, _stream_ptr(stream))
    return out.view(T, N)


def q4k_matmul_tc(x, w, N: int | None = None, out=None, stream=None):
    """As q4k_matmul on the tensor cores with bf16-rounded operands."""
    x2, T, K, N, out = _prep(x, w, None, lambda k: (k // Q4K_VALUES) * Q4K_BYTES, out, N)
    q4k_matmul_tc_ptr(x2.data_ptr(), w.data_ptr(), out.data_ptr(), K, N, T, _stream_ptr(stream))
    return out.view(T, N)


def q4k_matmul_tc_noalloc(x, w, N: int | None = None, out=None, stream=None):
    """As q4k_matmul_tc with its scratch in the library's fixed device array
    (no allocation; calls that overlap on the GPU race on that array)."""
    x2, T, K, N, out = _prep(x, w, None, lambda k: (k // Q4K_VALUES) * Q4K_BYTES, out, N)
    q4k_matmul_tc_noalloc_ptr(x2.data_ptr(), w.data_ptr(), out.data_ptr(), K, N, T, _stream_ptr(stream))
    return out.view(T, N)


TC_CHUNK_BYTES = 48  # relayouted bytes per row and 64 values
TC_TILE_ROWS = 256   # rows per tile of the relayouted layout


def tc_relayout_bytes(K: int, N: int) -> int:
    """Size of a relayouted K -> N weight (rows rounded up to whole tiles)."""
    return -(-N // TC_TILE_ROWS) * TC_TILE_ROWS * (K // 64) * TC_CHUNK_BYTES


def q4k_relayout_tc(w, K: int, N: int | None = None, out=None, stream=None):
    """The one-time relayout of a canonical Q4_K weight for
    q4k_matmul_tc_relayouted: a uint8 CUDA tensor of tc_relayout_bytes(K, N)
    bytes (tile-major, zero rows padding the last 256-row tile)."""
    import torch
    if w.dtype != torch.uint8 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("the packed weight must be a contiguous uint8 CUDA tensor")
    row = (K // Q4K_VALUES) * Q4K_BYTES
    if N is None:
        if row <= 0 or w.numel() % row:
            raise ValueError("weight size is not a whole number of rows")
        N = w.numel() // row
    nbytes = tc_relayout_bytes(K, N)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    elif out.dtype != torch.uint8 or not out.is_cuda or not out.is_contiguous() or out.numel() != nbytes:
        raise ValueError("out must be a contiguous uint8 CUDA tensor of tc_relayout_bytes(K, N) bytes")
    q4k_relayout_tc_ptr(w.data_ptr(), out.data_ptr(), K, N, _stream_ptr(stream))
    return out


def q4k_matmul_tc_relayouted(x, w_tc, N: int, out=None, stream=None):
    """q4k_matmul_tc on a weight relayouted by q4k_relayout_tc (N is
    required: the padded layout does not give it)."""
    if w_tc.numel() != tc_relayout_bytes(x.shape[-1], N):
        raise ValueError("w_tc size does not match tc_relayout_bytes(K, N)")
    x2, T, K, N, out = _prep(x, w_tc, None, lambda k: (k // 64) * TC_CHUNK_BYTES, out, N)
    q4k_matmul_tc_relayouted_ptr(x2.data_ptr(), w_tc.data_ptr(), out.data_ptr(), K, N, T, _stream_ptr(stream))
    return out.view(T, N)


Q40_VALUES, Q40_BYTES = 32, 18


def q4_0_gemv(x, w, N: int | None = None, out=None, stream=None):
    """y[T, N] = x[T, K] · dequant_q4_0(W)ᵀ in FP32 (up to 8 tokens per weight pass)."""
    x2, T, K, N, out = _prep(x, w, None, lambda k: (k // Q40_VALUES) * Q40_BYTES, out, N)
    q4_0_gemv_ptr(x2.data_ptr(), w.data_ptr(), out.data_ptr(), K, N, T, _stream_ptr(stream))
    return out.view(T, N)


Q6K_BYTES = 210


def q6k_gemv(x, w, N: int | None = None, out=None, stream=None):
    """y[T, N] = x[T, K] · dequant_q6k(W)ᵀ in FP32 (up to 8 tokens per weight pass)."""
    x2, T, K, N, out = _prep(x, w, None, lambda k: (k // Q4K_VALUES) * Q6K_BYTES, out, N)
    q6k_gemv_ptr(x2.data_ptr(), w.data_ptr(), out.data_ptr(), K, N, T, _stream_ptr(stream))
    return out.view(T, N)


def q4k_ffn_swiglu(x, w_gate, w_up, N: int | None = None, out=None, stream=None):
    """h[T, N] = silu(x · dequant(W_gate)ᵀ) · (x · dequant(W_up)ᵀ), both Q4_K."""
    x2, T, K, N, out = _prep(x, w_gate, None, lambda k: (k // Q4K_VALUES) * Q4K_BYTES, out, N)
    if (w_up.dtype != w_gate.dtype or w_up.numel() != w_gate.numel() or not w_up.is_cuda
            or not w_up.is_contiguous()):
        raise ValueError("w_up must be a contiguous CUDA uint8 tensor of the gate weight's size")
    q4k_ffn_swiglu_ptr(x2.data_ptr(), w_gate.data_ptr(), w_up.data_ptr(), out.data_ptr(),
                       K, N, T, _stream_ptr(stream))
    return out.view(T, N)


def ternary_gemv(x, w, scale: float = 1.0, N: int | None = None, out=None, stream=None):
    """y[T, N] = scale · x[T, K] · codes(W)ᵀ, BitNet b1.58 payload, FP32."""
    x2, T, K, N, out = _prep(x, w, None, lambda k: k // 4, out, N)
    ternary_gemv_ptr(x2.data_ptr(), w.data_ptr(), float(scale), out.data_ptr(), K, N, T,
                     _stream_ptr(stream))
    return out.view(T, N)
