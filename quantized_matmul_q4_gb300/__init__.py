"""GB300 (sm_103a) kernels for y = x·Wᵀ with an FP32 activation and a
block-quantized weight (Q4_K or BitNet b1.58 ternary), dequantized in-kernel.

This package is a thin Python binding over the C ABI of ``libq4mm.so``
(declared in ``include/q4mm.h``): it only marshals tensor pointers, sizes and
the current CUDA stream.  Every step of the computation runs in the CUDA
kernels; there is no CPU or PyTorch fallback, and importing the binding fails
loudly if the library has not been built
(``python quantized_matmul_q4_gb300/_build.py``).
"""
from ._binding import (  # noqa: F401
    Q4mmError,
    Q4K_BYTES,
    Q4K_VALUES,
    arm_wait_failure,
    device_status,
    last_error,
    library,
    library_path,
    q4k_matmul,
    q4k_matmul_ptr,
    q4k_matmul_tc,
    q4k_matmul_tc_ptr,
    q4k_matmul_tc_noalloc,
    q4k_matmul_tc_noalloc_ptr,
    q4k_relayout_tc,
    tc_relayout_bytes,
    q4k_relayout_tc_ptr,
    q4k_matmul_tc_relayouted,
    q4k_matmul_tc_relayouted_ptr,
    q4_0_gemv,
    q4_0_gemv_ptr,
    q6k_gemv,
    q6k_gemv_ptr,
    q4k_ffn_swiglu,
    q4k_ffn_swiglu_ptr,
    ternary_gemv,
    ternary_gemv_ptr,
    version,
)
