// Internal launchers behind the C ABI.  Each returns cudaSuccess or the
// launch error; arguments are already validated by capi.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

namespace q4mm {

struct LaunchCtx {
    cudaStream_t stream;
    int num_sms;
    int max_smem_optin;  // bytes of shared memory a CTA may opt into
    int *status;         // device status word (bounded-wait time-outs)
    bool pdl;            // launch with programmatic stream serialization
    long long wait_limit;  // SM cycles a bounded in-kernel wait lasts at most
    int withhold;          // test only: a weight stage never copied (-1: none)
};

// Q4_K decode GEMV, 1..8 tokens on the one-token kernel (bulk-copied weight
// rows, byte planes of x in registers; each compute warp serves one token).
// Returns cudaErrorNotSupported when the shape is outside its geometry.
cudaError_t launch_q4k_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                               int K, int N, int T = 1);

// Q4_0 decode GEMV, one token (same kernel as the Q4_K one with the Q4_0
// row format).  cudaErrorNotSupported when the shape is outside its geometry.
cudaError_t launch_q4_0_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                int K, int N, int T = 1);

// Q6_K decode GEMV, one token (the one-token kernel with the Q6_K row format).
cudaError_t launch_q6k_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N,
                              int T = 1);

// BitNet b1.58 ternary GEMV, 1..8 tokens, on the same one-token kernel with
// the byte-plane integer code-dot (K % 256 == 0, W 16-byte aligned; otherwise
// cudaErrorNotSupported).
cudaError_t launch_ternary_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float scale, float *y,
                                   int K, int N, int T = 1);

// Llama FFN input side, one token: h = silu(x·Wgᵀ)·(x·Wuᵀ), both Q4_K, in one
// launch of the one-token kernel (x split once for both weights).
cudaError_t launch_q4k_ffn_swiglu_t1(const LaunchCtx &c, const float *x, const uint8_t *Wg, const uint8_t *Wu,
                                     float *h, int K, int N);

// Q4_K decode GEMV for 1..8 tokens with x staged in shared memory.
cudaError_t launch_q4k_gemv_multi(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                  int K, int N, int T);
// The fused gate+up SwiGLU (h = silu(x·Wgᵀ) ⊙ (x·Wuᵀ)) for up to 8 tokens on
// the same kernel: one pass over both weights for all tokens.
cudaError_t launch_q4k_ffn_swiglu_multi(const LaunchCtx &c, const float *x, const uint8_t *Wg, const uint8_t *Wu,
                                        float *h, int K, int N, int T);

// Q4_K prefill, FP32 FMA (any token count, tiles of 64 tokens).
cudaError_t launch_q4k_mm_fp32(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                               int K, int N, int T);

// Q4_K prefill on tcgen05 tensor cores (bf16 operands, fp32 accumulate).
cudaError_t launch_q4k_mm_tc(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K,
                             int N, int T);

// The tensor-core prefill on a weight in the relayouted tensor-core layout
// (48 bytes per row and 64-value chunk), and the one-time relayout that
// makes it from a canonical Q4_K weight (q4k_relayout_tc_bytes(K, N) bytes).
cudaError_t launch_q4k_mm_tc_relayouted(const LaunchCtx &c, const float *x, const uint8_t *R, float *y, int K,
                                        int N, int T);
size_t q4k_relayout_tc_bytes(int K, int N);
cudaError_t launch_q4k_relayout_tc(const LaunchCtx &c, const uint8_t *W, uint8_t *R, int K, int N);

// The tensor-core prefill with its scratch in a fixed array of library
// memory (no allocation): bytes of scratch a call needs, and the launcher
// (cudaErrorInvalidValue if the need exceeds the array).
size_t q4k_mm_tc_scratch_bytes(int K, int N, int T);
cudaError_t launch_q4k_mm_tc_fixed_scratch(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                           int K, int N, int T);

// BitNet b1.58 ternary GEMV, any token count.
cudaError_t launch_ternary_gemv(const LaunchCtx &c, const float *x, const uint8_t *W, float scale,
                                float *y, int K, int N, int T);

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the attribute call is made only when the limit grows, so a
// warmed-up launch (for instance one being captured into a CUDA graph) issues
// nothing but the launch itself.
cudaError_t ensure_smem_limit(const void *kernel, size_t bytes);

template <typename... KArgs>
cudaError_t ensure_smem(void (*kernel)(KArgs...), size_t bytes) {
    return ensure_smem_limit(reinterpret_cast<const void *>(kernel), bytes);
}

// Launch helper: cudaLaunchKernelEx with optional programmatic serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const LaunchCtx &c, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                          size_t smem, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    int nattr = 0;
    if (c.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        nattr = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace q4mm
