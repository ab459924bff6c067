// C ABI of libq4mm.so: argument validation, dispatch to the kernels, error
// reporting.  Declarations and the contract of every entry point are in
// include/q4mm.h.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "q4mm.h"
#include "dispatch.h"
#include "kernels.h"
#include "sync.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int fail_cuda(cudaError_t e, const char *what) {
    return fail(Q4MM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Set by a kernel whose bounded wait gave up.
__device__ int g_device_status;

struct DeviceInfo {
    // Set (release) after the other fields are filled; read (acquire) without
    // the lock, so a thread that sees it set also sees those fields.
    std::atomic<bool> ready{false};
    int num_sms = 0;
    int max_smem_optin = 0;
    int *status = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Armed by q4mm_test_fail_next_wait for the calling thread's next compute
// call only.
struct TestFault {
    bool armed = false;
    int stage = -1;
    long long limit = 0;
};
thread_local TestFault g_test_fault;

// take_test_fault: a compute call (it consumes an armed test fault).
int device_ctx(q4mm_stream_t stream, q4mm::LaunchCtx *ctx, bool take_test_fault = true) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(Q4MM_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
            e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(shared memory)");
            e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status);
            if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(status)");
            d.ready.store(true, std::memory_order_release);
        }
    }
    ctx->stream = reinterpret_cast<cudaStream_t>(stream);
    ctx->num_sms = d.num_sms;
    ctx->max_smem_optin = d.max_smem_optin;
    ctx->status = d.status;
    // Programmatic dependent launch: a kernel may start its weight stream
    // while the previous kernel on the stream finishes.
    ctx->pdl = true;
    ctx->wait_limit = q4mm::kWaitLimitCycles;
    ctx->withhold = -1;
    if (take_test_fault && g_test_fault.armed) {
        ctx->wait_limit = g_test_fault.limit;
        ctx->withhold = g_test_fault.stage;
        g_test_fault.armed = false;
    }
    return Q4MM_OK;
}

// Runs a one-token-kernel launcher over the tokens in chunks of up to 8,
// halving a chunk whose geometry the kernel cannot hold.
template <class F>
cudaError_t token_chunks(F launch, const float *x, float *y, int K, int N, int tokens) {
    cudaError_t e = cudaSuccess;
    for (int t0 = 0; t0 < tokens && e == cudaSuccess;) {
        int tt = tokens - t0 < 8 ? tokens - t0 : 8;
        for (;;) {
            e = launch(x + (size_t)t0 * K, y + (size_t)t0 * N, tt);
            if (e != cudaErrorNotSupported || tt == 1) break;
            tt /= 2;
        }
        t0 += tt;
    }
    return e;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// w_bytes_per_row: the weight's bytes per output row; w_total_bytes, when
// nonzero, its whole size instead (a layout padded past N rows).
int check_common(const float *x, const void *w, const float *y, int K, int N, int T, int k_multiple,
                 size_t w_bytes_per_row, size_t w_align, size_t w_total_bytes = 0) {
    if (!x || !w || !y) return fail(Q4MM_ERR_NULL, "x, weight and y must be non-NULL");
    if (K <= 0 || N <= 0 || T <= 0)
        return fail(Q4MM_ERR_DIM, "inputDim (%d), outputDim (%d) and tokens (%d) must be positive", K, N, T);
    if (K % k_multiple)
        return fail(Q4MM_ERR_DIM, "inputDim %d is not a multiple of %d", K, k_multiple);
    if (K > Q4MM_MAX_INPUT_DIM)
        return fail(Q4MM_ERR_DIM, "inputDim %d exceeds the limit %d", K, Q4MM_MAX_INPUT_DIM);
    if (reinterpret_cast<uintptr_t>(x) % 16) return fail(Q4MM_ERR_ALIGN, "x must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(y) % 4) return fail(Q4MM_ERR_ALIGN, "y must be 4-byte aligned");
    if (reinterpret_cast<uintptr_t>(w) % w_align)
        return fail(Q4MM_ERR_ALIGN, "weight must be %zu-byte aligned", w_align);
    const size_t xb = (size_t)T * K * sizeof(float), yb = (size_t)T * N * sizeof(float);
    const size_t wb = w_total_bytes ? w_total_bytes : (size_t)N * w_bytes_per_row;
    if (overlap(x, xb, y, yb) || overlap(x, xb, w, wb) || overlap(w, wb, y, yb))
        return fail(Q4MM_ERR_ALIAS, "x, weight and y must not overlap");
    return Q4MM_OK;
}

}  // namespace

namespace q4mm {

cudaError_t ensure_smem_limit(const void *kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    struct Entry {
        int dev;
        const void *fn;
        size_t bytes;
    };
    static Entry table[256];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].dev == dev && table[i].fn == kernel && table[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    // The largest shared-memory configuration of the SM: kernels that pair a
    // CTA of the next launch with one of the current launch need both to fit.
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < used; ++i)
        if (table[i].dev == dev && table[i].fn == kernel) {
            table[i].bytes = bytes;
            return cudaSuccess;
        }
    if (used < 256) table[used++] = Entry{dev, kernel, bytes};
    return cudaSuccess;
}

}  // namespace q4mm

extern "C" {

int q4k_matmul(const float *x, const void *w_q4k, float *y, int inputDim, int outputDim, int tokens,
               q4mm_stream_t stream) {
    int rc = check_common(x, w_q4k, y, inputDim, outputDim, tokens, 256,
                          (size_t)(inputDim / 256) * 144, 16);
    if (rc) return rc;
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    const uint8_t *W = static_cast<const uint8_t *>(w_q4k);
    // The kernel for this token count (dispatch.h), each falling back to the
    // next where its geometry does not fit the shape.
    const q4mm::Q4kPath path = q4mm::q4k_matmul_path(tokens, outputDim, ctx.num_sms);
    cudaError_t e = cudaErrorNotSupported;
    if (path == q4mm::Q4kPath::kOneToken) e = q4mm::launch_q4k_gemv_t1(ctx, x, W, y, inputDim, outputDim, tokens);
    if (e == cudaErrorNotSupported && tokens <= 8)
        e = q4mm::launch_q4k_gemv_multi(ctx, x, W, y, inputDim, outputDim, tokens);
    if (e == cudaErrorNotSupported && path == q4mm::Q4kPath::kTileChunks) {
        e = cudaSuccess;
        for (int t0 = 0; t0 < tokens && e == cudaSuccess; t0 += 8) {
            const int tt = tokens - t0 < 8 ? tokens - t0 : 8;
            e = q4mm::launch_q4k_gemv_multi(ctx, x + (size_t)t0 * inputDim, W, y + (size_t)t0 * outputDim, inputDim,
                                            outputDim, tt);
            // A geometry the register-tile kernel cannot hold fails on the
            // first chunk, before anything is launched.
            if (e == cudaErrorNotSupported && t0 > 0) return fail_cuda(e, "q4k_matmul launch");
        }
    }
    if (e == cudaErrorNotSupported) e = q4mm::launch_q4k_mm_fp32(ctx, x, W, y, inputDim, outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "q4k_matmul launch");
    return Q4MM_OK;
}

int q4k_matmul_tc(const float *x, const void *w_q4k, float *y, int inputDim, int outputDim,
                  int tokens, q4mm_stream_t stream) {
    int rc = check_common(x, w_q4k, y, inputDim, outputDim, tokens, 256,
                          (size_t)(inputDim / 256) * 144, 16);
    if (rc) return rc;
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    cudaError_t e = q4mm::launch_q4k_mm_tc(ctx, x, static_cast<const uint8_t *>(w_q4k), y, inputDim,
                                           outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "q4k_matmul_tc launch");
    return Q4MM_OK;
}

int q4k_matmul_tc_noalloc(const float *x, const void *w_q4k, float *y, int inputDim, int outputDim,
                          int tokens, q4mm_stream_t stream) {
    int rc = check_common(x, w_q4k, y, inputDim, outputDim, tokens, 256,
                          (size_t)(inputDim / 256) * 144, 16);
    if (rc) return rc;
    const size_t need = q4mm::q4k_mm_tc_scratch_bytes(inputDim, outputDim, tokens);
    if (need > (size_t)Q4MM_TC_NOALLOC_SCRATCH_BYTES)
        return fail(Q4MM_ERR_DIM,
                    "q4k_matmul_tc_noalloc: %d tokens x inputDim %d x outputDim %d need %zu bytes of scratch, "
                    "more than the fixed %zu-byte array (use q4k_matmul_tc, or fewer tokens per call)",
                    tokens, inputDim, outputDim, need, (size_t)Q4MM_TC_NOALLOC_SCRATCH_BYTES);
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    cudaError_t e = q4mm::launch_q4k_mm_tc_fixed_scratch(ctx, x, static_cast<const uint8_t *>(w_q4k), y,
                                                         inputDim, outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "q4k_matmul_tc_noalloc launch");
    return Q4MM_OK;
}

int q4k_relayout_tc(const void *w_q4k, void *w_tc, int inputDim, int outputDim, q4mm_stream_t stream) {
    if (!w_q4k || !w_tc) return fail(Q4MM_ERR_NULL, "w_q4k and w_tc must be non-NULL");
    if (inputDim <= 0 || outputDim <= 0)
        return fail(Q4MM_ERR_DIM, "inputDim (%d) and outputDim (%d) must be positive", inputDim, outputDim);
    if (inputDim % 256) return fail(Q4MM_ERR_DIM, "inputDim %d is not a multiple of 256", inputDim);
    if (inputDim > Q4MM_MAX_INPUT_DIM)
        return fail(Q4MM_ERR_DIM, "inputDim %d exceeds the limit %d", inputDim, Q4MM_MAX_INPUT_DIM);
    if (reinterpret_cast<uintptr_t>(w_q4k) % 16 || reinterpret_cast<uintptr_t>(w_tc) % 16)
        return fail(Q4MM_ERR_ALIGN, "w_q4k and w_tc must be 16-byte aligned");
    const size_t wb = (size_t)outputDim * (inputDim / 256) * 144;
    if (overlap(w_q4k, wb, w_tc, Q4MM_TC_RELAYOUT_BYTES(inputDim, outputDim)))
        return fail(Q4MM_ERR_ALIAS, "w_q4k and w_tc must not overlap");
    q4mm::LaunchCtx ctx;
    int rc;
    if ((rc = device_ctx(stream, &ctx, false))) return rc;
    const cudaError_t e = q4mm::launch_q4k_relayout_tc(ctx, static_cast<const uint8_t *>(w_q4k),
                                                       static_cast<uint8_t *>(w_tc), inputDim, outputDim);
    if (e != cudaSuccess) return fail_cuda(e, "q4k_relayout_tc launch");
    return Q4MM_OK;
}

int q4k_matmul_tc_relayouted(const float *x, const void *w_tc, float *y, int inputDim, int outputDim, int tokens,
                             q4mm_stream_t stream) {
    // The weight-overlap check takes the padded layout's exact size.
    int rc = check_common(x, w_tc, y, inputDim, outputDim, tokens, 256, 0, 16,
                          inputDim > 0 && outputDim > 0 ? Q4MM_TC_RELAYOUT_BYTES(inputDim, outputDim) : 0);
    if (rc) return rc;
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    cudaError_t e = q4mm::launch_q4k_mm_tc_relayouted(ctx, x, static_cast<const uint8_t *>(w_tc), y, inputDim,
                                                      outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "q4k_matmul_tc_relayouted launch");
    return Q4MM_OK;
}

int q4_0_gemv(const float *x, const void *w_q4_0, float *y, int inputDim, int outputDim, int tokens,
              q4mm_stream_t stream) {
    int rc = check_common(x, w_q4_0, y, inputDim, outputDim, tokens, 256,
                          (size_t)(inputDim / 32) * 18, 16);
    if (rc) return rc;
    if (inputDim > Q4MM_Q4_0_MAX_INPUT_DIM)
        return fail(Q4MM_ERR_DIM, "inputDim %d exceeds the Q4_0 limit %d", inputDim, Q4MM_Q4_0_MAX_INPUT_DIM);
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    const uint8_t *W = static_cast<const uint8_t *>(w_q4_0);
    const cudaError_t e = token_chunks(
        [&](const float *xt, float *yt, int tt) {
            return q4mm::launch_q4_0_gemv_t1(ctx, xt, W, yt, inputDim, outputDim, tt);
        },
        x, y, inputDim, outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "q4_0_gemv launch");
    return Q4MM_OK;
}

int q6k_gemv(const float *x, const void *w_q6k, float *y, int inputDim, int outputDim, int tokens,
             q4mm_stream_t stream) {
    int rc = check_common(x, w_q6k, y, inputDim, outputDim, tokens, 256, (size_t)(inputDim / 256) * 210, 16);
    if (rc) return rc;
    if (inputDim > Q4MM_Q6K_MAX_INPUT_DIM)
        return fail(Q4MM_ERR_DIM, "inputDim %d exceeds the Q6_K limit %d", inputDim, Q4MM_Q6K_MAX_INPUT_DIM);
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    const uint8_t *W = static_cast<const uint8_t *>(w_q6k);
    const cudaError_t e = token_chunks(
        [&](const float *xt, float *yt, int tt) {
            return q4mm::launch_q6k_gemv_t1(ctx, xt, W, yt, inputDim, outputDim, tt);
        },
        x, y, inputDim, outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "q6k_gemv launch");
    return Q4MM_OK;
}

int q4k_ffn_swiglu(const float *x, const void *w_gate, const void *w_up, float *h, int inputDim,
                   int hiddenDim, int tokens, q4mm_stream_t stream) {
    const size_t row_bytes = (size_t)(inputDim / 256) * 144;
    int rc = check_common(x, w_gate, h, inputDim, hiddenDim, tokens, 256, row_bytes, 16);
    if (rc) return rc;
    if ((rc = check_common(x, w_up, h, inputDim, hiddenDim, tokens, 256, row_bytes, 16))) return rc;
    if (inputDim > Q4MM_FFN_MAX_INPUT_DIM)
        return fail(Q4MM_ERR_DIM, "inputDim %d exceeds the fused FFN limit %d", inputDim, Q4MM_FFN_MAX_INPUT_DIM);
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    const uint8_t *Wg = static_cast<const uint8_t *>(w_gate), *Wu = static_cast<const uint8_t *>(w_up);
    // From 3 tokens on: the FP32 register-tile kernel over both weights, up
    // to 8 tokens per pass; 1-2 tokens (or a geometry it cannot hold): the
    // one-token kernel, one launch per token.
    if (tokens >= 3) {
        cudaError_t e = cudaSuccess;
        for (int t0 = 0; t0 < tokens && e == cudaSuccess; t0 += 8) {
            const int tt = tokens - t0 < 8 ? tokens - t0 : 8;
            e = q4mm::launch_q4k_ffn_swiglu_multi(ctx, x + (size_t)t0 * inputDim, Wg, Wu, h + (size_t)t0 * hiddenDim,
                                                  inputDim, hiddenDim, tt);
            if (e == cudaErrorNotSupported && t0 == 0) break;  // nothing launched yet
        }
        if (e == cudaSuccess) return Q4MM_OK;
        if (e != cudaErrorNotSupported) return fail_cuda(e, "q4k_ffn_swiglu launch");
    }
    for (int t = 0; t < tokens; ++t) {
        const cudaError_t e = q4mm::launch_q4k_ffn_swiglu_t1(ctx, x + (size_t)t * inputDim, Wg, Wu,
                                                             h + (size_t)t * hiddenDim, inputDim, hiddenDim);
        if (e != cudaSuccess) return fail_cuda(e, "q4k_ffn_swiglu launch");
    }
    return Q4MM_OK;
}

int ternary_gemv(const float *x, const void *w_packed, float scale, float *y, int inputDim,
                 int outputDim, int tokens, q4mm_stream_t stream) {
    int rc = check_common(x, w_packed, y, inputDim, outputDim, tokens, 4, (size_t)inputDim / 4, 1);
    if (rc) return rc;
    q4mm::LaunchCtx ctx;
    if ((rc = device_ctx(stream, &ctx))) return rc;
    cudaError_t e = q4mm::launch_ternary_gemv(ctx, x, static_cast<const uint8_t *>(w_packed), scale, y,
                                              inputDim, outputDim, tokens);
    if (e != cudaSuccess) return fail_cuda(e, "ternary_gemv launch");
    return Q4MM_OK;
}

const char *q4mm_last_error(void) { return g_err; }

int q4mm_device_status(q4mm_stream_t stream, int clear) {
    q4mm::LaunchCtx ctx;
    int rc = device_ctx(stream, &ctx, false);
    if (rc) return rc;
    int host = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&host, ctx.status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "reading the device status word");
    if (clear && host) {
        const int zero = 0;
        e = cudaMemcpyAsync(ctx.status, &zero, sizeof(int), cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return fail_cuda(e, "clearing the device status word");
    }
    if (host) return fail(Q4MM_ERR_TIMEOUT, "a bounded in-kernel wait ran out (status word %d)", host);
    return Q4MM_OK;
}

int q4mm_test_fail_next_wait(int stage, long long limit_cycles) {
    if (stage == -1) {
        g_test_fault.armed = false;
        return Q4MM_OK;
    }
    if (stage < 0 || limit_cycles <= 0)
        return fail(Q4MM_ERR_DIM, "q4mm_test_fail_next_wait: stage (%d) must be >= 0 (or -1) and limit (%lld) > 0",
                    stage, limit_cycles);
    g_test_fault.armed = true;
    g_test_fault.stage = stage;
    g_test_fault.limit = limit_cycles;
    return Q4MM_OK;
}

int q4mm_version(void) { return 200; }

}  // extern "C"
