// BitNet b1.58 ternary GEMV, FP32, sm_103a.
//
// y[t][o] = scale · Σ_k x[t][k]·code(o,k) with code(o,i) = ((byte >> 2·(i%4))
// & 3) − 1 read from byte o·K/4 + i/4, accumulated in FP32, the scale applied
// once to the finished dot (SKaiNET issue #1138 "[ternary-f32] Phase 2:
// TernaryF32GemvNative SPI + reference ViewKernel + TernaryF32KernelPack",
// section "Tasks").  Rows of tokens advance by r·K in x and r·N in y.
//
// Decode: for field i of each byte of a 32-bit word, (w << (5 − 2i)) masked
// with 0x60606060 leaves field value c ∈ {0..3} in bits 5-6 of each byte; a
// byte permute places one such byte under the exponent byte 0x3F, giving the
// float 0.5 + c/8 (see field_biased).  With acc = Σ x·(0.5 + c/8) over a
// lane's positions and sx = Σ x over the same positions,
//   Σ x·(c − 1) = 8·acc − 5·sx,
// exact for integer activations (every partial sum is a multiple of 1/8 far
// below 2^21), so the code-dot is bit-exact there and the scale multiply is a
// single fp32 rounding.
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace q4mm {

namespace {

constexpr int kTernWarps = 8;
constexpr int kTernChunk = 4096;  // K values of x per shared-memory chunk (multiple of 16)

template <int k>
__device__ __forceinline__ float field_biased(uint32_t w) {
    return __uint_as_float(__byte_perm(w, 0x3F000000u, 0x7054u | (k << 8)));
}

template <int i>
__device__ __forceinline__ uint32_t field_bits(uint32_t w) {
    // Field i of every byte moved to bits 5-6 of that byte.
    if constexpr (i == 3)
        return (w >> 1) & 0x60606060u;
    else
        return (w << (5 - 2 * i)) & 0x60606060u;
}

template <bool kWordAligned>
__device__ __forceinline__ uint32_t load_word(const uint8_t *p) {
    if constexpr (kWordAligned) {
        return ld_stream_u32(p);
    } else {
        return ld_stream_u8(p) | (ld_stream_u8(p + 1) << 8) | (ld_stream_u8(p + 2) << 16) |
               (ld_stream_u8(p + 3) << 24);
    }
}

// One warp per output row per pass; lane l handles the 32-bit words
// l, l+32, l+64, … of the row's K/4 bytes (16 positions each), coalesced.
// x for one K-chunk of all T tokens sits in shared memory.
template <int T, bool kWordAligned>
__global__ void __launch_bounds__(32 * kTernWarps) ternary_gemv_kernel(
    const float *__restrict__ x, const uint8_t *__restrict__ W, float scale, float *__restrict__ y,
    int K, int N, int rows_per_cta) {
    extern __shared__ __align__(16) float tsm[];
    float *xsm = tsm;                  // [T][chunk]
    float *acc = tsm + T * kTernChunk; // [rows_per_cta][T]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * rows_per_cta;
    const int nrows = min(rows_per_cta, N - row0);
    const size_t row_bytes = (size_t)K / 4;

    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i < nrows * T; i += blockDim.x) acc[i] = 0.f;

    for (int c0 = 0; c0 < K; c0 += kTernChunk) {
        const int ck = min(kTernChunk, K - c0);  // multiple of 4
        __syncthreads();
        for (int i = threadIdx.x; i < T * (ck / 4); i += blockDim.x) {
            const int t = i / (ck / 4), u = i % (ck / 4);
            reinterpret_cast<float4 *>(xsm + t * kTernChunk)[u] =
                __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * K + c0) + u);
        }
        __syncthreads();

        const int full_words = ck / 16;     // words with 16 positions
        const int tail = (ck % 16) / 4;     // trailing bytes (< 4) of this chunk
        for (int rl = warp; rl < nrows; rl += kTernWarps) {
            const uint8_t *row = W + (size_t)(row0 + rl) * row_bytes + c0 / 4;
            float2 a[T];
            float sx[T];
#pragma unroll
            for (int t = 0; t < T; ++t) {
                a[t] = make_float2(0.f, 0.f);
                sx[t] = 0.f;
            }
            for (int wi = lane; wi < full_words; wi += 32) {
                const uint32_t w = load_word<kWordAligned>(row + 4 * wi);
                // Byte k of field_bits<i>(w) is the field of position 16wi + 4k + i.
                const uint32_t f0 = field_bits<0>(w), f1 = field_bits<1>(w);
                const uint32_t f2 = field_bits<2>(w), f3 = field_bits<3>(w);
                float c[16];
                c[0] = field_biased<0>(f0); c[1] = field_biased<0>(f1);
                c[2] = field_biased<0>(f2); c[3] = field_biased<0>(f3);
                c[4] = field_biased<1>(f0); c[5] = field_biased<1>(f1);
                c[6] = field_biased<1>(f2); c[7] = field_biased<1>(f3);
                c[8] = field_biased<2>(f0); c[9] = field_biased<2>(f1);
                c[10] = field_biased<2>(f2); c[11] = field_biased<2>(f3);
                c[12] = field_biased<3>(f0); c[13] = field_biased<3>(f1);
                c[14] = field_biased<3>(f2); c[15] = field_biased<3>(f3);
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float4 *xv = reinterpret_cast<const float4 *>(xsm + t * kTernChunk + 16 * wi);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 v = xv[q];
                        a[t] = ffma2(make_float2(v.x, v.y), make_float2(c[4 * q], c[4 * q + 1]), a[t]);
                        a[t] = ffma2(make_float2(v.z, v.w), make_float2(c[4 * q + 2], c[4 * q + 3]), a[t]);
                        sx[t] += (v.x + v.y) + (v.z + v.w);
                    }
                }
            }
            if (lane < tail) {
                // Remaining whole bytes (4 positions each) after the last word.
                const int byte_i = full_words * 4 + lane;
                const uint32_t bv = ld_stream_u8(row + byte_i);
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float *xv = xsm + t * kTernChunk + 4 * byte_i;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float cf = __uint_as_float(
                            __byte_perm((bv << 5 >> (2 * i)) & 0x60u, 0x3F000000u, 0x7054u));
                        a[t].x = fmaf(xv[i], cf, a[t].x);
                        sx[t] += xv[i];
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const float part = fmaf(8.f, a[t].x + a[t].y, -5.f * sx[t]);
                const float v = warp_sum(part);
                if (lane == 0) acc[rl * T + t] += v;
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nrows * T; i += blockDim.x) {
        const int rl = i / T, t = i % T;
        y[(size_t)t * N + row0 + rl] = acc[i] * scale;
    }
}

template <int T>
cudaError_t launch_t(const LaunchCtx &c, const float *x, const uint8_t *W, float scale, float *y,
                     int K, int N, bool aligned) {
    int grid = 2 * c.num_sms;
    int rows_per_cta = (N + grid - 1) / grid;
    grid = (N + rows_per_cta - 1) / rows_per_cta;
    const size_t smem = (size_t)T * kTernChunk * sizeof(float) + (size_t)rows_per_cta * T * sizeof(float);
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;
    if (aligned) {
        cudaError_t e = ensure_smem(ternary_gemv_kernel<T, true>, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(c, ternary_gemv_kernel<T, true>, dim3(grid), dim3(32 * kTernWarps), smem,
                             x, W, scale, y, K, N, rows_per_cta);
    }
    cudaError_t e = ensure_smem(ternary_gemv_kernel<T, false>, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(c, ternary_gemv_kernel<T, false>, dim3(grid), dim3(32 * kTernWarps), smem, x,
                         W, scale, y, K, N, rows_per_cta);
}

}  // namespace

cudaError_t launch_ternary_gemv(const LaunchCtx &c, const float *x, const uint8_t *W, float scale,
                                float *y, int K, int N, int T) {
    // Word loads need 4-byte aligned rows: row stride K/4 a multiple of 4 and W aligned.
    const bool aligned = (K % 16 == 0) && ((reinterpret_cast<uintptr_t>(W) & 3) == 0);
    // Token tiles of up to 8 (the weights are re-read per tile only above 8 tokens).
    cudaError_t e = cudaSuccess;
    for (int t0 = 0; t0 < T && e == cudaSuccess; t0 += 8) {
        const int tt = min(8, T - t0);
        const float *xt = x + (size_t)t0 * K;
        float *yt = y + (size_t)t0 * N;
        switch (tt) {
            case 1: e = launch_t<1>(c, xt, W, scale, yt, K, N, aligned); break;
            case 2: e = launch_t<2>(c, xt, W, scale, yt, K, N, aligned); break;
            case 3: e = launch_t<3>(c, xt, W, scale, yt, K, N, aligned); break;
            case 4: e = launch_t<4>(c, xt, W, scale, yt, K, N, aligned); break;
            case 5: e = launch_t<5>(c, xt, W, scale, yt, K, N, aligned); break;
            case 6: e = launch_t<6>(c, xt, W, scale, yt, K, N, aligned); break;
            case 7: e = launch_t<7>(c, xt, W, scale, yt, K, N, aligned); break;
            default: e = launch_t<8>(c, xt, W, scale, yt, K, N, aligned); break;
        }
    }
    return e;
}

}  // namespace q4mm
