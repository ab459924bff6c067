// Q4_K prefill matmul, FP32 FMA (the 1e-4 variant), sm_103a.
//
// y[t][o] = Σ_k x[t][k]·w[o][k], w = d·sc_s·q − dmin·m_s (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline").  Every weight byte is read once per call: a CTA owns
// BN output rows and all BM tokens of its tile, so the token dimension never
// causes a second pass over the weights (the rule behind llama.cpp PR #37
// "ggml-cpu: cache-aware tiling in ggml_compute_forward_mul_mat", item 1,
// applied to the GPU tile shape).
//
// Per K-step of 64 values (one 32-byte qs slab of one block): the weight slab
// of BN rows is dequantized to fp32 into shared memory (k-major), the matching
// 64 activations of BM tokens are staged k-major, and each thread accumulates
// a 4-row × 8-token register tile with fused multiply-adds.
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace q4mm {

namespace {

constexpr int kBN = 32;       // weight rows per CTA
constexpr int kBM = 64;       // tokens per CTA
constexpr int kKS = 64;       // K values per step (one slab)
constexpr int kThreads = 64;  // 8 row-groups of 4 rows × 8 token-groups of 8 tokens
constexpr int kPadW = kBN + 4;
constexpr int kPadX = kBM + 4;

__global__ void __launch_bounds__(kThreads) q4k_mm_fp32_kernel(const float *__restrict__ x,
                                                               const uint8_t *__restrict__ W,
                                                               float *__restrict__ y, int K, int N,
                                                               int T) {
    __shared__ __align__(16) float ws[kKS][kPadW];  // [k][row]
    __shared__ __align__(16) float xsm[kKS][kPadX]; // [k][token]

    const int tid = threadIdx.x;
    const int ty = tid / 8, tx = tid % 8;  // rows ty*4..+3, tokens tx*8..+7
    const int row0 = blockIdx.x * kBN, tok0 = blockIdx.y * kBM;
    const int nb = K / kQ4kValues;
    const size_t row_bytes = (size_t)nb * kQ4kBytes;

    pdl_launch_dependents();
    pdl_wait();

    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[i][t] = 0.f;

    for (int ks = 0; ks < K / kKS; ++ks) {
        const int b = ks / 4, j = ks % 4;
        // Dequantize the slab: thread → (row r = tid/2, half h = tid%2), each
        // half is one sub-block (h = 0: low nibbles, sub-block 2j; h = 1: high
        // nibbles, sub-block 2j+1), 32 values.
        {
            const int r = tid / 2, h = tid % 2;
            float vals[32];
            if (row0 + r < N) {
                const uint8_t *blk = W + (size_t)(row0 + r) * row_bytes + (size_t)b * kQ4kBytes;
                const uint4 hdr = ld_stream_u4(blk);
                const uint4 q0 = ld_stream_u4(blk + 16 + 32 * j);
                const uint4 q1 = ld_stream_u4(blk + 32 + 32 * j);
                const float2 dm = q4k_d_dmin(hdr.x);
                const Q4kScales u = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
                const int sb = 2 * j + h;
                const uint32_t scw = sb < 4 ? u.sc_lo : u.sc_hi;
                const uint32_t mw = sb < 4 ? u.m_lo : u.m_hi;
                const float scale = dm.x * byte_to_float(scw, sb & 3);
                const float offset = dm.y * byte_to_float(mw, sb & 3);
                const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const uint32_t v = h ? (qw[w] >> 4) : qw[w];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        vals[4 * w + k] = fmaf(scale, (float)((v >> (8 * k)) & 15u), -offset);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) vals[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) ws[32 * h + i][r] = vals[i];
        }
        // Stage the activations: 64 tokens × 64 values, k-major.
        for (int i = tid; i < kBM * (kKS / 4); i += kThreads) {
            const int t = i / (kKS / 4), u = i % (kKS / 4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tok0 + t < T)
                v = __ldg(reinterpret_cast<const float4 *>(x + (size_t)(tok0 + t) * K + ks * kKS) + u);
            xsm[4 * u + 0][t] = v.x;
            xsm[4 * u + 1][t] = v.y;
            xsm[4 * u + 2][t] = v.z;
            xsm[4 * u + 3][t] = v.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kKS; ++k) {
            const float4 wv = *reinterpret_cast<const float4 *>(&ws[k][ty * 4]);
            const float4 xa = *reinterpret_cast<const float4 *>(&xsm[k][tx * 8]);
            const float4 xb = *reinterpret_cast<const float4 *>(&xsm[k][tx * 8 + 4]);
            const float wr[4] = {wv.x, wv.y, wv.z, wv.w};
            const float xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int t = 0; t < 8; ++t) acc[i][t] = fmaf(wr[i], xr[t], acc[i][t]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int o = row0 + ty * 4 + i;
        if (o >= N) continue;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int tt = tok0 + tx * 8 + t;
            if (tt < T) y[(size_t)tt * N + o] = acc[i][t];
        }
    }
}

}  // namespace

cudaError_t launch_q4k_mm_fp32(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                               int K, int N, int T) {
    const dim3 grid((N + kBN - 1) / kBN, (T + kBM - 1) / kBM);
    return launch_kernel(c, q4k_mm_fp32_kernel, grid, dim3(kThreads), 0, x, W, y, K, N, T);
}

}  // namespace q4mm
