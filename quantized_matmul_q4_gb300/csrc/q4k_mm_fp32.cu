// Q4_K prefill matmul, FP32 FMA (the 1e-4 variant), sm_103a.
//
// y[t][o] = Σ_k x[t][k]·w[o][k], w = d·sc_s·q − dmin·m_s (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline").  A cluster of S = 3 CTAs owns 128 output rows and 64
// tokens, each CTA a third of K, so every weight byte is read once per call
// for up to 64 tokens (the rule behind llama.cpp PR #37 "ggml-cpu:
// cache-aware tiling in ggml_compute_forward_mul_mat", item 1, applied to the
// GPU tile shape) while 86 row tiles of an 11008-row weight keep 258 CTAs,
// two per SM, busy.
//
// Per chunk of 64 values of K, double-buffered in shared memory:
//  * thread (r, h) dequantizes qs bytes 16h..16h+15 of row r's slab to fp32
//    (d·sc·q − dmin·m with one rounding, the oracle's fp32 weight) and stores
//    them k-major, [k][row];
//  * thread (t, kq) stores x[t][16kq .. 16kq+15] k-major, [k][token];
//  * each thread accumulates an 8-row × 4-token register tile, one k at a
//    time from two 16-byte loads of weights and one of activations (lanes of
//    a warp share rows, so the weight loads are broadcasts), with paired FMAs
//    over adjacent rows.
// The global loads of chunk c+1 are issued before the FMAs of chunk c.
// Ranks 1, 2 then store their partial tiles into rank 0's shared memory
// (distributed shared memory), and rank 0 adds them in rank order, stages
// the tile and writes y row by row, so results do not depend on scheduling.
#include <utility>

#include "cluster.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace q4mm {

namespace {

constexpr int kFRows = 128;                 // weight rows per cluster tile
constexpr int kFTok = 64;                   // tokens per tile
constexpr int kFKc = 64;                    // K values per chunk (one qs slab)
constexpr int kFThreads = 256;
constexpr int kFS = 3;                      // CTAs per cluster (split of K)
constexpr int kFWPitch = kFRows + 4;        // [k][row], rows 16-byte aligned
constexpr int kFXPitch = kFTok + 4;         // [k][token]
constexpr int kFBufFloats = kFKc * (kFWPitch + kFXPitch);
constexpr size_t kFSmem = 2 * (size_t)kFBufFloats * sizeof(float);  // 102,400 bytes
// After the main loop: rank 0 receives (S − 1) partial tiles [128][64] and
// stages the summed tile [64 tokens][129].
constexpr int kFYPitch = kFRows + 1;
static_assert((size_t)((kFS - 1) * kFRows * kFTok + kFTok * kFYPitch) * sizeof(float) <= kFSmem,
              "the reduction reuses the chunk buffers");

// Row i (0..7) of the register tile, token t.
__device__ __forceinline__ float row_acc(const float2 (&acc)[4][4], int i, int t) {
    return (i & 1) ? acc[i >> 1][t].y : acc[i >> 1][t].x;
}

__global__ void __launch_bounds__(kFThreads, 2)
    q4k_mm_fp32_kernel(const float *__restrict__ x, const uint8_t *__restrict__ W, float *__restrict__ y, int K,
                       int N, int T) {
    extern __shared__ __align__(16) float fsm[];
    const int tid = threadIdx.x;
    const int S = (int)cluster_size(), rank = (int)cluster_rank();
    const int row0 = (blockIdx.x / S) * kFRows;
    const int nb = K / kQ4kValues;
    const size_t row_bytes = (size_t)nb * kQ4kBytes;
    const int nc_all = K / kFKc;
    const int c_base = rank * nc_all / S;
    const int nchunks = (rank + 1) * nc_all / S - c_base;

    // Dequant role: row r, byte half h.  Staging role: token tk, quarter kq.
    const int r = tid & (kFRows - 1), h = tid >> 7;
    const int tk = tid & (kFTok - 1), kq = tid >> 6;
    const bool row_ok = row0 + r < N;
    const bool tok_ok = tk < T;
    const uint8_t *wrow = W + (size_t)(row0 + (row_ok ? r : 0)) * row_bytes;
    const float *xrow = x + (size_t)(tok_ok ? tk : 0) * K;
    // Compute role: rows 8·rg .. +7, tokens 4·tg .. +3.
    const int rg = tid >> 4, tg = tid & 15;

    uint4 hdr = make_uint4(0, 0, 0, 0), q = hdr;
    float4 xv[4];
    auto load_w = [&](int c) {  // chunk c of this CTA
        if (row_ok) {
            const int ca = c_base + c, b = ca >> 2, j = ca & 3;
            const uint8_t *blk = wrow + (size_t)b * kQ4kBytes;
            hdr = ld_stream_u4(blk);
            q = ld_stream_u4(blk + 16 + 32 * j + 16 * h);
        }
    };
    auto load_x = [&](int c) {
        const float4 *src = reinterpret_cast<const float4 *>(xrow + (size_t)(c_base + c) * kFKc + 16 * kq);
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = tok_ok ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto store_chunk = [&](int c, float *buf) {
        float *ws = buf, *xs = buf + kFKc * kFWPitch;
        // Weights: 16 low-nibble values (sub-block 2j, k = 16h..) and 16 high
        // (2j+1, k = 32 + 16h..), each d·sc·q − dmin·m rounded once.
        const int j = (c_base + c) & 3;
        float lo_s = 0.f, lo_o = 0.f, hi_s = 0.f, hi_o = 0.f;
        if (row_ok) {
            const float2 dm = q4k_d_dmin(hdr.x);
            const Q4kScales u = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
            const int sl = 2 * j, sh = 2 * j + 1;
            lo_s = dm.x * byte_to_float(sl < 4 ? u.sc_lo : u.sc_hi, sl & 3);
            lo_o = dm.y * byte_to_float(sl < 4 ? u.m_lo : u.m_hi, sl & 3);
            hi_s = dm.x * byte_to_float(sh < 4 ? u.sc_lo : u.sc_hi, sh & 3);
            hi_o = dm.y * byte_to_float(sh < 4 ? u.m_lo : u.m_hi, sh & 3);
        }
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t byte = (qw[w] >> (8 * e)) & 0xFFu;
                const int k = 16 * h + 4 * w + e;
                ws[k * kFWPitch + r] = fmaf(lo_s, static_cast<float>(byte & 15u), -lo_o);
                ws[(32 + k) * kFWPitch + r] = fmaf(hi_s, static_cast<float>(byte >> 4), -hi_o);
            }
        }
        // Activations, k-major.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = 16 * kq + 4 * i;
            xs[(k + 0) * kFXPitch + tk] = xv[i].x;
            xs[(k + 1) * kFXPitch + tk] = xv[i].y;
            xs[(k + 2) * kFXPitch + tk] = xv[i].z;
            xs[(k + 3) * kFXPitch + tk] = xv[i].w;
        }
    };

    // acc[p][t] holds rows 8·rg + 2p and 8·rg + 2p + 1 of token 4·tg + t, so
    // one paired FMA takes a pair of adjacent weights against one activation.
    float2 acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[i][t] = make_float2(0.f, 0.f);

    pdl_launch_dependents();
    if (nchunks > 0) load_w(0);  // weights are never written by an earlier kernel
    // x may be produced by the previous kernel on the stream.
    pdl_wait();
    if (nchunks > 0) load_x(0);
    for (int c = 0; c < nchunks; ++c) {
        float *buf = fsm + (c & 1) * kFBufFloats;
        store_chunk(c, buf);
        if (c + 1 < nchunks) {
            load_w(c + 1);
            load_x(c + 1);
        }
        __syncthreads();
        const float *ws = buf, *xs = buf + kFKc * kFWPitch;
#pragma unroll 4
        for (int k = 0; k < kFKc; ++k) {
            const float4 wa = *reinterpret_cast<const float4 *>(ws + k * kFWPitch + 8 * rg);
            const float4 wb = *reinterpret_cast<const float4 *>(ws + k * kFWPitch + 8 * rg + 4);
            const float4 xt = *reinterpret_cast<const float4 *>(xs + k * kFXPitch + 4 * tg);
            const float2 wp[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w), make_float2(wb.x, wb.y),
                                  make_float2(wb.z, wb.w)};
            const float xr[4] = {xt.x, xt.y, xt.z, xt.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 xx = make_float2(xr[t], xr[t]);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[p][t] = __ffma2_rn(wp[p], xx, acc[p][t]);
            }
        }
    }

    // Split-K reduction in rank 0's shared memory: slices [S−1][128][64].
    __syncthreads();   // this CTA's chunk buffers are idle
    cluster_sync_all();  // ... and so are rank 0's
    if (rank != 0) {
        const uint32_t dst = map_to_rank(smem_addr(fsm), 0) +
                             (uint32_t)(((rank - 1) * kFRows * kFTok) * sizeof(float));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            st_cluster_v4(dst + (uint32_t)(((8 * rg + i) * kFTok + 4 * tg) * sizeof(float)),
                          make_float4(row_acc(acc, i, 0), row_acc(acc, i, 1), row_acc(acc, i, 2),
                                      row_acc(acc, i, 3)));
    }
    cluster_sync_all();
    if (rank == 0) {
        float *ysm = fsm + (kFS - 1) * kFRows * kFTok;  // [64 tokens][129]
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 v = make_float4(row_acc(acc, i, 0), row_acc(acc, i, 1), row_acc(acc, i, 2), row_acc(acc, i, 3));
            for (int s = 1; s < S; ++s) {
                const float4 p =
                    *reinterpret_cast<const float4 *>(fsm + (s - 1) * kFRows * kFTok + (8 * rg + i) * kFTok + 4 * tg);
                v.x += p.x;
                v.y += p.y;
                v.z += p.z;
                v.w += p.w;
            }
            ysm[(4 * tg + 0) * kFYPitch + 8 * rg + i] = v.x;
            ysm[(4 * tg + 1) * kFYPitch + 8 * rg + i] = v.y;
            ysm[(4 * tg + 2) * kFYPitch + 8 * rg + i] = v.z;
            ysm[(4 * tg + 3) * kFYPitch + 8 * rg + i] = v.w;
        }
        __syncthreads();
        const int ncols = min(kFRows, N - row0);
        for (int i = tid; i < T * kFRows; i += kFThreads) {
            const int t = i / kFRows, col = i % kFRows;
            if (col < ncols) y[(size_t)t * N + row0 + col] = ysm[t * kFYPitch + col];
        }
    }
}

}  // namespace

cudaError_t launch_q4k_mm_fp32(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                               int K, int N, int T) {
    cudaError_t e = ensure_smem(q4k_mm_fp32_kernel, kFSmem);
    if (e != cudaSuccess) return e;
    const int tiles = (N + kFRows - 1) / kFRows;
    for (int t0 = 0; t0 < T && e == cudaSuccess; t0 += kFTok) {
        const int tt = min(kFTok, T - t0);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(tiles * kFS);
        cfg.blockDim = dim3(kFThreads);
        cfg.dynamicSmemBytes = kFSmem;
        cfg.stream = c.stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kFS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        int nattr = 1;
        if (c.pdl) {
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            nattr = 2;
        }
        cfg.attrs = attr;
        cfg.numAttrs = nattr;
        e = cudaLaunchKernelEx(&cfg, q4k_mm_fp32_kernel, x + (size_t)t0 * K, W, y + (size_t)t0 * N, K, N, tt);
    }
    return e;
}

}  // namespace q4mm
