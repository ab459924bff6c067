// Q4_K decode GEMV kernels (1..8 tokens), FP32 arithmetic, sm_103a.
//
// Computes y[t][o] = Σ_k x[t][k]·w[o][k] with w = d·sc_s·q − dmin·m_s decoded
// on the fly from the 144-byte Q4_K super-blocks (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline").  As on that page, one load of a qs byte feeds both the
// low-nibble accumulator (sub-block 2j) and the high-nibble one (2j+1), and
// the min term is applied lazily once per sub-block from the sum of the
// inputs, never per weight.
//
// GPU design (not the page's): a "slab lane" owns one 32-byte qs slab j of
// one block b — 64 weights of sub-blocks 2j and 2j+1 — for every row it
// visits, so the 64 matching activations live in its registers for the whole
// kernel.  Weight rows are streamed once from HBM into a shared-memory ring by
// 1-D bulk copies (cp.async.bulk) that one producer thread issues before the
// kernel even waits for the previous kernel on the stream (weights are never
// written by it), so the stream of weight bytes starts at launch.
//
// Nibble decode: a masked code q in byte k of a word becomes the float
// 0.5 + q/256 with one byte permute (see nib_biased).  The bias 0.5·Σx is
// removed together with the lazy min term: per sub-block s the contribution
// is (256·d·sc_s)·acc_s − (128·d·sc_s + dmin·m_s)·Σx_s where
// acc_s = Σ x·(0.5 + q/256).
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace q4mm {

namespace {

// ----------------------------------------------------------------------------
// Shared slab arithmetic
// ----------------------------------------------------------------------------

// Per-lane constants for the two sub-blocks 2j and 2j+1 of a block:
// scale' = 256·d·sc and offset' = 128·d·sc + dmin·m.
struct SlabScales {
    float s0, s1, o0, o1;
};

__device__ __forceinline__ SlabScales slab_scales(uint4 hdr, int j) {
    const float2 dm = q4k_d_dmin(hdr.x);
    const Q4kScales u = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
    const bool upper = j >= 2;  // sub-blocks 4..7 use the split 6-bit fields
    const uint32_t scw = upper ? u.sc_hi : u.sc_lo;
    const uint32_t mw = upper ? u.m_hi : u.m_lo;
    const int k0 = 2 * (j & 1);
    const float d256 = dm.x * 256.0f;  // exact: power-of-two scaling
    SlabScales r;
    r.s0 = d256 * byte_to_float(scw, k0);  // exact: 11-bit × 6-bit
    r.s1 = d256 * byte_to_float(scw, k0 + 1);
    r.o0 = fmaf(dm.y, byte_to_float(mw, k0), 0.5f * r.s0);
    r.o1 = fmaf(dm.y, byte_to_float(mw, k0 + 1), 0.5f * r.s1);
    return r;
}

// Σ x·(0.5 + q/256) over the 32 low-nibble and the 32 high-nibble weights of a
// 32-byte slab (q0 = bytes 0..15, q1 = bytes 16..31), x from registers:
// xs[l] pairs with the low nibble of slab byte l, xs[32 + l] with its high
// nibble.
__device__ __forceinline__ void slab_dot(const float (&xs)[64], uint4 q0, uint4 q1, float &lo,
                                         float &hi) {
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float2 alo = make_float2(0.f, 0.f), ahi = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t l4 = qw[w] & 0x0F0F0F0Fu;
        const uint32_t h4 = (qw[w] >> 4) & 0x0F0F0F0Fu;
        alo = ffma2(make_float2(xs[4 * w], xs[4 * w + 1]),
                    make_float2(nib_biased<0>(l4), nib_biased<1>(l4)), alo);
        alo = ffma2(make_float2(xs[4 * w + 2], xs[4 * w + 3]),
                    make_float2(nib_biased<2>(l4), nib_biased<3>(l4)), alo);
        ahi = ffma2(make_float2(xs[32 + 4 * w], xs[32 + 4 * w + 1]),
                    make_float2(nib_biased<0>(h4), nib_biased<1>(h4)), ahi);
        ahi = ffma2(make_float2(xs[32 + 4 * w + 2], xs[32 + 4 * w + 3]),
                    make_float2(nib_biased<2>(h4), nib_biased<3>(h4)), ahi);
    }
    lo = alo.x + alo.y;
    hi = ahi.x + ahi.y;
}

// x in shared memory: 16-byte unit u (elements 4u..4u+3) is stored at unit
// u ^ ((u >> 4) & 7), so the eight slab lanes of a quarter warp, which read
// the same unit offset of eight consecutive 64-element slabs, hit eight
// different bank groups.
__device__ __forceinline__ int x_swz(int u) { return u ^ ((u >> 4) & 7); }

// ----------------------------------------------------------------------------
// One token: TMA-staged rows, x slab in registers
// ----------------------------------------------------------------------------

struct T1Params {
    const float *x;
    const uint8_t *W;
    float *y;
    int *status;
    int N;
    int nb;            // blocks per row (K/256)
    int wc;            // warps per row
    int lpr;           // lanes per row (power of two) when wc == 1
    int rpp;           // rows per warp pass (32/lpr when wc == 1, else 1)
    int rg;            // row groups: compute warps = wc·rg
    int rows_per_cta;  // contiguous rows per CTA
    int stage_rows;    // rows per ring slot (multiple of rpp·rg)
    int nslots;        // ring depth
    uint32_t row_bytes;
};

__global__ void __launch_bounds__(32 * 9, 2) q4k_gemv_t1_kernel(T1Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncw = p.wc * p.rg;
    const uint32_t slot_bytes = p.stage_rows * p.row_bytes;
    uint8_t *ring = smem;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + (size_t)p.nslots * slot_bytes);
    uint64_t *empty_bar = full_bar + p.nslots;
    float *xsm = reinterpret_cast<float *>(empty_bar + p.nslots);  // K floats, swizzled
    float *part = xsm + p.nb * kQ4kValues;                         // [rows_per_cta][wc]

    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int nstages = (nrows + p.stage_rows - 1) / p.stage_rows;

    // Bulk copies need a 16-byte aligned destination; never issue one otherwise.
    if (smem_addr(smem) & 15) {
        if (threadIdx.x == 0) flag_timeout(p.status);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], ncw);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        // Producer: stream this CTA's contiguous rows, stage by stage.
        if (lane == 0) {
            const uint8_t *src = p.W + (size_t)row0 * p.row_bytes;
            for (int st = 0; st < nstages; ++st) {
                const int slot = st % p.nslots;
                if (st >= p.nslots &&
                    !mbar_wait_bounded(&empty_bar[slot], ((st / p.nslots) - 1) & 1,
                                       kWaitLimitCycles)) {
                    abort_flag = 1;
                    flag_timeout(p.status);
                    break;
                }
                if (abort_flag) break;
                const int rows = min(p.stage_rows, nrows - st * p.stage_rows);
                const uint32_t bytes = rows * p.row_bytes;
                mbar_arrive_expect_tx(&full_bar[slot], bytes);
                bulk_g2s(ring + (size_t)slot * slot_bytes,
                         src + (size_t)st * p.stage_rows * p.row_bytes, bytes, &full_bar[slot]);
            }
        }
    } else {
        const int cw = warp - 1;
        const int wcol = cw % p.wc, rgi = cw / p.wc;
        int s, ro;
        if (p.wc == 1) {
            ro = lane / p.lpr;
            s = lane % p.lpr;
        } else {
            ro = 0;
            s = wcol * 32 + lane;
        }
        const bool active = s < 4 * p.nb;
        const int b = active ? (s >> 2) : 0, j = s & 3;

        // x may be produced by the previous kernel on the stream.
        pdl_wait();
        const int K = p.nb * kQ4kValues;
        for (int u = threadIdx.x - 32; u < K / 4; u += ncw * 32) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p.x) + u);
            reinterpret_cast<float4 *>(xsm)[x_swz(u)] = v;
        }
        named_bar_sync(1, ncw * 32);

        float xs[64];
        float sum_lo = 0.f, sum_hi = 0.f;
        {
            const int u0 = (b * kQ4kValues + j * 64) / 4;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (active) v = reinterpret_cast<const float4 *>(xsm)[x_swz(u0 + i)];
                xs[4 * i] = v.x;
                xs[4 * i + 1] = v.y;
                xs[4 * i + 2] = v.z;
                xs[4 * i + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                sum_lo += xs[i];
                sum_hi += xs[32 + i];
            }
        }

        for (int st = 0; st < nstages; ++st) {
            const int slot = st % p.nslots;
            if (abort_flag) break;
            if (!mbar_wait_bounded(&full_bar[slot], (st / p.nslots) & 1, kWaitLimitCycles)) {
                abort_flag = 1;
                flag_timeout(p.status);
                break;
            }
            const uint8_t *stage = ring + (size_t)slot * slot_bytes;
            const int rows = min(p.stage_rows, nrows - st * p.stage_rows);
            for (int pass = rgi; pass * p.rpp < rows; pass += p.rg) {
                const int rl = pass * p.rpp + ro;
                float partial = 0.f;
                if (active && rl < rows) {
                    const uint8_t *blk = stage + (size_t)rl * p.row_bytes + b * kQ4kBytes;
                    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j);
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * j);
                    const SlabScales sc = slab_scales(hdr, j);
                    float lo, hi;
                    slab_dot(xs, q0, q1, lo, hi);
                    partial = fmaf(sc.s0, lo, sc.s1 * hi) - fmaf(sc.o0, sum_lo, sc.o1 * sum_hi);
                }
                if (p.wc == 1) {
                    partial = group_sum(partial, p.lpr);
                    if (s == 0 && rl < rows) p.y[row0 + st * p.stage_rows + rl] = partial;
                } else {
                    partial = warp_sum(partial);
                    if (lane == 0 && rl < rows)
                        part[(st * p.stage_rows + rl) * p.wc + wcol] = partial;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
        }

        if (p.wc > 1) {
            named_bar_sync(1, ncw * 32);
            for (int i = threadIdx.x - 32; i < nrows; i += ncw * 32) {
                float acc = 0.f;
                for (int w = 0; w < p.wc; ++w) acc += part[i * p.wc + w];
                p.y[row0 + i] = acc;
            }
        }
    }

    // Never leave a bulk copy writing into shared memory of an exiting CTA.
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) {
        for (int st = max(0, nstages - p.nslots); st < nstages; ++st)
            (void)mbar_wait_bounded(&full_bar[st % p.nslots], (st / p.nslots) & 1,
                                    kWaitLimitCycles);
    }
}

// ----------------------------------------------------------------------------
// 1..8 tokens: x staged in shared memory by K-chunks, weights by plain loads
// ----------------------------------------------------------------------------

constexpr int kMultiWarps = 8;
constexpr int kMultiChunkBlocks = 8;  // blocks per K-chunk: one warp spans a row-chunk

struct MultiParams {
    const float *x;
    const uint8_t *W;
    float *y;
    int K, N;
    int nb;            // blocks per row
    int chunk_blocks;  // blocks per K-chunk (<= 8)
    int lpr;           // lanes per row-chunk (power of two, >= 4·chunk_blocks)
    int rows_per_cta;
};

template <int T>
__global__ void __launch_bounds__(32 * kMultiWarps) q4k_gemv_multi_kernel(MultiParams p) {
    extern __shared__ __align__(16) float msm[];
    float *xsm = msm;                                         // [T][chunk·256] swizzled
    float *acc = msm + T * p.chunk_blocks * kQ4kValues;       // [rows_per_cta][T]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rpp = 32 / p.lpr;
    const int ro = lane / p.lpr, s = lane % p.lpr;
    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const size_t row_bytes = (size_t)p.nb * kQ4kBytes;
    const int chunk_elems = p.chunk_blocks * kQ4kValues;

    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i < nrows * T; i += blockDim.x) acc[i] = 0.f;

    for (int c0 = 0; c0 < p.nb; c0 += p.chunk_blocks) {
        const int cb = min(p.chunk_blocks, p.nb - c0);
        __syncthreads();  // previous chunk's x no longer in use; acc zeroed
        for (int i = threadIdx.x; i < T * cb * 64; i += blockDim.x) {
            const int t = i / (cb * 64), u = i % (cb * 64);
            const float4 v =
                __ldg(reinterpret_cast<const float4 *>(p.x + (size_t)t * p.K + c0 * kQ4kValues) + u);
            reinterpret_cast<float4 *>(xsm + t * chunk_elems)[x_swz(u)] = v;
        }
        __syncthreads();

        const bool active = s < 4 * cb;
        const int b = active ? (s >> 2) : 0, j = s & 3;
        const int u0 = (b * kQ4kValues + j * 64) / 4;
        for (int pass = warp; pass * rpp < nrows; pass += kMultiWarps) {
            const int rl = pass * rpp + ro;
            float2 a[T];
#pragma unroll
            for (int t = 0; t < T; ++t) a[t] = make_float2(0.f, 0.f);
            if (active && rl < nrows) {
                const uint8_t *blk =
                    p.W + (size_t)(row0 + rl) * row_bytes + (size_t)(c0 + b) * kQ4kBytes;
                const uint4 hdr = ld_stream_u4(blk);
                const uint4 q0 = ld_stream_u4(blk + 16 + 32 * j);
                const uint4 q1 = ld_stream_u4(blk + 32 + 32 * j);
                const SlabScales sc = slab_scales(hdr, j);
                const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const uint32_t l4 = qw[w] & 0x0F0F0F0Fu;
                    const uint32_t h4 = (qw[w] >> 4) & 0x0F0F0F0Fu;
                    // Dequantized weights: scale'·(0.5 + q/256) − offset' = d·sc·q − dmin·m.
                    const float2 s0 = make_float2(sc.s0, sc.s0), n0 = make_float2(-sc.o0, -sc.o0);
                    const float2 s1 = make_float2(sc.s1, sc.s1), n1 = make_float2(-sc.o1, -sc.o1);
                    const float2 wl01 = ffma2(make_float2(nib_biased<0>(l4), nib_biased<1>(l4)), s0, n0);
                    const float2 wl23 = ffma2(make_float2(nib_biased<2>(l4), nib_biased<3>(l4)), s0, n0);
                    const float2 wh01 = ffma2(make_float2(nib_biased<0>(h4), nib_biased<1>(h4)), s1, n1);
                    const float2 wh23 = ffma2(make_float2(nib_biased<2>(h4), nib_biased<3>(h4)), s1, n1);
#pragma unroll
                    for (int t = 0; t < T; ++t) {
                        const float4 *xt = reinterpret_cast<const float4 *>(xsm + t * chunk_elems);
                        const float4 xl = xt[x_swz(u0 + w)];
                        const float4 xh = xt[x_swz(u0 + 8 + w)];
                        a[t] = ffma2(make_float2(xl.x, xl.y), wl01, a[t]);
                        a[t] = ffma2(make_float2(xl.z, xl.w), wl23, a[t]);
                        a[t] = ffma2(make_float2(xh.x, xh.y), wh01, a[t]);
                        a[t] = ffma2(make_float2(xh.z, xh.w), wh23, a[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const float v = group_sum(a[t].x + a[t].y, p.lpr);
                if (s == 0 && rl < nrows) acc[rl * T + t] += v;
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nrows * T; i += blockDim.x) {
        const int rl = i / T, t = i % T;
        p.y[(size_t)t * p.N + row0 + rl] = acc[i];
    }
}

int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

}  // namespace

cudaError_t launch_q4k_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                               int K, int N) {
    T1Params p;
    p.x = x;
    p.W = W;
    p.y = y;
    p.status = c.status;
    p.N = N;
    p.nb = K / kQ4kValues;
    p.row_bytes = (uint32_t)p.nb * kQ4kBytes;
    const int L = 4 * p.nb;
    if (L <= 32) {
        p.wc = 1;
        p.lpr = next_pow2(L);
        p.rpp = 32 / p.lpr;
    } else {
        p.wc = (L + 31) / 32;
        p.lpr = 32;
        p.rpp = 1;
    }
    // At most 8 compute warps (+1 producer): wider rows go to the generic kernel.
    if (p.wc > 8) return cudaErrorNotSupported;
    const int target_warps = 8;
    p.rg = max(1, target_warps / p.wc);
    const int ncw = p.wc * p.rg;
    const int group_rows = p.rpp * p.rg;
    const int m = max(1, 16384 / (int)(group_rows * p.row_bytes));
    p.stage_rows = m * group_rows;
    const size_t slot_bytes = (size_t)p.stage_rows * p.row_bytes;

    // Two CTAs per SM so that the next kernel's CTAs can start streaming while
    // this one drains; rows split evenly and contiguously.
    int grid = 2 * c.num_sms;
    p.rows_per_cta = (N + grid - 1) / grid;
    if (p.rows_per_cta < p.rpp) p.rows_per_cta = p.rpp;
    grid = (N + p.rows_per_cta - 1) / p.rows_per_cta;

    const size_t xs_bytes = (size_t)K * sizeof(float);
    const size_t part_bytes = p.wc > 1 ? (size_t)p.rows_per_cta * p.wc * sizeof(float) : 0;
    const size_t budget = 100 * 1024;
    size_t fixed = xs_bytes + part_bytes + 2 * 8 * 8;
    int nslots = (int)((budget > fixed ? budget - fixed : 0) / slot_bytes);
    const int stages_needed = (p.rows_per_cta + p.stage_rows - 1) / p.stage_rows;
    nslots = min(nslots, max(2, stages_needed));
    nslots = min(nslots, 8);
    if (nslots < 2) {
        nslots = 2;
    }
    p.nslots = nslots;
    const size_t smem = (size_t)nslots * slot_bytes + 2 * nslots * sizeof(uint64_t) + xs_bytes + part_bytes;
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;

    cudaError_t e = ensure_smem(q4k_gemv_t1_kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(c, q4k_gemv_t1_kernel, dim3(grid), dim3(32 * (1 + ncw)), smem, p);
}

cudaError_t launch_q4k_gemv_multi(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                  int K, int N, int T) {
    MultiParams p;
    p.x = x;
    p.W = W;
    p.y = y;
    p.K = K;
    p.N = N;
    p.nb = K / kQ4kValues;
    p.chunk_blocks = min(kMultiChunkBlocks, p.nb);
    p.lpr = next_pow2(4 * p.chunk_blocks);
    int grid = 2 * c.num_sms;
    p.rows_per_cta = (N + grid - 1) / grid;
    grid = (N + p.rows_per_cta - 1) / p.rows_per_cta;
    const size_t smem =
        (size_t)T * p.chunk_blocks * kQ4kValues * sizeof(float) + (size_t)p.rows_per_cta * T * sizeof(float);
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;

#define Q4MM_MULTI_CASE(TT)                                                                    \
    case TT: {                                                                                 \
        cudaError_t e = ensure_smem(q4k_gemv_multi_kernel<TT>, smem);                                       \
        if (e != cudaSuccess) return e;                                                        \
        return launch_kernel(c, q4k_gemv_multi_kernel<TT>, dim3(grid), dim3(32 * kMultiWarps), \
                             smem, p);                                                         \
    }
    switch (T) {
        Q4MM_MULTI_CASE(1)
        Q4MM_MULTI_CASE(2)
        Q4MM_MULTI_CASE(3)
        Q4MM_MULTI_CASE(4)
        Q4MM_MULTI_CASE(5)
        Q4MM_MULTI_CASE(6)
        Q4MM_MULTI_CASE(7)
        Q4MM_MULTI_CASE(8)
        default:
            return cudaErrorInvalidValue;
    }
#undef Q4MM_MULTI_CASE
}

}  // namespace q4mm
