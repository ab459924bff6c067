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
#include <cstdlib>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

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

// ---------------------------------------------------------------------------
// One token: streamed rows, x in registers.
//
// A CTA owns a contiguous range of rows; one producer thread streams them
// through a shared-memory ring with bulk copies (each stage a run of whole
// rows, issued before the wait on the previous kernel since the weights do
// not depend on it).  Compute warp c owns word column c % ncol (32
// consecutive 32-bit words, i.e. 512 positions, one word per lane) with the
// 16 activations of its word in registers, and row phase c / ncol.  Rows go
// in groups of 8: eight word loads, decode, FMAs, then a butterfly that
// leaves each row's column sum in one lane, stored as that column's partial
// of the row.  The partials are summed in column order at the end, so the
// result does not depend on scheduling.
// ---------------------------------------------------------------------------

constexpr int kTernT1Warps = 16;  // warp 0 produces, warps 1..15 compute
constexpr int kTernT1Cw = kTernT1Warps - 1;
constexpr int kTernT1Rows = 8;    // rows per group

struct TernT1Params {
    const float *x;
    const uint8_t *W;
    float *y;
    int *status;
    float scale;
    int K, N, row_bytes, rows_per_cta, stage_rows, nslots, ncol;
};

// Decode one 32-bit word of codes into the biased floats 0.5 + c/8 of its 16
// positions, in position order (position 4k + i is field i of byte k).
__device__ __forceinline__ void decode_word(uint32_t w, float (&c)[16]) {
    const uint32_t f0 = field_bits<0>(w), f1 = field_bits<1>(w);
    const uint32_t f2 = field_bits<2>(w), f3 = field_bits<3>(w);
    c[0] = field_biased<0>(f0);  c[1] = field_biased<0>(f1);
    c[2] = field_biased<0>(f2);  c[3] = field_biased<0>(f3);
    c[4] = field_biased<1>(f0);  c[5] = field_biased<1>(f1);
    c[6] = field_biased<1>(f2);  c[7] = field_biased<1>(f3);
    c[8] = field_biased<2>(f0);  c[9] = field_biased<2>(f1);
    c[10] = field_biased<2>(f2); c[11] = field_biased<2>(f3);
    c[12] = field_biased<3>(f0); c[13] = field_biased<3>(f1);
    c[14] = field_biased<3>(f2); c[15] = field_biased<3>(f3);
}

// Butterfly over the warp of V = 8 per-lane values: afterwards lane l holds,
// in v[0], the warp-wide sum of value index (l >> 2) & 7 reversed into the
// halving order (see row_of_lane); lanes differing only in bits 0–1 agree.
__device__ __forceinline__ float reduce8(float (&v)[8], int lane) {
#pragma unroll
    for (int o = 16, half = 4; o >= 4; o >>= 1, half >>= 1) {
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}

// Value index held by `lane` after reduce8: the halving steps at offsets
// 16, 8, 4 select the upper half (4, 2, 1) when the lane's bit is set.
__device__ __forceinline__ int row_of_lane(int lane) {
    return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

__global__ void __launch_bounds__(32 * kTernT1Warps, 1) ternary_t1_kernel(const TernT1Params p) {
    extern __shared__ __align__(128) uint8_t t1_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int nstages = (nrows + p.stage_rows - 1) / p.stage_rows;
    const uint32_t slot_bytes = (uint32_t)p.stage_rows * p.row_bytes;
    uint8_t *ring = t1_smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)p.nslots * slot_bytes);
    uint64_t *empty = full + p.nslots;
    float *part = reinterpret_cast<float *>(empty + p.nslots);  // [ncol][rows_per_cta]
    float *sx = part + (size_t)p.ncol * p.rows_per_cta;          // [ncol] Σ x per column

    // Warps beyond a whole number of column sets idle (they still take part
    // in the final barrier).
    const int nph = kTernT1Cw / p.ncol;
    const int nactive = nph * p.ncol;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nactive);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int s = 0; s < nstages; ++s, ++issued) {
                const int slot = s % p.nslots;
                if (s >= p.nslots &&
                    !mbar_wait_bounded(&empty[slot], ((s / p.nslots) - 1) & 1, kWaitLimitCycles)) {
                    flag_timeout(p.status);
                    break;
                }
                const int rows = min(p.stage_rows, nrows - s * p.stage_rows);
                const uint32_t bytes = (uint32_t)rows * p.row_bytes;
                mbar_arrive_expect_tx(&full[slot], bytes);
                bulk_g2s(ring + (size_t)slot * slot_bytes,
                         p.W + (size_t)(row0 + s * p.stage_rows) * p.row_bytes, bytes, &full[slot]);
            }
            // Never leave a copy writing into an exiting CTA: the last use of
            // each slot must have landed.
            for (int s = max(0, issued - p.nslots); s < issued; ++s)
                (void)mbar_wait_bounded(&full[s % p.nslots], (s / p.nslots) & 1, kWaitLimitCycles);
        }
        __syncwarp();
    } else if (warp - 1 < nactive) {
        const int cw = warp - 1;
        const int col = cw % p.ncol, ph = cw / p.ncol;
        const int words = p.row_bytes >> 2;
        const int wi = 32 * col + lane;           // this lane's word of every row
        const bool has = wi < words;
        pdl_wait();
        float xv[16];
        float xsum = 0.f;
        if (has) {
            const float4 *xp = reinterpret_cast<const float4 *>(p.x) + 4 * wi;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = __ldg(xp + q);
                xv[4 * q] = v.x; xv[4 * q + 1] = v.y; xv[4 * q + 2] = v.z; xv[4 * q + 3] = v.w;
                xsum += (v.x + v.y) + (v.z + v.w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) xv[j] = 0.f;
        }
        if (ph == 0) {
            xsum = warp_sum(xsum);
            if (lane == 0) sx[col] = xsum;
        }
        const int my_row = row_of_lane(lane);
        for (int s = 0; s < nstages; ++s) {
            const int slot = s % p.nslots;
            // Warp-uniform, so that the warp stays converged for the shuffles.
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (s / p.nslots) & 1, kWaitLimitCycles))) {
                flag_timeout(p.status);
                break;
            }
            const uint8_t *stage = ring + (size_t)slot * slot_bytes;
            const int rows = min(p.stage_rows, nrows - s * p.stage_rows);
            for (int g = ph * kTernT1Rows; g < rows; g += nph * kTernT1Rows) {
                float acc[kTernT1Rows];
#pragma unroll
                for (int i = 0; i < kTernT1Rows; ++i) {
                    const int r = g + i;
                    uint32_t w = 0x55555555u;  // all codes 1 (value 0) for absent rows/words
                    if (has && r < rows)
                        w = *reinterpret_cast<const uint32_t *>(stage + (size_t)r * p.row_bytes + 4 * wi);
                    float c[16];
                    decode_word(w, c);
                    float2 a = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        a = ffma2(make_float2(xv[j], xv[j + 1]), make_float2(c[j], c[j + 1]), a);
                    acc[i] = a.x + a.y;
                }
                const float v = reduce8(acc, lane);
                const int r = g + my_row;
                if ((lane & 3) == 0 && r < rows) part[(size_t)col * p.rows_per_cta + s * p.stage_rows + r] = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    __syncthreads();
    float sxt = 0.f;
    for (int cl = 0; cl < p.ncol; ++cl) sxt += sx[cl];
    for (int i = threadIdx.x; i < nrows; i += blockDim.x) {
        float a = 0.f;
        for (int cl = 0; cl < p.ncol; ++cl) a += part[(size_t)cl * p.rows_per_cta + i];
        p.y[row0 + i] = p.scale * fmaf(8.f, a, -5.f * sxt);
    }
}

// ---------------------------------------------------------------------------
// Several tokens: register tiles of 8 rows × TT tokens.
//
// A CTA owns 8·kTernTileWarps rows and TT tokens; per K chunk it copies the
// rows' code bytes and the tokens' activations into shared memory, then warp
// w accumulates rows 8w..8w+7 for all TT tokens with lane l on words
// l, l+32, … of the chunk, rows in pairs by packed FMAs.  Each word's 16
// positions go in four quads; the
// lanes take the quads in a rotated order ((q + l/2) mod 4) so that the
// activation reads of a quarter-warp fall in distinct banks.  A butterfly
// over the 8·TT accumulators finishes the sums.
// ---------------------------------------------------------------------------

constexpr int kTernTileWarps = 6;
constexpr int kTernTileRows = 8 * kTernTileWarps;

struct TernTileParams {
    const float *x;
    const uint8_t *W;
    float *y;
    int *status;
    float scale;
    int K, N, T, kc;  // kc: K values per chunk (multiple of 64)
};

template <int TT>
__global__ void __launch_bounds__(32 * kTernTileWarps, 2) ternary_tile_kernel(const TernTileParams p) {
    extern __shared__ __align__(128) uint8_t tile_smem[];
    float *xs = reinterpret_cast<float *>(tile_smem);                     // [TT][kc]
    uint8_t *ws = tile_smem + (size_t)TT * p.kc * sizeof(float);          // [rows][kc/4]
    uint64_t *bar = reinterpret_cast<uint64_t *>(ws + (size_t)kTernTileRows * (p.kc / 4));
    float *sxs = reinterpret_cast<float *>(bar + 1);                      // [TT] Σ x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kTernTileRows;
    const int t0 = blockIdx.y * TT;
    const int nrows = min(kTernTileRows, p.N - row0);
    const int ntok = min(TT, p.T - t0);
    const size_t row_bytes = (size_t)p.K / 4;

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < TT) sxs[threadIdx.x] = 0.f;
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();

    float2 acc2[4][TT];  // rows (2rp, 2rp+1) × token t
#pragma unroll
    for (int rp = 0; rp < 4; ++rp)
#pragma unroll
        for (int t = 0; t < TT; ++t) acc2[rp][t] = make_float2(0.f, 0.f);
    float xsum[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) xsum[t] = 0.f;

    const int nchunks = (p.K + p.kc - 1) / p.kc;
    bool ok = true;
    for (int ch = 0; ch < nchunks && ok; ++ch) {
        const int k0 = ch * p.kc;
        const int kn = min(p.kc, p.K - k0);  // multiple of 64
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(bar, (uint32_t)(nrows * (kn / 4) + ntok * kn * 4));
            for (int r = 0; r < nrows; ++r)
                bulk_g2s(ws + (size_t)r * (p.kc / 4), p.W + (size_t)(row0 + r) * row_bytes + k0 / 4, kn / 4,
                         bar);
            for (int t = 0; t < ntok; ++t)
                bulk_g2s(xs + (size_t)t * p.kc, p.x + (size_t)(t0 + t) * p.K + k0, kn * 4, bar);
        }
        // CTA-uniform, so that every thread leaves the loop together.
        ok = __syncthreads_and(mbar_wait_bounded(bar, ch & 1, kWaitLimitCycles));
        if (!ok) {
            flag_timeout(p.status);
            break;
        }
        const int words = kn / 16;
        const int rot = (lane >> 1) & 3;
        for (int wi = lane; wi < words; wi += 32) {
            uint32_t fb[8][4];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int rr = warp * 8 + r;
                const uint32_t w = rr < nrows
                                       ? *reinterpret_cast<const uint32_t *>(ws + (size_t)rr * (p.kc / 4) + 4 * wi)
                                       : 0x55555555u;
                fb[r][0] = field_bits<0>(w);
                fb[r][1] = field_bits<1>(w);
                fb[r][2] = field_bits<2>(w);
                fb[r][3] = field_bits<3>(w);
            }
#pragma unroll
            for (int qi = 0; qi < 4; ++qi) {
                const int q = (qi + rot) & 3;  // positions 16wi + 4q + i, i = 0..3: byte q, field i
                const uint32_t sel = 0x7054u | ((uint32_t)q << 8);
                float xq[TT][4];
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    const float4 v = *reinterpret_cast<const float4 *>(xs + (size_t)t * p.kc + 16 * wi + 4 * q);
                    xq[t][0] = v.x; xq[t][1] = v.y; xq[t][2] = v.z; xq[t][3] = v.w;
                    if (warp == 0) xsum[t] += (v.x + v.y) + (v.z + v.w);
                }
#pragma unroll
                for (int rp = 0; rp < 4; ++rp) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 c = make_float2(__uint_as_float(__byte_perm(fb[2 * rp][i], 0x3F000000u, sel)),
                                                     __uint_as_float(__byte_perm(fb[2 * rp + 1][i], 0x3F000000u, sel)));
#pragma unroll
                        for (int t = 0; t < TT; ++t) acc2[rp][t] = ffma2(make_float2(xq[t][i], xq[t][i]), c, acc2[rp][t]);
                    }
                }
            }
        }
        __syncthreads();  // the chunk buffers are refilled next
    }
    if (warp == 0) {
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float v = warp_sum(xsum[t]);
            if (lane == 0) sxs[t] = v;
        }
    }
    __syncthreads();
    if (!ok) return;
    // Butterfly over the 8·TT accumulators; then each value is in 32/(8·TT)
    // lanes (or one lane when 8·TT >= 32).
    constexpr int V = 8 * TT;
    float v[V];
#pragma unroll
    for (int rp = 0; rp < 4; ++rp)
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            v[(2 * rp) * TT + t] = acc2[rp][t].x;
            v[(2 * rp + 1) * TT + t] = acc2[rp][t].y;
        }
    int idx = 0;
    int n = V;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const int half = n >> 1;
            const bool up = lane & o;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = up ? v[i] : v[i + half];
                    const float keep = up ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (up) idx += half;
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    // Lane holds indices idx .. idx + n − 1; when n == 1 and V < 32 the lanes
    // sharing idx hold the same sum and only the first writes.
    const bool writer = V >= 32 || (lane & (32 / V - 1)) == 0;
    if (writer) {
#pragma unroll
        for (int i = 0; i < (V >= 32 ? V / 32 : 1); ++i) {
            const int id = idx + i;
            const int r = id / TT, t = id % TT;
            const int row = row0 + warp * 8 + r;
            if (warp * 8 + r < nrows && t < ntok)
                p.y[(size_t)(t0 + t) * p.N + row] = p.scale * fmaf(8.f, v[i], -5.f * sxs[t]);
        }
    }
}

cudaError_t launch_ternary_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float scale, float *y,
                              int K, int N) {
    TernT1Params p;
    p.x = x; p.W = W; p.y = y; p.status = c.status; p.scale = scale; p.K = K; p.N = N;
    p.row_bytes = K / 4;
    p.ncol = (p.row_bytes / 4 + 31) / 32;
    if (p.ncol > kTernT1Cw) return cudaErrorNotSupported;
    int grid = min(c.num_sms, (N + kTernT1Rows - 1) / kTernT1Rows);
    p.rows_per_cta = (N + grid - 1) / grid;
    grid = (N + p.rows_per_cta - 1) / p.rows_per_cta;
    p.stage_rows = max(1, min(p.rows_per_cta, 16384 / p.row_bytes));
    const int stages = (p.rows_per_cta + p.stage_rows - 1) / p.stage_rows;
    const size_t slot_bytes = (size_t)p.stage_rows * p.row_bytes;
    p.nslots = (int)max((size_t)2, min((size_t)stages, (size_t)(160 * 1024) / slot_bytes));
    const size_t smem = (size_t)p.nslots * slot_bytes + 2 * p.nslots * sizeof(uint64_t) +
                        ((size_t)p.ncol * p.rows_per_cta + p.ncol) * sizeof(float);
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;
    cudaError_t e = ensure_smem(ternary_t1_kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(c, ternary_t1_kernel, dim3(grid), dim3(32 * kTernT1Warps), smem, p);
}

template <int TT>
cudaError_t launch_tile(const LaunchCtx &c, const TernTileParams &p) {
    const size_t smem = (size_t)TT * p.kc * sizeof(float) + (size_t)kTernTileRows * (p.kc / 4) +
                        sizeof(uint64_t) + TT * sizeof(float);
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;
    cudaError_t e = ensure_smem(ternary_tile_kernel<TT>, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((p.N + kTernTileRows - 1) / kTernTileRows, (p.T + TT - 1) / TT);
    return launch_kernel(c, ternary_tile_kernel<TT>, grid, dim3(32 * kTernTileWarps), smem, p);
}

cudaError_t launch_ternary_tile(const LaunchCtx &c, const float *x, const uint8_t *W, float scale, float *y,
                                int K, int N, int T) {
    TernTileParams p;
    p.x = x; p.W = W; p.y = y; p.status = c.status; p.scale = scale; p.K = K; p.N = N; p.T = T;
    const int tt = T <= 2 ? 2 : T <= 4 ? 4 : 8;
    // Chunk: activation and code tiles within 112 KB, a multiple of 64 values.
    const int kc_max = (112 * 1024) / (tt * (int)sizeof(float) + kTernTileRows / 4);
    p.kc = min(K, max(64, kc_max / 64 * 64));
    switch (tt) {
        case 2: return launch_tile<2>(c, p);
        case 4: return launch_tile<4>(c, p);
        default: return launch_tile<8>(c, p);
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
    // The streamed kernels copy whole 16-byte runs of code bytes: rows of
    // K/4 bytes must be a multiple of 16 (K % 64 == 0) and W 16-byte aligned.
    const bool bulk = (K % 64 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0);
    if (bulk) {
        cudaError_t e = cudaErrorNotSupported;
        // K % 256 == 0 and up to 3 tokens: the shared one-token kernel
        // (byte-plane integer code-dot, one token per compute warp).  From 4
        // tokens on the FP32 register-tile kernel is as fast or faster
        // (2560 -> 6912, GB300: 1 token 5.1 vs 5.6 us, 2: 7.4 vs 8.9,
        // 3: 10.0 vs 11.8, 4: 11.7 vs 11.8, 8: 19.1 vs 13.3).  Otherwise the
        // float one-token kernel (one token) or the register-tile kernel.
        if (K % 256 == 0 && T <= 3) {
            e = launch_ternary_gemv_t1(c, x, W, scale, y, K, N, T);
            if (e == cudaErrorNotSupported && T > 1) {
                // Too wide for T tokens at once: one token at a time if that fits.
                e = cudaSuccess;
                for (int t = 0; t < T && e == cudaSuccess; ++t)
                    e = launch_ternary_gemv_t1(c, x + (size_t)t * K, W, scale, y + (size_t)t * N, K, N, 1);
            }
        }
        if (T == 1 && e == cudaErrorNotSupported) e = launch_ternary_t1(c, x, W, scale, y, K, N);
        if (e == cudaErrorNotSupported) e = launch_ternary_tile(c, x, W, scale, y, K, N, T);
        if (e != cudaErrorNotSupported) return e;
    }
    // Any alignment: word loads need 4-byte aligned rows (K % 16 == 0 and W
    // aligned), otherwise bytes.  Token tiles of up to 8.
    const bool aligned = (K % 16 == 0) && ((reinterpret_cast<uintptr_t>(W) & 3) == 0);
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
