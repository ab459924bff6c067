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
#include <cstdlib>
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

// ----------------------------------------------------------------------------
// One token: bulk-copied rows, slab lanes, exact int8 activation planes
// ----------------------------------------------------------------------------
//
// Roles in a CTA (a contiguous range of output rows):
//  * warp 0, lane 0 streams the rows into a shared-memory ring with 1-D bulk
//    copies of whole stages (weights are never written by an earlier kernel,
//    so this starts before the wait on the previous kernel);
//  * the other warps are "slab lanes": lane (b, j) owns the 32-byte qs slab j
//    of block b of every row it visits (32 low nibbles of sub-block 2j, 32
//    high nibbles of 2j+1) and decodes the two 6-bit scale/min pairs it needs
//    from the block header.  Passes of two rows are numbered across the whole
//    CTA, so different warps work on different stages at once.
//
// The code-dot Σ x·q of a sub-block runs on integer dot-product instructions
// (four byte products per instruction).  Each 256-value block of x is split,
// once per CTA, into three int8 planes under a power-of-two block scale s_b:
//   x = s_b·(p1 + p2/128 + p3/16384) + e,  |e| ≤ 2^-15·s_b ≤ 2^-21·max|x_b|,
// with |p1| ≤ 127 and |p2|, |p3| ≤ 64; every step of the split is exact
// (power-of-two scalings and exact fp32 subtractions), so activations with at
// most 21 significant bits below their block maximum (integers included) are
// represented exactly.  The 4-bit codes are used as they are (no bias), the
// integer sums are exact, and scales, mins and the final combination are fp32.
// kNB (blocks per row) is a template constant for common widths so that row
// and stage address arithmetic folds at compile time; 0 reads it at run time.

// Scale d·sc and offset dmin·m of the two sub-blocks 2j and 2j+1 of a block
// (lane-constant j), from the 16-byte block header.
struct SlabScalesRaw {
    float s0, s1, o0, o1;
};

__device__ __forceinline__ SlabScalesRaw slab_scales_raw(uint4 hdr, int j) {
    const float2 dm = q4k_d_dmin(hdr.x);
    const Q4kScales u = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
    const bool upper = j >= 2;
    const uint32_t scw = upper ? u.sc_hi : u.sc_lo;
    const uint32_t mw = upper ? u.m_hi : u.m_lo;
    const int k0 = 2 * (j & 1);
    SlabScalesRaw r;
    r.s0 = dm.x * byte_to_float(scw, k0);  // exact: 11-bit × 6-bit
    r.s1 = dm.x * byte_to_float(scw, k0 + 1);
    r.o0 = dm.y * byte_to_float(mw, k0);
    r.o1 = dm.y * byte_to_float(mw, k0 + 1);
    return r;
}

// Integer code-dots of one slab against the three activation planes:
// d_lo[p] = Σ_l q_lo(l)·plane_p[l], d_hi[p] likewise for the high nibbles.
// Slab byte l pairs with plane byte l of the low 32 positions (words 0..7)
// and with plane byte l of the high 32 positions (words 8..15).
__device__ __forceinline__ void slab_dot_planes(const int (&pl)[3][16], uint4 q0, uint4 q1,
                                                int (&d_lo)[3], int (&d_hi)[3]) {
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int l4 = (int)(qw[w] & 0x0F0F0F0Fu);
        const int h4 = (int)((qw[w] >> 4) & 0x0F0F0F0Fu);
#pragma unroll
        for (int pp = 0; pp < 3; ++pp) {
            d_lo[pp] = __dp4a(l4, pl[pp][w], d_lo[pp]);
            d_hi[pp] = __dp4a(h4, pl[pp][8 + w], d_hi[pp]);
        }
    }
}

// Σ q·x in units of the block scale from the three plane sums.
__device__ __forceinline__ float plane_combine(const int (&d)[3]) {
    const int d01 = d[0] * 128 + d[1];  // |d01| < 2^23: exact in fp32
    return fmaf(static_cast<float>(d[2]), 1.0f / 16384.0f, static_cast<float>(d01) * (1.0f / 128.0f));
}

// Round to nearest (ties to even) for |v| < 2^22 with the 1.5·2^23 shifter;
// the low byte of the shifted value's bits is the result as an int8.
__device__ __forceinline__ float shifted(float v) { return v + 12582912.0f; }

struct T1Params {
    const float *x;
    const uint8_t *W;
    float *y;
    int *status;
    int N;
    int nb;            // blocks per row (K/256)
    int rg;            // row groups: compute warps = wc·rg
    int rows_per_cta;  // contiguous rows per CTA
    int stage_rows;    // rows per ring slot (multiple of the pass size)
    int nslots;        // ring depth
};

constexpr int kT1RoleWarps = 1;  // the copy warp

template <int kNB>
__global__ void __launch_bounds__(32 * 16, 1) q4k_gemv_t1_kernel(T1Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int abort_flag;

    // Row geometry: compile-time when kNB > 0.
    const int nb = kNB > 0 ? kNB : p.nb;
    const int K = nb * kQ4kValues;
    const int nslabs = 4 * nb;                     // 64-value slabs per row
    const uint32_t row_bytes = (uint32_t)nb * kQ4kBytes;
    const int L = 4 * nb;                          // slab lanes per row
    const bool wide = L > 32;                      // a row spans several warps
    const int wc = wide ? (L + 31) / 32 : 1;       // warps per row
    int lpr = 32;                                  // lanes per row slot when !wide
    if (!wide) {
        lpr = 4;
        while (lpr < L) lpr <<= 1;
    }
    const int rpp = wide ? 1 : 32 / lpr;           // row slots per warp pass
    const int pass_rows = 2 * rpp;
    const int half = wide ? 16 : lpr / 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncw = wc * p.rg;
    const uint32_t slot_bytes = p.stage_rows * row_bytes;
    int8_t *planes = reinterpret_cast<int8_t *>(smem);                // 3 planes of K bytes
    float *sx = reinterpret_cast<float *>(planes + 3 * K);            // K/32 sub-block sums
    float *sb = sx + K / 32;                                          // K/256 block scales
    uint8_t *ring = reinterpret_cast<uint8_t *>(sb) + ((nb * 4 + 15) & ~15);
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(ring + (size_t)p.nslots * slot_bytes);
    uint64_t *empty_bar = full_bar + p.nslots;
    float *part = reinterpret_cast<float *>(empty_bar + p.nslots);  // [rows_per_cta][wc]

    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int nstages = (nrows + p.stage_rows - 1) / p.stage_rows;
    const int passes_per_stage = p.stage_rows / pass_rows;

    // Bulk copies need a 16-byte aligned destination; never issue one otherwise.
    if (smem_addr(smem) & 15) {
        if (threadIdx.x == 0) flag_timeout(p.status);
        return;
    }
    if (threadIdx.x == 0) {
        // Warm L2 with x: a hint that returns no data, so it may run before
        // the wait on the kernel that produces x.
        bulk_prefetch_l2(p.x, (uint32_t)K * sizeof(float));
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full_bar[s], 1);
            // Every pass of a stage is worked by the wc warps of a row.
            mbar_init(&empty_bar[s], passes_per_stage * wc);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            const uint8_t *src = p.W + (size_t)row0 * row_bytes;
            int st = 0;
            for (; st < min(nstages, p.nslots); ++st) {
                const int rows = min(p.stage_rows, nrows - st * p.stage_rows);
                mbar_arrive_expect_tx(&full_bar[st], rows * row_bytes);
                bulk_g2s(ring + (size_t)st * slot_bytes, src + (size_t)st * p.stage_rows * row_bytes,
                         rows * row_bytes, &full_bar[st]);
            }
            for (; st < nstages; ++st) {
                const int slot = st % p.nslots;
                if (abort_flag) break;
                if (!mbar_wait_bounded(&empty_bar[slot], ((st / p.nslots) - 1) & 1,
                                       kWaitLimitCycles)) {
                    abort_flag = 1;
                    flag_timeout(p.status);
                    break;
                }
                const int rows = min(p.stage_rows, nrows - st * p.stage_rows);
                mbar_arrive_expect_tx(&full_bar[slot], rows * row_bytes);
                bulk_g2s(ring + (size_t)slot * slot_bytes, src + (size_t)st * p.stage_rows * row_bytes,
                         rows * row_bytes, &full_bar[slot]);
            }
        }
        __syncwarp();
    } else {
        const int cw = warp - kT1RoleWarps;
        const int wcol = cw % wc, rgi = cw / wc;
        const int ro = wide ? 0 : lane / lpr;
        const int s = wide ? wcol * 32 + lane : lane % lpr;
        const bool active = s < L;
        const int b = active ? (s >> 2) : 0, j = s & 3;

        // x may be produced by the previous kernel on the stream.
        pdl_wait();
        // x → three int8 planes under power-of-two block scales, plus the
        // fp32 sub-block sums.  Thread ct takes half sub-blocks (16 values);
        // the 16 threads of a block (an aligned 16-lane group) share its
        // maximum through shuffles, and the two halves of a sub-block sit in
        // neighbouring lanes.
        {
            const int ct = threadIdx.x - 32 * kT1RoleWarps, nth = ncw * 32, nh = K / 16;
            for (int h0 = 0; h0 < nh; h0 += nth) {
                const int h = h0 + ct;
                const bool on = h < nh;
                float v[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 t = on ? __ldg(reinterpret_cast<const float4 *>(p.x) + 4 * h + k)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[4 * k] = t.x;
                    v[4 * k + 1] = t.y;
                    v[4 * k + 2] = t.z;
                    v[4 * k + 3] = t.w;
                }
                float amax = 0.f, sum = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    amax = fmaxf(amax, fabsf(v[i]));
                    sum += v[i];
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                // s_b = 2^e with amax / 2^e < 127 (1 when the block is zero).
                int e = 0;
                if (amax > 0.f) (void)frexpf(amax * (1.0f / 127.0f), &e);
                e = max(e, -120);  // keeps 2^-e finite; such blocks still scale below 127
                const float inv = ldexpf(1.0f, -e);
                uint32_t w1[4], w2[4], w3[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t b1[4], b2[4], b3[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float a = v[4 * k + i] * inv;  // exact
                        const float s1 = shifted(a);
                        const float r1 = (a - (s1 - 12582912.0f)) * 128.0f;  // exact
                        const float s2 = shifted(r1);
                        const float r2 = (r1 - (s2 - 12582912.0f)) * 128.0f;  // exact
                        const float s3 = shifted(r2);
                        b1[i] = __float_as_uint(s1);
                        b2[i] = __float_as_uint(s2);
                        b3[i] = __float_as_uint(s3);
                    }
                    // Low byte of each shifted value, four to a word.
                    w1[k] = __byte_perm(__byte_perm(b1[0], b1[1], 0x0040), __byte_perm(b1[2], b1[3], 0x0040), 0x5410);
                    w2[k] = __byte_perm(__byte_perm(b2[0], b2[1], 0x0040), __byte_perm(b2[2], b2[3], 0x0040), 0x5410);
                    w3[k] = __byte_perm(__byte_perm(b3[0], b3[1], 0x0040), __byte_perm(b3[2], b3[3], 0x0040), 0x5410);
                }
                if (on) {
                    // Unit-major layout: 16-byte unit u (0..11) of slab S at
                    // index u·nslabs + S, with u = 4·plane + (h & 3) and
                    // S = h / 4, so the eight lanes of a quarter warp read
                    // eight consecutive units.
                    uint4 *pu = reinterpret_cast<uint4 *>(planes) + (h & 3) * nslabs + (h >> 2);
                    pu[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    pu[4 * nslabs] = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                    pu[8 * nslabs] = make_uint4(w3[0], w3[1], w3[2], w3[3]);
                    if ((h & 1) == 0) sx[h / 2] = sum;
                    if ((h & 15) == 0) sb[h / 16] = ldexpf(1.0f, e);
                }
            }
        }
        named_bar_sync(1, ncw * 32);
        int pl[3][16];
        float s_blk, sum_lo, sum_hi;
        {
            // This slab's 64 plane bytes per plane: positions 64j..64j+31
            // (low nibbles) then 64j+32..64j+63 (high nibbles) of block b.
            const uint4 *src = reinterpret_cast<const uint4 *>(planes) + (4 * b + j);
#pragma unroll
            for (int pp = 0; pp < 3; ++pp) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 t = active ? src[(4 * pp + i) * nslabs] : make_uint4(0u, 0u, 0u, 0u);
                    pl[pp][4 * i] = (int)t.x;
                    pl[pp][4 * i + 1] = (int)t.y;
                    pl[pp][4 * i + 2] = (int)t.z;
                    pl[pp][4 * i + 3] = (int)t.w;
                }
            }
            s_blk = active ? sb[b] : 0.f;
            sum_lo = active ? sx[8 * b + 2 * j] : 0.f;
            sum_hi = active ? sx[8 * b + 2 * j + 1] : 0.f;
        }

        const int npasses = (nrows + pass_rows - 1) / pass_rows;
        // Stage, slot and phase of the current pass, advanced without
        // divisions as the pass index steps by rg.
        int pin = rgi, st = 0;
        while (pin >= passes_per_stage) {
            pin -= passes_per_stage;
            ++st;
        }
        int slot = st % p.nslots;
        uint32_t phase = (st / p.nslots) & 1;
        int waited_stage = -1;
        const uint8_t *stage_base = ring;
        int rows = 0;
        for (int pass = rgi; pass < npasses; pass += p.rg) {
            if (st != waited_stage) {
                if (abort_flag) break;
                if (!mbar_wait_bounded(&full_bar[slot], phase, kWaitLimitCycles)) {
                    abort_flag = 1;
                    flag_timeout(p.status);
                    break;
                }
                waited_stage = st;
                stage_base = ring + (size_t)slot * slot_bytes + b * kQ4kBytes;
                rows = min(p.stage_rows, nrows - st * p.stage_rows);
            }
            const int ra = pin * pass_rows + 2 * ro, rb = ra + 1;
            const uint8_t *ba = stage_base + min(ra, rows - 1) * row_bytes;
            const uint8_t *bb = stage_base + min(rb, rows - 1) * row_bytes;
            const uint4 ha = *reinterpret_cast<const uint4 *>(ba);
            const uint4 hb = *reinterpret_cast<const uint4 *>(bb);
            const uint4 a0 = *reinterpret_cast<const uint4 *>(ba + 16 + 32 * j);
            const uint4 a1 = *reinterpret_cast<const uint4 *>(ba + 32 + 32 * j);
            const uint4 b0 = *reinterpret_cast<const uint4 *>(bb + 16 + 32 * j);
            const uint4 b1 = *reinterpret_cast<const uint4 *>(bb + 32 + 32 * j);
            const SlabScalesRaw sa = slab_scales_raw(ha, j), sc_b = slab_scales_raw(hb, j);
            int da_lo[3] = {0, 0, 0}, da_hi[3] = {0, 0, 0}, db_lo[3] = {0, 0, 0}, db_hi[3] = {0, 0, 0};
            slab_dot_planes(pl, a0, a1, da_lo, da_hi);
            slab_dot_planes(pl, b0, b1, db_lo, db_hi);
            float pa = s_blk * fmaf(sa.s0, plane_combine(da_lo), sa.s1 * plane_combine(da_hi)) -
                       fmaf(sa.o0, sum_lo, sa.o1 * sum_hi);
            float pb = s_blk * fmaf(sc_b.s0, plane_combine(db_lo), sc_b.s1 * plane_combine(db_hi)) -
                       fmaf(sc_b.o0, sum_lo, sc_b.o1 * sum_hi);
            if (!active || ra >= rows) pa = 0.f;
            if (!active || rb >= rows) pb = 0.f;
            // Two-row butterfly: lanes with (lane & half) == 0 finish with
            // row a, the others with row b.
            const bool up = (lane & half) != 0;
            float v = (up ? pb : pa) + __shfl_xor_sync(0xFFFFFFFFu, up ? pa : pb, half);
            for (int o = half >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            const int r = up ? rb : ra;
            const int rl = st * p.stage_rows + r;
            if (wide) {
                if ((lane & (half - 1)) == 0 && r < rows) part[rl * wc + wcol] = v;
            } else {
                if (s == (up ? half : 0) && r < rows) p.y[row0 + rl] = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
            pin += p.rg;
            while (pin >= passes_per_stage) {
                pin -= passes_per_stage;
                ++st;
                if (++slot == p.nslots) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
        }

        if (wide) {
            named_bar_sync(1, ncw * 32);
            for (int i = threadIdx.x - 32 * kT1RoleWarps; i < nrows; i += ncw * 32) {
                float acc = 0.f;
                for (int w = 0; w < wc; ++w) acc += part[i * wc + w];
                p.y[row0 + i] = acc;
            }
        }
    }

    // Never leave a bulk copy writing into shared memory of an exiting CTA.
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        for (int st = max(0, nstages - p.nslots); st < nstages; ++st)
            (void)mbar_wait_bounded(&full_bar[st % p.nslots], (st / p.nslots) & 1,
                                    kWaitLimitCycles);
    }
}

// ----------------------------------------------------------------------------
// 2..8 tokens: bulk-copied row groups, word lanes, register tiles
// ----------------------------------------------------------------------------
//
// A CTA owns a contiguous range of rows in groups of four; one producer
// thread streams each group (four whole rows) into its own ring slot with a
// bulk copy, before the wait on the previous kernel.  Compute warp c takes
// groups c, c + kMultiCw, …, and for each group walks all blocks of the rows:
// lane l owns qs word l of every block — 4 low-nibble weights of sub-block
// 2j and 4 high-nibble weights of 2j+1 (j = l/8) — with the 8 matching
// activations of all TT tokens loaded once per block and reused by the four
// rows.  Each weight is dequantized once (scale'·(0.5 + q/256) − offset') and
// multiplied into TT token accumulators, two positions per paired FMA.  A
// butterfly over the 4·TT sums at the end of the group finishes the rows.

constexpr int kMultiWarps = 8;                    // copy warp + 7 compute warps
constexpr int kMultiCw = kMultiWarps - 1;
constexpr int kMultiRows = 4;                     // rows per group (one ring slot)

struct MultiParams {
    const float *x;
    const uint8_t *W;
    float *y;
    int *status;
    int K, N, T;       // T: tokens of this launch (<= TT)
    int nb;            // blocks per row
    int rows_per_cta;  // multiple of kMultiRows
    int nslots;        // ring depth (groups in flight)
};

template <int TT>
__global__ void __launch_bounds__(32 * kMultiWarps, 1) q4k_gemv_multi_kernel(MultiParams p) {
    extern __shared__ __align__(128) uint8_t msmem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t row_bytes = (uint32_t)p.nb * kQ4kBytes;
    const uint32_t slot_bytes = kMultiRows * row_bytes;
    uint8_t *ring = msmem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)p.nslots * slot_bytes);
    uint64_t *empty = full + p.nslots;
    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int ngroups = (nrows + kMultiRows - 1) / kMultiRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int g = 0; g < ngroups; ++g, ++issued) {
                const int slot = g % p.nslots;
                if (g >= p.nslots &&
                    !mbar_wait_bounded(&empty[slot], ((g / p.nslots) - 1) & 1, kWaitLimitCycles)) {
                    flag_timeout(p.status);
                    break;
                }
                const uint32_t bytes = (uint32_t)min(kMultiRows, nrows - g * kMultiRows) * row_bytes;
                mbar_arrive_expect_tx(&full[slot], bytes);
                bulk_g2s(ring + (size_t)slot * slot_bytes,
                         p.W + (size_t)(row0 + g * kMultiRows) * row_bytes, bytes, &full[slot]);
            }
            // Never leave a copy writing into an exiting CTA.
            for (int g = max(0, issued - p.nslots); g < issued; ++g)
                (void)mbar_wait_bounded(&full[g % p.nslots], (g / p.nslots) & 1, kWaitLimitCycles);
        }
        __syncwarp();
        return;
    }

    const int cw = warp - 1;
    const int j = lane >> 3, wq = lane & 7;   // slab and word within it
    // x may be produced by the previous kernel on the stream.
    pdl_wait();
    for (int g = cw; g < ngroups; g += kMultiCw) {
        const int slot = g % p.nslots;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (g / p.nslots) & 1, kWaitLimitCycles))) {
            flag_timeout(p.status);
            break;
        }
        const uint8_t *grp = ring + (size_t)slot * slot_bytes;
        const int rows = min(kMultiRows, nrows - g * kMultiRows);
        float2 acc[kMultiRows][TT];
#pragma unroll
        for (int r = 0; r < kMultiRows; ++r)
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[r][t] = make_float2(0.f, 0.f);

        for (int b = 0; b < p.nb; ++b) {
            // Activations of this lane's 8 positions for every token.
            float4 xl[TT], xh[TT];
            const int k0 = b * kQ4kValues + 64 * j + 4 * wq;
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                if (t < p.T) {
                    const float *xt = p.x + (size_t)t * p.K + k0;
                    xl[t] = __ldg(reinterpret_cast<const float4 *>(xt));
                    xh[t] = __ldg(reinterpret_cast<const float4 *>(xt + 32));
                } else {
                    xl[t] = make_float4(0.f, 0.f, 0.f, 0.f);
                    xh[t] = xl[t];
                }
            }
#pragma unroll
            for (int r = 0; r < kMultiRows; ++r) {
                // Absent rows of a short last group read row 0 of the slot;
                // their sums are never stored.
                const uint8_t *blk = grp + (size_t)(r < rows ? r : 0) * row_bytes + (size_t)b * kQ4kBytes;
                const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
                const uint32_t q = *reinterpret_cast<const uint32_t *>(blk + 16 + 32 * j + 4 * wq);
                const SlabScales sc = slab_scales(hdr, j);
                const uint32_t l4 = q & 0x0F0F0F0Fu;
                const uint32_t h4 = (q >> 4) & 0x0F0F0F0Fu;
                const float2 s0 = make_float2(sc.s0, sc.s0), n0 = make_float2(-sc.o0, -sc.o0);
                const float2 s1 = make_float2(sc.s1, sc.s1), n1 = make_float2(-sc.o1, -sc.o1);
                const float2 wl01 = ffma2(make_float2(nib_biased<0>(l4), nib_biased<1>(l4)), s0, n0);
                const float2 wl23 = ffma2(make_float2(nib_biased<2>(l4), nib_biased<3>(l4)), s0, n0);
                const float2 wh01 = ffma2(make_float2(nib_biased<0>(h4), nib_biased<1>(h4)), s1, n1);
                const float2 wh23 = ffma2(make_float2(nib_biased<2>(h4), nib_biased<3>(h4)), s1, n1);
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    acc[r][t] = ffma2(make_float2(xl[t].x, xl[t].y), wl01, acc[r][t]);
                    acc[r][t] = ffma2(make_float2(xl[t].z, xl[t].w), wl23, acc[r][t]);
                    acc[r][t] = ffma2(make_float2(xh[t].x, xh[t].y), wh01, acc[r][t]);
                    acc[r][t] = ffma2(make_float2(xh[t].z, xh[t].w), wh23, acc[r][t]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        // Butterfly over the 4·TT sums: afterwards lane l holds value index
        // idx .. idx + n − 1 (see the halving below), summed over the warp.
        constexpr int V = kMultiRows * TT;
        float v[V];
#pragma unroll
        for (int r = 0; r < kMultiRows; ++r)
#pragma unroll
            for (int t = 0; t < TT; ++t) v[r * TT + t] = acc[r][t].x + acc[r][t].y;
        int idx = 0, n = V;
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
        const bool writer = V >= 32 || (lane & (32 / V - 1)) == 0;
        if (writer) {
#pragma unroll
            for (int i = 0; i < (V >= 32 ? V / 32 : 1); ++i) {
                const int id = idx + i;
                const int r = id / TT, t = id % TT;
                if (r < rows && t < p.T) p.y[(size_t)t * p.N + row0 + g * kMultiRows + r] = v[i];
            }
        }
    }
}

// Geometry knobs of the one-token kernel (environment, read once): compute
// warps per CTA, resident CTAs per SM, bytes per ring slot, ring budget.
struct T1Tuning {
    int warps = 14;
    int ctas_per_sm = 1;
    int stage_bytes = 16384;
    int ring_bytes = 200 * 1024;
};

int env_int(const char *name, int dflt, int lo, int hi) {
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    const int x = atoi(v);
    return x < lo ? lo : (x > hi ? hi : x);
}

const T1Tuning &t1_tuning() {
    static const T1Tuning t = [] {
        T1Tuning r;
        r.warps = env_int("Q4MM_T1_WARPS", r.warps, 1, 15);
        r.ctas_per_sm = env_int("Q4MM_T1_CTAS_PER_SM", r.ctas_per_sm, 1, 8);
        r.stage_bytes = env_int("Q4MM_T1_STAGE_BYTES", r.stage_bytes, 1024, 65536);
        r.ring_bytes = env_int("Q4MM_T1_RING_BYTES", r.ring_bytes, 8192, 200 * 1024);
        return r;
    }();
    return t;
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
    const int row_bytes = p.nb * kQ4kBytes;
    const int L = 4 * p.nb;  // slab lanes per row
    const bool wide = L > 32;
    const int wc = wide ? (L + 31) / 32 : 1;
    const int pass_rows = wide ? 2 : 2 * (32 / next_pow2(max(L, 4)));
    // At most 15 compute warps (+1 copy warp): wider rows go to the generic kernel.
    if (wc > 15) return cudaErrorNotSupported;
    const T1Tuning &tun = t1_tuning();
    p.rg = max(1, tun.warps / wc);
    const int ncw = wc * p.rg;
    // Stage: whole passes, at least stage_bytes of weights (bulk copies of
    // 16 KB and more run at full HBM bandwidth).
    p.stage_rows = pass_rows * max(1, (tun.stage_bytes + pass_rows * row_bytes - 1) /
                                          (pass_rows * row_bytes));

    int grid = tun.ctas_per_sm * c.num_sms;
    p.rows_per_cta = (N + grid - 1) / grid;
    if (p.rows_per_cta < pass_rows) p.rows_per_cta = pass_rows;
    if (p.stage_rows > p.rows_per_cta)
        p.stage_rows = pass_rows * ((p.rows_per_cta + pass_rows - 1) / pass_rows);
    grid = (N + p.rows_per_cta - 1) / p.rows_per_cta;
    const size_t slot_bytes = (size_t)p.stage_rows * row_bytes;

    const size_t xs_bytes = 3 * (size_t)K + (size_t)(K / 32) * sizeof(float) + (size_t)((p.nb * 4 + 15) & ~15);
    const size_t part_bytes = wide ? (size_t)p.rows_per_cta * wc * sizeof(float) : 0;
    const size_t fixed = xs_bytes + part_bytes + 2 * 8 * sizeof(uint64_t);
    const size_t budget = tun.ring_bytes;
    int nslots = (int)((budget > fixed ? budget - fixed : 0) / slot_bytes);
    const int stages_needed = (p.rows_per_cta + p.stage_rows - 1) / p.stage_rows;
    nslots = max(2, min(nslots, min(stages_needed, 8)));
    p.nslots = nslots;
    const size_t smem = xs_bytes + (size_t)nslots * slot_bytes + 2 * nslots * sizeof(uint64_t) + part_bytes;
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;

    const dim3 block(32 * (kT1RoleWarps + ncw));
    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e = ensure_smem(kernel, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(c, kernel, dim3(grid), block, smem, p);
    };
    switch (p.nb) {
        case 4: return go(q4k_gemv_t1_kernel<4>);
        case 8: return go(q4k_gemv_t1_kernel<8>);
        case 16: return go(q4k_gemv_t1_kernel<16>);
        case 32: return go(q4k_gemv_t1_kernel<32>);
        case 43: return go(q4k_gemv_t1_kernel<43>);
        default: return go(q4k_gemv_t1_kernel<0>);
    }
}

cudaError_t launch_q4k_gemv_multi(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                  int K, int N, int T) {
    MultiParams p;
    p.x = x;
    p.W = W;
    p.y = y;
    p.status = c.status;
    p.K = K;
    p.N = N;
    p.T = T;
    p.nb = K / kQ4kValues;
    const size_t row_bytes = (size_t)p.nb * kQ4kBytes;
    const size_t slot_bytes = kMultiRows * row_bytes;
    const int groups = (N + kMultiRows - 1) / kMultiRows;
    int grid = min(c.num_sms, groups);
    p.rows_per_cta = kMultiRows * ((groups + grid - 1) / grid);
    grid = (N + p.rows_per_cta - 1) / p.rows_per_cta;
    const int cta_groups = p.rows_per_cta / kMultiRows;
    // Ring: up to 200 KB, at least two slots, never more slots than groups.
    p.nslots = (int)min((size_t)min(cta_groups, 16), max((size_t)2, (size_t)(200 * 1024) / slot_bytes));
    p.nslots = max(p.nslots, min(cta_groups, 2));
    const size_t smem = (size_t)p.nslots * slot_bytes + 2 * (size_t)p.nslots * sizeof(uint64_t);
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;

#define Q4MM_MULTI_CASE(TT)                                                                    \
    {                                                                                          \
        cudaError_t e = ensure_smem(q4k_gemv_multi_kernel<TT>, smem);                          \
        if (e != cudaSuccess) return e;                                                        \
        return launch_kernel(c, q4k_gemv_multi_kernel<TT>, dim3(grid), dim3(32 * kMultiWarps), \
                             smem, p);                                                         \
    }
    if (T <= 2) Q4MM_MULTI_CASE(2)
    if (T <= 4) Q4MM_MULTI_CASE(4)
    if (T <= 8) Q4MM_MULTI_CASE(8)
#undef Q4MM_MULTI_CASE
    return cudaErrorInvalidValue;
}

}  // namespace q4mm
