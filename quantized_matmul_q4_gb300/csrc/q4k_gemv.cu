// Q4_K, Q4_0, Q6_K and ternary decode GEMV on the one-token kernel (1 token;
// up to 4 tokens for Q4_K, up to 8 for Q4_0 and Q6_K, 3 for ternary), and the
// fused gate+up SwiGLU, sm_103a.
//
// Computes y[t][o] = Σ_k x[t][k]·w[o][k] with w = d·sc_s·q − dmin·m_s decoded
// on the fly from the 144-byte Q4_K super-blocks (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline").  As on that page, one load of a qs byte feeds both the
// low-nibble codes (sub-block 2j) and the high-nibble ones (2j+1), and the
// min term is applied lazily once per sub-block from the sum of the inputs,
// never per weight.
//
// GPU design (not the page's): a "slab lane" owns one 32-byte qs slab j of
// one block b — 64 weights of sub-blocks 2j and 2j+1 — for every row it
// visits, so the 64 matching activations live in its registers (as exact
// byte planes) for the whole kernel.  Weight rows are streamed once from HBM
// into a shared-memory ring by 1-D bulk copies (cp.async.bulk) that one
// producer thread issues right after the activation copy.  The 2..8 token
// kernel is in q4k_gemv_multi.cu.
#include <cstdlib>
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"
#include "t1_geometry.h"

namespace q4mm {

namespace {

// ----------------------------------------------------------------------------
// One token: bulk-copied rows, slab lanes, exact int8 activation planes
// ----------------------------------------------------------------------------
//
// Roles in a CTA (a contiguous range of output rows):
//  * warp 0, lane 0 streams the rows into a shared-memory ring with 1-D bulk
//    copies of whole stages.  It first waits for the previous kernel on the
//    stream (which may write x), copies x into shared memory with one bulk
//    copy, and only then issues the weight stages: an activation fetch that
//    queues behind the CTA's weight stream arrives late, and everything after
//    it (plane split, code-dots) waits for it, while the weights have the
//    plane split's time to land.  (pre_stages > 0 sends that many stages
//    ahead of the wait instead; measured slower on GB300.)  Above 64 KB of x
//    the compute threads load x themselves and all stages go out first;
//  * the other warps are "slab lanes": lane (b, j) owns the 32-byte qs slab j
//    of block b of every row it visits (32 low nibbles of sub-block 2j, 32
//    high nibbles of 2j+1) and decodes the two 6-bit scale/min pairs it needs
//    from the block header.  Passes of two rows are numbered across the whole
//    CTA, so different warps work on different stages at once.
//
// The code-dot Σ x·q of a sub-block runs on integer dot-product instructions
// (four byte products per instruction).  Each 256-value block of x is split,
// once per CTA, into three byte planes under a power-of-two block scale s_b:
//   n = rint(x·2^15/s_b),  |n| < 127·2^15 < 2^22,
//   n = 65536·p2 + 256·p1 + p0  (p0, p1 unsigned bytes, p2 a signed byte),
// so x = s_b·2^-15·n + e with |e| ≤ 2^-16·s_b ≤ 2^-15·max|x_b|/127 (s_b is at
// most 2·max|x_b|/127; the bound is about 2.4e-7·max|x_b|).  The rounding is a
// single FMA against the 1.5·2^23 shifter (the product by a power of two is
// exact), whose low bytes are the digits of n; the grid step 2^-15·s_b is at
// most 2^-20 of the leading power of two of max|x_b|, so activations with at
// most 21 significant bits below that leading bit (integers below 2^21
// included) are represented exactly.  Low-nibble codes enter the dot products as they are;
// high-nibble codes enter as 16·q (the byte masked in place, no shift) and
// the factor 16 is taken out of that sub-block's scale.  The integer sums are
// exact; scales, mins and the final combination are fp32.
// kNB (blocks per row) is a template constant for common widths so that row
// and stage address arithmetic folds at compile time; 0 reads it at run time.

// Lane-constant selectors that pick the two 6-bit scale/min pairs of
// sub-blocks 2j and 2j+1 out of the 12 packed bytes (ggml canonical packing:
// sub-blocks 0..3 in the low 6 bits of bytes 0..3 / 4..7; sub-blocks 4..7
// from the nibbles of bytes 8..11 plus the top 2 bits of bytes 0..3 / 4..7).
struct LaneScaleSel {
    uint32_t mask_lo;   // nibble field of bytes 8..11 (upper sub-blocks only)
    uint32_t mask_hi;   // 6-bit field (lower) or top-2-bit field (upper)
    uint32_t sh_hi;     // shift bringing the top 2 bits to bits 4..5
    uint32_t sh_min;    // the mins' nibbles sit in bits 4..7 of bytes 8..11
    uint32_t sel0, sel1;  // byte permutes: byte k of a word → float 2^23 + byte
};

__device__ __forceinline__ LaneScaleSel lane_scale_sel(int j) {
    const bool upper = j >= 2;
    const uint32_t k0 = 2 * (j & 1);
    LaneScaleSel r;
    r.mask_lo = upper ? 0x0F0F0F0Fu : 0u;
    r.mask_hi = upper ? 0x30303030u : 0x3F3F3F3Fu;
    r.sh_hi = upper ? 2u : 0u;
    r.sh_min = upper ? 4u : 0u;
    r.sel0 = 0x7440u | k0;
    r.sel1 = 0x7440u | (k0 + 1);
    return r;
}

// Scales and mins of sub-blocks 2j and 2j+1 of one block: s0 = d·sc_2j,
// s1 = d·sc_2j+1 / 16 (the high-nibble sums carry a factor 16), o = dmin·m.
// A 6-bit field becomes the float 2^23 + v by one byte permute, and d·v comes
// exactly out of one FMA against −d·2^23.
struct RowScales {
    float s0, s1, o0, o1;
};

__device__ __forceinline__ RowScales row_scales(uint4 h, const LaneScaleSel &L) {
    const float2 dm = q4k_d_dmin(h.x);
    const float d = dm.x;
    const float d16 = d * 0.0625f;
    const uint32_t scw = (h.w & L.mask_lo) | ((h.y >> L.sh_hi) & L.mask_hi);
    const uint32_t mw = ((h.w >> L.sh_min) & L.mask_lo) | ((h.z >> L.sh_hi) & L.mask_hi);
    constexpr float kTwo23 = 8388608.0f;
    RowScales r;
    r.s0 = fmaf(d, __uint_as_float(__byte_perm(scw, 0x4B000000u, L.sel0)), -d * kTwo23);
    r.s1 = fmaf(d16, __uint_as_float(__byte_perm(scw, 0x4B000000u, L.sel1)), -d16 * kTwo23);
    r.o0 = fmaf(dm.y, __uint_as_float(__byte_perm(mw, 0x4B000000u, L.sel0)), -dm.y * kTwo23);
    r.o1 = fmaf(dm.y, __uint_as_float(__byte_perm(mw, 0x4B000000u, L.sel1)), -dm.y * kTwo23);
    return r;
}

// d = c + Σ a_i·b_i with a as four unsigned bytes and b as four signed bytes.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = c + Σ a_i·b_i with a and b as four unsigned bytes each.
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Integer code-dots of one slab against the three activation planes:
// d_lo[p] = Σ_l q_lo(l)·plane_p[l], d_hi[p] = 16·Σ_l q_hi(l)·plane_p[32 + l]
// (planes 0 and 1 unsigned, plane 2 signed).  Slab byte l pairs with plane
// byte l of the low 32 positions (words 0..7) and with plane byte l of the
// high 32 positions (words 8..15).  |d| < 2^21.
__device__ __forceinline__ void slab_dot_planes(const int (&pl)[3][16], uint4 q0, uint4 q1,
                                                int (&d_lo)[3], int (&d_hi)[3]) {
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t l4 = qw[w] & 0x0F0F0F0Fu;
        const uint32_t h4 = qw[w] & 0xF0F0F0F0u;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            d_lo[pp] = dp4a_uu(l4, (uint32_t)pl[pp][w], d_lo[pp]);
            d_hi[pp] = dp4a_uu(h4, (uint32_t)pl[pp][8 + w], d_hi[pp]);
        }
        d_lo[2] = dp4a_us(l4, pl[2][w], d_lo[2]);
        d_hi[2] = dp4a_us(h4, pl[2][8 + w], d_hi[2]);
    }
}

// 65536·d2 + 256·d1 + d0, i.e. Σ q·x in units of s_b·2^-15: the last two
// terms are an exact integer (|·| < 2^29), the sum takes one rounding.
__device__ __forceinline__ float plane_combine(const int (&d)[3]) {
    const int d01 = d[1] * 256 + d[0];
    return fmaf(static_cast<float>(d[2]), 65536.0f, static_cast<float>(d01));
}

// One row's contribution from one slab lane: scales, code-dots (times the
// plane unit s_b·2^-15, a power of two), lazy mins.
__device__ __forceinline__ float slab_row(const uint8_t *blk, int j, const LaneScaleSel &L, float unit,
                                          const int (&pl)[3][16], float sum_lo, float sum_hi) {
    const uint4 h = *reinterpret_cast<const uint4 *>(blk);
    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * j);
    const RowScales r = row_scales(h, L);
    int dl[3] = {0, 0, 0}, dh[3] = {0, 0, 0};
    slab_dot_planes(pl, q0, q1, dl, dh);
    return fmaf(unit, fmaf(r.s0, plane_combine(dl), r.s1 * plane_combine(dh)),
                -fmaf(r.o0, sum_lo, r.o1 * sum_hi));
}

// Row formats of the one-token kernel.  Both spend 144 bytes on every 256
// values of a row, so rows, stages and slab lanes have the same geometry;
// lane (b, j) covers values 64j..64j+63 of the 256-value group b, and
// row() returns that lane's share of one row, given the group's first byte.

// Q4_K: the group is one super-block; the lane reads the header and qs slab j.
struct FmtQ4K {
    static constexpr int kGroupBytes = 144;  // bytes per 256 values of a row
    __device__ static void prep_planes(int (&)[3][16]) {}
    struct Lane {
        LaneScaleSel sel;
        int j;
    };
    __device__ static void unit_of(int j, int i, int &slab, int &pos) { slab = j, pos = i; }
    __device__ static Lane lane(int j, const float *) { return Lane{lane_scale_sel(j), j}; }
    __device__ static float row(const uint8_t *grp, const Lane &L, float unit, const int (&pl)[3][16],
                                float sum_lo, float sum_hi) {
        return slab_row(grp, L.j, L.sel, unit, pl, sum_lo, sum_hi);
    }
};

// Q4_0: the group is eight 18-byte blocks; the lane's 64 values are blocks
// 2j and 2j+1 (bytes 36j..36j+35, 4-byte aligned): block A = values 0..31
// (its 16 qs bytes start 2 bytes in, so its words come out of funnel shifts),
// block B = values 32..63 (qs 4-byte aligned at byte 20).  Per block,
// Σ w·x = d·(Σ q·x − 8·Σ x).
struct FmtQ40 {
    static constexpr int kGroupBytes = 144;
    __device__ static void prep_planes(int (&)[3][16]) {}
    struct Lane {
        int j;
    };
    __device__ static void unit_of(int j, int i, int &slab, int &pos) { slab = j, pos = i; }
    __device__ static Lane lane(int j, const float *) { return Lane{j}; }
    __device__ static float row(const uint8_t *grp, const Lane &L, float unit, const int (&pl)[3][16],
                                float sum_lo, float sum_hi) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(grp + 36 * L.j);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = p[i];
        const float2 dd = __half22float2(__halves2half2(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)),
                                                        __ushort_as_half((unsigned short)(w[4] >> 16))));
        uint32_t qa[4], qb[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            qa[k] = __funnelshift_r(w[k], w[k + 1], 16);
            qb[k] = w[5 + k];
        }
        int da_lo[3] = {0, 0, 0}, da_hi[3] = {0, 0, 0}, db_lo[3] = {0, 0, 0}, db_hi[3] = {0, 0, 0};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t al = qa[k] & 0x0F0F0F0Fu, ah = qa[k] & 0xF0F0F0F0u;
            const uint32_t bl = qb[k] & 0x0F0F0F0Fu, bh = qb[k] & 0xF0F0F0F0u;
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                da_lo[pp] = dp4a_uu(al, (uint32_t)pl[pp][k], da_lo[pp]);
                da_hi[pp] = dp4a_uu(ah, (uint32_t)pl[pp][4 + k], da_hi[pp]);
                db_lo[pp] = dp4a_uu(bl, (uint32_t)pl[pp][8 + k], db_lo[pp]);
                db_hi[pp] = dp4a_uu(bh, (uint32_t)pl[pp][12 + k], db_hi[pp]);
            }
            da_lo[2] = dp4a_us(al, pl[2][k], da_lo[2]);
            da_hi[2] = dp4a_us(ah, pl[2][4 + k], da_hi[2]);
            db_lo[2] = dp4a_us(bl, pl[2][8 + k], db_lo[2]);
            db_hi[2] = dp4a_us(bh, pl[2][12 + k], db_hi[2]);
        }
        const float qa_x = fmaf(plane_combine(da_hi), 0.0625f, plane_combine(da_lo));
        const float qb_x = fmaf(plane_combine(db_hi), 0.0625f, plane_combine(db_lo));
        return fmaf(dd.x, fmaf(unit, qa_x, -8.0f * sum_lo), dd.y * fmaf(unit, qb_x, -8.0f * sum_hi));
    }
};

// BitNet b1.58 ternary (SKaiNET issue #1138 "[ternary-f32] Phase 2:
// TernaryF32GemvNative SPI + reference ViewKernel + TernaryF32KernelPack",
// section "Tasks"): 256 values in 64 bytes, four 2-bit fields per byte,
// code = field − 1.  The lane's 64 values are bytes 16j..16j+15 of the group
// (one 16-byte load); byte k of word w holds values 16w + 4k + i in field i.
// prep_planes transposes each 16-value run of the plane words so that plane
// word 4w + i holds values 16w + i, 16w + 4 + i, 16w + 8 + i, 16w + 12 + i,
// the order in which field i of word w meets them.  Σ x·code = Σ x·field − Σ x,
// the scale is applied after the dot (T1Params::out_scale).
struct FmtTern {
    static constexpr int kGroupBytes = 64;
    __device__ static void prep_planes(int (&pl)[3][16]) {
#pragma unroll
        for (int pp = 0; pp < 3; ++pp)
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t i0 = (uint32_t)pl[pp][4 * w], i1 = (uint32_t)pl[pp][4 * w + 1];
                const uint32_t i2 = (uint32_t)pl[pp][4 * w + 2], i3 = (uint32_t)pl[pp][4 * w + 3];
                const uint32_t t0 = __byte_perm(i0, i1, 0x5140), t1 = __byte_perm(i0, i1, 0x7362);
                const uint32_t t2 = __byte_perm(i2, i3, 0x5140), t3 = __byte_perm(i2, i3, 0x7362);
                pl[pp][4 * w] = (int)__byte_perm(t0, t2, 0x5410);
                pl[pp][4 * w + 1] = (int)__byte_perm(t0, t2, 0x7632);
                pl[pp][4 * w + 2] = (int)__byte_perm(t1, t3, 0x5410);
                pl[pp][4 * w + 3] = (int)__byte_perm(t1, t3, 0x7632);
            }
    }
    struct Lane {
        int j;
    };
    __device__ static void unit_of(int j, int i, int &slab, int &pos) { slab = j, pos = i; }
    __device__ static Lane lane(int j, const float *) { return Lane{j}; }
    __device__ static float row(const uint8_t *grp, const Lane &L, float unit, const int (&pl)[3][16],
                                float sum_lo, float sum_hi) {
        const uint4 q = *reinterpret_cast<const uint4 *>(grp + 16 * L.j);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        int d[3] = {0, 0, 0};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t f = (qw[w] >> (2 * i)) & 0x03030303u;
                d[0] = dp4a_uu(f, (uint32_t)pl[0][4 * w + i], d[0]);
                d[1] = dp4a_uu(f, (uint32_t)pl[1][4 * w + i], d[1]);
                d[2] = dp4a_us(f, pl[2][4 * w + i], d[2]);
            }
        }
        return fmaf(unit, plane_combine(d), -(sum_lo + sum_hi));
    }
};

// Q6_K (the other follow-up named by SKaiNET PR #562, section "Out of
// scope"; byte layout read as ggml's): 256 values in 210 bytes — ql[128]
// (low 4 bits), qh[64] (high 2 bits, four codes per byte), 16 signed 8-bit
// sub-block scales, fp16 d last; w = d·scale·(q − 32).  Lane j = 2n + h takes,
// in half n, the values 128n + 32g + 16h + l for g = 0..3 and l < 16: bytes
// 16h..16h+15 of the runs ql[64n..], ql[64n + 32..] and qh[32n..], one
// sub-block (and scale) per g.  Blocks start at any even byte, so every
// 16-byte run is read as five aligned words and funnel-shifted.
struct FmtQ6K {
    static constexpr int kGroupBytes = 210;
    __device__ static void prep_planes(int (&)[3][16]) {}
    __device__ static void unit_of(int j, int i, int &slab, int &pos) {
        slab = 2 * (j >> 1) + (i >> 1);
        pos = 2 * (i & 1) + (j & 1);
    }
    struct Lane {
        int n, h;
        float s16[4];  // Σ x over each of the lane's four 16-value sub-blocks
    };
    __device__ static Lane lane(int j, const float *bsx16) {
        Lane L;
        L.n = j >> 1;
        L.h = j & 1;
#pragma unroll
        for (int g = 0; g < 4; ++g) L.s16[g] = bsx16[8 * L.n + 2 * g + L.h];
        return L;
    }
    // Four words starting `off` bytes after the 4-byte aligned `base`, shifted
    // right by `sh` bits across word boundaries.
    __device__ static void run16(const uint32_t *base, int off, uint32_t sh, uint32_t (&o)[4]) {
        const uint32_t *p = base + off / 4;
        uint32_t w[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) w[i] = p[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[i], w[i + 1], sh);
    }
    __device__ static float row(const uint8_t *grp, const Lane &L, float unit, const int (&pl)[3][16], float,
                                float) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(grp);
        const uint32_t *base = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
        const uint32_t sh = (uint32_t)(a & 3) * 8;
        uint32_t qa[4], qb[4], qh[4], sw[4];
        run16(base, 64 * L.n + 16 * L.h, sh, qa);
        run16(base, 64 * L.n + 32 + 16 * L.h, sh, qb);
        run16(base, 128 + 32 * L.n + 16 * L.h, sh, qh);
        run16(base, 192, sh, sw);  // the 16 scales
        const uint32_t dbits = (base[52] >> sh) & 0xFFFFu;  // bytes 208..209
        const float d = __half2float(__ushort_as_half((unsigned short)dbits));
        // Scale g of this lane is scale byte 8n + h + 2g: word 2n (g < 2) or
        // 2n + 1, byte h + 2(g & 1).  Signed byte v → the float 2^23 + 128 + v
        // by one XOR and one byte permute, minus 2^23 + 128 (exact: both are
        // integers below 2^24), times d (exact: 11 × 8 significant bits).
        const uint32_t s0 = (L.n ? sw[2] : sw[0]) ^ 0x80808080u, s1 = (L.n ? sw[3] : sw[1]) ^ 0x80808080u;
        float sc[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t word = g < 2 ? s0 : s1;
            const uint32_t sel = 0x7440u | (uint32_t)(L.h + 2 * (g & 1));
            sc[g] = d * (__uint_as_float(__byte_perm(word, 0x4B000000u, sel)) - 8388736.0f);
        }
        float acc = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            int dd[3] = {0, 0, 0};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t src = (g & 1) ? qb[k] : qa[k];
                const uint32_t lo = (g & 2) ? ((src >> 4) & 0x0F0F0F0Fu) : (src & 0x0F0F0F0Fu);
                const uint32_t hs = g == 0 ? (qh[k] << 4) : g == 1 ? (qh[k] << 2) : g == 2 ? qh[k] : (qh[k] >> 2);
                const uint32_t code = (hs & 0x30303030u) | lo;  // 6-bit codes, four bytes
                dd[0] = dp4a_uu(code, (uint32_t)pl[0][4 * g + k], dd[0]);
                dd[1] = dp4a_uu(code, (uint32_t)pl[1][4 * g + k], dd[1]);
                dd[2] = dp4a_us(code, pl[2][4 * g + k], dd[2]);
            }
            acc = fmaf(sc[g], fmaf(unit, plane_combine(dd), -32.0f * L.s16[g]), acc);
        }
        return acc;
    }
};

// L2 eviction policies for the weight stream.  Weights are read once per
// call: evict_first keeps them from displacing data that is read again
// (activations, outputs, whatever the caller keeps hot in L2).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global → shared with an L2 cache policy, completion counted
// on `bar` in bytes; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Round to nearest (ties to even) for |v| < 2^22 with the 1.5·2^23 shifter:
// the float's bits are 0x4B400000 + rint(v).
constexpr float kShifter = 12582912.0f;
constexpr uint32_t kShifterBits = 0x4B400000u;

// Bytes per 64-value slab in the plane area: 12 units of 16 bytes (3 planes
// × 4 quarters) plus 16 bytes of padding, so that the eight slabs read by a
// quarter warp start in eight different bank groups.
constexpr int kPlaneSlabBytes = 208;

struct T1Params {
    const float *x;
    const uint8_t *W;
    const uint8_t *W2;  // SwiGLU: the up projection (W is the gate projection)
    float *y;
    int *status;
    int N;
    int nb;            // blocks per row (K/256)
    int rg;            // row groups: compute warps = wc·rg
    int rows_per_cta;  // contiguous rows per CTA
    int stage_rows;    // rows per ring slot (multiple of the pass size)
    int nslots;        // ring depth
    int pre_stages;    // stages issued before the wait on the previous kernel
    int x_staged;      // 1: x arrives by one bulk copy into shared memory
    float out_scale;   // y = out_scale · (row result); 1 except for the ternary scale
    int T;             // tokens (x [T][K], y [T][N]); each compute warp serves one token
    int l2_evict_first;  // 1: weight copies carry the L2 evict_first policy
};

constexpr int kT1RoleWarps = 1;  // the copy warp
static_assert(kPlaneSlabBytes == kT1PlaneSlabBytes, "plane layout of the kernel and its geometry");

// kSwiGLU: the CTA's rows of W (gate) and then the same rows of W2 (up) form
// one list of 2·nrows virtual rows through the same ring and passes; every
// row result goes to shared memory and y[o] = silu(g[o])·u[o] at the end.
template <class Fmt, int kNB, bool kSwiGLU>
__global__ void __launch_bounds__(32 * (kT1RoleWarps + kT1MaxCw), 1) gemv_t1_kernel(T1Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int abort_flag;
    __shared__ int issued;  // weight stages issued so far (for the abort drain)
    __shared__ __align__(8) uint64_t x_bar;

    // Row geometry: compile-time when kNB > 0.
    const int nb = kNB > 0 ? kNB : p.nb;
    const int K = nb * kQ4kValues;
    const int nslabs = 4 * nb;                     // 64-value slabs per row
    const uint32_t row_bytes = (uint32_t)nb * Fmt::kGroupBytes;
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
    // Tokens: the planes, sums and block scales of token t follow those of
    // token t − 1, so the split indexes them by its flat position in x [T][K].
    const int T = kSwiGLU ? 1 : p.T;
    const int TK = T * K;
    const int ncw = T * wc * p.rg;
    const uint32_t slot_bytes = p.stage_rows * row_bytes;
    uint8_t *planes = smem;                                           // T·nslabs × 208 bytes
    float *sx = reinterpret_cast<float *>(planes + T * nslabs * kPlaneSlabBytes);  // T·K/32 sub-block sums
    float *sx16 = sx + TK / 32;                                       // T·K/16 half-sub-block sums
    float *sb = sx16 + TK / 16;                                       // T·K/256 block scales
    float *xst = sb + ((T * nb + 3) & ~3);                            // x (when staged)
    uint8_t *ring = reinterpret_cast<uint8_t *>(xst + (p.x_staged ? TK : 0));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(ring + (size_t)p.nslots * slot_bytes);
    uint64_t *empty_bar = full_bar + p.nslots;
    float *part = reinterpret_cast<float *>(empty_bar + p.nslots);  // [T][virtual rows][wc]

    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int nv = kSwiGLU ? 2 * nrows : nrows;  // rows streamed through the ring
    const bool to_smem = wide || kSwiGLU;        // row results go to part[]
    const int nstages = (nv + p.stage_rows - 1) / p.stage_rows;
    const int passes_per_stage = p.stage_rows / pass_rows;

    // Bulk copies need a 16-byte aligned destination; never issue one otherwise.
    if (smem_addr(smem) & 15) {
        if (threadIdx.x == 0) flag_timeout(p.status);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full_bar[s], 1);
            // Every pass of a stage is worked by the wc warps of a row, per token.
            mbar_init(&empty_bar[s], passes_per_stage * wc * T);
        }
        mbar_init(&x_bar, 1);
        abort_flag = 0;
        issued = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // Weights are read once: streamed with evict_first so that they
            // do not displace activations and outputs from L2.
            const uint64_t wpol = p.l2_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
            auto issue = [&](int st, int slot) {
                const int v0 = st * p.stage_rows, v1 = min(v0 + p.stage_rows, nv);
                uint8_t *dst = ring + (size_t)slot * slot_bytes;
                // Gate (or only) rows [v0, min(v1, nrows)), then up rows.
                const int g1 = kSwiGLU ? min(v1, nrows) : v1;
                if (g1 > v0) {
                    const uint8_t *src = p.W + (size_t)(row0 + v0) * row_bytes;
                    const uint32_t bytes = (uint32_t)(g1 - v0) * row_bytes;
                    // Rows of a format whose row size is not a multiple of 16
                    // start stages on 8-row boundaries (16-byte aligned); only
                    // the last stage of the matrix can end off the 16-byte
                    // grid: its last bytes go by plain loads, ahead of the
                    // arrive that publishes the stage.
                    const uint32_t bulk = bytes & ~15u;
                    if (bulk != bytes) {
                        for (uint32_t i = bulk; i < bytes; ++i) dst[i] = __ldg(src + i);
                        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(v1 - v0) * row_bytes - (bytes - bulk));
                    } else {
                        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(v1 - v0) * row_bytes);
                    }
                    bulk_g2s_hint(dst, src, bulk, &full_bar[slot], wpol);
                } else {
                    mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(v1 - v0) * row_bytes);
                }
                if (kSwiGLU && v1 > nrows) {
                    const int u0 = max(v0, nrows);
                    bulk_g2s_hint(dst + (size_t)(u0 - v0) * row_bytes,
                                  p.W2 + (size_t)(row0 + u0 - nrows) * row_bytes, (uint32_t)(v1 - u0) * row_bytes,
                                  &full_bar[slot], wpol);
                }
                issued = st + 1;
            };
            const int first = min(nstages, p.nslots);
            const int pre = min(first, p.pre_stages);
            int st = 0;
            for (; st < pre; ++st) issue(st, st);
            // x may be written by the previous kernel on the stream.
            pdl_wait();
            if (p.x_staged) {
                mbar_arrive_expect_tx(&x_bar, (uint32_t)TK * sizeof(float));
                bulk_g2s(xst, p.x, (uint32_t)TK * sizeof(float), &x_bar);
            }
            for (; st < first; ++st) issue(st, st);
            for (; st < nstages; ++st) {
                const int slot = st % p.nslots;
                if (abort_flag) break;
                if (!mbar_wait_bounded(&empty_bar[slot], ((st / p.nslots) - 1) & 1,
                                       kWaitLimitCycles)) {
                    abort_flag = 1;
                    flag_timeout(p.status);
                    break;
                }
                issue(st, slot);
            }
        }
        __syncwarp();
    } else {
        const int cw = warp - kT1RoleWarps;
        const int tok = cw / (wc * p.rg), cwt = cw % (wc * p.rg);
        const int wcol = cwt % wc, rgi = cwt / wc;
        const int ro = wide ? 0 : lane / lpr;
        const int s = wide ? wcol * 32 + lane : lane % lpr;
        const bool active = s < L;
        const int b = active ? (s >> 2) : 0, j = s & 3;

        // x may be produced by the previous kernel on the stream.
        pdl_wait();
        const float *xsrc = p.x;
        if (p.x_staged) {
            if (!mbar_wait_bounded(&x_bar, 0, kWaitLimitCycles)) {
                abort_flag = 1;
                flag_timeout(p.status);
            }
            xsrc = xst;
        }
        // x → three byte planes under power-of-two block scales, plus the
        // fp32 sub-block sums.  Thread ct takes eighths of sub-blocks (8
        // values): the 32 threads of a block form one warp and share its
        // maximum; the four threads of a sub-block are neighbouring lanes.
        {
            const int ct = threadIdx.x - 32 * kT1RoleWarps, nth = ncw * 32, ne = TK / 8;
            for (int e0 = 0; e0 < ne; e0 += nth) {
                const int e = e0 + ct;
                const bool on = e < ne && !abort_flag;
                float v[8];
                {
                    const float4 *src = reinterpret_cast<const float4 *>(xsrc) + 2 * e;
                    const float4 t0 = on ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 t1 = on ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[0] = t0.x; v[1] = t0.y; v[2] = t0.z; v[3] = t0.w;
                    v[4] = t1.x; v[5] = t1.y; v[6] = t1.z; v[7] = t1.w;
                }
                float amax = 0.f, sum = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    amax = fmaxf(amax, fabsf(v[i]));
                    sum += v[i];
                }
                // Non-negative floats order like their bit patterns.
                amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax)));
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                const float sum16 = sum;
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
                // s_b = 2^ex with amax / 2^ex <= 127 (1 when the block is
                // zero): ex is the binary exponent of amax/127 written as
                // m·2^ex with m in [0.5, 1), read from the float's exponent
                // field; -112 bounds it below so that 2^(15-ex) stays a
                // normal float (such blocks still scale below 127).
                const int ebits = (int)(__float_as_uint(amax * (1.0f / 127.0f)) >> 23);
                const int ex = amax > 0.f ? max(ebits - 126, -112) : 0;
                const float inv = __uint_as_float((uint32_t)(127 + 15 - ex) << 23);  // 2^(15-ex)
                // n = rint(v·2^(15-ex)) with one FMA (exact product, one
                // rounding); its three low bytes are the planes' digits.
                uint32_t nb_[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) nb_[i] = __float_as_uint(fmaf(v[i], inv, kShifter)) - kShifterBits;
                uint32_t w[3][2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint32_t *n4 = nb_ + 4 * k;
                    w[0][k] = __byte_perm(__byte_perm(n4[0], n4[1], 0x0040), __byte_perm(n4[2], n4[3], 0x0040), 0x5410);
                    w[1][k] = __byte_perm(__byte_perm(n4[0], n4[1], 0x0051), __byte_perm(n4[2], n4[3], 0x0051), 0x5410);
                    w[2][k] = __byte_perm(__byte_perm(n4[0], n4[1], 0x0062), __byte_perm(n4[2], n4[3], 0x0062), 0x5410);
                }
                if (on) {
                    // Slab-major layout: slab S = e/8 holds 12 units of 16
                    // bytes, unit 4p + i covering plane p of values
                    // 16i..16i+15 of the slab; this thread writes the half
                    // e % 2 of unit i = (e/2) % 4 of each plane.
                    uint2 *pu = reinterpret_cast<uint2 *>(planes + (e >> 3) * kPlaneSlabBytes) +
                                2 * ((e >> 1) & 3) + (e & 1);
                    pu[0] = make_uint2(w[0][0], w[0][1]);
                    pu[8] = make_uint2(w[1][0], w[1][1]);
                    pu[16] = make_uint2(w[2][0], w[2][1]);
                    if ((e & 1) == 0) sx16[e / 2] = sum16;
                    if ((e & 3) == 0) sx[e / 4] = sum;
                    if ((e & 31) == 0) sb[e / 32] = __uint_as_float((uint32_t)(127 + ex) << 23);
                }
            }
        }
        named_bar_sync(1, ncw * 32);
        int pl[3][16];
        float s_blk, sum_lo, sum_hi;
        {
            // This slab's 64 plane bytes per plane: positions 64j..64j+31
            // (low nibbles) then 64j+32..64j+63 (high nibbles) of block b.
            // (Fmt::unit_of names the slab and 16-value unit of each of the
            // lane's four runs; the Q4 and ternary lanes take slab j in order.)
#pragma unroll
            for (int pp = 0; pp < 3; ++pp) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int us, up;
                    Fmt::unit_of(j, i, us, up);
                    const uint4 *src =
                        reinterpret_cast<const uint4 *>(planes + (tok * nslabs + 4 * b + us) * kPlaneSlabBytes);
                    const uint4 t = active ? src[4 * pp + up] : make_uint4(0u, 0u, 0u, 0u);
                    pl[pp][4 * i] = (int)t.x;
                    pl[pp][4 * i + 1] = (int)t.y;
                    pl[pp][4 * i + 2] = (int)t.z;
                    pl[pp][4 * i + 3] = (int)t.w;
                }
            }
            s_blk = active ? sb[tok * nb + b] : 0.f;
            sum_lo = active ? sx[tok * K / 32 + 8 * b + 2 * j] : 0.f;
            sum_hi = active ? sx[tok * K / 32 + 8 * b + 2 * j + 1] : 0.f;
        }
        Fmt::prep_planes(pl);
        const typename Fmt::Lane lfmt = Fmt::lane(j, sx16 + tok * K / 16 + 16 * b);
        const float unit = s_blk * (1.0f / 32768.0f);

        const int npasses = (nv + pass_rows - 1) / pass_rows;
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
                stage_base = ring + (size_t)slot * slot_bytes + b * Fmt::kGroupBytes;
                rows = min(p.stage_rows, nv - st * p.stage_rows);
            }
            const int ra = pin * pass_rows + 2 * ro, rb = ra + 1;
            float pa = Fmt::row(stage_base + min(ra, rows - 1) * row_bytes, lfmt, unit, pl, sum_lo, sum_hi);
            float pb = Fmt::row(stage_base + min(rb, rows - 1) * row_bytes, lfmt, unit, pl, sum_lo, sum_hi);
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
                if ((lane & (half - 1)) == 0 && r < rows) part[(tok * nv + rl) * wc + wcol] = v;
            } else if (kSwiGLU) {
                if (s == (up ? half : 0) && r < rows) part[rl] = v;
            } else {
                if (s == (up ? half : 0) && r < rows) p.y[(size_t)tok * p.N + row0 + rl] = p.out_scale * v;
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

        if (to_smem) {
            named_bar_sync(1, ncw * 32);
            for (int it = threadIdx.x - 32 * kT1RoleWarps; it < T * nrows; it += ncw * 32) {
                const int t = it / nrows, i = it % nrows;
                const float *pt = part + (size_t)t * nv * wc;
                float acc = 0.f;
                for (int w = 0; w < wc; ++w) acc += pt[i * wc + w];
                if (kSwiGLU) {
                    float up = 0.f;
                    for (int w = 0; w < wc; ++w) up += pt[(nrows + i) * wc + w];
                    acc = acc / (1.0f + expf(-acc)) * up;  // silu(g)·u
                }
                p.y[(size_t)t * p.N + row0 + i] = p.out_scale * acc;
            }
        }
    }

    // Never leave a bulk copy writing into shared memory of an exiting CTA.
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        for (int st = max(0, issued - p.nslots); st < issued; ++st)
            (void)mbar_wait_bounded(&full_bar[st % p.nslots], (st / p.nslots) & 1,
                                    kWaitLimitCycles);
        if (p.x_staged) (void)mbar_wait_bounded(&x_bar, 0, kWaitLimitCycles);
    }
}

// Geometry knobs of the one-token kernel (T1Tuning, t1_geometry.h) from the
// environment, read once; out-of-range values are clamped.
int env_int(const char *name, int dflt, int lo, int hi) {
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    const int x = atoi(v);
    return x < lo ? lo : (x > hi ? hi : x);
}

const T1Tuning &t1_tuning() {
    static const T1Tuning t = [] {
        T1Tuning r;
        r.warps = env_int("Q4MM_T1_WARPS", r.warps, 1, kT1MaxCw);
        r.ctas_per_sm = env_int("Q4MM_T1_CTAS_PER_SM", r.ctas_per_sm, 1, 8);
        r.stage_bytes = env_int("Q4MM_T1_STAGE_BYTES", r.stage_bytes, 1024, 65536);
        r.ring_bytes = env_int("Q4MM_T1_RING_BYTES", r.ring_bytes, 8192, 200 * 1024);
        r.pre_stages = env_int("Q4MM_T1_PRE_STAGES", r.pre_stages, 0, 64);
        r.x_stage_max = env_int("Q4MM_T1_X_STAGE_MAX", r.x_stage_max, 0, 65536);
        r.l2_evict_first = env_int("Q4MM_T1_L2_EVICT_FIRST", r.l2_evict_first, 0, 1);
        r.max_grid = env_int("Q4MM_T1_MAX_GRID", r.max_grid, 0, 4096);
        r.spare_sms = env_int("Q4MM_T1_SPARE_SMS", r.spare_sms, 0, 64);
        r.spare_max_bytes = env_int("Q4MM_T1_SPARE_MAX_BYTES", r.spare_max_bytes, 0, 1 << 30);
        return r;
    }();
    return t;
}

}  // namespace

template <class Fmt, bool kSwiGLU = false>
cudaError_t launch_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N,
                           const uint8_t *W2 = nullptr, float out_scale = 1.0f, int T = 1) {
    const T1Tuning &tun = t1_tuning();
    const T1Geometry g =
        plan_gemv_t1(Fmt::kGroupBytes, K, N, T, kSwiGLU ? 2 : 1, c.num_sms, c.max_smem_optin, tun);
    if (!g.ok) return cudaErrorNotSupported;
    T1Params p;
    p.T = T;
    p.x = x;
    p.W = W;
    p.W2 = W2;
    p.out_scale = out_scale;
    p.y = y;
    p.status = c.status;
    p.N = N;
    p.nb = K / kQ4kValues;
    p.rg = g.rg;
    p.rows_per_cta = g.rows_per_cta;
    p.stage_rows = g.stage_rows;
    p.nslots = g.nslots;
    p.pre_stages = g.pre_stages;
    p.x_staged = g.x_staged;
    p.l2_evict_first = tun.l2_evict_first;
    const int grid = g.grid;
    const size_t smem = g.smem;

    const dim3 block(32 * (kT1RoleWarps + g.ncw));
    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e = ensure_smem(kernel, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(c, kernel, dim3(grid), block, smem, p);
    };
    if constexpr (kSwiGLU) {
        switch (p.nb) {
            case 16: return go(gemv_t1_kernel<Fmt, 16, true>);
            default: return go(gemv_t1_kernel<Fmt, 0, true>);
        }
    } else if constexpr (std::is_same<Fmt, FmtQ6K>::value) {
        switch (p.nb) {
            case 16: return go(gemv_t1_kernel<Fmt, 16, false>);
            default: return go(gemv_t1_kernel<Fmt, 0, false>);
        }
    } else if constexpr (std::is_same<Fmt, FmtTern>::value) {
        switch (p.nb) {
            case 10: return go(gemv_t1_kernel<Fmt, 10, false>);
            default: return go(gemv_t1_kernel<Fmt, 0, false>);
        }
    } else if constexpr (std::is_same<Fmt, FmtQ4K>::value) {
        switch (p.nb) {
            case 4: return go(gemv_t1_kernel<Fmt, 4, false>);
            case 8: return go(gemv_t1_kernel<Fmt, 8, false>);
            case 16: return go(gemv_t1_kernel<Fmt, 16, false>);
            case 32: return go(gemv_t1_kernel<Fmt, 32, false>);
            case 43: return go(gemv_t1_kernel<Fmt, 43, false>);
            case 56: return go(gemv_t1_kernel<Fmt, 56, false>);
            case 64: return go(gemv_t1_kernel<Fmt, 64, false>);
            default: return go(gemv_t1_kernel<Fmt, 0, false>);
        }
    } else {
        switch (p.nb) {
            case 16: return go(gemv_t1_kernel<Fmt, 16, false>);
            case 43: return go(gemv_t1_kernel<Fmt, 43, false>);
            default: return go(gemv_t1_kernel<Fmt, 0, false>);
        }
    }
}

cudaError_t launch_q4k_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N,
                               int T) {
    return launch_gemv_t1<FmtQ4K>(c, x, W, y, K, N, nullptr, 1.0f, T);
}

cudaError_t launch_q4_0_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N,
                                int T) {
    return launch_gemv_t1<FmtQ40>(c, x, W, y, K, N, nullptr, 1.0f, T);
}

cudaError_t launch_q6k_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N,
                              int T) {
    return launch_gemv_t1<FmtQ6K>(c, x, W, y, K, N, nullptr, 1.0f, T);
}

cudaError_t launch_ternary_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float scale, float *y,
                                   int K, int N, int T) {
    return launch_gemv_t1<FmtTern>(c, x, W, y, K, N, nullptr, scale, T);
}

cudaError_t launch_q4k_ffn_swiglu_t1(const LaunchCtx &c, const float *x, const uint8_t *Wg, const uint8_t *Wu,
                                     float *h, int K, int N) {
    return launch_gemv_t1<FmtQ4K, true>(c, x, Wg, h, K, N, Wu);
}

}  // namespace q4mm
