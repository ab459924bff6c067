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
// producer thread issues.  The 2..8 token kernel is in q4k_gemv_multi.cu.
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"
#include "t1_geometry.h"

namespace q4mm {

namespace {

// ----------------------------------------------------------------------------
// One token: bulk-copied rows, slab lanes, byte planes of the activations
// ----------------------------------------------------------------------------
//
// Roles in a CTA (a contiguous range of output rows, 16 warps, all of them
// computing: an SM sub-partition then runs 4 warps of up to 128 registers):
//  * thread 0 issues the first ring stages: 1-D bulk copies of whole stages
//    of rows.  Weights are never written by an earlier kernel on the stream,
//    so stages may go out before the wait on the previous kernel; with x
//    staged in shared memory (up to 64 KB of it) x is copied first, right
//    after that wait, and the first stages follow (an activation fetch
//    queued behind the CTA's own weight stream arrives late, and everything
//    after it waits for it).  Above 64 KB of x the compute threads load x
//    themselves and the stages go out first;
//  * every warp splits its share of x into byte planes; then the first ncw
//    warps are "slab lanes": lane (b, j) owns the 32-byte qs slab j of block
//    b of every row it visits (32 low nibbles of sub-block 2j, 32 high
//    nibbles of 2j+1) and decodes the two 6-bit scale/min pairs it needs
//    from the block header.  A row group takes passes r, r + rg, ... of the
//    CTA's rows, kRP rows per row slot and pass;
//  * the warp that finishes the last pass of a ring slot's stage issues the
//    stage that next uses the slot (a per-slot pass counter with
//    release/acquire ordering and an async-proxy fence before the copy), so
//    no thread is set aside for copying.
//
// The code-dot Σ x·q of a sub-block runs on integer dot-product instructions
// (four byte products per instruction).  Each 32-value group g of x is split,
// once per CTA, into P = kT1Planes byte planes under a power-of-two scale
// s_g = 2^e ≥ max|x_g|/255 (so s_g < 2·max|x_g|/255), with S = 8P − 9:
//   n = rint(x·2^S/s_g),  |n| < 255·2^S < 2^(8P−1),
//   n = Σ_p 2^(8p)·d_p  (the low digits unsigned bytes, the top one signed),
// so x = s_g·2^-S·n + e with |e| ≤ 2^-(S+1)·s_g < 2^-S·max|x_g|/255 (s_g is
// at least 2^(S−126), so groups below 255·2^(S−126) have |e| ≤ 2^-127
// instead).  The product by a power of two is exact and the conversion
// rounds once; every x_g value of magnitude at least s_g (within a factor of
// about 255 of the group's largest) is represented exactly, and only smaller
// ones carry the error above.  A group's scale depends on its own 32 values
// only, so a large activation elsewhere in the row changes nothing here.
// Q4_K codes enter the dot products unsigned (high nibbles masked in place as
// 16·q, the factor taken out of the sub-block's scale) and the min term uses
// the fp32 group sums; formats whose zero point is a fixed code (Q4_0, Q6_K,
// ternary) enter as signed bytes c − zero, so their sums are exact integers.
// The planes' sums are combined with two fp32 roundings, and scales, mins
// and the final sum are fp32.
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

// d = c + Σ a_i·b_i over four byte pairs; a (the codes) and b (a plane)
// each unsigned (u) or signed (s).
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Activation planes of one lane: kT1Planes planes of 16 words (the lane's 64
// values, four per word); the last plane holds signed bytes.
using Planes = int[kT1Planes][16];
using Acc = int[kT1Planes];

// Four code bytes (four values) against word w of every plane.  kSigned:
// the codes are signed bytes (formats whose zero point is a fixed code).
template <bool kSigned = false>
__device__ __forceinline__ void dot4(uint32_t codes, const Planes &pl, int w, Acc &d) {
#pragma unroll
    for (int p = 0; p + 1 < kT1Planes; ++p)
        d[p] = kSigned ? dp4a_su(codes, (uint32_t)pl[p][w], d[p]) : dp4a_uu(codes, (uint32_t)pl[p][w], d[p]);
    constexpr int t = kT1Planes - 1;
    d[t] = kSigned ? dp4a_ss(codes, (uint32_t)pl[t][w], d[t]) : dp4a_us(codes, (uint32_t)pl[t][w], d[t]);
}

// Σ c·n in units of the group's step: Σ_p 2^(8p)·d_p, as 2^16·hi + lo with
// hi = 256·d3 + d2 (four planes) or d2 (three) and lo = 256·d1 + d0.  For
// the 4-bit and 2-bit codes hi has at most 24 significant bits (times a
// power of two when the codes carry one), so its conversion is exact; lo
// takes one rounding, the sum another (Q6_K's 6-bit codes over 16 values can
// take hi to 25 bits: one more rounding there).
__device__ __forceinline__ float plane_combine(const Acc &d) {
    const int hi = kT1Planes == 4 ? d[kT1Planes - 1] * 256 + d[2] : d[2];
    const int lo = d[1] * 256 + d[0];
    return fmaf(static_cast<float>(hi), 65536.0f, static_cast<float>(lo));
}

// The plane split's scale: n = rint(x·2^kShift/s_g) fills 8·kT1Planes − 1 bits.
constexpr int kShift = 8 * kT1Planes - 9;

// Row formats of the one-token kernel.  Each spends group_bytes on every 256
// values of a row, so rows, stages and slab lanes have the same geometry;
// lane (b, j) covers values 64j..64j+63 of the 256-value group b (Q6_K
// interleaves, see its unit_of), and row() returns that lane's share of one
// row, given the group's first byte.

// Q4_K: the group is one super-block; the lane reads the header and qs slab j.
struct FmtQ4K {
    static constexpr int kGroupBytes = 144;  // bytes per 256 values of a row
    static constexpr bool kSums = true;      // needs Σx per 32-value group (the min term)
    __device__ static void prep_planes(Planes &) {}
    struct Lane {
        LaneScaleSel sel;
        int j;
        float u_lo, u_hi, s_lo, s_hi;
    };
    __device__ static void unit_of(int j, int i, int &slab, int &pos) { slab = j, pos = i; }
    // u32 / sx32 point at block b's first entries (8 groups of 32 per block).
    __device__ static Lane lane(int j, const float *u32, const float *sx32) {
        Lane L;
        L.sel = lane_scale_sel(j);
        L.j = j;
        L.u_lo = u32[2 * j];
        L.u_hi = u32[2 * j + 1];
        L.s_lo = sx32[2 * j];
        L.s_hi = sx32[2 * j + 1];
        return L;
    }
    __device__ static float row(const uint8_t *blk, const Lane &L, const Planes &pl) {
        const uint4 h = *reinterpret_cast<const uint4 *>(blk);
        const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * L.j);
        const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * L.j);
        const RowScales r = row_scales(h, L.sel);
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        // Slab byte l pairs with plane byte l of the low 32 positions (words
        // 0..7) and with plane byte l of the high 32 positions (words 8..15).
        Acc dl = {}, dh = {};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            dot4(qw[w] & 0x0F0F0F0Fu, pl, w, dl);
            dot4(qw[w] & 0xF0F0F0F0u, pl, 8 + w, dh);
        }
        return fmaf(r.s0 * L.u_lo, plane_combine(dl), (r.s1 * L.u_hi) * plane_combine(dh)) -
               fmaf(r.o0, L.s_lo, r.o1 * L.s_hi);
    }
};

// Q4_0: the group is eight 18-byte blocks; the lane's 64 values are blocks
// 2j and 2j+1 (bytes 36j..36j+35, 4-byte aligned): block A = values 0..31
// (its 16 qs bytes start 2 bytes in, so its words come out of funnel shifts),
// block B = values 32..63 (qs 4-byte aligned at byte 20).  The zero point is
// the code 8 (w = d·(q − 8)), so the codes enter the dot products as the
// signed bytes 16·(q − 8) — a nibble in a byte's high half XOR 0x80 — and the
// block's sum Σ 16·(q − 8)·n is an exact integer: a zero weight adds nothing,
// whatever its activation.
struct FmtQ40 {
    static constexpr int kGroupBytes = 144;
    static constexpr bool kSums = false;
    __device__ static void prep_planes(Planes &) {}
    struct Lane {
        int j;
        float u16_a, u16_b;  // the steps of blocks A and B, over 16 (the codes carry 16)
    };
    __device__ static void unit_of(int j, int i, int &slab, int &pos) { slab = j, pos = i; }
    __device__ static Lane lane(int j, const float *u32, const float *) {
        Lane L;
        L.j = j;
        L.u16_a = u32[2 * j] * 0.0625f;
        L.u16_b = u32[2 * j + 1] * 0.0625f;
        return L;
    }
    __device__ static float row(const uint8_t *grp, const Lane &L, const Planes &pl) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(grp + 36 * L.j);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) w[i] = p[i];
        const float2 dd = __half22float2(__halves2half2(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)),
                                                        __ushort_as_half((unsigned short)(w[4] >> 16))));
        // Low nibbles (values 0..15 of a block) shifted into the high half,
        // high nibbles (values 16..31) masked in place.
        Acc a = {}, b = {};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t qa = __funnelshift_r(w[k], w[k + 1], 16), qb = w[5 + k];
            dot4<true>(((qa << 4) & 0xF0F0F0F0u) ^ 0x80808080u, pl, k, a);
            dot4<true>((qa & 0xF0F0F0F0u) ^ 0x80808080u, pl, 4 + k, a);
            dot4<true>(((qb << 4) & 0xF0F0F0F0u) ^ 0x80808080u, pl, 8 + k, b);
            dot4<true>((qb & 0xF0F0F0F0u) ^ 0x80808080u, pl, 12 + k, b);
        }
        return fmaf(dd.x * L.u16_a, plane_combine(a), (dd.y * L.u16_b) * plane_combine(b));
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
    static constexpr bool kSums = false;
    __device__ static void prep_planes(Planes &pl) {
#pragma unroll
        for (int pp = 0; pp < kT1Planes; ++pp)
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
        float u_lo, u_hi;
    };
    __device__ static void unit_of(int j, int i, int &slab, int &pos) { slab = j, pos = i; }
    __device__ static Lane lane(int j, const float *u32, const float *) {
        Lane L;
        L.j = j;
        L.u_lo = u32[2 * j];
        L.u_hi = u32[2 * j + 1];
        return L;
    }
    __device__ static float row(const uint8_t *grp, const Lane &L, const Planes &pl) {
        const uint4 q = *reinterpret_cast<const uint4 *>(grp + 16 * L.j);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        // Words 0, 1 hold values 0..31 (the low group), words 2, 3 values 32..63.
        // Each field f becomes the signed byte f − 1 (a bytewise subtraction
        // with no borrow between bytes: bit 7 set first, then cleared), so
        // the code-dot is an exact integer and a zero code adds nothing.
        Acc dl = {}, dh = {};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t f = ((qw[w] >> (2 * i)) & 0x03030303u) | 0x80808080u;
                const uint32_t c = (f - 0x01010101u) ^ 0x80808080u;
                dot4<true>(c, pl, 4 * w + i, w < 2 ? dl : dh);
            }
        }
        return fmaf(L.u_lo, plane_combine(dl), L.u_hi * plane_combine(dh));
    }
};

// Q6_K (the other follow-up named by SKaiNET PR #562, section "Out of
// scope"; byte layout read as ggml's): 256 values in 210 bytes — ql[128]
// (low 4 bits), qh[64] (high 2 bits, four codes per byte), 16 signed 8-bit
// sub-block scales, fp16 d last; w = d·scale·(q − 32).  Lane j = 2n + h takes,
// in half n, the values 128n + 32g + 16h + l for g = 0..3 and l < 16: bytes
// 16h..16h+15 of the runs ql[64n..], ql[64n + 32..] and qh[32n..], one
// sub-block (and scale) per g, each run in 32-value group 4n + g of the
// block.  Blocks start at any even byte, so every 16-byte run is read as
// five aligned words and funnel-shifted.
struct FmtQ6K {
    static constexpr int kGroupBytes = 210;
    static constexpr bool kSums = false;
    __device__ static void prep_planes(Planes &) {}
    __device__ static void unit_of(int j, int i, int &slab, int &pos) {
        slab = 2 * (j >> 1) + (i >> 1);
        pos = 2 * (i & 1) + (j & 1);
    }
    struct Lane {
        int n, h;
        float u4[4];  // per run g: the step of its 32-value group, over 4 (the codes carry 4)
    };
    __device__ static Lane lane(int j, const float *u32, const float *) {
        Lane L;
        L.n = j >> 1;
        L.h = j & 1;
#pragma unroll
        for (int g = 0; g < 4; ++g) L.u4[g] = u32[4 * L.n + g] * 0.25f;
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
    __device__ static float row(const uint8_t *grp, const Lane &L, const Planes &pl) {
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
        float acc = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t word = g < 2 ? s0 : s1;
            const uint32_t sel = 0x7440u | (uint32_t)(L.h + 2 * (g & 1));
            const float sc = d * (__uint_as_float(__byte_perm(word, 0x4B000000u, sel)) - 8388736.0f);
            // The zero point is the code 32: codes enter as the signed bytes
            // 4·(q − 32), i.e. 4·q XOR 0x80, and the sum is an exact integer.
            Acc dd = {};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t src = (g & 1) ? qb[k] : qa[k];
                const uint32_t lo = (g & 2) ? ((src >> 2) & 0x3C3C3C3Cu) : ((src << 2) & 0x3C3C3C3Cu);
                const uint32_t hs = g == 0 ? (qh[k] << 6) : g == 1 ? (qh[k] << 4) : g == 2 ? (qh[k] << 2) : qh[k];
                const uint32_t code4 = ((hs & 0xC0C0C0C0u) | lo) ^ 0x80808080u;  // 4·(q − 32), four bytes
                dot4<true>(code4, pl, 4 * g + k, dd);
            }
            acc = fmaf(sc * L.u4[g], plane_combine(dd), acc);
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

// Bytes per 64-value slab in the plane area: 4·kT1Planes units of 16 bytes
// (planes × quarters) plus 16 bytes of padding, so that the eight slabs read
// by a quarter warp start in eight different bank groups.
constexpr int kPlaneSlabBytes = 64 * kT1Planes + 16;

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
    int slot_bytes;    // bytes per ring slot (16 more when rows are off the 16-byte grid)
    int nslots;        // ring depth
    int pre_stages;    // stages issued before the wait on the previous kernel
    int x_staged;      // 1: x arrives by one bulk copy into shared memory
    float out_scale;   // y = out_scale · (row result); 1 except for the ternary scale
    int T;             // tokens (x [T][K], y [T][N]); each compute warp serves one token
    int l2_evict_first;  // 1: weight copies carry the L2 evict_first policy
    long long wait_limit;  // SM cycles a bounded wait lasts at most
    int withhold;          // test only: a stage whose copy is never issued (-1: none)
};

// Split of x into planes, group steps and (kSums) group sums, by every
// thread: thread ct takes 8 consecutive values of x [T][K] per step; the
// four threads of a 32-value group are neighbouring lanes and share its
// maximum.
template <bool kSums>
__device__ __forceinline__ void split_x(const float *xsrc, int TK, int ct, int nth, volatile int &abort_flag,
                                        uint8_t *planes, float *u32, float *sx32) {
    const int n8 = TK / 8;
    // Up to four steps' loads go out together (x may come from L2 or HBM).
    constexpr int kBatch = 4;
    for (int i00 = 0; i00 < n8; i00 += kBatch * nth) {
        float4 ld[kBatch][2];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i00 + u * nth + ct;
            const bool on = i < n8 && !abort_flag;
            const float4 *src = reinterpret_cast<const float4 *>(xsrc) + 2 * i;
            ld[u][0] = on ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
            ld[u][1] = on ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (i00 + u * nth >= n8) break;  // uniform over the CTA
            const int i = i00 + u * nth + ct;
            const bool on = i < n8 && !abort_flag;
            float v[8];
            v[0] = ld[u][0].x; v[1] = ld[u][0].y; v[2] = ld[u][0].z; v[3] = ld[u][0].w;
            v[4] = ld[u][1].x; v[5] = ld[u][1].y; v[6] = ld[u][1].z; v[7] = ld[u][1].w;
            float amax = 0.f, sum = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                amax = fmaxf(amax, fabsf(v[k]));
                if (kSums) sum += v[k];
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            if (kSums) {
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            }
            // s_g = 2^ex with amax / 2^ex < 255 (1 when the group is zero): ex is
            // the binary exponent of amax/255 written as m·2^ex with m in [0.5, 1),
            // read from the float's exponent field.  The lower bound kShift − 126
            // keeps both 2^(kShift-ex) and the step 2^(ex-kShift) normal floats
            // (such groups still scale below 255).  A product amax·(1/255) rounded
            // down across a power of two gives ex one too small and |n| at most
            // 255·2^kShift·(1 + 2^-23), still inside the planes.
            const int ebits = (int)(__float_as_uint(amax * (1.0f / 255.0f)) >> 23);
            const int ex = amax > 0.f ? max(ebits - 126, kShift - 126) : 0;
            const float mul = __uint_as_float((uint32_t)(127 + kShift - ex) << 23);  // 2^(kShift-ex)
            int n[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) n[k] = __float2int_rn(v[k] * mul);
            if (on) {
                // Slab-major layout: slab S = i/8 holds 4·kT1Planes units of 16
                // bytes, unit 4p + q covering plane p of values 16q..16q+15 of the
                // slab; this thread writes half i % 2 of quarter (i % 8)/2 of each
                // plane: a 4×4 byte transpose per four values (byte p of n is
                // plane p; with three planes byte 2 is already the signed top
                // digit).
                uint2 *pu = reinterpret_cast<uint2 *>(planes + (i >> 3) * kPlaneSlabBytes) + (i & 7);
                uint32_t P[4][2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t n0 = (uint32_t)n[4 * q], n1 = (uint32_t)n[4 * q + 1];
                    const uint32_t n2 = (uint32_t)n[4 * q + 2], n3 = (uint32_t)n[4 * q + 3];
                    const uint32_t t0 = __byte_perm(n0, n1, 0x5140), t1 = __byte_perm(n0, n1, 0x7362);
                    const uint32_t t2 = __byte_perm(n2, n3, 0x5140), t3 = __byte_perm(n2, n3, 0x7362);
                    P[0][q] = __byte_perm(t0, t2, 0x5410);
                    P[1][q] = __byte_perm(t0, t2, 0x7632);
                    P[2][q] = __byte_perm(t1, t3, 0x5410);
                    P[3][q] = __byte_perm(t1, t3, 0x7632);
                }
#pragma unroll
                for (int p = 0; p < kT1Planes; ++p) pu[8 * p] = make_uint2(P[p][0], P[p][1]);
                if ((i & 3) == 0) {
                    if (kSums) sx32[i >> 2] = sum;
                    u32[i >> 2] = __uint_as_float((uint32_t)(127 + ex - kShift) << 23);  // 2^(ex-kShift)
                }
            }
        }
    }
}

// Wait until *tag == want (a ring slot's stage tag), bounded; false on
// time-out or when another thread of the CTA has given up.
__device__ __forceinline__ bool wait_tag(const int *tag, int want, long long limit, const volatile int *abort) {
    const volatile int *t = tag;
    if (*t == want) return true;
    const long long t0 = clock64();
    while (*t != want) {
        if (*abort || clock64() - t0 > limit) return false;
        __nanosleep(64);
    }
    return true;
}

// Sum of kRP (2 or 4) row partials v[] over a slot of G lanes (G a power of
// two, at least kRP; slots are aligned lane groups): exchange levels leave
// each lane with one row, the rest is a butterfly.  Lane l of the slot ends
// with row (l % G) / (G / kRP) summed over the slot.
template <int kRP>
__device__ __forceinline__ float reduce_rows(const float (&v)[kRP], int lane, int G) {
    float b;
    int o;
    if constexpr (kRP == 4) {
        const bool hi = (lane & (G >> 1)) != 0, lo = (lane & (G >> 2)) != 0;
        float a0 = hi ? v[2] : v[0], a1 = hi ? v[3] : v[1];
        const float s0 = hi ? v[0] : v[2], s1 = hi ? v[1] : v[3];
        a0 += __shfl_xor_sync(0xFFFFFFFFu, s0, G >> 1);
        a1 += __shfl_xor_sync(0xFFFFFFFFu, s1, G >> 1);
        b = lo ? a1 : a0;
        b += __shfl_xor_sync(0xFFFFFFFFu, lo ? a0 : a1, G >> 2);
        o = G >> 3;
    } else {
        const bool hi = (lane & (G >> 1)) != 0;
        b = (hi ? v[1] : v[0]) + __shfl_xor_sync(0xFFFFFFFFu, hi ? v[0] : v[1], G >> 1);
        o = G >> 2;
    }
    for (; o > 0; o >>= 1) b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
    return b;
}

// kSwiGLU: the CTA's rows of W (gate) and then the same rows of W2 (up) form
// one list of 2·nrows virtual rows through the same ring and passes; every
// row result goes to shared memory and y[o] = silu(g[o])·u[o] at the end.
// kRP: rows a row slot takes per pass (4, or 2 where 4-row stages do not fit
// shared memory).  All kT1Cw warps compute; thread 0 issues the first
// stages, and each later stage is issued by the warp that finishes the last
// pass of the stage before it in the same slot.
template <class Fmt, int kNB, bool kSwiGLU, int kRP>
__global__ void __launch_bounds__(32 * kT1Cw, 1) gemv_t1_kernel(T1Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int abort_flag;
    __shared__ __align__(8) uint64_t x_bar;

    // Row geometry: compile-time when kNB > 0.
    const int nb = kNB > 0 ? kNB : p.nb;
    const int K = nb * kQ4kValues;
    const int nslabs = 4 * nb;                     // 64-value slabs per row
    const uint32_t row_bytes = (uint32_t)nb * Fmt::kGroupBytes;
    const int L = 4 * nb;                          // slab lanes per row
    const bool wide = L > 32;                      // a row spans several warps
    const int wc = wide ? (L + 31) / 32 : 1;       // warps per row
    int lpr = 32;                                  // lanes per row slot
    if (!wide) {
        lpr = 4;
        while (lpr < L) lpr <<= 1;
    }
    const int rpp = wide ? 1 : 32 / lpr;           // row slots per warp
    const int pass_rows = kRP * rpp;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tokens: the planes, sums and group steps of token t follow those of
    // token t − 1, so the split indexes them by its flat position in x [T][K].
    const int T = kSwiGLU ? 1 : p.T;
    const int TK = T * K;
    const int ncw = T * wc * p.rg;
    const uint32_t slot_bytes = p.slot_bytes;
    uint8_t *planes = smem;                                           // T·nslabs slabs
    float *u32 = reinterpret_cast<float *>(planes + T * nslabs * kPlaneSlabBytes);  // T·K/32 steps
    float *sx32 = u32 + TK / 32;                                      // T·K/32 group sums (kSums)
    float *xst = sx32 + (Fmt::kSums ? TK / 32 : 0);                   // x (when staged)
    uint8_t *ring = reinterpret_cast<uint8_t *>(xst + (p.x_staged ? TK : 0));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(ring + (size_t)p.nslots * slot_bytes);
    int *done = reinterpret_cast<int *>(full_bar + p.nslots);        // passes finished in each slot's stage
    int *holds = done + p.nslots;                                     // stage last issued into each slot
    float *part = reinterpret_cast<float *>(holds + p.nslots);        // [T][virtual rows][wc]

    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int nv = kSwiGLU ? 2 * nrows : nrows;  // rows streamed through the ring
    const bool to_smem = wide || kSwiGLU;        // row results go to part[]
    const int nstages = (nv + p.stage_rows - 1) / p.stage_rows;
    const int passes_per_stage = p.stage_rows / pass_rows;
    // Every pass of a full stage is worked by the wc warps of a row, per token.
    const int slot_passes = passes_per_stage * wc * T;

    // Bulk copies need a 16-byte aligned destination; never issue one otherwise.
    if (smem_addr(smem) & 15) {
        if (threadIdx.x == 0) flag_timeout(p.status);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full_bar[s], 1);
            done[s] = 0;
            holds[s] = -1;
        }
        mbar_init(&x_bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // Stage st into ring slot `slot` (one thread).  Weights are read once:
    // streamed with evict_first so that they do not displace activations and
    // outputs from L2.
    auto issue = [&](int st, int slot) {
        const uint64_t wpol = p.l2_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
        const int v0 = st * p.stage_rows, v1 = min(v0 + p.stage_rows, nv);
        uint8_t *dst = ring + (size_t)slot * slot_bytes;
        // (A test may ask for one stage never to arrive, to see a wait run
        // out; nothing then writes into the slot.)
        if (st == p.withhold) return;
        *reinterpret_cast<volatile int *>(&holds[slot]) = st;
        // Gate (or only) rows [v0, min(v1, nrows)), then up rows.
        const int g1 = kSwiGLU ? min(v1, nrows) : v1;
        if (g1 > v0) {
            // The stage's bytes start `mis` bytes into the slot: the copy
            // starts at the 16-byte boundary below them (W is 16-byte
            // aligned, so that is still inside W) and its last bytes off the
            // 16-byte grid go by plain loads, ahead of the arrive that
            // publishes the stage, so nothing past the rows is read.
            const uint8_t *src = p.W + (size_t)(row0 + v0) * row_bytes;
            const uint32_t mis = (uint32_t)(((size_t)(row0 + v0) * row_bytes) & 15);
            const uint32_t total = mis + (uint32_t)(g1 - v0) * row_bytes;
            const uint32_t bulk = total & ~15u;
            for (uint32_t i = bulk; i < total; ++i) dst[i] = __ldg(src - mis + i);
            mbar_arrive_expect_tx(&full_bar[slot], bulk + (uint32_t)(v1 - g1) * row_bytes);
            if (bulk) bulk_g2s_hint(dst, src - mis, bulk, &full_bar[slot], wpol);
        } else {
            mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(v1 - v0) * row_bytes);
        }
        if (kSwiGLU && v1 > nrows) {
            const int u0 = max(v0, nrows);
            bulk_g2s_hint(dst + (size_t)(u0 - v0) * row_bytes, p.W2 + (size_t)(row0 + u0 - nrows) * row_bytes,
                          (uint32_t)(v1 - u0) * row_bytes, &full_bar[slot], wpol);
        }
    };

    if (warp == 0) {
        // The first stages of the ring, before or after x as the geometry
        // says (x may be written by the previous kernel on the stream), one
        // lane each: a bulk copy holds its issuing thread for a few hundred
        // cycles, so one thread issuing them in turn would delay the last
        // stage by thousands.
        const int first = min(nstages, p.nslots);
        const int pre = min(first, p.pre_stages);
        if (lane < pre) issue(lane, lane);
        __syncwarp();
        if (lane == 0) {
            pdl_wait();
            if (p.x_staged) {
                mbar_arrive_expect_tx(&x_bar, (uint32_t)TK * sizeof(float));
                bulk_g2s(xst, p.x, (uint32_t)TK * sizeof(float), &x_bar);
            }
        }
        __syncwarp();
        if (lane >= pre && lane < first) issue(lane, lane);
    }

    const bool worker = warp < ncw;  // warps past ncw only help with the split
    const int cwc = worker ? warp : 0;
    const int tok = cwc / (wc * p.rg), cwt = cwc % (wc * p.rg);
    const int wcol = cwt % wc, rgi = cwt / wc;
    const int ro = wide ? 0 : lane / lpr;      // row slot of this lane
    const int s = wide ? wcol * 32 + lane : lane % lpr;
    const bool active = s < L;
    const int b = active ? (s >> 2) : 0, j = s & 3;

    // x may be produced by the previous kernel on the stream.
    pdl_wait();
    const float *xsrc = p.x;
    if (p.x_staged) {
        if (!mbar_wait_bounded(&x_bar, 0, p.wait_limit)) {
            abort_flag = 1;
            flag_timeout(p.status);
        }
        xsrc = xst;
    }
    split_x<Fmt::kSums>(xsrc, TK, threadIdx.x, kT1Cw * 32, abort_flag, planes, u32, sx32);
    __syncthreads();
    if (worker) {
        Planes pl;
        {
            // This slab's 64 plane bytes per plane: positions 64j..64j+31
            // (low nibbles) then 64j+32..64j+63 (high nibbles) of block b.
            // (Fmt::unit_of names the slab and 16-value unit of each of the
            // lane's four runs; the Q4 and ternary lanes take slab j in order.)
#pragma unroll
            for (int pp = 0; pp < kT1Planes; ++pp) {
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
        }
        Fmt::prep_planes(pl);
        // Steps and sums of block b (8 groups of 32).
        const int gb = tok * K / 32 + 8 * b;
        const typename Fmt::Lane lfmt = Fmt::lane(j, u32 + gb, sx32 + gb);

        // Rows: pass q of a stage covers rows pass_rows·q ..; this lane's row
        // slot ro takes kRP consecutive rows of it.  Rows past the stage's
        // last are computed from ring bytes of the slot (never outside it)
        // and not stored.
        const int G = wide ? 32 : lpr;
        const int ri = (lane % G) / (G / kRP);   // row of the slot this lane finishes
        // (A lane past the row's last slab adds zeros but may still hold a
        // finished row.)
        const bool writer = (lane % (G / kRP)) == 0;
        const int npasses = (nv + pass_rows - 1) / pass_rows;
        int pin = rgi, st = 0;
        while (pin >= passes_per_stage) {
            pin -= passes_per_stage;
            ++st;
        }
        int slot = st % p.nslots;
        uint32_t phase = (st / p.nslots) & 1;
        for (int pass = rgi; pass < npasses;) {
            if (abort_flag) break;
            // The slot's tag names the stage last issued into it; a stage is
            // issued only once the slot's previous stage has been consumed,
            // so once the tag names this stage the parity wait below refers
            // to it, whichever group consumed the previous one.
            if (!wait_tag(&holds[slot], st, p.wait_limit, &abort_flag) ||
                !mbar_wait_abortable(&full_bar[slot], phase, p.wait_limit, &abort_flag)) {
                abort_flag = 1;
                flag_timeout(p.status);
                break;
            }
            // Rows of a width off the 16-byte grid start `mis` bytes into
            // their slot (see issue()).
            const uint32_t mis = (uint32_t)(((size_t)(row0 + st * p.stage_rows) * row_bytes) & 15);
            const uint8_t *stage_base = ring + (size_t)slot * slot_bytes + mis + b * Fmt::kGroupBytes;
            const int rows = min(p.stage_rows, nv - st * p.stage_rows);
            int finished = 0;  // passes of this warp in this stage
            // Every pass of this group in this stage.
            do {
                const int r0 = pin * pass_rows + kRP * ro;
                const uint8_t *rp = stage_base + r0 * row_bytes;
                float v[kRP];
#pragma unroll
                for (int i = 0; i < kRP; ++i) v[i] = Fmt::row(rp + i * row_bytes, lfmt, pl);
                if (!active) {
#pragma unroll
                    for (int i = 0; i < kRP; ++i) v[i] = 0.f;
                }
                const float sum = reduce_rows<kRP>(v, lane, G);
                const int r = r0 + ri;
                if (writer && r < rows) {
                    const int rl = st * p.stage_rows + r;
                    if (wide) {
                        part[(tok * nv + rl) * wc + wcol] = sum;
                    } else if (kSwiGLU) {
                        part[rl] = sum;
                    } else {
                        p.y[(size_t)tok * p.N + row0 + rl] = p.out_scale * sum;
                    }
                }
                ++finished;
                pass += p.rg;
                pin += p.rg;
            } while (pin < passes_per_stage && pass < npasses);
            // Release the slot: the warp whose passes complete the stage's
            // count issues the stage nslots further on into it.  Every lane's
            // reads of the slot come before lane 0's release (warp barrier,
            // CTA-scope fence), the count's last increment reads them all
            // (acquire fence), and the proxy fence orders them before the
            // bulk copy's writes.
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&done[slot], finished) + finished == slot_passes) {
                    done[slot] = 0;
                    __threadfence_block();
                    const int nxt = st + p.nslots;
                    if (nxt < nstages && !abort_flag) {
                        fence_async_proxy();
                        issue(nxt, slot);
                    }
                }
            }
            while (pin >= passes_per_stage) {
                pin -= passes_per_stage;
                ++st;
                if (++slot == p.nslots) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
        }
    }

    if (to_smem) {
        __syncthreads();
        for (int it = threadIdx.x; it < T * nrows; it += kT1Cw * 32) {
            const int t = it / nrows, i = it % nrows;
            const float *pt = part + (size_t)t * nv * wc;
            float acc = 0.f;
            for (int w = 0; w < wc; ++w) acc += pt[i * wc + w];
            if (kSwiGLU) {
                float upv = 0.f;
                for (int w = 0; w < wc; ++w) upv += pt[(nrows + i) * wc + w];
                acc = acc / (1.0f + expf(-acc)) * upv;  // silu(g)·u
            }
            p.y[(size_t)t * p.N + row0 + i] = p.out_scale * acc;
        }
    }

    // Never leave a bulk copy writing into shared memory of an exiting CTA:
    // after a time-out, wait (bounded) for the last stage issued into each
    // slot (the earlier ones were consumed, so they had landed) and for x.
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) {
        for (int sl = 0; sl < p.nslots; ++sl)
            if (holds[sl] >= 0)
                (void)mbar_wait_bounded(&full_bar[sl], (holds[sl] / p.nslots) & 1, p.wait_limit);
        if (p.x_staged) (void)mbar_wait_bounded(&x_bar, 0, p.wait_limit);
    }
}

}  // namespace

template <class Fmt, bool kSwiGLU = false>
cudaError_t launch_gemv_t1(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N,
                           const uint8_t *W2 = nullptr, float out_scale = 1.0f, int T = 1) {
    const T1Tuning tun;
    const T1Geometry g =
        plan_gemv_t1(Fmt::kGroupBytes, Fmt::kSums ? 1 : 0, K, N, T, kSwiGLU ? 2 : 1, c.num_sms, c.max_smem_optin,
                     tun);
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
    p.slot_bytes = (int)g.slot_bytes;
    p.nslots = g.nslots;
    p.pre_stages = g.pre_stages;
    p.x_staged = g.x_staged;
    p.l2_evict_first = tun.l2_evict_first;
    p.wait_limit = c.wait_limit;
    p.withhold = c.withhold;
    const int grid = g.grid;
    const size_t smem = g.smem;

    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e = ensure_smem(kernel, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(c, kernel, dim3(grid), dim3(32 * kT1Cw), smem, p);
    };
    // Blocks-per-row specialisations for common widths (4-row passes); the
    // general width (kNB = 0) also takes 2-row passes.
    auto pick = [&](auto nbc) -> cudaError_t {
        constexpr int kNB = decltype(nbc)::value;
        if (g.slot_rows == kT1SlotRows) return go(gemv_t1_kernel<Fmt, kNB, kSwiGLU, kT1SlotRows>);
        if constexpr (kNB == 0) return go(gemv_t1_kernel<Fmt, 0, kSwiGLU, kT1SlotRowsWide>);
        return cudaErrorNotSupported;
    };
    using I0 = std::integral_constant<int, 0>;
    if (g.slot_rows != kT1SlotRows) return pick(I0{});
    if constexpr (kSwiGLU) {
        return pick(I0{});
    } else if constexpr (std::is_same<Fmt, FmtQ6K>::value) {
        return p.nb == 16 ? pick(std::integral_constant<int, 16>{}) : pick(I0{});
    } else if constexpr (std::is_same<Fmt, FmtTern>::value) {
        return p.nb == 10 ? pick(std::integral_constant<int, 10>{}) : pick(I0{});
    } else if constexpr (std::is_same<Fmt, FmtQ4K>::value) {
        switch (p.nb) {
            case 4: return pick(std::integral_constant<int, 4>{});
            case 16: return pick(std::integral_constant<int, 16>{});
            case 43: return pick(std::integral_constant<int, 43>{});
            default: return pick(I0{});
        }
    } else {
        return p.nb == 16 ? pick(std::integral_constant<int, 16>{}) : pick(I0{});
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
