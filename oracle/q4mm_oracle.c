/*
 * Plain CPU oracle for the two quantized x·Wᵀ products.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the tests, the smoke check and the benchmark's CPU-baseline / reference arm
 * may load it.  It shares no code, header, table or constant with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Everything is written from the definitions on the pages, slowly and in
 * double precision:
 *
 *  - Q4_K super-block (SKaiNET PR #562 "SIMD-fused Q4_K matmul kernel +
 *    Q4KMatmulKernel SPI", section "Pipeline": canonical ggml strided layout,
 *    sub-block 2j in the low nibbles and 2j+1 in the high nibbles of the same
 *    32 bytes; the per-value formula w = d·sc·q − dmin·m and the lazy-dmin
 *    identity acc += scale·codeSum − offset·inputSum).  Block bytes: fp16 d,
 *    fp16 dmin, 12 bytes of packed 6-bit scales and mins, 128 bytes of qs.
 *    The 6-bit packing is not printed on the pages; the oracle uses the ggml
 *    canonical packing that the page says the gold reference was validated
 *    against (section "Test plan").
 *  - Dequantize-then-matmul shape of the oracle: the same PR, section
 *    "Benchmark numbers" (scalar dequant-then-matmul baseline) and "Test plan"
 *    (gold reference).
 *  - BitNet b1.58 ternary payload (SKaiNET issue #1138 "[ternary-f32] Phase 2:
 *    TernaryF32GemvNative SPI …", section "Tasks": gemvPacked computes
 *    out[o] = Σ_k in[k]·code(o,k) with the scale NOT applied, inputDim % 4 == 0,
 *    code = ((byte >> 2·(i%4)) & 3) − 1, fp32 accumulate, then one multiply by
 *    the BitNet scale; prefill loops rows advancing by r·k and r·n).
 *  - Q4_0, the 32-value / 18-byte block named as the follow-up in the same
 *    PR (section "Out of scope"); layout read as ggml's (see its section).
 *  - Q6_K, the other follow-up of that section; layout read as ggml's.
 *  - x·Wᵀ with W stored [out, in] and used in place (SKaiNET docs "Eager
 *    execution: backends and kernels", the paragraph on the dense x·Wᵀ row).
 *
 * Layouts: x is [T][K] fp32 row-major, W is N rows of K/256 blocks of 144
 * bytes (Q4_K) or N rows of K/4 bytes (ternary), y is [T][N].
 *
 * Parallelism: the timed entry points split independent output rows across
 * OpenMP threads.  No sum is blocked, fused or reordered: every output is one
 * sequential loop over k with a double accumulator.  Build without
 * -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define Q4K_VALUES 256
#define Q4K_BYTES 144

/* IEEE 754 binary16 (little-endian bit pattern) to double, exactly.
 * Subnormals are honoured; Inf/NaN map to Inf/NaN. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 31;
    int mantissa = h & 1023;
    double v;
    if (exponent == 0)
        v = ldexp((double)mantissa, -24);              /* 0.m × 2^-14 */
    else if (exponent == 31)
        v = mantissa ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mantissa), exponent - 25); /* 1.m × 2^(e-15) */
    return sign ? -v : v;
}

/* Round a float to bfloat16 (round to nearest, ties to even) and return it
 * as a float.  Finite inputs only. */
float oracle_round_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
    memcpy(&f, &u, 4);
    return f;
}

/* 6-bit scale and min of sub-block s (0..7) from the 12 packed bytes. */
static void q4k_scale_min(const uint8_t *packed, int s, int *sc, int *m)
{
    if (s < 4) {
        *sc = packed[s] & 63;
        *m = packed[s + 4] & 63;
    } else {
        *sc = (packed[s + 4] & 15) | ((packed[s - 4] >> 6) << 4);
        *m = (packed[s + 4] >> 4) | ((packed[s] >> 6) << 4);
    }
}

/* 4-bit code of element e (0..255) of a block: slab j = e/64 holds elements
 * 64j..64j+31 in the low nibbles and 64j+32..64j+63 in the high nibbles of
 * the same 32 bytes qs[32j .. 32j+31]. */
static int q4k_code(const uint8_t *qs, int e)
{
    int j = e / 64, l = e % 64;
    if (l < 32)
        return qs[32 * j + l] & 15;
    return qs[32 * j + (l - 32)] >> 4;
}

static double q4k_d(const uint8_t *blk)
{
    return oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
}

static double q4k_dmin(const uint8_t *blk)
{
    return oracle_fp16_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
}

/* Dequantize one 144-byte block: w[e] = d·sc_s·q_e − dmin·m_s with s = e/32,
 * evaluated exactly in double (every term has at most 21 significant bits)
 * and rounded once to float. */
void oracle_q4k_dequant_block(const uint8_t *blk, float w[Q4K_VALUES])
{
    double d = q4k_d(blk), dmin = q4k_dmin(blk);
    const uint8_t *packed = blk + 4, *qs = blk + 16;
    for (int e = 0; e < Q4K_VALUES; ++e) {
        int sc, m;
        q4k_scale_min(packed, e / 32, &sc, &m);
        w[e] = (float)(d * sc * q4k_code(qs, e) - dmin * m);
    }
}

/*
 * One-time relayout of a Q4_K weight for the tensor-core prefill (SKaiNET
 * docs "Eager execution: backends and kernels", the paragraph on weights
 * relayouted once when they are registered rather than on every call).  The
 * page does not fix a target layout; this one is the library's own: every
 * 64-value slab j of a block (the 32 bytes qs[32j..32j+31], sub-blocks 2j and
 * 2j+1) becomes a 48-byte chunk
 *     fp32 d·sc(2j), fp32 dmin·m(2j), fp32 d·sc(2j+1), fp32 dmin·m(2j+1),
 *     the 32 code bytes unchanged,
 * and the chunks are stored tile-major: the rows form tiles of 256 (the last
 * one padded with zero rows), and chunk c (values 64c..64c+63) of the 256
 * rows of tile t is one contiguous run of 256·48 bytes at
 *     ((t·(K/64) + c)·256 + row mod 256)·48.
 * Each product has at most 17 significant bits and lies within fp32's normal
 * range, so it is exact in fp32 and the relayouted weight dequantizes to the
 * same fp32 matrix.  The layout keeps products, not factors: d and sc (and
 * dmin and m) cannot be recovered separately, so the inverse is defined on
 * the matrix (oracle_q4k_tc_dequant), not on the bytes of the scale field.
 * Floats are stored little-endian.
 */
#define Q4K_TC_CHUNK_BYTES 48
#define Q4K_TC_TILE_ROWS 256

static void put_f32(uint8_t *dst, double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    dst[0] = (uint8_t)u;
    dst[1] = (uint8_t)(u >> 8);
    dst[2] = (uint8_t)(u >> 16);
    dst[3] = (uint8_t)(u >> 24);
}

static double get_f32(const uint8_t *src)
{
    uint32_t u = (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) |
                 ((uint32_t)src[3] << 24);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Bytes of the relayouted weight: the rows rounded up to whole tiles. */
int64_t oracle_q4k_tc_bytes(int64_t K, int64_t N)
{
    if (K <= 0 || N <= 0 || K % Q4K_VALUES)
        return -1;
    int64_t tiles = (N + Q4K_TC_TILE_ROWS - 1) / Q4K_TC_TILE_ROWS;
    return tiles * Q4K_TC_TILE_ROWS * (K / 64) * Q4K_TC_CHUNK_BYTES;
}

/* Offset of chunk c of row o. */
static int64_t tc_chunk_offset(int64_t K, int64_t o, int64_t c)
{
    int64_t t = o / Q4K_TC_TILE_ROWS, r = o % Q4K_TC_TILE_ROWS;
    return ((t * (K / 64) + c) * Q4K_TC_TILE_ROWS + r) * Q4K_TC_CHUNK_BYTES;
}

/* W [N][K/256 blocks of 144 B] → R (oracle_q4k_tc_bytes(K, N) bytes).
 * Returns 0, or -1 on bad sizes. */
int oracle_q4k_tc_relayout(const uint8_t *W, int64_t K, int64_t N, uint8_t *R)
{
    int64_t total = oracle_q4k_tc_bytes(K, N);
    if (total < 0)
        return -1;
    memset(R, 0, (size_t)total);
    int64_t nb = K / Q4K_VALUES;
    for (int64_t o = 0; o < N; ++o) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = W + (o * nb + b) * Q4K_BYTES;
            double d = q4k_d(blk), dmin = q4k_dmin(blk);
            for (int j = 0; j < 4; ++j) {
                uint8_t *ch = R + tc_chunk_offset(K, o, 4 * b + j);
                for (int h = 0; h < 2; ++h) {
                    int sc, m;
                    q4k_scale_min(blk + 4, 2 * j + h, &sc, &m);
                    put_f32(ch + 8 * h, d * sc);
                    put_f32(ch + 8 * h + 4, dmin * m);
                }
                memcpy(ch + 16, blk + 16 + 32 * j, 32);
            }
        }
    }
    return 0;
}

/* R → out [N][K] fp32: value i < 32 of chunk c is s_lo·(qs[i] & 15) − o_lo,
 * value 32 + i is s_hi·(qs[i] >> 4) − o_hi, evaluated in double and rounded
 * once to float.  Returns 0, or -1 on bad sizes. */
int oracle_q4k_tc_dequant(const uint8_t *R, int64_t K, int64_t N, float *out)
{
    if (oracle_q4k_tc_bytes(K, N) < 0)
        return -1;
    int64_t nc = K / 64;
    for (int64_t o = 0; o < N; ++o) {
        for (int64_t c = 0; c < nc; ++c) {
            const uint8_t *ch = R + tc_chunk_offset(K, o, c);
            double s_lo = get_f32(ch), o_lo = get_f32(ch + 4);
            double s_hi = get_f32(ch + 8), o_hi = get_f32(ch + 12);
            float *w = out + o * K + c * 64;
            for (int i = 0; i < 32; ++i) {
                w[i] = (float)(s_lo * (ch[16 + i] & 15) - o_lo);
                w[32 + i] = (float)(s_hi * (ch[16 + i] >> 4) - o_hi);
            }
        }
    }
    return 0;
}

/* W [N][K/256 blocks] → out [N][K] fp32. Returns 0, or -1 on bad sizes. */
int oracle_q4k_dequant(const uint8_t *W, int64_t K, int64_t N, float *out)
{
    if (K <= 0 || N <= 0 || K % Q4K_VALUES)
        return -1;
    int64_t nb = K / Q4K_VALUES;
    for (int64_t o = 0; o < N; ++o)
        for (int64_t b = 0; b < nb; ++b)
            oracle_q4k_dequant_block(W + (o * nb + b) * Q4K_BYTES, out + o * K + b * Q4K_VALUES);
    return 0;
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* y[t][o] = Σ_k x[t][k]·w[o][k] with w the fp32 dequantized weight, summed
 * sequentially in k with a double accumulator.  bf16 != 0 first rounds both
 * x and w to bfloat16 (the operand precision of the tensor-core path). */
static int q4k_matmul_impl(const float *x, const uint8_t *W, int64_t K, int64_t N,
                           int64_t T, double *y, int nthreads, int bf16)
{
    if (K <= 0 || N <= 0 || T <= 0 || K % Q4K_VALUES)
        return -1;
    int64_t nb = K / Q4K_VALUES;
    int nt = set_threads(nthreads);
    int failed = 0;
#pragma omp parallel num_threads(nt)
    {
        float *w = (float *)malloc((size_t)K * sizeof(float));
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t o = 0; o < N; ++o) {
            if (!w)
                continue;
            for (int64_t b = 0; b < nb; ++b)
                oracle_q4k_dequant_block(W + (o * nb + b) * Q4K_BYTES, w + b * Q4K_VALUES);
            for (int64_t t = 0; t < T; ++t) {
                const float *xt = x + t * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    float xv = xt[k], wv = w[k];
                    if (bf16) {
                        xv = oracle_round_bf16(xv);
                        wv = oracle_round_bf16(wv);
                    }
                    acc += (double)xv * (double)wv;
                }
                y[t * N + o] = acc;
            }
        }
        free(w);
    }
    return failed ? -2 : 0;
}

int oracle_q4k_matmul(const float *x, const uint8_t *W, int64_t K, int64_t N, int64_t T,
                      double *y, int nthreads)
{
    return q4k_matmul_impl(x, W, K, N, T, y, nthreads, 0);
}

int oracle_q4k_matmul_bf16(const float *x, const uint8_t *W, int64_t K, int64_t N, int64_t T,
                           double *y, int nthreads)
{
    return q4k_matmul_impl(x, W, K, N, T, y, nthreads, 1);
}

/* Llama feed-forward input side with SwiGLU: g = x·W_gateᵀ and u = x·W_upᵀ
 * (both Q4_K, each exactly as oracle_q4k_matmul computes it), then
 * h = silu(g)·u with silu(z) = z / (1 + e^(−z)), in double.  The pages name
 * this fused operation only as the llama.cpp benchmark "ffn_swiglu" (PR #37
 * "ggml-cpu: cache-aware tiling in ggml_compute_forward_mul_mat", section
 * "Measured impact"); the formula is the standard Llama FFN.  g and u are
 * returned too when their pointers are non-NULL. */
int oracle_q4k_ffn_swiglu(const float *x, const uint8_t *Wg, const uint8_t *Wu, int64_t K, int64_t N,
                          int64_t T, double *g, double *u, double *h, int nthreads)
{
    if (K <= 0 || N <= 0 || T <= 0 || K % Q4K_VALUES)
        return -1;
    double *gg = (double *)malloc((size_t)(T * N) * sizeof(double));
    double *uu = (double *)malloc((size_t)(T * N) * sizeof(double));
    int rc = (gg && uu) ? 0 : -2;
    if (!rc)
        rc = q4k_matmul_impl(x, Wg, K, N, T, gg, nthreads, 0);
    if (!rc)
        rc = q4k_matmul_impl(x, Wu, K, N, T, uu, nthreads, 0);
    if (!rc) {
        for (int64_t i = 0; i < T * N; ++i) {
            double z = gg[i];
            h[i] = z / (1.0 + exp(-z)) * uu[i];
            if (g)
                g[i] = z;
            if (u)
                u[i] = uu[i];
        }
    }
    free(gg);
    free(uu);
    return rc;
}

/* The pages' lazy-dmin form, in double: per sub-block s of each block,
 *   acc += (d·sc_s)·Σ_e x_e·q_e − (dmin·m_s)·Σ_e x_e
 * with the "scale" d·sc_s and "offset" dmin·m_s applied once per
 * sub-block × super-block.  Mathematically equal to the direct form. */
int oracle_q4k_matmul_lazy(const float *x, const uint8_t *W, int64_t K, int64_t N, int64_t T,
                           double *y, int nthreads)
{
    if (K <= 0 || N <= 0 || T <= 0 || K % Q4K_VALUES)
        return -1;
    int64_t nb = K / Q4K_VALUES;
    int nt = set_threads(nthreads);
#pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t o = 0; o < N; ++o) {
        for (int64_t t = 0; t < T; ++t) {
            const float *xt = x + t * K;
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = W + (o * nb + b) * Q4K_BYTES;
                double d = q4k_d(blk), dmin = q4k_dmin(blk);
                for (int s = 0; s < 8; ++s) {
                    int sc, m;
                    q4k_scale_min(blk + 4, s, &sc, &m);
                    double code_sum = 0.0, input_sum = 0.0;
                    for (int l = 0; l < 32; ++l) {
                        int e = 32 * s + l;
                        double xv = xt[b * Q4K_VALUES + e];
                        code_sum += xv * q4k_code(blk + 16, e);
                        input_sum += xv;
                    }
                    acc += (d * sc) * code_sum - (dmin * m) * input_sum;
                }
            }
            y[t * N + o] = acc;
        }
    }
    return 0;
}

/* Ternary code of element i of a row: ((byte >> 2·(i%4)) & 3) − 1. The field
 * value 3 decodes to +2 by the literal formula. */
static int ternary_code(const uint8_t *row, int64_t i)
{
    return ((row[i / 4] >> (2 * (i % 4))) & 3) - 1;
}

/* dot[t][o] = Σ_k x[t][k]·code(o,k) (double, sequential in k; scale not
 * applied), y[t][o] = (float)(scale · dot) — the single round-to-nearest
 * fp32 product of the fp32 code-dot and the scale. */
int oracle_ternary_gemv(const float *x, const uint8_t *W, float scale, int64_t K, int64_t N,
                        int64_t T, double *dot, float *y, int nthreads)
{
    if (K <= 0 || N <= 0 || T <= 0 || K % 4)
        return -1;
    int64_t row_bytes = K / 4;
    int nt = set_threads(nthreads);
#pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t o = 0; o < N; ++o) {
        const uint8_t *row = W + o * row_bytes;
        for (int64_t t = 0; t < T; ++t) {
            const float *xt = x + t * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)xt[k] * ternary_code(row, k);
            if (dot)
                dot[t * N + o] = acc;
            if (y)
                y[t * N + o] = (float)((double)scale * (double)(float)acc);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Q4_0 (SKaiNET PR #562, section "Out of scope": the simpler 32-value,
 * 18-byte block that runs the same algorithm).  The page gives only the block
 * size; the byte layout is the ggml canonical one the PR builds on: fp16 d
 * (little-endian), then 16 bytes qs; element l (l < 16) is the low nibble of
 * qs[l] and element 16 + l its high nibble (the same strided pattern as the
 * Q4_K slabs), and w = d·(q − 8).  In the page's lazy form this is scale d
 * and offset 8·d per block.
 * ------------------------------------------------------------------------ */
#define Q40_VALUES 32
#define Q40_BYTES 18

static int q40_code(const uint8_t *qs, int e)
{
    return e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);
}

/* Dequantize one 18-byte block: w[e] = d·(q_e − 8), exact in double (11-bit
 * d times a 4-bit integer) and rounded once to float. */
void oracle_q4_0_dequant_block(const uint8_t *blk, float w[Q40_VALUES])
{
    double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int e = 0; e < Q40_VALUES; ++e)
        w[e] = (float)(d * (q40_code(blk + 2, e) - 8));
}

/* W [N][K/32 blocks] → out [N][K] fp32. Returns 0, or -1 on bad sizes. */
int oracle_q4_0_dequant(const uint8_t *W, int64_t K, int64_t N, float *out)
{
    if (K <= 0 || N <= 0 || K % Q40_VALUES)
        return -1;
    int64_t nb = K / Q40_VALUES;
    for (int64_t o = 0; o < N; ++o)
        for (int64_t b = 0; b < nb; ++b)
            oracle_q4_0_dequant_block(W + (o * nb + b) * Q40_BYTES, out + o * K + b * Q40_VALUES);
    return 0;
}

/* y[t][o] = Σ_k x[t][k]·w[o][k], w the fp32 dequantized Q4_0 weight, summed
 * sequentially in k with a double accumulator (dequantize-then-matmul). */
int oracle_q4_0_matmul(const float *x, const uint8_t *W, int64_t K, int64_t N, int64_t T,
                       double *y, int nthreads)
{
    if (K <= 0 || N <= 0 || T <= 0 || K % Q40_VALUES)
        return -1;
    int64_t nb = K / Q40_VALUES;
    int nt = set_threads(nthreads);
    int failed = 0;
#pragma omp parallel num_threads(nt)
    {
        float *w = (float *)malloc((size_t)K * sizeof(float));
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t o = 0; o < N; ++o) {
            if (!w)
                continue;
            for (int64_t b = 0; b < nb; ++b)
                oracle_q4_0_dequant_block(W + (o * nb + b) * Q40_BYTES, w + b * Q40_VALUES);
            for (int64_t t = 0; t < T; ++t) {
                const float *xt = x + t * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (double)xt[k] * (double)w[k];
                y[t * N + o] = acc;
            }
        }
        free(w);
    }
    return failed ? -2 : 0;
}

/* ------------------------------------------------------------------------
 * Q6_K (SKaiNET PR #562, section "Out of scope": "ql + qh with the
 * 4-codes-per-qh-byte half-interleaved layout").  The page names the parts;
 * the byte layout is ggml's: 256 values in 210 bytes, ql[128] (low 4 bits),
 * qh[64] (high 2 bits), 16 signed 8-bit sub-block scales, fp16 d (little-
 * endian) last.  Half n (values 128n..128n+127) uses ql[64n..64n+63],
 * qh[32n..32n+31] and scales[8n..8n+7]; for l < 32 and group g (0..3), value
 * 128n + 32g + l takes the low nibble of ql[64n + l] (g = 0), of
 * ql[64n + 32 + l] (g = 1), the high nibble of ql[64n + l] (g = 2), of
 * ql[64n + 32 + l] (g = 3), plus bits 2g..2g+1 of qh[32n + l] as bits 4..5;
 * its sub-block is 8n + 2g + l/16 and w = d·scale·(q − 32).
 * ------------------------------------------------------------------------ */
#define Q6K_VALUES 256
#define Q6K_BYTES 210

static int q6k_code(const uint8_t *blk, int v)
{
    int n = v / 128, g = (v % 128) / 32, l = v % 32;
    const uint8_t *ql = blk + 64 * n, *qh = blk + 128 + 32 * n;
    int lo = (g & 1) ? ql[32 + l] : ql[l];
    lo = (g & 2) ? (lo >> 4) : (lo & 15);
    int hi = (qh[l] >> (2 * g)) & 3;
    return lo | (hi << 4);
}

/* Dequantize one 210-byte block: w[v] = d·scale_s·(q_v − 32), exact in double
 * (11-bit d × 8-bit scale × 6-bit code) and rounded once to float. */
void oracle_q6k_dequant_block(const uint8_t *blk, float w[Q6K_VALUES])
{
    double d = oracle_fp16_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
    const int8_t *sc = (const int8_t *)(blk + 192);
    for (int v = 0; v < Q6K_VALUES; ++v) {
        int n = v / 128, g = (v % 128) / 32, l = v % 32;
        int s = 8 * n + 2 * g + l / 16;
        w[v] = (float)(d * sc[s] * (q6k_code(blk, v) - 32));
    }
}

int oracle_q6k_dequant(const uint8_t *W, int64_t K, int64_t N, float *out)
{
    if (K <= 0 || N <= 0 || K % Q6K_VALUES)
        return -1;
    int64_t nb = K / Q6K_VALUES;
    for (int64_t o = 0; o < N; ++o)
        for (int64_t b = 0; b < nb; ++b)
            oracle_q6k_dequant_block(W + (o * nb + b) * Q6K_BYTES, out + o * K + b * Q6K_VALUES);
    return 0;
}

/* y[t][o] = Σ_k x[t][k]·w[o][k], w the fp32 dequantized Q6_K weight, summed
 * sequentially in k with a double accumulator. */
int oracle_q6k_matmul(const float *x, const uint8_t *W, int64_t K, int64_t N, int64_t T, double *y,
                      int nthreads)
{
    if (K <= 0 || N <= 0 || T <= 0 || K % Q6K_VALUES)
        return -1;
    int64_t nb = K / Q6K_VALUES;
    int nt = set_threads(nthreads);
    int failed = 0;
#pragma omp parallel num_threads(nt)
    {
        float *w = (float *)malloc((size_t)K * sizeof(float));
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t o = 0; o < N; ++o) {
            if (!w)
                continue;
            for (int64_t b = 0; b < nb; ++b)
                oracle_q6k_dequant_block(W + (o * nb + b) * Q6K_BYTES, w + b * Q6K_VALUES);
            for (int64_t t = 0; t < T; ++t) {
                const float *xt = x + t * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (double)xt[k] * (double)w[k];
                y[t * N + o] = acc;
            }
        }
        free(w);
    }
    return failed ? -2 : 0;
}

/* Encoders, used only to build hand-worked fixtures in the tests. */

/* Pack one Q6_K block from d's fp16 bits, 16 scales (−128..127) and 256 codes
 * (0..63), inverse of the unpacking above. */
void oracle_q6k_pack_block(uint16_t d_bits, const int sc[16], const int q[Q6K_VALUES],
                           uint8_t out[Q6K_BYTES])
{
    memset(out, 0, Q6K_BYTES);
    for (int v = 0; v < Q6K_VALUES; ++v) {
        int n = v / 128, g = (v % 128) / 32, l = v % 32;
        int lo = q[v] & 15, hi = (q[v] >> 4) & 3;
        uint8_t *ql = out + 64 * n + ((g & 1) ? 32 : 0) + l;
        *ql |= (uint8_t)((g & 2) ? (lo << 4) : lo);
        out[128 + 32 * n + l] |= (uint8_t)(hi << (2 * g));
    }
    for (int s = 0; s < 16; ++s)
        out[192 + s] = (uint8_t)(int8_t)sc[s];
    out[208] = d_bits & 255;
    out[209] = d_bits >> 8;
}

/* Pack one Q4_0 block from d's fp16 bits and 32 codes (0..15). */
void oracle_q4_0_pack_block(uint16_t d_bits, const int q[Q40_VALUES], uint8_t out[Q40_BYTES])
{
    out[0] = d_bits & 255;
    out[1] = d_bits >> 8;
    for (int l = 0; l < 16; ++l)
        out[2 + l] = (uint8_t)((q[l] & 15) | ((q[16 + l] & 15) << 4));
}

/* Pack one Q4_K block from its parts (inverse of the unpacking above). */
void oracle_q4k_pack_block(uint16_t d_bits, uint16_t dmin_bits, const int sc[8], const int m[8],
                           const int q[Q4K_VALUES], uint8_t out[Q4K_BYTES])
{
    memset(out, 0, Q4K_BYTES);
    out[0] = d_bits & 255;
    out[1] = d_bits >> 8;
    out[2] = dmin_bits & 255;
    out[3] = dmin_bits >> 8;
    uint8_t *packed = out + 4, *qs = out + 16;
    for (int s = 0; s < 4; ++s) {
        packed[s] = (uint8_t)((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
        packed[s + 4] = (uint8_t)((m[s] & 63) | ((m[s + 4] >> 4) << 6));
        packed[s + 8] = (uint8_t)((sc[s + 4] & 15) | ((m[s + 4] & 15) << 4));
    }
    for (int j = 0; j < 4; ++j)
        for (int l = 0; l < 32; ++l)
            qs[32 * j + l] = (uint8_t)((q[64 * j + l] & 15) | ((q[64 * j + 32 + l] & 15) << 4));
}

/* Pack ternary codes (each −1, 0 or +1) four to a byte, element i in bits
 * 2·(i%4) of byte i/4.  n % 4 == 0. */
void oracle_ternary_pack(const int *codes, int64_t n, uint8_t *out)
{
    for (int64_t b = 0; b < n / 4; ++b) {
        int v = 0;
        for (int i = 0; i < 4; ++i)
            v |= ((codes[4 * b + i] + 1) & 3) << (2 * i);
        out[b] = (uint8_t)v;
    }
}

int oracle_max_threads(void)
{
    return set_threads(0);
}
