// Q4_K prefill on the tcgen05 tensor cores: bf16 operands, fp32 accumulation
// in tensor memory (sm_103a).
//
// y[t][o] = Σ_k x[t][k]·w[o][k] with w = d·sc_s·q − dmin·m_s (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline"), evaluated as D[o][t] = A[o][k]·B[t][k] with
//   A = the dequantized weights rounded to bf16, M = 128 weight rows per
//       MMA, held in TENSOR MEMORY: the dequant warps write each chunk of A
//       there with tcgen05.st, so the dequantized operand never passes
//       through shared memory,
//   B = the activations rounded to bf16 (N = the tile's tokens rounded up to
//       16, at most 128), K-major in shared memory with the 128-byte swizzle,
//   D = fp32 in tensor memory, one 128 × N accumulator per 128 weight rows.
// Putting the tokens on N sizes every MMA to the tile: 64 tokens run
// 128 × 64 × 16 instructions (measured on GB300: 46 cycles each, 70% of the
// tensor pipe's rate; N = 128 and 256 run at the full rate), with no padded
// token rows.
//
// Weights stream through a ring of chunk stages (256 rows × 64 values of K,
// 12 KB): in the canonical 144-byte Q4_K layout a stage is two 2-D tensor
// copies (the 16-byte header of every row's block and the 32 code bytes of
// the chunk's slab: 256 short pieces, one per row); in the relayouted
// tensor-core layout (48 bytes per row and chunk: fp32 d·sc and dmin·m of
// the slab's two sub-blocks, then its 32 code bytes; tile-major, so that a
// chunk of a 256-row tile is one 12 KB run) it is one plain bulk copy of
// contiguous bytes, a CTA's whole weight range is one run in memory, and
// the scales arrive already decoded.
//
// Up to 128 tokens (one tile) the dequant warps also read fp32 x, round it
// to bf16 and write each chunk's activation tile in the swizzled layout the
// MMA reads, one chunk ahead of use; nothing is allocated.  Above 128 tokens
// a small kernel first rounds x to bf16 once into a stream-ordered scratch
// buffer (2·T·K bytes, allocated and freed on the call's stream), and each
// 128-token tile loads its activation tiles from it by TMA with the hardware
// 128-byte swizzle.
//
// Grid: clusters of S CTAs (3, or 4 above K = 49152) per 256-row tile, CTA
// rank r of a cluster taking 64-value chunks [r·nc/S, (r+1)·nc/S) of K, so
// that the 43 row tiles of an 11008-row weight spread over 129 SMs.  Each
// CTA accumulates its K range in tensor memory (at most 16384 values of K,
// within which the tensor core's fp32 accumulation stays far inside the
// stated tolerance).  Rank s of a cluster owns the tile's rows
// [floor(256·s/S), floor(256·(s+1)/S)): every rank writes its accumulators to
// a row-major shared tile, one thread sends each other rank the rows it owns
// with one shared-to-cluster bulk copy, and each rank adds the S partial sums
// of its rows in rank order from local shared memory and writes y, so the
// result does not depend on scheduling and no partial sum goes through
// global memory.
//
// Tensor memory (512 columns, one CTA per SM): D of row half m at columns
// c_D·m .. c_D·m + N, with c_D = 64 up to 64 tokens and 128 above; A of
// operand stage s, row half m at 2·c_D + 64·s + 32·m (32 columns: 64 bf16
// values of K per lane, two per column, lower K in the low half).  The
// operand ring is as deep as the remaining columns allow: 6 stages up to 64
// tokens, 4 above.  A stage is released when its MMAs complete, so the ring
// must cover the MMAs' completion latency as well as the dequantization of
// the next chunks.
//
// Roles in a CTA:
//  * warp 16 (one thread) issues the weight chunk copies, before the wait on
//    the previous kernel, and (from the bf16 copy) the activation tiles after
//    it, each as soon as its ring slot is free.
//  * warps 0–15 dequantize: warp w serves tensor-memory lane quarter w mod 4
//    of row half (w / 4) mod 2, and the chunks c ≡ w / 8 (mod 2); each thread
//    turns the 32 code bytes of its row's chunk into 64 bf16 values: each
//    nibble becomes a float with one logic op (2^23 + q·2^p), one paired FMA
//    with the scale at 2^-p and −scale·2^(23−p) gives scale·q exactly, one
//    paired add removes the min term (the single rounding of the fp32
//    dequantization), and one conversion packs two bf16.  With fused
//    activations the same threads also write the chunk's activation tile.
//  * warp 17 allocates tensor memory; the first threads of warps 17 and 18
//    issue the chunk's MMAs of row half 0 and 1 (four K steps of 16 each)
//    and commit them to the chunk's ring stage.  An MMA instruction is
//    accepted only about as fast as the tensor pipe runs it (measured on
//    GB300), so whatever one issuer does between chunks leaves the pipe idle
//    unless the other issuer fills that time.
//  * warps 0–15 then read the accumulators (tcgen05.ld) into the shared
//    tile, and every thread takes part in the local sum.
// All mbarrier waits are bounded; a time-out sets the device status word and
// every thread still reaches the cluster barriers of every epilogue pass.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>
#include <utility>

#include "q4mm.h"
#include "cluster.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace q4mm {

namespace {

constexpr int kTcRows = 256;                       // weight rows per CTA: two MMAs of M = 128
constexpr int kTcM = 128;                          // MMA M: weight rows of one tensor-memory accumulator
constexpr int kTcTok = 128;                        // token rows per tile (MMA N at most)
constexpr int kTcKc = 64;                          // K per chunk: a 128-byte row of bf16
constexpr int kTcDqWarps = 16;                     // dequant + epilogue warps
constexpr int kTcWarpTma = kTcDqWarps;             // TMA producer warp
constexpr int kTcWarpMma = kTcDqWarps + 1;         // MMA issuer warps: kTcWarpMma + m for row half m
constexpr int kTcThreads = 32 * (kTcDqWarps + 3);
constexpr int kTcGroupWarps = kTcDqWarps / 2;      // warps per chunk (alternate chunks per group)
constexpr int kTcWStages = 8;                      // weight chunk stages in flight
constexpr int kTcStagesMax = 6;                    // operand stages (A in tensor memory, B in shared memory):
                                                   // 6 up to 64 tokens, 4 above (tensor-memory columns)
constexpr int kTcChunkBytes = 48;                  // relayouted bytes per row and chunk
constexpr uint32_t kTcWStageBytes = kTcRows * kTcChunkBytes;  // 12288: both layouts
constexpr uint32_t kTcXTileBytes = kTcTok * 128;              // 16384: the largest activation tile
constexpr uint32_t kTcXRegion = 4 * kTcXTileBytes;            // 4 tiles of 128 tokens or 6 of 64
constexpr int kTcMaxKPerCta = 16384;               // one accumulator per CTA
constexpr uint32_t kTcTmemCols = 512;              // the whole of tensor memory

struct TcLayout {
    static constexpr uint32_t off_x = 0;
    static constexpr uint32_t off_w = off_x + kTcXRegion;
    static constexpr uint32_t off_bar = off_w + kTcWStages * kTcWStageBytes;
    static constexpr uint32_t n_bars = 2 * kTcWStages + 3 * kTcStagesMax + 2;
    static constexpr uint32_t off_misc = off_bar + 8 * n_bars;
    static constexpr uint32_t total = off_misc + 16;
    static_assert(off_w % 1024 == 0, "activation tiles must be 1024-byte aligned");
    // The epilogue's tiles (own: 256 rows x 72 token slots; receive: S - 1
    // slots of at most 86 rows, S = 3, or 64 rows, S = 4, x 68) reuse the rings.
    static_assert((kTcRows * 72 + 2 * 86 * 68) * 4 <= off_bar && (kTcRows * 72 + 3 * 64 * 68) * 4 <= off_bar,
                  "epilogue tiles must fit the rings");
};

// Tokens per launch tile: the token rows of one MMA.
constexpr int kTcMaxTokens = kTcTok;

// tcgen05 shared-memory matrix descriptor for a K-major operand in the
// 128-byte swizzle layout: rows of 128 bytes, 8-row atoms 1024 bytes apart,
// the 16-byte chunk c of row r stored at chunk c ^ (r % 8).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                          // leading byte offset (unused here): 16 B
    d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: 8 rows × 128 B
    d |= (uint64_t)1u << 46;                          // descriptor version for tcgen05
    d |= (uint64_t)2u << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major,
// M = 128, N = n (a multiple of 16, 16..256).
__device__ __forceinline__ uint32_t mma_idesc_m128(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Bulk copy from this CTA's shared memory to another CTA's of the cluster
// (cluster addresses dst and bar), completing on that CTA's barrier.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// D (tensor memory) (+)= A·Bᵀ with A read from tensor memory at column
// address a_tmem and B from shared memory through its descriptor.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Sixteen 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 2^23 + (w & mask) as a float: the masked nibble sits in the mantissa.
__device__ __forceinline__ float magic(uint32_t w, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, 0x4B000000, 0xEA;" : "=r"(r) : "r"(w), "r"(mask));  // (a & b) | c
    return __uint_as_float(r);
}

// Per sub-block constants: for a nibble at bit p of its word, built as
// f = 2^23 + q·2^p, fma(s·2^-p, f, −s·2^(23−p)) = s·q exactly, then − o.
struct NibScale {
    float2 s01, c01, s23, c23, no;
};

// Low nibbles: bytes 0,1 at bits 0 and 8; bytes 2,3 at bit 16 (byte 3 after
// a shift by 8).  High nibbles: bytes 0,1 at bits 4 and 12; bytes 2,3 at bit
// 12 (after shifts by 8 and 16).
__device__ __forceinline__ NibScale nib_scale_lo(float s, float o) {
    NibScale r;
    r.s01 = make_float2(s, s * 0x1p-8f);
    r.c01 = make_float2(s * -0x1p23f, s * -0x1p15f);
    r.s23 = make_float2(s * 0x1p-16f, s * 0x1p-16f);
    r.c23 = make_float2(s * -0x1p7f, s * -0x1p7f);
    r.no = make_float2(-o, -o);
    return r;
}
__device__ __forceinline__ NibScale nib_scale_hi(float s, float o) {
    NibScale r;
    r.s01 = make_float2(s * 0x1p-4f, s * 0x1p-12f);
    r.c01 = make_float2(s * -0x1p19f, s * -0x1p11f);
    r.s23 = make_float2(s * 0x1p-12f, s * 0x1p-12f);
    r.c23 = make_float2(s * -0x1p11f, s * -0x1p11f);
    r.no = make_float2(-o, -o);
    return r;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    return __fadd2_rn(a, b);
}

// One qs word → two bf16x2 words of its low-nibble values (bytes 0,1 and
// 2,3), or of its high-nibble values.
__device__ __forceinline__ void dequant_lo(uint32_t v, const NibScale &lo, uint32_t &l01, uint32_t &l23) {
    const uint32_t v8 = __umulhi(v, 1u << 24);  // v >> 8, on the FMA pipe
    const float2 tl01 = __ffma2_rn(make_float2(magic(v, 0xFu), magic(v, 0xF00u)), lo.s01, lo.c01);
    const float2 tl23 = __ffma2_rn(make_float2(magic(v, 0xF0000u), magic(v8, 0xF0000u)), lo.s23, lo.c23);
    l01 = pack_bf16x2(fadd2(tl01, lo.no));
    l23 = pack_bf16x2(fadd2(tl23, lo.no));
}
__device__ __forceinline__ void dequant_hi(uint32_t v, const NibScale &hi, uint32_t &h01, uint32_t &h23) {
    const uint32_t v8 = __umulhi(v, 1u << 24);   // v >> 8
    const uint32_t v16 = __umulhi(v, 1u << 16);  // v >> 16
    const float2 th01 = __ffma2_rn(make_float2(magic(v, 0xF0u), magic(v, 0xF000u)), hi.s01, hi.c01);
    const float2 th23 = __ffma2_rn(make_float2(magic(v8, 0xF000u), magic(v16, 0xF000u)), hi.s23, hi.c23);
    h01 = pack_bf16x2(fadd2(th01, hi.no));
    h23 = pack_bf16x2(fadd2(th23, hi.no));
}

// Scale d·sc and offset dmin·m of sub-block `sb` of a block header (ggml
// canonical 6-bit packing), both exact in fp32.  Called with sb constant
// after unrolling, so the byte selection folds.
__device__ __forceinline__ float2 sub_scale(int sb, uint4 hdr, float2 dm) {
    uint32_t sc, m;
    if (sb < 4) {
        sc = (hdr.y >> (8 * sb)) & 63u;
        m = (hdr.z >> (8 * sb)) & 63u;
    } else {
        const uint32_t hi = (hdr.w >> (8 * (sb - 4))) & 0xFFu;
        sc = (hi & 15u) | (((hdr.y >> (8 * (sb - 4) + 6)) & 3u) << 4);
        m = (hi >> 4) | (((hdr.z >> (8 * (sb - 4) + 6)) & 3u) << 4);
    }
    return make_float2(dm.x * static_cast<float>(sc), dm.y * static_cast<float>(m));
}

// fp32 → bf16 activations, round to nearest even, four values per thread step.
__global__ void x_to_bf16_kernel(const float4 *__restrict__ x, uint2 *__restrict__ xb, size_t n4) {
    pdl_launch_dependents();
    pdl_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = x[i];
        xb[i] = make_uint2(pack_bf16x2(make_float2(v.x, v.y)), pack_bf16x2(make_float2(v.z, v.w)));
    }
}

// kXRows = 0: activation tiles come by TMA from a bf16 copy of x (tm_x).
// Otherwise the dequant warps read fp32 x themselves (kXRows token rows per
// thread and chunk: 2 for up to 64 tokens, 4 for up to 128), round it and
// write the activation tile of each chunk, published with the chunk's A.
// kRelay: weights in the relayouted tensor-core layout (tm_w: one 48-byte
// box per row and chunk); otherwise canonical Q4_K (tm_w: the 16-byte block
// header of each row, tm_q: the chunk's 32 code bytes of each row).
template <int kXRows, bool kRelay>
__global__ void __launch_bounds__(kTcThreads, 1)
    q4k_mm_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_x, const uint8_t *__restrict__ w_tc,
                     const float *__restrict__ x, float *__restrict__ y, int K, int N, int T, int *status,
                     long long wait_limit, int withhold) {
    using L = TcLayout;
    extern __shared__ uint8_t tc_smem_raw[];
    __shared__ volatile int abort_flag;
    // Operand tiles need 1024-byte aligned swizzle atoms.
    const uint32_t raw = smem_addr(tc_smem_raw);
    uint8_t *smem = tc_smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full_w = bars, *empty_w = full_w + kTcWStages;
    uint64_t *full_x = empty_w + kTcWStages, *full_a = full_x + kTcStagesMax, *empty_a = full_a + kTcStagesMax;
    uint64_t *done = empty_a + kTcStagesMax;
    uint64_t *recv_bar = done + 1;  // epilogue: slices received from the other ranks
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_misc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = (int)cluster_size(), rank = (int)cluster_rank();
    const int row0 = (blockIdx.x / S) * kTcRows;
    const int nc_all = K / kTcKc;
    const int c_base = rank * nc_all / S;                 // first chunk of K (absolute)
    const int nchunks = (rank + 1) * nc_all / S - c_base;
    const int n_mma = (T + 15) & ~15;                     // MMA N: tokens rounded up to 16
    // Tensor-memory columns of one accumulator (64 up to 64 tokens, else
    // 128); the rest of the 512 holds the operand stages, 64 columns each,
    // and an activation tile has dcols token rows.  Tiles from the bf16
    // copy are always 128 tokens high.
    const int dcols = (kXRows > 0 && T <= 64) ? 64 : 128;
    const int nst = (int)(kTcTmemCols - 2 * dcols) / 64;  // 6 or 4
    const uint32_t xt_bytes = (uint32_t)dcols * 128;
    const uint32_t tmem_a = 2 * dcols;                    // first column of the A stages

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcWStages; ++s) {
            mbar_init(&full_w[s], 1);
            mbar_init(&empty_w[s], kTcGroupWarps);
        }
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&full_a[s], kTcGroupWarps);
            mbar_init(&empty_a[s], 2);  // one commit per MMA issuer
        }
        mbar_init(done, 2);
        mbar_init(recv_bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kTcWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == kTcWarpTma) {
        int nw = 0, nx = 0;
        auto issue_w = [&](int c) {
            const int ws = c % kTcWStages;
            const uint32_t dst = sbase + L::off_w + ws * kTcWStageBytes;
            const int ca = c_base + c;
            mbar_arrive_expect_tx(&full_w[ws], kTcWStageBytes);
            if constexpr (kRelay) {
                // Tile-major relayout: the chunk's 256 rows are one run.
                bulk_g2s(smem + L::off_w + ws * kTcWStageBytes,
                         w_tc + ((size_t)(row0 / kTcRows) * nc_all + ca) * kTcWStageBytes, kTcWStageBytes, &full_w[ws]);
            } else {
                const int b = ca >> 2, j = ca & 3;
                tma_load_2d(dst, &tm_w, b * kQ4kBytes, row0, &full_w[ws]);
                tma_load_2d(dst + kTcRows * 16, &tm_q, b * kQ4kBytes + 16 + 32 * j, row0, &full_w[ws]);
            }
        };
        auto issue_x = [&](int c) {
            const int st = c % nst;
            mbar_arrive_expect_tx(&full_x[st], xt_bytes);
            tma_load_2d(sbase + L::off_x + st * xt_bytes, &tm_x, (c_base + c) * kTcKc, 0, &full_x[st]);
        };
        if (lane == 0) {
            // (A test may ask for one weight chunk never to arrive, to see
            // the waits on it run out; nothing then writes into its slot.)
            for (; nw < min(nchunks, kTcWStages); ++nw)
                if (nw != withhold) issue_w(nw);
            if constexpr (kXRows == 0) {
                // The bf16 activations come from the previous kernel on the stream.
                pdl_wait();
                for (; nx < min(nchunks, nst); ++nx) issue_x(nx);
                // Weight chunks and activation tiles, each as soon as its
                // slot is free: poll both, backing off while neither moves.
                long long t_last = clock64();
                while ((nw < nchunks || nx < nchunks) && !abort_flag) {
                    bool progressed = false;
                    if (nw < nchunks &&
                        mbar_try_wait(&empty_w[nw % kTcWStages], ((nw / kTcWStages) - 1) & 1)) {
                        if (nw != withhold) issue_w(nw);
                        ++nw;
                        progressed = true;
                    }
                    if (nx < nchunks && mbar_try_wait(&empty_a[nx % nst], ((nx / nst) - 1) & 1)) {
                        issue_x(nx);
                        ++nx;
                        progressed = true;
                    }
                    if (progressed) {
                        t_last = clock64();
                    } else if (clock64() - t_last > wait_limit) {
                        abort_flag = 1;
                        flag_timeout(status);
                    } else {
                        __nanosleep(200);
                    }
                }
            } else {
                // Only weight chunks to issue: wait (suspended, bounded) for
                // each slot in turn.
                nx = nchunks;
                for (; nw < nchunks && !abort_flag; ++nw) {
                    const int ws = nw % kTcWStages;
                    if (!mbar_wait_abortable(&empty_w[ws], ((nw / kTcWStages) - 1) & 1, wait_limit, &abort_flag)) {
                        abort_flag = 1;
                        flag_timeout(status);
                        break;
                    }
                    if (nw != withhold) issue_w(nw);
                }
            }
            // Never leave a tensor copy writing into shared memory that is
            // about to be reused: the last use of each ring slot must land.
            for (int c = max(0, nw - kTcWStages); c < nw; ++c)
                if (c != withhold)
                    (void)mbar_wait_bounded(&full_w[c % kTcWStages], (c / kTcWStages) & 1, wait_limit);
            if constexpr (kXRows == 0) {
                for (int c = max(0, nx - nst); c < nx; ++c)
                    (void)mbar_wait_bounded(&full_x[c % nst], (c / nst) & 1, wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == kTcWarpMma || warp == kTcWarpMma + 1) {
        // One issuer per row half (accumulator), in warps on different SM
        // sub-partitions: an MMA instruction is accepted only about as fast
        // as the tensor pipe runs it, so the few instructions an issuer runs
        // between chunks (its wait, descriptors, commit) leave the pipe idle
        // unless the other issuer fills that time; and the dequantizing warps
        // that share a sub-partition with an issuer take most of its issue
        // slots.  Each accumulator still receives its MMAs from one thread in
        // K order, so the sums do not depend on scheduling.
        const int mh = warp - kTcWarpMma;
        if (lane == 0) {
            const uint32_t idesc = mma_idesc_m128(n_mma);
            // A descriptor's address field counts 16-byte units; every tile
            // lies below 256 KB, so stepping it by addition carries nowhere.
            const uint64_t x_desc0 = sw128_desc(sbase + L::off_x);
            int st = 0;
            uint32_t ph = 0;
            for (int c = 0; c < nchunks; ++c) {
                bool ok = true;
                if constexpr (kXRows == 0) ok = mbar_spin_abortable(&full_x[st], ph, wait_limit, &abort_flag);
                ok = ok && mbar_spin_abortable(&full_a[st], ph, wait_limit, &abort_flag);
                if (!ok) {
                    abort_flag = 1;
                    flag_timeout(status);
                    break;
                }
                tc_fence_after();
                const uint64_t bd = x_desc0 + (uint64_t)(st * (xt_bytes >> 4));
                const uint32_t ad = tmem + tmem_a + 64 * st + 32 * mh;
#pragma unroll
                for (int kk = 0; kk < kTcKc / 16; ++kk)
                    tc_mma_ts(tmem + dcols * mh, ad + 8 * kk, bd + 2 * kk, idesc, (c | kk) != 0);
                tc_commit(&empty_a[st]);
                if (++st == nst) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            // Always signal completion of whatever was issued, and wait for
            // it, so that tensor memory is never read or released with MMAs
            // in flight.
            tc_commit(done);
            (void)mbar_wait_bounded(done, 0, wait_limit);
        }
        __syncwarp();
    } else {
        // Warp w: tensor-memory lane quarter q = w mod 4 of row half
        // mh = (w / 4) mod 2, chunks c ≡ w / 8 (mod 2).  Thread (w, lane)
        // dequantizes weight row r = 128·mh + 32·q + lane of its chunks.
        const int q = warp & 3, mh = (warp >> 2) & 1, grp = warp >> 3;
        const int r = kTcM * mh + 32 * q + lane;
        const uint32_t t_lane = (uint32_t)(32 * q) << 16;
        // Fused activations: in each of its chunks, thread i of a group
        // rounds 16-byte segment i mod 8 of token rows i/8 + 32j, j <
        // kXRows, loaded when the group's previous chunk is written so that
        // the L2 latency hides behind it.
        const int gi = threadIdx.x & (32 * kTcGroupWarps - 1);
        const int aseg = gi & 7, arow = gi >> 3;
        // Token rows past T are read as a copy of row T - 1: they fill only
        // accumulator columns that are never stored, and every access stays
        // inside x and inside the activation tile.
        constexpr int kXR = kXRows > 0 ? kXRows : 1;
        const float *xp = x + (size_t)c_base * kTcKc + 8 * aseg;
        int xro[kXR];
#pragma unroll
        for (int i = 0; i < kXR; ++i) xro[i] = min(arow + 32 * i, T - 1) * K;
        float4 xr[2 * kXR];
        auto load_x = [&](int cc) {
#pragma unroll
            for (int i = 0; i < kXR; ++i) {
                if (kXRows > 0) {
                    const float4 *src = reinterpret_cast<const float4 *>(xp + xro[i] + cc * kTcKc);
                    xr[2 * i] = __ldg(src);
                    xr[2 * i + 1] = __ldg(src + 1);
                }
            }
        };
        if constexpr (kXRows > 0) {
            // x may be written by the previous kernel on the stream.
            pdl_wait();
            if (grp < nchunks) load_x(grp);
        }
        bool good = true;
        // Operand stage st = c mod nst of round c / nst, advanced by 2 per chunk.
        int st = grp, round = 0;
        for (int c = grp; c < nchunks; c += 2) {
            const int ws = c % kTcWStages;
            bool ok = mbar_wait_abortable(&full_w[ws], (c / kTcWStages) & 1, wait_limit, &abort_flag);
            // Operand stage st is free once the MMAs of chunk c - nst are done.
            if (ok && round > 0) ok = mbar_wait_abortable(&empty_a[st], (round - 1) & 1, wait_limit, &abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                good = false;
                break;
            }
            tc_fence_after();
            if constexpr (kXRows > 0) {
                uint8_t *ap = smem + L::off_x + st * xt_bytes + arow * 128 + ((aseg ^ (arow & 7)) << 4);
#pragma unroll
                for (int i = 0; i < kXRows; ++i)
                    *reinterpret_cast<uint4 *>(ap + 32 * 128 * i) =
                        make_uint4(pack_bf16x2(make_float2(xr[2 * i].x, xr[2 * i].y)),
                                   pack_bf16x2(make_float2(xr[2 * i].z, xr[2 * i].w)),
                                   pack_bf16x2(make_float2(xr[2 * i + 1].x, xr[2 * i + 1].y)),
                                   pack_bf16x2(make_float2(xr[2 * i + 1].z, xr[2 * i + 1].w)));
                if (c + 2 < nchunks) load_x(c + 2);
            }
            const uint8_t *wst = smem + L::off_w + ws * kTcWStageBytes;
            float4 sc;  // scale and offset of the low-nibble and the high-nibble sub-block
            uint4 q0, q1;
            if constexpr (kRelay) {
                const uint8_t *row = wst + r * kTcChunkBytes;
                sc = *reinterpret_cast<const float4 *>(row);
                q0 = *reinterpret_cast<const uint4 *>(row + 16);
                q1 = *reinterpret_cast<const uint4 *>(row + 32);
            } else {
                const uint4 hdr = *reinterpret_cast<const uint4 *>(wst + r * 16);
                q0 = *reinterpret_cast<const uint4 *>(wst + kTcRows * 16 + r * 32);
                q1 = *reinterpret_cast<const uint4 *>(wst + kTcRows * 16 + r * 32 + 16);
                const float2 dm = q4k_d_dmin(hdr.x);
                float2 sl, sh;
                switch ((c_base + c) & 3) {  // the same for the whole warp
                    case 0: sl = sub_scale(0, hdr, dm); sh = sub_scale(1, hdr, dm); break;
                    case 1: sl = sub_scale(2, hdr, dm); sh = sub_scale(3, hdr, dm); break;
                    case 2: sl = sub_scale(4, hdr, dm); sh = sub_scale(5, hdr, dm); break;
                    default: sl = sub_scale(6, hdr, dm); sh = sub_scale(7, hdr, dm); break;
                }
                sc = make_float4(sl.x, sl.y, sh.x, sh.y);
            }
            // Columns of this lane: low-nibble values k = 0..31 of the chunk
            // at 0..15, high-nibble values k = 32..63 at 16..31.
            const uint32_t ta = tmem + t_lane + tmem_a + 64 * st + 32 * mh;
            uint32_t o[16];
            {
                const NibScale lo = nib_scale_lo(sc.x, sc.y);
                dequant_lo(q0.x, lo, o[0], o[1]);
                dequant_lo(q0.y, lo, o[2], o[3]);
                dequant_lo(q0.z, lo, o[4], o[5]);
                dequant_lo(q0.w, lo, o[6], o[7]);
                dequant_lo(q1.x, lo, o[8], o[9]);
                dequant_lo(q1.y, lo, o[10], o[11]);
                dequant_lo(q1.z, lo, o[12], o[13]);
                dequant_lo(q1.w, lo, o[14], o[15]);
                tc_st16(ta, o);
            }
            {
                const NibScale hi = nib_scale_hi(sc.z, sc.w);
                dequant_hi(q0.x, hi, o[0], o[1]);
                dequant_hi(q0.y, hi, o[2], o[3]);
                dequant_hi(q0.z, hi, o[4], o[5]);
                dequant_hi(q0.w, hi, o[6], o[7]);
                dequant_hi(q1.x, hi, o[8], o[9]);
                dequant_hi(q1.y, hi, o[10], o[11]);
                dequant_hi(q1.z, hi, o[12], o[13]);
                dequant_hi(q1.w, hi, o[14], o[15]);
                tc_st16(ta + 16, o);
            }
            // Publish the chunk's A (and activation tile) to the MMA issuers,
            // and release the weight stage (its words are consumed above) to
            // the next copy.
            tc_wait_st();
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full_a[st]);
                mbar_arrive(&empty_w[ws]);
            }
            st += 2;
            if (st >= nst) {
                st -= nst;
                ++round;
            }
        }
        if (!good) {
            abort_flag = 1;
            flag_timeout(status);
        }
    }

    // The accumulators are complete once every MMA this CTA issued has finished.
    const bool have_acc = __syncthreads_and(mbar_wait_bounded(done, 0, wait_limit) ? 1 : 0) != 0;
    tc_fence_after();

    // Epilogue: the split-K sum over the cluster, in passes of up to 64
    // tokens.  Rank s owns the tile's rows [lo(s), lo(s+1)), lo(s) =
    // floor(256·s/S).  In a pass every rank writes its accumulators to a
    // local tile own[row][token] (token pitch tp = the pass's tokens rounded
    // up to 4, plus 4, which keeps 16-byte rows and spreads consecutive rows
    // over the banks); after a cluster barrier (which also marks every rank
    // done with its rings, which the tiles reuse) one thread sends the rows
    // each other rank owns, one contiguous slice per rank, with a bulk copy
    // into that rank's receive slot (recv[slot][row - lo][token], one slot per
    // sender), completing on the receiver's barrier.  Bulk copies move the
    // data far faster than per-thread loads or stores to distributed shared
    // memory, measured on GB300.  Each rank then adds the S partial sums of
    // its rows in rank order, all from local shared memory, and writes its
    // rows of y.  A second cluster barrier keeps every sender's tile until
    // its copies have landed.  The result does not depend on scheduling.
    const int rows_cap = (kTcRows + S - 1) / S;
    auto lo_of = [&](int s_) { return s_ * kTcRows / S; };
    float *own = reinterpret_cast<float *>(smem);
    float *recv = own + kTcRows * (64 + 8);  // after the largest own tile
    const int lo = lo_of(rank), rows = lo_of(rank + 1) - lo;
    const int ncols = min(kTcRows, N - row0);
    for (int p0 = 0, pass = 0; p0 < T; p0 += 64, ++pass) {
        const int tpass = min(64, T - p0);
        const int tp = ((tpass + 3) & ~3) + 4;
        if (warp < kTcDqWarps) {
            const int q = warp & 3, mh = (warp >> 2) & 1;
            const int o = kTcM * mh + 32 * q + lane;
#pragma unroll 1
            for (int tb = (p0 >> 4) + (warp >> 3); 16 * tb < p0 + tpass; tb += 2) {  // warp-uniform
                float v[16];
                if (have_acc && nchunks > 0) {
                    tc_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(dcols * mh + 16 * tb), v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                const int tl = 16 * tb - p0;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (tl + 4 * k < tpass)
                        *reinterpret_cast<float4 *>(own + (size_t)o * tp + tl + 4 * k) =
                            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            }
        }
        // The tile is read next by bulk copies (the async proxy).
        fence_async_smem();
        tc_fence_before();
        cluster_sync_all();
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(recv_bar, (uint32_t)((S - 1) * rows * tp * 4));
            for (int s_ = 0; s_ < S; ++s_) {
                if (s_ == rank) continue;
                const int slo = lo_of(s_), srows = lo_of(s_ + 1) - slo;
                const int slot = rank < s_ ? rank : rank - 1;
                const uint32_t dst = map_to_rank(smem_addr(recv + (size_t)slot * rows_cap * tp), (uint32_t)s_);
                const uint32_t bar = map_to_rank(smem_addr(recv_bar), (uint32_t)s_);
                bulk_s2cluster(dst, smem_addr(own + (size_t)slo * tp), (uint32_t)(srows * tp * 4), bar);
            }
        }
        const bool got = mbar_wait_bounded(recv_bar, pass & 1, wait_limit);
        if (!got && threadIdx.x == 0) flag_timeout(status);
        // The output may be read by the previous kernel on the stream.
        if (pass == 0) pdl_wait();
        const int ngroups = (tpass + 3) / 4;
        for (int i = threadIdx.x; got && i < rows * ngroups; i += kTcThreads) {
            const int ol = i % rows, t0 = 4 * (i / rows);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s_ = 0; s_ < S; ++s_) {
                const float *src = s_ == rank ? own + (size_t)(lo + ol) * tp
                                              : recv + ((size_t)(s_ < rank ? s_ : s_ - 1) * rows_cap + ol) * tp;
                const float4 v = *reinterpret_cast<const float4 *>(src + t0);
                if (s_ == 0) {
                    acc = v;
                } else {
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
            }
            const int col = lo + ol;
            if (col < ncols) {
                float *dst = y + (size_t)(p0 + t0) * N + row0 + col;
                dst[0] = acc.x;
                if (t0 + 1 < tpass) dst[N] = acc.y;
                if (t0 + 2 < tpass) dst[2 * (size_t)N] = acc.z;
                if (t0 + 3 < tpass) dst[3 * (size_t)N] = acc.w;
            }
        }
        // Every rank has received its slices, so every sender's tile has
        // been read: the next pass (or exit) may proceed.
        __syncthreads();
        cluster_sync_all();
    }
    if (warp == kTcWarpMma) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// One launch over a tile of at most 128 tokens: activations either from the
// bf16 copy xb by TMA (xb != nullptr) or from fp32 x, rounded in the kernel.
// relay: W is in the relayouted tensor-core layout.
cudaError_t launch_tile(const LaunchCtx &c, const __nv_bfloat16 *xb, const float *x, const uint8_t *W, bool relay,
                        float *y, int K, int N, int T, int S) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    alignas(64) CUtensorMap tm_w, tm_q, tm_x;
    std::memset(&tm_q, 0, sizeof(tm_q));
    std::memset(&tm_x, 0, sizeof(tm_x));
    auto map_w = [&](CUtensorMap *m, cuuint64_t row_bytes, cuuint32_t box_bytes) {
        const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)N};
        const cuuint64_t strides[1] = {row_bytes};
        const cuuint32_t box[2] = {box_bytes, (cuuint32_t)kTcRows};
        const cuuint32_t estr[2] = {1, 1};
        return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(W), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (relay) {
        // Tile-major: each chunk of a 256-row tile is one 12 KB run, copied
        // by a plain bulk copy; no tensor map.
        std::memset(&tm_w, 0, sizeof(tm_w));
    } else {
        // Rows of K/256 blocks of 144 bytes; boxes of the 16-byte headers and
        // of one chunk's 32 code bytes, 256 rows each.
        const cuuint64_t row_bytes = (cuuint64_t)(K / kQ4kValues) * kQ4kBytes;
        if (!map_w(&tm_w, row_bytes, 16) || !map_w(&tm_q, row_bytes, 32)) return cudaErrorInvalidValue;
    }
    if (xb) {
        // bf16 activations [T][K]: a 64-value (128-byte) by 128-token box with
        // the 128-byte swizzle is exactly one K-major MMA operand tile; token
        // rows past T read as zero.
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
        const cuuint64_t strides[1] = {(cuuint64_t)K * sizeof(__nv_bfloat16)};
        const cuuint32_t box[2] = {(cuuint32_t)kTcKc, (cuuint32_t)kTcTok};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(xb), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const size_t smem = TcLayout::total + 1024;
    if (smem > (size_t)c.max_smem_optin) return cudaErrorNotSupported;
    decltype(&q4k_mm_tc_kernel<0, false>) kernel;
    if (relay)
        kernel = xb ? q4k_mm_tc_kernel<0, true> : (T <= 64 ? q4k_mm_tc_kernel<2, true> : q4k_mm_tc_kernel<4, true>);
    else
        kernel = xb ? q4k_mm_tc_kernel<0, false> : (T <= 64 ? q4k_mm_tc_kernel<2, false> : q4k_mm_tc_kernel<4, false>);
    cudaError_t e = ensure_smem(kernel, smem);
    if (e != cudaSuccess) return e;
    const int tiles = (N + kTcRows - 1) / kTcRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * S);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
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
    return cudaLaunchKernelEx(&cfg, kernel, tm_w, tm_q, tm_x, relay ? W : nullptr, x, y, K, N, T, c.status,
                              c.wait_limit, c.withhold);
}

// Tiles of 128 tokens over the bf16 copy xb of x (several tiles), or one
// tile that rounds x itself (xb == nullptr, at most 128 tokens).
cudaError_t launch_tiles(const LaunchCtx &c, const float *x, __nv_bfloat16 *xb, const uint8_t *W, bool relay,
                         float *y, int K, int N, int T, int S) {
    if (!xb) return launch_tile(c, nullptr, x, W, relay, y, K, N, T, S);
    const size_t n = (size_t)T * K;
    cudaError_t e;
    {
        const size_t n4 = n / 4;
        const int grid = (int)min((size_t)4 * c.num_sms, (n4 + 255) / 256);
        e = launch_kernel(c, x_to_bf16_kernel, dim3(grid), dim3(256), 0,
                          reinterpret_cast<const float4 *>(x), reinterpret_cast<uint2 *>(xb), n4);
    }
    for (int t0 = 0; t0 < T && e == cudaSuccess; t0 += kTcMaxTokens) {
        const int tt = min(kTcMaxTokens, T - t0);
        e = launch_tile(c, xb + (size_t)t0 * K, nullptr, W, relay, y + (size_t)t0 * N, K, N, tt, S);
    }
    return e;
}

// One-time relayout, canonical Q4_K → tile-major tensor-core chunks: one
// thread per (tile row, chunk) of the padded layout, 16-byte loads and
// stores (both buffers 16-byte aligned).  Thread i writes the 48 bytes at
// 48·i: chunk c = (i / 256) mod nc of tile (i / 256) / nc, row i mod 256 of
// the tile; rows past N are zero.  The products d·sc and dmin·m are exact in
// fp32, so the relayouted weight dequantizes to the same fp32 matrix.
__global__ void q4k_relayout_tc_kernel(const uint8_t *__restrict__ W, uint8_t *__restrict__ R, int K, int N) {
    const int nc = K / kTcKc, nb = K / kQ4kValues;
    const size_t tiles = ((size_t)N + kTcRows - 1) / kTcRows;
    const size_t total = tiles * nc * kTcRows;
    pdl_launch_dependents();
    pdl_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t run = i / kTcRows;
        const int r = (int)(i % kTcRows), ca = (int)(run % nc);
        const size_t o = (run / nc) * kTcRows + r;
        uint4 *dst = reinterpret_cast<uint4 *>(R + i * kTcChunkBytes);
        if (o >= (size_t)N) {
            dst[0] = dst[1] = dst[2] = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const int b = ca >> 2, j = ca & 3;
        const uint8_t *blk = W + (o * nb + b) * kQ4kBytes;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        const float2 dm = q4k_d_dmin(hdr.x);
        float2 sl, sh;
        switch (j) {
            case 0: sl = sub_scale(0, hdr, dm); sh = sub_scale(1, hdr, dm); break;
            case 1: sl = sub_scale(2, hdr, dm); sh = sub_scale(3, hdr, dm); break;
            case 2: sl = sub_scale(4, hdr, dm); sh = sub_scale(5, hdr, dm); break;
            default: sl = sub_scale(6, hdr, dm); sh = sub_scale(7, hdr, dm); break;
        }
        dst[0] = make_uint4(__float_as_uint(sl.x), __float_as_uint(sl.y), __float_as_uint(sh.x), __float_as_uint(sh.y));
        dst[1] = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j);
        dst[2] = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * j);
    }
}

// Split of K over the cluster: at least 3 CTAs per row tile, and at most
// kTcMaxKPerCta values of K per CTA; 0 when the reduction (at most four
// ranks) cannot take it.
int tc_split(int K) {
    const int S = max(3, (K + kTcMaxKPerCta - 1) / kTcMaxKPerCta);
    return S > 4 ? 0 : S;
}

}  // namespace

size_t q4k_mm_tc_scratch_bytes(int K, int N, int T) {
    (void)N;
    if (T <= kTcMaxTokens) return 0;
    return ((size_t)T * K * sizeof(__nv_bfloat16) + 255) / 256 * 256;
}

namespace {

cudaError_t launch_mm_tc(const LaunchCtx &c, const float *x, const uint8_t *W, bool relay, float *y, int K, int N,
                         int T) {
    const int S = tc_split(K);
    if (S == 0) return cudaErrorNotSupported;
    // Up to 128 tokens: one launch that rounds x itself, nothing allocated.
    // More: x is rounded to bf16 once into stream-ordered scratch (freed on
    // the same stream after the last tile) and the weights are re-read once
    // per tile of 128 tokens.
    const size_t bytes = q4k_mm_tc_scratch_bytes(K, N, T);
    if (bytes == 0) return launch_tiles(c, x, nullptr, W, relay, y, K, N, T, S);
    void *scratch = nullptr;
    cudaError_t e = cudaMallocAsync(&scratch, bytes, c.stream);
    if (e != cudaSuccess) return e;
    e = launch_tiles(c, x, static_cast<__nv_bfloat16 *>(scratch), W, relay, y, K, N, T, S);
    const cudaError_t ef = cudaFreeAsync(scratch, c.stream);
    return e != cudaSuccess ? e : ef;
}

}  // namespace

cudaError_t launch_q4k_mm_tc(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K, int N, int T) {
    return launch_mm_tc(c, x, W, false, y, K, N, T);
}

cudaError_t launch_q4k_mm_tc_relayouted(const LaunchCtx &c, const float *x, const uint8_t *R, float *y, int K, int N,
                                        int T) {
    return launch_mm_tc(c, x, R, true, y, K, N, T);
}

size_t q4k_relayout_tc_bytes(int K, int N) {
    return ((size_t)N + kTcRows - 1) / kTcRows * kTcRows * (size_t)(K / kTcKc) * kTcChunkBytes;
}

cudaError_t launch_q4k_relayout_tc(const LaunchCtx &c, const uint8_t *W, uint8_t *R, int K, int N) {
    const size_t total = ((size_t)N + kTcRows - 1) / kTcRows * kTcRows * (K / kTcKc);
    const int grid = (int)min((size_t)8 * c.num_sms, (total + 255) / 256);
    return launch_kernel(c, q4k_relayout_tc_kernel, dim3(grid), dim3(256), 0, W, R, K, N);
}

// ----------------------------------------------------------------------------
// The same product with its scratch in a fixed array of library memory, for
// callers that cannot allocate during a call (q4k_matmul_tc_noalloc).
// ----------------------------------------------------------------------------

namespace {

// Module memory: every GPU that loads the library holds it until the process
// exits.  In host code this name is only a stand-in for the device object;
// kernels get the address that cudaGetSymbolAddress returns for the current
// device.
static __device__ __align__(256) uint8_t g_tc_fixed_scratch[Q4MM_TC_NOALLOC_SCRATCH_BYTES];

constexpr int kFixedMaxDevices = 64;

struct FixedScratch {
    bool ready = false;
    uint8_t *ptr = nullptr;
};
FixedScratch g_fixed[kFixedMaxDevices];
std::mutex g_fixed_mu;

// Device address of the array on the current device, looked up once per
// device (with that device current) and kept.
cudaError_t fixed_scratch(uint8_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kFixedMaxDevices) return cudaErrorInvalidDevice;
    FixedScratch &f = g_fixed[dev];
    std::lock_guard<std::mutex> lock(g_fixed_mu);
    if (!f.ready) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&f.ptr), g_tc_fixed_scratch);
        if (e != cudaSuccess) return e;
        f.ready = true;
    }
    *out = f.ptr;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_q4k_mm_tc_fixed_scratch(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                           int K, int N, int T) {
    const int S = tc_split(K);
    if (S == 0) return cudaErrorNotSupported;
    const size_t bytes = q4k_mm_tc_scratch_bytes(K, N, T);
    if (bytes > (size_t)Q4MM_TC_NOALLOC_SCRATCH_BYTES) return cudaErrorInvalidValue;
    // The lookup runs on every call, so the first call on a device makes it
    // whatever its size.
    uint8_t *scratch = nullptr;
    cudaError_t e = fixed_scratch(&scratch);
    if (e != cudaSuccess) return e;
    // As in launch_q4k_mm_tc, the scratch (above 128 tokens) holds x rounded
    // to bf16.  Nothing needs clearing: the pre-pass writes all of it.
    return launch_tiles(c, x, bytes ? reinterpret_cast<__nv_bfloat16 *>(scratch) : nullptr, W, false, y, K, N, T, S);
}

}  // namespace q4mm
