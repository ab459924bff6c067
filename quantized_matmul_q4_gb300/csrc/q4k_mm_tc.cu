// Q4_K prefill on the tcgen05 tensor cores: bf16 operands, fp32 accumulation
// in tensor memory (sm_103a).
//
// y[t][o] = Σ_k x[t][k]·w[o][k] with w = d·sc_s·q − dmin·m_s (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline"), evaluated as D[t][o] = A[t][k]·B[o][k] with
//   A = the activations rounded to bf16 (M = 128 token rows; tokens past the
//       tile's count read as zero),
//   B = the dequantized weights rounded to bf16 (N = 256 output rows),
//   D = fp32 in tensor memory, K = 16 per MMA instruction.
// A tcgen05.mma instruction's time grows far less than its size (measured
// on GB300: 108 cycles at 128 × 128 × 16, 130 at 128 × 256 × 16), so each
// instruction is made as large as the tile allows: 128 × 256 × 16.
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
// CTA accumulates its K range in one tensor-memory accumulator (at most
// 16384 values of K, within which the tensor core's fp32 accumulation stays
// far inside the stated tolerance).  Every rank copies its accumulator into
// its own shared memory; after a cluster barrier each rank takes one S-th of
// the tile's outputs, adds the S ranks' values in rank order through
// distributed shared memory and writes them to y, so the result does not
// depend on scheduling and no partial sum goes through global memory.
//
// Roles in a CTA:
//  * warp 16 (one thread) issues 2-D TMA tensor loads: a Q4_K block column
//    (256 rows × 144 bytes) per 256 values of K, before the wait on the
//    previous kernel, and (tiles of the bf16 copy) a bf16 activation tile
//    (128 tokens × 64 values) per chunk of 64 values, after it, each as soon
//    as its ring slot is free.
//  * warps 0–15 dequantize: thread (r, h), r = t mod 256 and h = t / 256,
//    turns qs bytes 16h..16h+15 of row r's slab into 16 low-nibble values of
//    sub-block 2j and 16 high-nibble values of 2j+1.  Each nibble becomes a float with one logic op (2^23 + q·2^p), one
//    paired FMA with the scale at 2^-p and −scale·2^(23−p) gives scale·q
//    exactly, one paired add removes the min term (the single rounding of the
//    fp32 dequantization), and one conversion packs two bf16.  Results go in
//    the 128-byte-swizzled K-major layout; with fused activations the same
//    threads also write the chunk's activation tile.  The writes are fenced
//    to the async proxy before the chunk's barrier arrive.
//  * warp 17 allocates the accumulator in tensor memory; its first thread
//    issues four 128×256×16 MMAs per chunk and commits them to the chunk's
//    activation and weight slots.
//  * warps 0–15 then read the accumulator (tcgen05.ld) into shared memory,
//    and every thread takes part in the cluster-wide reduction.
// All mbarrier waits are bounded; a time-out sets the device status word and
// every thread still reaches the two cluster barriers.
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

constexpr int kTcRows = 256;                       // MMA N: weight rows per CTA
constexpr int kTcTok = 128;                        // MMA M: token rows per tile
constexpr int kTcKc = 64;                          // K per chunk: a 128-byte row of bf16
constexpr int kTcDqWarps = 16;                     // dequant + epilogue warps
constexpr int kTcWarpTma = kTcDqWarps;             // TMA producer warp
constexpr int kTcWarpMma = kTcDqWarps + 1;         // MMA issuer warp
constexpr int kTcThreads = 32 * (kTcDqWarps + 2);
constexpr int kTcDq = 32 * kTcDqWarps;             // dequant threads (two per weight row)
constexpr int kTcWStages = 2;                      // Q4_K block-column tiles in flight
constexpr int kTcAStages = 3;                      // bf16 activation tiles in flight
constexpr int kTcBStages = 3;                      // bf16 weight operand tiles in flight
static_assert(kTcAStages == kTcBStages, "fused activation tiles share the weight ring's slots");
constexpr uint32_t kTcWTileBytes = kTcRows * kQ4kBytes;  // 36864
constexpr uint32_t kTcATileBytes = kTcTok * 128;         // 16384
constexpr uint32_t kTcBTileBytes = kTcRows * 128;        // 32768
constexpr int kTcMaxKPerCta = 16384;               // one accumulator per CTA
constexpr uint32_t kTcTmemCols = kTcRows;          // fp32 accumulator columns

struct TcLayout {
    static constexpr uint32_t off_a = 0;
    static constexpr uint32_t off_b = off_a + kTcAStages * kTcATileBytes;
    static constexpr uint32_t off_w = off_b + kTcBStages * kTcBTileBytes;
    static constexpr uint32_t off_bar = off_w + kTcWStages * kTcWTileBytes;
    static constexpr uint32_t n_bars = 2 * kTcWStages + 2 * kTcAStages + 2 * kTcBStages + 1;
    static constexpr uint32_t off_misc = off_bar + 8 * n_bars;
    static constexpr uint32_t total = off_misc + 16;
    static_assert(off_b % 1024 == 0 && off_w % 1024 == 0, "operand tiles must be 1024-byte aligned");
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
// M × N.
template <int M, int N>
__device__ __forceinline__ uint32_t mma_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
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

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
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

// One qs word → two bf16x2 words of low-nibble values (bytes 0,1 and 2,3)
// and two of high-nibble values.
__device__ __forceinline__ void dequant_word(uint32_t v, const NibScale &lo, const NibScale &hi,
                                             uint32_t &l01, uint32_t &l23, uint32_t &h01,
                                             uint32_t &h23) {
    const uint32_t v8 = __umulhi(v, 1u << 24);   // v >> 8, on the FMA pipe
    const uint32_t v16 = __umulhi(v, 1u << 16);  // v >> 16
    const float2 tl01 = __ffma2_rn(make_float2(magic(v, 0xFu), magic(v, 0xF00u)), lo.s01, lo.c01);
    const float2 tl23 = __ffma2_rn(make_float2(magic(v, 0xF0000u), magic(v8, 0xF0000u)), lo.s23, lo.c23);
    const float2 th01 = __ffma2_rn(make_float2(magic(v, 0xF0u), magic(v, 0xF000u)), hi.s01, hi.c01);
    const float2 th23 = __ffma2_rn(make_float2(magic(v8, 0xF000u), magic(v16, 0xF000u)), hi.s23, hi.c23);
    l01 = pack_bf16x2(fadd2(tl01, lo.no));
    l23 = pack_bf16x2(fadd2(tl23, lo.no));
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
// write the activation tile of each chunk next to its weight tile, and one
// barrier (full_b) publishes both.
template <int kXRows>
__global__ void __launch_bounds__(kTcThreads, 1)
    q4k_mm_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
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
    uint64_t *full_a = empty_w + kTcWStages, *empty_a = full_a + kTcAStages;
    uint64_t *full_b = empty_a + kTcAStages, *empty_b = full_b + kTcBStages;
    uint64_t *done = empty_b + kTcBStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_misc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = (int)cluster_size(), rank = (int)cluster_rank();
    const int row0 = (blockIdx.x / S) * kTcRows;
    const int nc_all = K / kTcKc;
    const int c_base = rank * nc_all / S;                 // first chunk of K (absolute)
    const int nchunks = (rank + 1) * nc_all / S - c_base; // may be 0 when K is short
    // Q4_K blocks touched: the first may be entered at chunk j0 > 0.
    const int b_begin = c_base / 4;
    const int j0 = c_base % 4;
    const int nblocks = nchunks > 0 ? (c_base + nchunks + 3) / 4 - b_begin : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcWStages; ++s) {
            mbar_init(&full_w[s], 1);
            mbar_init(&empty_w[s], kTcDq);
        }
        for (int s = 0; s < kTcAStages; ++s) {
            mbar_init(&full_a[s], 1);
            mbar_init(&empty_a[s], 1);
        }
        for (int s = 0; s < kTcBStages; ++s) {
            mbar_init(&full_b[s], kTcDq / 2);
            mbar_init(&empty_b[s], 1);
        }
        mbar_init(done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (kXRows > 0) {
        // Token rows T..127 of every activation stage stay zero.
        const int pad16 = (kTcTok - T) * 128 / 16;
        for (int s = 0; s < kTcAStages; ++s) {
            uint4 *p = reinterpret_cast<uint4 *>(smem + L::off_a + s * kTcATileBytes + T * 128);
            for (int i = threadIdx.x; i < pad16; i += kTcThreads) p[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();
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
        if (lane == 0) {
            // Weight tiles and activation tiles are issued independently, each
            // as soon as its ring slot is free.
            int nw = 0, nx = 0;
            // (A test may ask for one weight tile never to arrive, to see
            // the waits on it run out; nothing then writes into its slot.)
            for (; nw < min(nblocks, kTcWStages); ++nw) {
                if (nw == withhold) continue;
                mbar_arrive_expect_tx(&full_w[nw], kTcWTileBytes);
                tma_load_2d(sbase + L::off_w + nw * kTcWTileBytes, &tm_w, (b_begin + nw) * kQ4kBytes, row0,
                            &full_w[nw]);
            }
            if constexpr (kXRows == 0) {
                // The bf16 activations come from the previous kernel on the stream.
                pdl_wait();
                for (; nx < min(nchunks, kTcAStages); ++nx) {
                    mbar_arrive_expect_tx(&full_a[nx], kTcATileBytes);
                    tma_load_2d(sbase + L::off_a + nx * kTcATileBytes, &tm_x, (c_base + nx) * kTcKc, 0,
                                &full_a[nx]);
                }
            } else {
                nx = nchunks;  // the dequant warps write the activation tiles
            }
            if constexpr (kXRows > 0) {
                // Only weight tiles to issue: wait (suspended, bounded) for
                // each slot in turn; a busy poll here would take issue slots
                // from the dequant warps on this scheduler.
                for (; nw < nblocks && !abort_flag; ++nw) {
                    const int ws = nw % kTcWStages;
                    if (!mbar_wait_abortable(&empty_w[ws], ((nw / kTcWStages) - 1) & 1, wait_limit, &abort_flag)) {
                        abort_flag = 1;
                        flag_timeout(status);
                        break;
                    }
                    if (nw != withhold) {
                        mbar_arrive_expect_tx(&full_w[ws], kTcWTileBytes);
                        tma_load_2d(sbase + L::off_w + ws * kTcWTileBytes, &tm_w, (b_begin + nw) * kQ4kBytes, row0,
                                    &full_w[ws]);
                    }
                }
            } else {
                // Weight and activation tiles, each as soon as its slot is
                // free: poll both, backing off while neither moves.
                long long t_last = clock64();
                while ((nw < nblocks || nx < nchunks) && !abort_flag) {
                    bool progressed = false;
                    if (nw < nblocks) {
                        const int ws = nw % kTcWStages;
                        if (mbar_try_wait(&empty_w[ws], ((nw / kTcWStages) - 1) & 1)) {
                            if (nw != withhold) {
                                mbar_arrive_expect_tx(&full_w[ws], kTcWTileBytes);
                                tma_load_2d(sbase + L::off_w + ws * kTcWTileBytes, &tm_w,
                                            (b_begin + nw) * kQ4kBytes, row0, &full_w[ws]);
                            }
                            ++nw;
                            progressed = true;
                        }
                    }
                    if (nx < nchunks) {
                        const int as = nx % kTcAStages;
                        if (mbar_try_wait(&empty_a[as], ((nx / kTcAStages) - 1) & 1)) {
                            mbar_arrive_expect_tx(&full_a[as], kTcATileBytes);
                            tma_load_2d(sbase + L::off_a + as * kTcATileBytes, &tm_x, (c_base + nx) * kTcKc, 0,
                                        &full_a[as]);
                            ++nx;
                            progressed = true;
                        }
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
            }
            // Never leave a tensor copy writing into shared memory that is
            // about to be reused: the last use of each ring slot must land.
            for (int b = max(0, nw - kTcWStages); b < nw; ++b)
                if (b != withhold)
                    (void)mbar_wait_bounded(&full_w[b % kTcWStages], (b / kTcWStages) & 1, wait_limit);
            if constexpr (kXRows == 0) {
                for (int c = max(0, nx - kTcAStages); c < nx; ++c)
                    (void)mbar_wait_bounded(&full_a[c % kTcAStages], (c / kTcAStages) & 1, wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == kTcWarpMma) {
        if (lane == 0) {
            const uint32_t idesc = mma_idesc<kTcTok, kTcRows>();
            // One thread's dependent chain sits between the chunks' MMAs, so
            // the loop keeps it short: stage, phase and descriptors advance by
            // additions (a descriptor's address field counts 16-byte units;
            // every tile lies below 256 KB, so no carry leaves the field).
            const uint64_t a_desc0 = sw128_desc(sbase + L::off_a), b_desc0 = sw128_desc(sbase + L::off_b);
            int st = 0;
            uint32_t ph = 0;
            for (int c = 0; c < nchunks; ++c) {
                bool ok = true;
                if constexpr (kXRows == 0) ok = mbar_wait_bounded(&full_a[st], ph, wait_limit);
                ok = ok && mbar_wait_bounded(&full_b[st], ph, wait_limit);
                if (!ok) {
                    abort_flag = 1;
                    flag_timeout(status);
                    break;
                }
                tc_fence_after();
                const uint64_t ad = a_desc0 + (uint64_t)(st * (kTcATileBytes >> 4));
                const uint64_t bd = b_desc0 + (uint64_t)(st * (kTcBTileBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < kTcKc / 16; ++kk)
                    tc_mma(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (c | kk) != 0);
                if constexpr (kXRows == 0) tc_commit(&empty_a[st]);
                tc_commit(&empty_b[st]);
                if (++st == kTcBStages) {
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
        // Two groups of 256 threads take alternate chunks: thread t of group
        // g = t / 256 dequantizes all 64 values of weight row r = t mod 256 in
        // the chunks c ≡ g (mod 2) of the CTA.
        const int r = threadIdx.x & (kTcRows - 1), grp = threadIdx.x >> 8;
        // Fused activations: in each of its chunks, thread r of a group
        // rounds 16-byte segment r mod 8 of token rows r/8 + 32i, i <
        // kXRows, loaded when the group's previous chunk is written so that
        // the L2 latency hides behind it.
        const int aseg = r & 7, arow = r >> 3;
        const float *xrow = x + (size_t)arow * K + (size_t)c_base * kTcKc + 8 * aseg;
        constexpr int kXR = kXRows > 0 ? kXRows : 1;
        float4 xr[2 * kXR];
        auto load_x = [&](int cc) {
#pragma unroll
            for (int i = 0; i < kXR; ++i) {
                if (kXRows > 0 && arow + 32 * i < T) {
                    const float4 *src = reinterpret_cast<const float4 *>(xrow + (size_t)(32 * i) * K + (size_t)cc * kTcKc);
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
        int c = 0;  // chunk of this CTA
        for (int b = 0; b < nblocks && good; ++b) {
            const int ws = b % kTcWStages;
            const uint8_t *blk = smem + L::off_w + ws * kTcWTileBytes + r * kQ4kBytes;
            // Chunks of this block within the CTA's range.
            const int jb = b == 0 ? j0 : 0;
            const int je = min(4, jb + (nchunks - c));
            // Every thread waits for the block, even one with no chunk of it,
            // before releasing it below: no thread can then release a ring
            // slot twice in one phase.
            if (__any_sync(0xffffffffu, abort_flag != 0) ||
                !__all_sync(0xffffffffu, mbar_wait_bounded(&full_w[ws], (b / kTcWStages) & 1, wait_limit))) {
                good = false;
                break;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < jb || j >= je) continue;
                const int cc = c + (j - jb);
                if ((cc & 1) != grp) continue;
                const int bs = cc % kTcBStages;
                if (__any_sync(0xffffffffu, abort_flag != 0)) {
                    good = false;
                    break;
                }
                bool ok = true;
                if (cc >= kTcBStages)
                    ok = mbar_wait_bounded(&empty_b[bs], ((cc / kTcBStages) - 1) & 1, wait_limit);
                if (!__all_sync(0xffffffffu, ok)) {
                    good = false;
                    break;
                }
                if constexpr (kXRows > 0) {
                    uint8_t *ap = smem + L::off_a + bs * kTcATileBytes + arow * 128 + ((aseg ^ (arow & 7)) << 4);
#pragma unroll
                    for (int i = 0; i < kXRows; ++i) {
                        if (arow + 32 * i < T)
                            *reinterpret_cast<uint4 *>(ap + 32 * 128 * i) = make_uint4(
                                pack_bf16x2(make_float2(xr[2 * i].x, xr[2 * i].y)),
                                pack_bf16x2(make_float2(xr[2 * i].z, xr[2 * i].w)),
                                pack_bf16x2(make_float2(xr[2 * i + 1].x, xr[2 * i + 1].y)),
                                pack_bf16x2(make_float2(xr[2 * i + 1].z, xr[2 * i + 1].w)));
                    }
                    if (cc + 2 < nchunks) load_x(cc + 2);
                }
                const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
                const float2 dm = q4k_d_dmin(hdr.x);
                const float2 slo = sub_scale(2 * j, hdr, dm);
                const float2 shi = sub_scale(2 * j + 1, hdr, dm);
                const NibScale lo = nib_scale_lo(slo.x, slo.y), hi = nib_scale_hi(shi.x, shi.y);
                uint8_t *brow = smem + L::off_b + bs * kTcBTileBytes + r * 128;
                const int sw = r & 7;
                // Half hh: qs bytes 16hh..16hh+15 give low values k = 16hh..
                // (logical 16-byte chunks 2hh, 2hh+1) and high values k =
                // 32+16hh.. (chunks 4+2hh, 5+2hh).
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * j + 16 * hh);
                    uint32_t lw[8], hw[8];
                    dequant_word(q.x, lo, hi, lw[0], lw[1], hw[0], hw[1]);
                    dequant_word(q.y, lo, hi, lw[2], lw[3], hw[2], hw[3]);
                    dequant_word(q.z, lo, hi, lw[4], lw[5], hw[4], hw[5]);
                    dequant_word(q.w, lo, hi, lw[6], lw[7], hw[6], hw[7]);
                    *reinterpret_cast<uint4 *>(brow + (((2 * hh) ^ sw) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    *reinterpret_cast<uint4 *>(brow + (((2 * hh + 1) ^ sw) << 4)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                    *reinterpret_cast<uint4 *>(brow + (((4 + 2 * hh) ^ sw) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(brow + (((5 + 2 * hh) ^ sw) << 4)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                }
                fence_async_smem();
                mbar_arrive(&full_b[bs]);
            }
            c += je - jb;
            // Every dequant thread releases the block once.
            if (good) mbar_arrive(&empty_w[ws]);
        }
        if (!good) {
            abort_flag = 1;
            flag_timeout(status);
        }
    }

    // The accumulator is complete once every MMA this CTA issued has finished.
    const bool have_acc = __syncthreads_and(mbar_wait_bounded(done, 0, wait_limit) ? 1 : 0) != 0;
    tc_fence_after();

    // Epilogue.  Warps w, w+4, w+8, w+12 share TMEM lane quarter w % 4
    // (tokens 32·quarter..) and read 64 of the 256 columns each into a shared
    // tile [T][260]; the rings are idle by now.  After a cluster barrier every
    // rank takes one S-th of the tile's outputs, adds the S ranks' values in
    // rank order, read straight from their shared memory (distributed shared
    // memory, 16 bytes per load), and writes them to y with consecutive
    // threads on consecutive columns.  A second barrier keeps each tile in
    // place until every rank has read it.
    // Row pitch of the shared tile: 260 floats keeps every row on a 16-byte
    // boundary, and eight lanes of consecutive tokens storing 16 bytes at
    // the same column land on eight distinct bank groups.
    constexpr int kPitch = kTcRows + 4;
    float *ysm = reinterpret_cast<float *>(smem);
    const int quarter = warp & 3, cq = warp >> 2;
    const int tok = 32 * quarter + lane;
    if (warp < kTcDqWarps && 32 * quarter < T) {  // warp-uniform
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            float v[16];
            if (have_acc && nchunks > 0) {
                tc_ld16(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(64 * cq + 16 * g), v);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            }
            if (tok < T) {
                float4 *dst = reinterpret_cast<float4 *>(ysm + tok * kPitch + 64 * cq + 16 * g);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
        }
    }
    tc_fence_before();
    cluster_sync_all();
    {
        // Outputs in groups of four columns; rank r takes groups
        // [r·G/S, (r+1)·G/S) of the tile's G = T·64.
        constexpr int kGroupsPerRow = kTcRows / 4;
        const int n_g = T * kGroupsPerRow;
        const int g0 = rank * n_g / S, g1 = (rank + 1) * n_g / S;
        const int ncols = min(kTcRows, N - row0);
        const bool vec_y = (reinterpret_cast<uintptr_t>(y) & 15) == 0 && (N & 3) == 0;
        const uint32_t local = smem_addr(ysm);
        uint32_t tile_of[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) tile_of[s] = map_to_rank(local, (uint32_t)min(s, S - 1));
        // The output may be read by the previous kernel on the stream.
        pdl_wait();
        // kU groups per thread step, every remote load issued before the
        // adds so that their latencies overlap.
        constexpr int kU = 4;
        for (int i0 = g0 + (int)threadIdx.x; i0 < g1; i0 += kU * kTcThreads) {
            float4 v[4][kU];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = min(i0 + u * kTcThreads, g1 - 1);
                    const uint32_t off = 4u * (uint32_t)((i / kGroupsPerRow) * kPitch + 4 * (i % kGroupsPerRow));
                    v[s][u] = s < S ? ld_cluster_v4(tile_of[s] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + u * kTcThreads;
                if (i < g1) {
                    const int t = i / kGroupsPerRow, col = 4 * (i % kGroupsPerRow);
                    float4 acc = v[0][u];
#pragma unroll
                    for (int s = 1; s < 4; ++s) {
                        if (s < S) {
                            acc.x += v[s][u].x;
                            acc.y += v[s][u].y;
                            acc.z += v[s][u].z;
                            acc.w += v[s][u].w;
                        }
                    }
                    float *dst = y + (size_t)t * N + row0 + col;
                    if (vec_y && col + 3 < ncols) {
                        *reinterpret_cast<float4 *>(dst) = acc;
                    } else {
                        if (col < ncols) dst[0] = acc.x;
                        if (col + 1 < ncols) dst[1] = acc.y;
                        if (col + 2 < ncols) dst[2] = acc.z;
                        if (col + 3 < ncols) dst[3] = acc.w;
                    }
                }
            }
        }
    }
    cluster_sync_all();
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
cudaError_t launch_tile(const LaunchCtx &c, const __nv_bfloat16 *xb, const float *x, const uint8_t *W, float *y,
                        int K, int N, int T, int S) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    alignas(64) CUtensorMap tm_w, tm_x;
    std::memset(&tm_x, 0, sizeof(tm_x));
    const cuuint64_t row_bytes = (cuuint64_t)(K / kQ4kValues) * kQ4kBytes;
    {
        const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)N};
        const cuuint64_t strides[1] = {row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)kQ4kBytes, (cuuint32_t)kTcRows};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(W), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
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
    auto kernel = xb ? q4k_mm_tc_kernel<0> : (T <= 64 ? q4k_mm_tc_kernel<2> : q4k_mm_tc_kernel<4>);
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
    return cudaLaunchKernelEx(&cfg, kernel, tm_w, tm_x, x, y, K, N, T, c.status, c.wait_limit, c.withhold);
}

// Tiles of 128 tokens over the bf16 copy xb of x (several tiles), or one
// tile that rounds x itself (xb == nullptr, at most 128 tokens).
cudaError_t launch_tiles(const LaunchCtx &c, const float *x, __nv_bfloat16 *xb, const uint8_t *W, float *y, int K,
                         int N, int T, int S) {
    if (!xb) return launch_tile(c, nullptr, x, W, y, K, N, T, S);
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
        e = launch_tile(c, xb + (size_t)t0 * K, nullptr, W, y + (size_t)t0 * N, K, N, tt, S);
    }
    return e;
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

cudaError_t launch_q4k_mm_tc(const LaunchCtx &c, const float *x, const uint8_t *W, float *y, int K,
                             int N, int T) {
    const int S = tc_split(K);
    if (S == 0) return cudaErrorNotSupported;
    // Up to 128 tokens: one launch that rounds x itself, nothing allocated.
    // More: x is rounded to bf16 once into stream-ordered scratch (freed on
    // the same stream after the last tile) and the weights are re-read once
    // per tile of 128 tokens.
    const size_t bytes = q4k_mm_tc_scratch_bytes(K, N, T);
    if (bytes == 0) return launch_tiles(c, x, nullptr, W, y, K, N, T, S);
    void *scratch = nullptr;
    cudaError_t e = cudaMallocAsync(&scratch, bytes, c.stream);
    if (e != cudaSuccess) return e;
    e = launch_tiles(c, x, static_cast<__nv_bfloat16 *>(scratch), W, y, K, N, T, S);
    const cudaError_t ef = cudaFreeAsync(scratch, c.stream);
    return e != cudaSuccess ? e : ef;
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
    return launch_tiles(c, x, bytes ? reinterpret_cast<__nv_bfloat16 *>(scratch) : nullptr, W, y, K, N, T, S);
}

}  // namespace q4mm
