// Q4_K decode GEMV for 3..8 tokens (FP32 register tiles; also 1..2 where the
// one-token kernel's geometry does not fit), sm_103a.
//
// Computes y[t][o] = Σ_k x[t][k]·w[o][k] with w = d·sc_s·q − dmin·m_s decoded
// on the fly from the 144-byte Q4_K super-blocks (SKaiNET PR #562
// "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
// section "Pipeline"); each weight is dequantized once and used by every
// token, so the weights stream from HBM once per call.
//
// Nibble decode: a masked code q in byte k of a word becomes the float
// 0.5 + q/256 with one byte permute (see nib_biased).  The bias 0.5·Σx is
// removed together with the lazy min term: per sub-block s the contribution
// is (256·d·sc_s)·acc_s − (128·d·sc_s + dmin·m_s)·Σx_s where
// acc_s = Σ x·(0.5 + q/256); here the dequantized weight
// scale'·(0.5 + q/256) − offset' is formed once and multiplied into every
// token's accumulator.
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "multi_geometry.h"
#include "sync.cuh"

namespace q4mm {

namespace {

// ----------------------------------------------------------------------------
// Block scales of one lane
// ----------------------------------------------------------------------------

// Constants of slab j (the two sub-blocks 2j and 2j+1) of a block, decoded
// into a warp's scale table: scale' = 256·d·sc and offset' = 128·d·sc + dmin·m.
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
// Row groups in a bulk-copy ring, word lanes, register tiles
// ----------------------------------------------------------------------------
//
// A CTA owns a contiguous range of rows in groups of four; the producer warp
// streams each group (four whole rows) into its own ring slot with a bulk
// copy (the first lap's copies one per lane, the refills from lane 0).
// Compute warp c takes groups c, c + n, … (n consumer warps, see the
// kernel), and for each group
// walks all blocks of the rows:
// lane l owns qs word l of every block — 4 low-nibble weights of sub-block
// 2j and 4 high-nibble weights of 2j+1 (j = l/8) — with the 8 matching
// activations of all TT tokens loaded once per block and reused by the four
// rows.  Each weight is dequantized once (scale'·(0.5 + q/256) − offset') and
// multiplied into TT token accumulators (TT ∈ {2, 3, 4, 6, 8}), two
// positions per paired FMA.  A butterfly over the 4·TT sums (padded to a
// power of two) at the end of the group finishes the rows.
//
// The eight lanes of a slab share its two sub-blocks' scale' and offset', so
// the warp decodes the block headers once into its own shared table (4 rows
// × kMultiTabBlocks blocks × 4 slabs of (s0, o0, s1, o1)) before walking
// those blocks, and each lane then reads its pair with one 16-byte load.

struct MultiParams {
    const float *x;
    const uint8_t *W;
    const uint8_t *W2;  // kSwiGLU: the up weight (W is the gate weight)
    float *y;
    int *status;
    int K, N, T;       // T: tokens of this launch (<= TT)
    int nb;            // blocks per row
    int rows_per_cta;  // multiple of kMultiRows
    int nslots;        // ring depth (groups in flight)
    long long wait_limit;  // SM cycles a bounded wait lasts at most
    int withhold;          // test only: a group whose copy is never issued (-1: none)
};

// kXs: x is staged in shared memory by one bulk copy (its T·K fp32 values
// fit beside the ring), so the per-block activation loads are shared-memory
// loads instead of L2 round trips.

// kSplit (up to 4 tokens): each group is taken by a pair of compute warps,
// the first over blocks [0, nb/2) of its rows, the second over the rest; the
// second hands its partial sums to the first through shared memory, which
// adds them (first + second, so the result does not depend on timing) and
// stores the rows.  Twice the warps hide more of each warp's latencies.

// kSwiGLU: the fused Llama FFN input side, y = silu(x·Wᵀ) ⊙ (x·W2ᵀ): a
// ring slot holds a group's four gate rows and then the same four rows of
// the up weight; a warp takes the gate part and then the up part of its
// group and combines the two sums of each row.

template <int TT, bool kXs, bool kSplit, bool kSwiGLU>
__global__ void __launch_bounds__(32 * (kSplit ? kMultiSplitWarps : kMultiWarps), 1)
    q4k_gemv_multi_kernel(MultiParams p) {
    constexpr int kParts = kSwiGLU ? 2 : 1;
    extern __shared__ __align__(128) uint8_t msmem[];
    __shared__ volatile int abort_flag;  // set by the first warp whose wait runs out
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t row_bytes = (uint32_t)p.nb * kQ4kBytes;
    const uint32_t slot_bytes = kParts * kMultiRows * row_bytes;
    float4 *tabs = reinterpret_cast<float4 *>(msmem);  // the compute warps' tables
    float *pair_buf = reinterpret_cast<float *>(msmem + kMultiCw * kMultiTabBytes);  // [pair][2][32]
    uint64_t *pair_bar = reinterpret_cast<uint64_t *>(pair_buf + kMultiCw * 2 * 32);  // [pair][2]
    uint8_t *ring = msmem + kMultiCw * kMultiTabBytes + kMultiPairBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)p.nslots * slot_bytes);
    uint64_t *empty = full + p.nslots;
    uint64_t *x_bar = empty + p.nslots;
    float *xs = reinterpret_cast<float *>(x_bar + 2);  // [T][K] when staged
    const int row0 = blockIdx.x * p.rows_per_cta;
    const int nrows = min(p.rows_per_cta, p.N - row0);
    const int ngroups = (nrows + kMultiRows - 1) / kMultiRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kSplit ? 2 : 1);  // both warps of a pair
        }
        if (kSplit)
            for (int i = 0; i < 2 * kMultiCw; ++i) mbar_init(&pair_bar[i], 1);
        mbar_init(x_bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == 0) {
        // (A test may ask for one group never to arrive, to see a wait run
        // out; nothing then writes into its slot.)
        auto issue = [&](int g, int slot) {
            const uint32_t bytes = (uint32_t)min(kMultiRows, nrows - g * kMultiRows) * row_bytes;
            const size_t off = (size_t)(row0 + g * kMultiRows) * row_bytes;
            uint8_t *dst = ring + (size_t)slot * slot_bytes;
            mbar_arrive_expect_tx(&full[slot], kParts * bytes);
            bulk_g2s(dst, p.W + off, bytes, &full[slot]);
            if (kSwiGLU) bulk_g2s(dst + kMultiRows * row_bytes, p.W2 + off, bytes, &full[slot]);
        };
        // Staged x first (the previous kernel on the stream may write it),
        // then the ring's first groups, one lane each: a bulk copy holds its
        // issuing thread for a few hundred cycles, so one thread issuing
        // them in turn would delay the last by thousands.  Then the rest of
        // the groups as slots free up, from lane 0.
        const int first = min(ngroups, p.nslots);
        if (kXs && lane == 0) {
            pdl_wait();
            mbar_arrive_expect_tx(x_bar, (uint32_t)(p.T * p.K) * sizeof(float));
            bulk_g2s(xs, p.x, (uint32_t)(p.T * p.K) * sizeof(float), x_bar);
        }
        __syncwarp();
        if (lane < first && lane != p.withhold) issue(lane, lane);
        __syncwarp();
        if (lane == 0) {
            int issued = first;
            for (int g = first; g < ngroups; ++g, ++issued) {
                const int slot = g % p.nslots;
                if (!mbar_wait_abortable(&empty[slot], ((g / p.nslots) - 1) & 1, p.wait_limit, &abort_flag)) {
                    abort_flag = 1;
                    flag_timeout(p.status);
                    break;
                }
                if (g != p.withhold) issue(g, slot);
            }
            // Never leave a copy writing into an exiting CTA: the last
            // groups issued (a withheld one has nothing in flight), and x.
            for (int g = max(0, issued - p.nslots); g < issued; ++g)
                if (g != p.withhold)
                    (void)mbar_wait_bounded(&full[g % p.nslots], (g / p.nslots) & 1, p.wait_limit);
            if (kXs) (void)mbar_wait_bounded(x_bar, 0, p.wait_limit);
        }
        __syncwarp();
        return;
    }

    // Consumers: min(kMultiCw, nslots) warps taking groups in turn, with
    // nslots a multiple of their count (the launcher rounds it), so that
    // slot s belongs to warp s mod ncons alone.  A warp's successive groups
    // in its slot are then one ring lap apart and it has consumed the
    // slot's previous phase itself, so its parity wait can never match an
    // older phase (a warp reaching group g before group g − nslots, held by
    // another warp, has landed would read the slot's previous contents).
    //
    // With kSplit the consumers are pairs of warps (the slot rule holds per
    // pair), and the first warp of a pair releases its slot only after it
    // has read the second's partial sums of the group: the second can then
    // be at most one group ahead, so each of the pair's two buffers (group
    // parity) and barriers is reused only after its previous use is done.
    const int ncons = min(kMultiCw, p.nslots);
    const int cw = warp - 1;
    const int unit = kSplit ? cw >> 1 : cw;  // the pair (kSplit) or the warp
    const bool second = kSplit && (cw & 1);  // the pair's second warp
    if (unit >= ncons) return;
    const int kb0 = second ? p.nb / 2 : 0, kb1 = (kSplit && !second) ? p.nb / 2 : p.nb;  // this warp's blocks
    const int j = lane >> 3, wq = lane & 7;   // slab and word within it
    // x may be produced by the previous kernel on the stream.
    pdl_wait();
    if (kXs && !__all_sync(0xffffffffu, mbar_wait_abortable(x_bar, 0, p.wait_limit, &abort_flag))) {
        abort_flag = 1;
        flag_timeout(p.status);
        return;
    }
    const float *xsrc = kXs ? xs : p.x;
    constexpr int kTB = kSplit ? kMultiTabBlocks / 2 : kMultiTabBlocks;  // blocks per table chunk
    constexpr int kTabEntries = kMultiRows * kTB * 4;
    float4 *tab = tabs + (size_t)cw * kTabEntries;
    float *pbuf = pair_buf + unit * 2 * 32;
    uint64_t *pbar = pair_bar + unit * 2;
    int lg = 0;  // this pair's (warp's) group count so far
    for (int g = unit; g < ngroups; g += ncons, ++lg) {
        const int slot = g % p.nslots;
        if (!__all_sync(0xffffffffu, mbar_wait_abortable(&full[slot], (g / p.nslots) & 1, p.wait_limit, &abort_flag))) {
            abort_flag = 1;
            flag_timeout(p.status);
            break;
        }
        const uint8_t *grp = ring + (size_t)slot * slot_bytes;
        const int rows = min(kMultiRows, nrows - g * kMultiRows);
        constexpr int TP = TT <= 2 ? 2 : TT <= 4 ? 4 : 8;
        constexpr int V = kMultiRows * TP;
        static_assert(V <= 32, "one value per writer lane");
        float res0 = 0.f, res1 = 0.f;  // this lane's row sum of the gate (or only) part and of the up part
        int idx = 0;                   // the value index it belongs to
#pragma unroll 1
        for (int part = 0; part < kParts; ++part) {
            const uint8_t *base = grp + (size_t)part * kMultiRows * row_bytes;
            float2 acc[kMultiRows][TT];
#pragma unroll
            for (int r = 0; r < kMultiRows; ++r)
#pragma unroll
                for (int t = 0; t < TT; ++t) acc[r][t] = make_float2(0.f, 0.f);

            for (int b0 = kb0; b0 < kb1; b0 += kTB) {
                const int nbc = min(kTB, kb1 - b0);
                // Entry e = (r·kTB + bb)·4 + slab; every lane keeps its
                // slab (e mod 4 = lane mod 4), so the table fill is branch-free.
                __syncwarp();  // the previous chunk's reads are done
#pragma unroll
                for (int i = 0; i < kTabEntries / 32; ++i) {
                    const int e = lane + 32 * i;
                    const int bb = (e >> 2) % kTB, r = e / (4 * kTB);
                    if (bb < nbc) {
                        const uint8_t *blk = base + (size_t)(r < rows ? r : 0) * row_bytes + (size_t)(b0 + bb) * kQ4kBytes;
                        const SlabScales sc = slab_scales(*reinterpret_cast<const uint4 *>(blk), e & 3);
                        tab[e] = make_float4(sc.s0, sc.o0, sc.s1, sc.o1);
                    }
                }
                __syncwarp();
                for (int bb = 0; bb < nbc; ++bb) {
                    const int b = b0 + bb;
                    // Activations of this lane's 8 positions for every token.
                    float4 xl[TT], xh[TT];
                    const int k0 = b * kQ4kValues + 64 * j + 4 * wq;
#pragma unroll
                    for (int t = 0; t < TT; ++t) {
                        if (t < p.T) {
                            const float *xt = xsrc + (size_t)t * p.K + k0;
                            if constexpr (kXs) {
                                xl[t] = *reinterpret_cast<const float4 *>(xt);
                                xh[t] = *reinterpret_cast<const float4 *>(xt + 32);
                            } else {
                                xl[t] = __ldg(reinterpret_cast<const float4 *>(xt));
                                xh[t] = __ldg(reinterpret_cast<const float4 *>(xt + 32));
                            }
                        } else {
                            xl[t] = make_float4(0.f, 0.f, 0.f, 0.f);
                            xh[t] = xl[t];
                        }
                    }
#pragma unroll
                    for (int r = 0; r < kMultiRows; ++r) {
                        // Absent rows of a short last group read row 0 of the slot;
                        // their sums are never stored.
                        const uint8_t *blk = base + (size_t)(r < rows ? r : 0) * row_bytes + (size_t)b * kQ4kBytes;
                        const uint32_t q = *reinterpret_cast<const uint32_t *>(blk + 16 + 32 * j + 4 * wq);
                        const float4 sc = tab[(r * kTB + bb) * 4 + j];  // (s0, o0, s1, o1)
                        const uint32_t l4 = q & 0x0F0F0F0Fu;
                        const uint32_t h4 = (q >> 4) & 0x0F0F0F0Fu;
                        const float2 s0 = make_float2(sc.x, sc.x), n0 = make_float2(-sc.y, -sc.y);
                        const float2 s1 = make_float2(sc.z, sc.z), n1 = make_float2(-sc.w, -sc.w);
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
            }
            // Butterfly over the 4·TP sums (TP: TT rounded up to a power of two,
            // the padding sums zero): afterwards lane l holds value index
            // idx .. idx + n − 1 (see the halving below), summed over the warp.
            float v[V];
#pragma unroll
            for (int r = 0; r < kMultiRows; ++r)
#pragma unroll
                for (int t = 0; t < TP; ++t) v[r * TP + t] = t < TT ? acc[r][t].x + acc[r][t].y : 0.f;
            idx = 0;
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
            if (part == 0)
                res0 = v[0];
            else
                res1 = v[0];
        }
        __syncwarp();
        if (lane == 0 && (!kSplit || second)) mbar_arrive(&empty[slot]);
        const bool writer = V >= 32 || (lane & (32 / V - 1)) == 0;
        if constexpr (kSplit) {
            static_assert(V <= 16, "a pair buffer part holds 16 sums");
            float *pb = pbuf + (lg & 1) * 32;
            if (second) {
                if (writer) {
                    pb[idx] = res0;
                    if (kSwiGLU) pb[16 + idx] = res1;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&pbar[lg & 1]);
                continue;
            }
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&pbar[lg & 1], (lg >> 1) & 1, p.wait_limit, &abort_flag))) {
                abort_flag = 1;
                flag_timeout(p.status);
                break;
            }
            if (writer) {
                res0 += pb[idx];
                if (kSwiGLU) res1 += pb[16 + idx];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        if (writer) {
            const int r = idx / TP, t = idx % TP;
            float out = res0;
            if constexpr (kSwiGLU) out = out / (1.0f + expf(-out)) * res1;  // silu(g)·u
            if (r < rows && t < p.T) p.y[(size_t)t * p.N + row0 + g * kMultiRows + r] = out;
        }
    }
}

}  // namespace

namespace {

template <bool kSwiGLU>
cudaError_t launch_multi(const LaunchCtx &c, const float *x, const uint8_t *W, const uint8_t *W2, float *y, int K,
                         int N, int T) {
    MultiParams p;
    p.x = x;
    p.W = W;
    p.W2 = W2;
    p.y = y;
    p.status = c.status;
    p.K = K;
    p.N = N;
    p.T = T;
    p.nb = K / kQ4kValues;
    p.wait_limit = c.wait_limit;
    p.withhold = c.withhold;
    const MultiGeometry g =
        plan_gemv_multi(K, N, c.num_sms, c.max_smem_optin, kMultiRingBytes, T, kSwiGLU ? 2 : 1);
    if (!g.ok) return cudaErrorNotSupported;
    p.rows_per_cta = g.rows_per_cta;
    p.nslots = g.nslots;
    const int grid = g.grid;
    const size_t smem = g.smem;

#define Q4MM_MULTI_CASE(TT, SPLIT)                                                                    \
    {                                                                                                 \
        auto kernel = g.x_staged ? q4k_gemv_multi_kernel<TT, true, SPLIT, kSwiGLU>                    \
                                 : q4k_gemv_multi_kernel<TT, false, SPLIT, kSwiGLU>;                  \
        cudaError_t e = ensure_smem(kernel, smem);                                                    \
        if (e != cudaSuccess) return e;                                                               \
        return launch_kernel(c, kernel, dim3(grid), dim3(32 * (SPLIT ? kMultiSplitWarps : kMultiWarps)), \
                             smem, p);                                                                \
    }
    if constexpr (!kSwiGLU) {
        if (T <= 2) Q4MM_MULTI_CASE(2, true)
        if (T <= 3) Q4MM_MULTI_CASE(3, true)
        if (T <= 4) Q4MM_MULTI_CASE(4, true)
        if (T <= 6) Q4MM_MULTI_CASE(6, false)
        if (T <= 8) Q4MM_MULTI_CASE(8, false)
    } else {
        if (T <= 4) Q4MM_MULTI_CASE(4, true)
        if (T <= 8) Q4MM_MULTI_CASE(8, false)
    }
#undef Q4MM_MULTI_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_q4k_gemv_multi(const LaunchCtx &c, const float *x, const uint8_t *W, float *y,
                                  int K, int N, int T) {
    return launch_multi<false>(c, x, W, nullptr, y, K, N, T);
}

cudaError_t launch_q4k_ffn_swiglu_multi(const LaunchCtx &c, const float *x, const uint8_t *Wg, const uint8_t *Wu,
                                        float *h, int K, int N, int T) {
    return launch_multi<true>(c, x, Wg, Wu, h, K, N, T);
}

}  // namespace q4mm
