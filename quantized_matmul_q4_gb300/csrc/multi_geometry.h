// Launch geometry of the 2-8 token Q4_K GEMV kernel (q4k_gemv_multi.cu):
// CTA rows and the weight ring.  Plain host C++ (no CUDA types), so that the
// CPU tests compile this same header and check its invariants.
#pragma once

#include <cstddef>
#include <cstdint>

namespace q4mm {

constexpr int kMultiWarps = 8;  // copy warp + 7 compute warps
constexpr int kMultiCw = kMultiWarps - 1;
constexpr int kMultiRows = 4;   // rows per group (one ring slot)
constexpr int kMultiRingBytes = 200 * 1024;  // ring budget the library launches with
constexpr int kMultiTabBlocks = 16;          // blocks per scale-table chunk
// Per compute warp: the decoded (scale', offset') of 8 sub-blocks of 4 rows ×
// kMultiTabBlocks blocks, fp32 pairs.  (Up to 4 tokens a group is taken by a
// pair of warps, each over half of the row's blocks, with tables of half
// that many blocks: the same bytes for twice the warps.)
constexpr size_t kMultiTabBytes = (size_t)kMultiRows * kMultiTabBlocks * 8 * 2 * sizeof(float);
constexpr int kMultiSplitWarps = 1 + 2 * kMultiCw;  // copy warp + a pair per consumer (up to 4 tokens)
// The pairs' exchange of partial sums: per pair two buffers of 32 floats
// (16 sums of each of up to two weights) and two barriers, padded to 2 KB.
constexpr size_t kMultiPairBytes = 2048;

struct MultiGeometry {
    int ok = 0;            // 0: the ring does not fit shared memory
    int grid = 0;
    int rows_per_cta = 0;  // multiple of kMultiRows
    int nslots = 0;        // ring depth (groups in flight)
    int consumers = 0;     // compute warps that take groups: min(kMultiCw, nslots)
    int x_staged = 0;      // x copied into shared memory (T·K fp32 beside the ring)
    size_t smem = 0;       // dynamic shared memory per CTA
};

// Shared memory: the compute warps' scale tables | pair exchange | ring |
// barriers | x.
// ring_bytes: byte budget of the ring (the library passes kMultiRingBytes; the
// CPU tests also check smaller budgets).  T: tokens (x is staged in shared
// memory when its T·K fp32 values fit beside a ring of one slot per
// consumer warp; T = 0 never stages).  vrow_mult: 2 for the fused gate+up
// (a slot holds the group's rows of both weights).
inline MultiGeometry plan_gemv_multi(int K, int N, int num_sms, int max_smem_optin, int ring_bytes, int T = 0,
                                     int vrow_mult = 1) {
    MultiGeometry g;
    const size_t row_bytes = (size_t)(K / 256) * 144;
    const size_t slot_bytes = (size_t)vrow_mult * kMultiRows * row_bytes;  // a group's rows of each weight
    const int groups = (N + kMultiRows - 1) / kMultiRows;
    const int grid = num_sms < groups ? num_sms : groups;
    g.rows_per_cta = kMultiRows * ((groups + grid - 1) / grid);
    g.grid = (N + g.rows_per_cta - 1) / g.rows_per_cta;
    const int cta_groups = g.rows_per_cta / kMultiRows;
    const size_t bars = 2 * sizeof(uint64_t);  // x barrier (+ padding)
    const size_t tab = (size_t)kMultiCw * kMultiTabBytes + kMultiPairBytes;  // scale tables, pair exchange
    const size_t x_bytes = (size_t)T * K * sizeof(float);
    auto plan = [&](size_t budget) {
        // Ring: up to budget, at least two slots, never more slots than groups.
        size_t fit = budget / slot_bytes;
        if (fit < 2) fit = 2;
        int n = cta_groups < 16 ? cta_groups : 16;
        if ((size_t)n > fit) n = (int)fit;
        const int least = cta_groups < 2 ? cta_groups : 2;
        if (n < least) n = least;
        // Every slot has one consumer warp (see the kernel): from kMultiCw slots
        // on, a multiple of kMultiCw; below that, one warp per slot.
        if (n >= kMultiCw) n = n / kMultiCw * kMultiCw;
        g.nslots = n;
        g.consumers = n < kMultiCw ? n : kMultiCw;
        g.smem = tab + (size_t)n * slot_bytes + 2 * (size_t)n * sizeof(uint64_t) + bars;
    };
    const int want_slots = cta_groups < kMultiCw ? cta_groups : kMultiCw;
    if (T > 0 && tab + x_bytes + (size_t)want_slots * slot_bytes + 2 * (size_t)want_slots * sizeof(uint64_t) + bars +
                         1024 <=
                     (size_t)max_smem_optin) {
        plan((size_t)max_smem_optin - 1024 - tab - x_bytes - bars - 2 * 16 * sizeof(uint64_t));
        g.x_staged = 1;
        g.smem += x_bytes;
    } else {
        const size_t room = (size_t)max_smem_optin - 1024 - tab - bars - 2 * 16 * sizeof(uint64_t);
        plan((size_t)ring_bytes < room ? (size_t)ring_bytes : room);
    }
    g.ok = g.smem <= (size_t)max_smem_optin ? 1 : 0;
    return g;
}

}  // namespace q4mm
