// Launch geometry of the one-token GEMV kernel (gemv_t1_kernel in
// q4k_gemv.cu): CTA rows, ring stages and depth, shared-memory layout.
// Plain host C++ (no CUDA types), so that the CPU tests compile this same
// header and check its invariants over many shapes.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

namespace q4mm {

// Geometry knobs (the library reads them from the environment once):
// compute warps per CTA, resident CTAs per SM, bytes per ring slot, ring
// budget, stages issued before the wait, largest x staged by one bulk copy,
// L2 policy of the weight stream, grid cap, spare SMs of short launches.
struct T1Tuning {
    int warps = 16;
    int ctas_per_sm = 1;
    int stage_bytes = 16384;
    int ring_bytes = 200 * 1024;
    int pre_stages = 0;        // weight stages issued before the activation copy
    int x_stage_max = 65536;   // bytes of x staged by a bulk copy (0: plain loads)
    int l2_evict_first = 1;    // weight copies with the L2 evict_first policy
    int max_grid = 0;          // CTAs per launch at most (0: no limit)
    int spare_sms = 4;         // SMs left without a CTA of a short launch
    int spare_max_bytes = 256 * 1024;  // "short": at most this many weight bytes per CTA
};

constexpr int kT1MaxCw = 16;           // compute warps at most
constexpr int kT1PlaneSlabBytes = 208; // byte planes of 64 activations, padded

struct T1Geometry {
    int ok = 0;            // 0: the kernel cannot take this shape
    int wide = 0;          // a row spans several warps
    int wc = 1;            // warps per row
    int pass_rows = 2;     // rows of one pass (whole CTA)
    int rg = 1;            // row groups per token
    int ncw = 0;           // compute warps
    int rq = 1;            // rows whose bytes are a multiple of 16
    int stage_rows = 0;    // rows per ring slot
    int rows_per_cta = 0;
    int grid = 0;
    int x_staged = 0;      // x arrives by one bulk copy
    int nslots = 0;        // ring depth
    int pre_stages = 0;
    size_t xs_bytes = 0;   // planes, sums, block scales and (staged) x
    size_t part_bytes = 0; // per-row partial sums of wide rows / SwiGLU
    size_t slot_bytes = 0;
    size_t smem = 0;       // dynamic shared memory per CTA
};

inline int t1_next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Row group r takes passes r, r + rg, r + 2·rg, … (pps passes per stage) and
// waits on the full barrier of each stage it has a pass in, by phase parity.
// A wait on a reused slot is sound when the group itself consumed the slot's
// previous stage: that phase has then completed and the parity names the
// stage awaited.  Otherwise a previous stage that has not landed yet has the
// other parity, the wait returns at once and the group would read the old
// contents.  True when every wait of every group is sound that way.
inline bool t1_ring_covered(int npasses, int pps, int rg, int nslots) {
    const int nstages = (npasses + pps - 1) / pps;
    if (nslots >= nstages) return true;          // no slot is reused
    if (pps % rg == 0) return true;              // every group has a pass in every stage
    if (rg % pps == 0) return nslots % (rg / pps) == 0;  // group r: stages r/pps + i·rg/pps
    std::vector<char> seen(nstages);
    for (int r = 0; r < rg; ++r) {
        for (int s = 0; s < nstages; ++s) seen[s] = 0;
        for (int p = r; p < npasses; p += rg) {
            const int st = p / pps;
            if (st >= nslots && !seen[st - nslots]) return false;
            seen[st] = 1;
        }
    }
    return true;
}

// group_bytes: bytes per 256 values of a row in the format (144 Q4_K and
// Q4_0, 210 Q6_K, 64 ternary).  vrow_mult: 2 for the fused gate+up (the
// gate rows and then the same rows of the up weight through one ring).
inline T1Geometry plan_gemv_t1(int group_bytes, int K, int N, int T, int vrow_mult, int num_sms,
                               int max_smem_optin, const T1Tuning &tun) {
    T1Geometry g;
    const int nb = K / 256;
    const int row_bytes = nb * group_bytes;
    const int L = 4 * nb;  // slab lanes per row
    g.wide = L > 32;
    g.wc = g.wide ? (L + 31) / 32 : 1;
    g.pass_rows = g.wide ? 2 : 2 * (32 / t1_next_pow2(L > 4 ? L : 4));
    // At most kT1MaxCw compute warps: wider rows go to another kernel.
    if (g.wc > kT1MaxCw) return g;
    // Each token gets warps / T compute warps: whole rows (wc warps each).
    if (tun.warps / T < g.wc) return g;
    g.rg = (tun.warps / T) / g.wc;
    g.ncw = T * g.wc * g.rg;
    // Stage: whole passes, at least stage_bytes of weights (bulk copies of
    // 16 KB and more run at full HBM bandwidth).  A row size off the 16-byte
    // grid (Q6_K) keeps CTA and stage boundaries on multiples of rq rows,
    // the fewest whose bytes are a multiple of 16 (row_bytes = 2·odd·nb, so
    // rq = 8 / gcd(nb, 8)).
    if (row_bytes % 16) {
        g.rq = 8;
        while (g.rq > 1 && (g.rq / 2) * row_bytes % 16 == 0) g.rq /= 2;
    }
    const int sq = g.pass_rows > g.rq ? g.pass_rows : g.rq;  // both powers of two
    int stage_rows = sq * ((tun.stage_bytes + sq * row_bytes - 1) / (sq * row_bytes));
    if (stage_rows < sq) stage_rows = sq;

    // Grid.  A CTA of the next launch on the stream can only start where a
    // CTA of this one has exited, and one that starts after this launch has
    // completed gets through its wait on it ~0.7 µs later than the CTAs
    // already resident: with a CTA on every SM, the CTAs of each launch that
    // start last also finish last and delay the next launch the same way.
    // For a short launch (few weight bytes per CTA) leaving spare_sms SMs
    // free lets every CTA of the next launch be resident before this one
    // completes; a long launch keeps every SM for the weight stream.
    int grid = tun.ctas_per_sm * num_sms;
    const double cta_bytes = (double)vrow_mult * N * row_bytes / grid;
    if (cta_bytes <= tun.spare_max_bytes) grid = grid - tun.spare_sms > 1 ? grid - tun.spare_sms : 1;
    if (tun.max_grid > 0 && tun.max_grid < grid) grid = tun.max_grid;
    int rows = (N + grid - 1) / grid;
    rows = (rows + g.rq - 1) / g.rq * g.rq;
    if (rows < g.pass_rows) rows = g.pass_rows;
    g.rows_per_cta = rows;
    g.grid = (N + rows - 1) / rows;

    const size_t TK = (size_t)T * K;
    const int vrows = vrow_mult * rows;
    const int npasses = (vrows + g.pass_rows - 1) / g.pass_rows;
    // Ring for a given stage size: x staging, fixed areas, depth.
    auto ring = [&](int srows) {
        if (srows > rows) srows = sq * ((rows + sq - 1) / sq);
        g.stage_rows = srows;
        g.slot_bytes = (size_t)srows * row_bytes;
        g.x_staged = TK * sizeof(float) <= (size_t)tun.x_stage_max ? 1 : 0;
        // Large rows at an 8-row stage quantum can leave no room for x: then
        // the compute threads load x themselves.
        if (g.x_staged && TK * sizeof(float) + 2 * g.slot_bytes + (TK / 64) * kT1PlaneSlabBytes >
                              (size_t)max_smem_optin - 8192)
            g.x_staged = 0;
        g.xs_bytes = (TK / 64) * kT1PlaneSlabBytes + (TK / 32 + TK / 16) * sizeof(float) +
                     (size_t)((T * nb * 4 + 15) & ~15) + (g.x_staged ? TK * sizeof(float) : 0);
        g.part_bytes = (g.wide || vrow_mult > 1) ? (size_t)T * vrows * g.wc * sizeof(float) : 0;
        const size_t fixed = g.xs_bytes + g.part_bytes + 2 * 8 * sizeof(uint64_t);
        const size_t budget = tun.ring_bytes;
        int n = (int)((budget > fixed ? budget - fixed : 0) / g.slot_bytes);
        const int stages_needed = (vrows + srows - 1) / srows;
        const int cap = stages_needed < 8 ? stages_needed : 8;
        n = n < cap ? n : cap;
        return n > 2 ? n : 2;
    };
    const int nslots_max = ring(stage_rows);
    // Ring depth and row groups: the deepest ring whose every reuse is
    // covered (see t1_ring_covered); where no depth of two or more is, fewer
    // row groups (one row group, or any count dividing the passes of a
    // stage, has a pass in every stage and covers every depth).
    const int pps = g.stage_rows / g.pass_rows;
    int nslots = nslots_max;
    for (;;) {
        nslots = nslots_max;
        while (nslots >= 2 && !t1_ring_covered(npasses, pps, g.rg, nslots)) --nslots;
        if (nslots >= 2 || g.rg == 1) break;
        --g.rg;
    }
    if (nslots < 2) return g;
    g.ncw = T * g.wc * g.rg;
    g.nslots = nslots;
    // With plain activation loads nothing needs to go out ahead of the rest.
    g.pre_stages = g.x_staged ? tun.pre_stages : nslots;
    g.smem = g.xs_bytes + (size_t)nslots * g.slot_bytes + 2 * nslots * sizeof(uint64_t) + g.part_bytes;
    if (g.smem > (size_t)max_smem_optin) return g;
    g.ok = 1;
    return g;
}

}  // namespace q4mm
