// Launch geometry of the one-token GEMV kernel (gemv_t1_kernel in
// q4k_gemv.cu): CTA rows, ring stages and depth, shared-memory layout.
// Plain host C++ (no CUDA types), so that the CPU tests compile this same
// header and check its invariants over many shapes.
#pragma once

#include <cstddef>
#include <cstdint>

namespace q4mm {

// Geometry constants of the library's launches (the CPU tests use the same
// defaults).  A CTA has `warps` = 16 warps, all of them computing (a thread
// may then hold 128 registers: each SM sub-partition runs 4 of them); the
// ring's refills are issued by the warp that finishes a slot last.  One CTA
// per SM; the weights stream through a ring of stages in shared memory.
struct T1Tuning {
    int warps = 16;
    int stage_bytes = 16384;           // weight bytes per ring stage, at least
    int ring_bytes = 231424;           // shared-memory budget of a CTA (all but 1 KB)
    int x_stage_max = 65536;           // bytes of x staged by one bulk copy (0: plain loads)
    int l2_evict_first = 1;            // weight copies with the L2 evict_first policy
    int spare_sms = 4;                 // SMs left without a CTA of a short launch
    int spare_max_bytes = 256 * 1024;  // "short": at most this many weight bytes per CTA
};

constexpr int kT1Cw = 16;               // warps of a CTA (all compute)
constexpr int kT1Planes = 4;            // byte planes of the activation split
constexpr int kT1PlaneSlabBytes = 64 * kT1Planes + 16;  // the planes of 64 activations + 16 B padding
constexpr int kT1SlotRows = 4;          // rows a row slot (a warp's lanes of one row) takes per pass
constexpr int kT1SlotRowsWide = 2;      // the same where 4-row stages do not fit shared memory
constexpr int kT1MaxSlots = 16;         // ring depth at most

struct T1Geometry {
    int ok = 0;            // 0: the kernel cannot take this shape
    int cw = 0;            // warps of the launched kernel (kT1Cw)
    int wide = 0;          // a row spans several warps
    int wc = 1;            // warps per row
    int slot_rows = 4;     // rows a row slot takes per pass (kT1SlotRows or kT1SlotRowsWide)
    int pass_rows = 4;     // rows of one pass: slot_rows per row slot of a warp
    int rg = 1;            // row groups per token
    int ncw = 0;           // compute warps doing passes (<= cw)
    int stage_rows = 0;    // rows per ring slot (a multiple of pass_rows)
    int rows_per_cta = 0;
    int grid = 0;
    int x_staged = 0;      // x arrives by one bulk copy
    int nslots = 0;        // ring depth
    int nstages = 0;       // stages of the CTA's rows
    int pre_stages = 0;    // stages issued before the wait on the previous kernel
    size_t xs_bytes = 0;   // planes, group steps and sums, and (staged) x
    size_t part_bytes = 0; // per-row partial sums of wide rows / SwiGLU
    size_t slot_bytes = 0;
    size_t smem = 0;       // dynamic shared memory per CTA
};

inline int t1_next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Shared memory of the activation side: the byte planes of every 64 values,
// one step (and, for Q4_K's min term, one sum) per 32 values, and x itself
// when staged.
inline size_t t1_xs_bytes(size_t TK, int sums, bool x_staged) {
    return (TK / 64) * kT1PlaneSlabBytes + (TK / 32) * (sums ? 2 : 1) * sizeof(float) +
           (x_staged ? TK * sizeof(float) : 0);
}

// One form of the kernel: slot_rows rows per slot and pass.
inline T1Geometry plan_gemv_t1_form(int group_bytes, int sums, int K, int N, int T, int vrow_mult,
                                    int num_sms, int max_smem_optin, const T1Tuning &tun, int slot_rows) {
    T1Geometry g;
    g.cw = kT1Cw;
    g.slot_rows = slot_rows;
    const int warps = tun.warps;
    const int nb = K / 256;
    const int row_bytes = nb * group_bytes;
    const int L = 4 * nb;  // slab lanes per row
    g.wide = L > 32;
    g.wc = g.wide ? (L + 31) / 32 : 1;
    g.pass_rows = slot_rows * (g.wide ? 1 : 32 / t1_next_pow2(L > 4 ? L : 4));
    // At most `warps` compute warps: wider rows go to another kernel.
    if (g.wc > warps) return g;
    // Each token gets warps / T compute warps: whole rows (wc warps each).
    if (warps / T < g.wc) return g;
    g.rg = (warps / T) / g.wc;
    g.ncw = T * g.wc * g.rg;
    // Stage: whole passes, at least stage_bytes of weights (bulk copies of
    // 16 KB and more run at full HBM bandwidth).  A ring slot is refilled by
    // the warp that finishes its stage, and every consumer first waits for
    // the slot's stage tag to name the stage it wants before its parity wait,
    // so a ring of any depth is sound, whichever row group consumed a slot's
    // previous stage (without the tag, a ring whose depth is not a multiple
    // of the groups' stage stride measured up to 10% slower on 4096 → 11008:
    // its rings had to be cut to a depth where every wait followed the
    // waiting group's own consumption of the slot).  A row size off the 16-byte grid (Q6_K) lets a stage
    // start anywhere: its slot holds the bytes from the 16-byte boundary
    // below the stage's first byte, so it is 16 bytes longer.
    const size_t slot_pad = row_bytes % 16 ? 16 : 0;

    // Grid.  A CTA of the next launch on the stream can only start where a
    // CTA of this one has exited, and one that starts after this launch has
    // completed gets through its wait on it ~0.7 µs later than the CTAs
    // already resident: with a CTA on every SM, the CTAs of each launch that
    // start last also finish last and delay the next launch the same way.
    // For a short launch (few weight bytes per CTA) leaving spare_sms SMs
    // free lets every CTA of the next launch be resident before this one
    // completes; a long launch keeps every SM for the weight stream.
    int grid = num_sms;
    const double cta_bytes = (double)vrow_mult * N * row_bytes / grid;
    if (cta_bytes <= tun.spare_max_bytes) grid = grid - tun.spare_sms > 1 ? grid - tun.spare_sms : 1;
    int rows = (N + grid - 1) / grid;
    if (rows < g.pass_rows) rows = g.pass_rows;
    g.rows_per_cta = rows;
    g.grid = (N + rows - 1) / rows;

    const size_t TK = (size_t)T * K;
    const int vrows = vrow_mult * rows;
    g.x_staged = TK * sizeof(float) <= (size_t)tun.x_stage_max ? 1 : 0;
    g.part_bytes = (g.wide || vrow_mult > 1) ? (size_t)T * vrows * g.wc * sizeof(float) : 0;
    int nstages = 0, nslots = 0;
    // Per slot: the ring bytes, a full barrier, a counter of finished passes
    // and the stage it holds.
    auto smem_for = [&](int ns) {
        return g.xs_bytes + (size_t)ns * (g.slot_bytes + sizeof(uint64_t) + 2 * sizeof(int)) + g.part_bytes;
    };
    // Stages of sq rows (a multiple of sq, at least stage_bytes, at most the
    // CTA's rows rounded up), slots that fit the budget.
    auto plan_ring = [&](int sq) {
        int stage_rows = sq * ((tun.stage_bytes + sq * row_bytes - 1) / (sq * row_bytes));
        if (stage_rows < sq) stage_rows = sq;
        if (stage_rows > vrows) stage_rows = sq * ((vrows + sq - 1) / sq);
        g.stage_rows = stage_rows;
        g.slot_bytes = ((size_t)stage_rows * row_bytes + 15) / 16 * 16 + slot_pad;
        nstages = (vrows + stage_rows - 1) / stage_rows;
        // Large rows can leave no room for x: then the compute threads load
        // x themselves.
        if (g.x_staged && TK * sizeof(float) + 2 * g.slot_bytes + (TK / 64) * kT1PlaneSlabBytes >
                              (size_t)max_smem_optin - 8192)
            g.x_staged = 0;
        g.xs_bytes = t1_xs_bytes(TK, sums, g.x_staged != 0);
        const size_t fixed = smem_for(0);
        const size_t budget = (size_t)tun.ring_bytes;
        nslots = (int)((budget > fixed ? budget - fixed : 0) / (g.slot_bytes + 16));
        nslots = nslots < nstages ? nslots : nstages;
        nslots = nslots < kT1MaxSlots ? nslots : kT1MaxSlots;
    };
    plan_ring(g.pass_rows);
    if (nslots < nstages && nslots < 4 && g.x_staged) {
        // Staged x can cost the ring its fourth pass-sized slot (16384-wide
        // rows: 64 KB of x): the threads then load x themselves if that
        // gives four (16384²: 4658 against 4567 GB/s with two stages of a
        // pass of both row groups and x staged).
        g.x_staged = 0;
        plan_ring(g.pass_rows);
        if (nslots < nstages && nslots < 4) {
            g.x_staged = 1;
            plan_ring(g.pass_rows);
        }
    }
    if (nslots < nstages && nslots < 4) {
        // A ring of fewer than 4 pass-sized slots leaves each row group one
        // stage in flight at a time, idle while its next stage streams in:
        // then a stage holds a pass of every row group, all groups work on
        // the same stage and the other slot is prefetch (measured at 16384²:
        // 4587 GB/s against 3940 with 2-row passes and six slots).
        plan_ring(g.pass_rows * g.rg);
    }
    if (nslots < 2) nslots = nstages == 1 ? 1 : 2;
    // Last resort for very large stages: one slot, its stages in turn.
    if (smem_for(nslots) > (size_t)max_smem_optin) nslots = 1;
    g.ncw = T * g.wc * g.rg;
    g.nslots = nslots;
    g.nstages = nstages;
    // With plain activation loads nothing needs to go out ahead of the rest.
    g.pre_stages = g.x_staged ? 0 : nslots;
    g.smem = smem_for(nslots);
    if (g.smem > (size_t)max_smem_optin) return g;
    g.ok = 1;
    return g;
}

// group_bytes: bytes per 256 values of a row in the format (144 Q4_K and
// Q4_0, 210 Q6_K, 64 ternary); sums: 1 for Q4_K (group sums of x for the min
// term).  vrow_mult: 2 for the fused gate+up (the gate rows and then the
// same rows of the up weight through one ring).  Passes of 4 rows per slot
// where they fit, else of 2.
inline T1Geometry plan_gemv_t1(int group_bytes, int sums, int K, int N, int T, int vrow_mult, int num_sms,
                               int max_smem_optin, const T1Tuning &tun) {
    const T1Geometry g =
        plan_gemv_t1_form(group_bytes, sums, K, N, T, vrow_mult, num_sms, max_smem_optin, tun, kT1SlotRows);
    if (g.ok) return g;
    return plan_gemv_t1_form(group_bytes, sums, K, N, T, vrow_mult, num_sms, max_smem_optin, tun,
                             kT1SlotRowsWide);
}

}  // namespace q4mm
