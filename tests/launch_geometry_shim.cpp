// Host shim for the CPU tests: exposes the launch geometry of the one-token
// and the 2-8 token GEMV kernels (the library's own headers, default tuning)
// through a C ABI.
#include "../quantized_matmul_q4_gb300/csrc/multi_geometry.h"
#include "../quantized_matmul_q4_gb300/csrc/dispatch.h"
#include "../quantized_matmul_q4_gb300/csrc/t1_geometry.h"

extern "C" int t1_plan(int group_bytes, int sums, int K, int N, int T, int vrow_mult, int num_sms, int max_smem,
                       long long *out) {
    const q4mm::T1Tuning tun;
    const q4mm::T1Geometry g =
        q4mm::plan_gemv_t1(group_bytes, sums, K, N, T, vrow_mult, num_sms, max_smem, tun);
    const long long v[] = {g.ok,         g.wide,       g.wc,       g.pass_rows,  g.rg,
                           g.ncw,        g.stage_rows, g.rows_per_cta, g.grid,
                           g.x_staged,   g.nslots,     g.pre_stages, (long long)g.xs_bytes,
                           (long long)g.part_bytes, (long long)g.slot_bytes, (long long)g.smem,
                           g.cw,         g.slot_rows};
    for (int i = 0; i < (int)(sizeof(v) / sizeof(v[0])); ++i) out[i] = v[i];
    return g.ok;
}

extern "C" int multi_plan(int K, int N, int num_sms, int max_smem, int ring_bytes, int T, int vrow_mult,
                          long long *out) {
    const q4mm::MultiGeometry g = q4mm::plan_gemv_multi(K, N, num_sms, max_smem, ring_bytes, T, vrow_mult);
    const long long v[] = {g.ok, g.grid, g.rows_per_cta, g.nslots, g.consumers, (long long)g.smem, g.x_staged};
    for (int i = 0; i < (int)(sizeof(v) / sizeof(v[0])); ++i) out[i] = v[i];
    return g.ok;
}

extern "C" int q4k_path(int tokens, int outputDim, int num_sms) {
    return (int)q4mm::q4k_matmul_path(tokens, outputDim, num_sms);
}
