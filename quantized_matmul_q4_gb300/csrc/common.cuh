// Device helpers shared by the q4mm kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace q4mm {

constexpr int kQ4kValues = 256;  // values per Q4_K super-block
constexpr int kQ4kBytes = 144;   // bytes per Q4_K super-block

// Streaming 16-byte load of weight bytes: read once, so keep them out of L1.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const void *p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Programmatic dependent launch: wait for the previous kernel on the stream
// (its writes become visible), and allow the next one to start its prologue.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// A 4-bit code q held in byte `k` (0..3) of `w` (high nibble of that byte
// already cleared) becomes the float 0.5 + q/256: the byte lands in bits
// 16..23 under the exponent byte 0x3F (value 2^-1·(1 + q·2^-7)).  One byte
// permute per value instead of an integer-to-float conversion.  The bias
// 0.5 per value is removed later through the per-sub-block input sums.
template <int k>
__device__ __forceinline__ float nib_biased(uint32_t w) {
    return __uint_as_float(__byte_perm(w, 0x3F000000u, 0x7054u | (k << 8)));
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    return __ffma2_rn(a, b, c);
}

// Q4_K header (first 16 bytes of a block): d and dmin as fp32.
__device__ __forceinline__ float2 q4k_d_dmin(uint32_t word0) {
    __half2 h = *reinterpret_cast<__half2 *>(&word0);
    return __half22float2(h);
}

// The eight 6-bit scales and mins of a Q4_K block, four per 32-bit word:
// sc[0..3] = bytes of sc_lo, sc[4..7] = bytes of sc_hi, likewise m.
// Packing (ggml canonical): bytes 0-3 hold sc0-3 in bits 0-5, bytes 4-7 hold
// m0-3 in bits 0-5; bytes 8-11 hold the low 4 bits of sc4-7 (bits 0-3) and
// of m4-7 (bits 4-7); the top 2 bits of bytes 0-3 / 4-7 are the high 2 bits
// of sc4-7 / m4-7.
struct Q4kScales {
    uint32_t sc_lo, sc_hi, m_lo, m_hi;
};

__device__ __forceinline__ Q4kScales q4k_unpack_scales(uint32_t s0, uint32_t s1, uint32_t s2) {
    Q4kScales r;
    r.sc_lo = s0 & 0x3F3F3F3Fu;
    r.m_lo = s1 & 0x3F3F3F3Fu;
    r.sc_hi = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
    r.m_hi = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
    return r;
}

__device__ __forceinline__ float byte_to_float(uint32_t w, int k) {
    return static_cast<float>((w >> (8 * k)) & 0xFFu);
}

// Sum of `v` over all 32 lanes (fixed butterfly order: bit-identical runs).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Sum over aligned groups of `width` lanes (width a power of two <= 32).
__device__ __forceinline__ float group_sum(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace q4mm
