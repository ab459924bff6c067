// Which kernel q4k_matmul runs for a token count: plain host C++ (no CUDA
// types), so that the CPU tests compile this same header and check the rule.
// Each choice falls back to the next one where a kernel's geometry does not
// fit the shape (capi.cu).
#pragma once

namespace q4mm {

enum class Q4kPath {
    kOneToken,       // byte-plane dp4a kernel, one token per compute warp (1-2 tokens)
    kRegisterTile,   // FP32 register-tile kernel, all tokens in one pass (3-8 tokens)
    kTileChunks,     // the same kernel in chunks of 8 tokens
    kFp32Tiles,      // FP32 tile kernel, 64-token tiles in clusters of 3 CTAs per 128 rows
};

// Measured on GB300 (chains of distinct weight copies in a CUDA graph):
//  * 2 tokens: the byte-plane kernel 7.4 against 7.7 us at 4096x4096, 13.5
//    against 17.5 us at 4096 -> 11008; from 3 tokens on the register-tile
//    kernel is as fast or faster (4 tokens: 9.3 against 12.6 us and 21.8
//    against 24.1 us);
//  * above 8 tokens the tile kernel computes whole 64-token tiles whatever
//    the tokens, and with fewer CTAs than SMs (outputDim below about 6,500)
//    leaves SMs idle: up to 32 tokens, or with that few CTAs, 8-token chunks
//    of the register-tile kernel are faster (4096x4096 at 16 tokens 27
//    against 163 us, at 64 tokens 107 against 183 us; 4096 -> 11008 at 32
//    tokens 131 against 178 us, at 64 tokens 262 against 198 us, where the
//    tile kernel keeps 258 CTAs busy).
inline Q4kPath q4k_matmul_path(int tokens, int outputDim, int num_sms) {
    if (tokens <= 2) return Q4kPath::kOneToken;
    if (tokens <= 8) return Q4kPath::kRegisterTile;
    const long long tile_ctas = 3LL * ((outputDim + 127) / 128);
    if (tokens <= 32 || tile_ctas < num_sms) return Q4kPath::kTileChunks;
    return Q4kPath::kFp32Tiles;
}

}  // namespace q4mm
