"""Planted mistakes: each test copies the oracle's C source, plants one
plausible mistake (a swapped nibble, a wrong sign, a wrong index, a transposed
operand, a dropped term, a wrong rounding), builds the copy on the CPU and
checks that at least one pin rejects it.  This shows the pins are strong
enough to catch such mistakes in the real oracle."""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "low_nibble_from_high": ("return qs[32 * j + l] & 15;", "return qs[32 * j + l] >> 4;"),
    "halves_swapped": ("int j = e / 64, l = e % 64;", "int j = e / 64, l = (e + 32) % 64;"),
    "dmin_sign": ("w[e] = (float)(d * sc * q4k_code(qs, e) - dmin * m);",
                  "w[e] = (float)(d * sc * q4k_code(qs, e) + dmin * m);"),
    "sub_block_index": ("q4k_scale_min(packed, e / 32, &sc, &m);",
                        "q4k_scale_min(packed, (e / 32) ^ 1, &sc, &m);"),
    "scale_high_bits_byte": ("*sc = (packed[s + 4] & 15) | ((packed[s - 4] >> 6) << 4);",
                             "*sc = (packed[s + 4] & 15) | ((packed[s] >> 6) << 4);"),
    "min_low_bits_nibble": ("*m = (packed[s + 4] >> 4) |", "*m = (packed[s + 4] & 15) |"),
    "d_dmin_swapped": ("double d = q4k_d(blk), dmin = q4k_dmin(blk);",
                       "double dmin = q4k_d(blk), d = q4k_dmin(blk);"),
    "fp16_bias": ("exponent - 25", "exponent - 24"),
    "fp16_subnormal": ("ldexp((double)mantissa, -24)", "ldexp((double)mantissa, -25)"),
    "output_transposed": ("y[t * N + o] = acc;", "y[o * T + t] = acc;"),
    "activation_row": ("const float *xt = x + t * K;\n                double acc",
                       "const float *xt = x + t;\n                double acc"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) {\n                    float xv",
                          "for (int64_t k = 0; k < K - 1; ++k) {\n                    float xv"),
    "lazy_offset_dropped": ("acc += (d * sc) * code_sum - (dmin * m) * input_sum;",
                            "acc += (d * sc) * code_sum;"),
    "ternary_field_order": ("return ((row[i / 4] >> (2 * (i % 4))) & 3) - 1;",
                            "return ((row[i / 4] >> (2 * (3 - i % 4))) & 3) - 1;"),
    "ternary_offset": ("return ((row[i / 4] >> (2 * (i % 4))) & 3) - 1;",
                       "return ((row[i / 4] >> (2 * (i % 4))) & 3);"),
    "bf16_truncates": ("u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;", "u = u & 0xFFFF0000u;"),
    "swiglu_sigmoid_sign": ("h[i] = z / (1.0 + exp(-z)) * uu[i];", "h[i] = z / (1.0 + exp(z)) * uu[i];"),
    "swiglu_gate_up_swapped": ("rc = q4k_matmul_impl(x, Wg, K, N, T, gg, nthreads, 0);",
                               "rc = q4k_matmul_impl(x, Wu, K, N, T, gg, nthreads, 0);"),
    "q6k_qh_shift": ("int hi = (qh[l] >> (2 * g)) & 3;", "int hi = (qh[l] >> g) & 3;"),
    "q6k_ql_halves": ("int lo = (g & 1) ? ql[32 + l] : ql[l];", "int lo = (g & 2) ? ql[32 + l] : ql[l];"),
    "q6k_sub_block": ("int s = 8 * n + 2 * g + l / 16;", "int s = 8 * n + g + l / 16;"),
    "q6k_offset": ("w[v] = (float)(d * sc[s] * (q6k_code(blk, v) - 32));",
                   "w[v] = (float)(d * sc[s] * (q6k_code(blk, v) - 31));"),
    "q6k_scales_unsigned": ("const int8_t *sc = (const int8_t *)(blk + 192);",
                            "const uint8_t *sc = (const uint8_t *)(blk + 192);"),
    "q4_0_nibble_halves": ("return e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);",
                           "return e < 16 ? (qs[e] >> 4) : (qs[e - 16] & 15);"),
    "q4_0_offset": ("w[e] = (float)(d * (q40_code(blk + 2, e) - 8));",
                    "w[e] = (float)(d * (q40_code(blk + 2, e) - 7));"),
    "q4_0_d_bytes": ("double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));\n    for (int e = 0; e < Q40_VALUES",
                     "double d = oracle_fp16_to_double((uint16_t)(blk[1] | (blk[0] << 8)));\n    for (int e = 0; e < Q40_VALUES"),
    "q4_0_block_stride": ("oracle_q4_0_dequant_block(W + (o * nb + b) * Q40_BYTES, w + b * Q40_VALUES);",
                          "oracle_q4_0_dequant_block(W + (o * nb + b) * 16, w + b * Q40_VALUES);"),
    "tc_sub_block_swapped": ("q4k_scale_min(blk + 4, 2 * j + h, &sc, &m);",
                             "q4k_scale_min(blk + 4, 2 * j + 1 - h, &sc, &m);"),
    "tc_scale_min_swapped": ("put_f32(ch + 8 * h, d * sc);\n                    put_f32(ch + 8 * h + 4, dmin * m);",
                             "put_f32(ch + 8 * h + 4, d * sc);\n                    put_f32(ch + 8 * h, dmin * m);"),
    "tc_slab_order": ("memcpy(ch + 16, blk + 16 + 32 * j, 32);", "memcpy(ch + 16, blk + 16 + 32 * (3 - j), 32);"),
    "tc_row_major": ("return ((t * (K / 64) + c) * Q4K_TC_TILE_ROWS + r) * Q4K_TC_CHUNK_BYTES;",
                     "return (o * (K / 64) + c) * Q4K_TC_CHUNK_BYTES;"),
    "tc_offset_sign": ("w[i] = (float)(s_lo * (ch[16 + i] & 15) - o_lo);",
                       "w[i] = (float)(s_lo * (ch[16 + i] & 15) + o_lo);"),
    "tc_high_nibble": ("w[32 + i] = (float)(s_hi * (ch[16 + i] >> 4) - o_hi);",
                       "w[32 + i] = (float)(s_hi * (ch[16 + i] & 15) - o_hi);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert old in src, f"mutation target for {name} no longer in the oracle source"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new, 1))
    lib_path = oracle.build(str(mutant_src), str(tmp_path / "libmutant.so"), force=True)
    lib = oracle.load(lib_path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, RuntimeError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
