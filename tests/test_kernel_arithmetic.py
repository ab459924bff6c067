"""CPU checks of two arithmetic recipes the CUDA kernels rely on, restated in
numpy and compared with the oracle (no GPU; nothing here is shared with the
kernels or the oracle).

1. Tensor-core prefill, bf16 weight operand.  A nibble q at bit p of its qs
   word becomes the float 2^23 + q·2^p (the masked word OR-ed into the bits
   of 2^23); one fused multiply-add with (s·2^-p, −s·2^(23−p)), s = d·sc,
   gives s·q exactly; one fp32 subtraction of o = dmin·m is the single
   rounding of the dequantized weight, and round-to-nearest-even to bf16
   follows.  The claim: the result equals the oracle's fp32 weight rounded to
   bf16, bit for bit, so the kernel's B operand is the oracle's bf16 variant
   of the weight (the Q4_K value d·sc·q − dmin·m of SKaiNET PR #562
   "feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
   section "Pipeline").

2. One-token GEMV, activation split.  Each 256-value block of x is rounded to
   n = rint(x·2^15 / s_b) with s_b = 2^e the power of two just above
   max|x_b| / 127 (its exponent read from the float's exponent field), so n
   fits 22 bits and splits into two unsigned byte digits and one signed one.
   The claims: |x − s_b·2^-15·n| ≤ 2^-15·max|x_b|/127 for every value (s_b is
   at most 2·max|x_b|/127), and values with at most 21 significant bits below
   the leading bit of max|x_b| are exact (the grid step is 2^-21 or 2^-20 of
   that leading power of two).
"""
import numpy as np

import oracle
import synth

F32 = np.float32


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of fp32 values to bf16 (finite inputs), as bits."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _header_scales(blk: np.ndarray):
    """d, dmin (fp16 → fp32) and the eight 6-bit (sc, m) pairs of one block,
    ggml canonical packing of the 12 scale bytes."""
    d = np.frombuffer(blk[0:2].tobytes(), "<f2")[0].astype(F32)
    dmin = np.frombuffer(blk[2:4].tobytes(), "<f2")[0].astype(F32)
    s = blk[4:16].astype(np.uint32)
    sc, m = [], []
    for j in range(8):
        if j < 4:
            sc.append(s[j] & 63)
            m.append(s[j + 4] & 63)
        else:
            sc.append((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4))
            m.append((s[j + 4] >> 4) | ((s[j] >> 6) << 4))
    return d, dmin, np.array(sc, np.uint32), np.array(m, np.uint32)


def _tc_recipe(q: np.ndarray, p: np.ndarray, s: F32, o: F32) -> np.ndarray:
    """bf16 bits of the tensor-core dequantization of codes q at bit positions p."""
    f = ((np.uint32(0x4B000000) | (q.astype(np.uint32) << p.astype(np.uint32))).view(F32)).astype(np.float64)
    a = (np.float64(s) * np.exp2(-p.astype(np.float64))).astype(F32)   # s·2^-p, exact
    c = (-np.float64(s) * np.exp2(23.0 - p)).astype(F32)                # −s·2^(23−p), exact
    # Fused multiply-add: the exact a·f + c (every term fits a double), one rounding.
    t = (a.astype(np.float64) * f + c.astype(np.float64)).astype(F32)
    w = t + F32(-o)                                                      # fp32 add, one rounding
    return _bf16_bits(w)


def _check_tc_blocks(W: np.ndarray, K: int, N: int):
    ref = _bf16_bits(oracle.q4k_dequant(W, K, N))
    blocks = W.reshape(N, K // 256, 144)
    # The kernel's bit positions: low nibbles at bits 0, 8, 16 (bytes 0, 1 and
    # 2 / 3 after a shift), high nibbles at bits 4 and 12.
    lo_pos = np.array([0, 8, 16, 16], np.uint32)
    hi_pos = np.array([4, 12, 12, 12], np.uint32)
    for r in range(N):
        for b in range(K // 256):
            blk = blocks[r, b]
            d, dmin, sc, m = _header_scales(blk)
            qs = blk[16:144]
            for jj in range(4):  # slab jj: sub-blocks 2jj (low) and 2jj+1 (high)
                slab = qs[32 * jj:32 * jj + 32].astype(np.uint32)
                for sub, q, pos in ((2 * jj, slab & 15, lo_pos), (2 * jj + 1, slab >> 4, hi_pos)):
                    s = F32(d * F32(sc[sub]))       # exact: 11-bit × 6-bit
                    o = F32(dmin * F32(m[sub]))
                    p = np.tile(pos, 8)             # byte l of the slab sits in word byte l % 4
                    got = _tc_recipe(q, p, s, o)
                    k0 = 256 * b + 32 * sub
                    want = ref[r, k0:k0 + 32]
                    assert np.array_equal(got, want), (r, b, sub)


def test_tc_dequant_recipe_matches_oracle_bf16_random_blocks():
    # 64 rows × 1024 values = 65,536 weights of the workloads' generator.
    g = synth.rng(11)
    K, N = 1024, 64
    _check_tc_blocks(synth.q4k_weights(g, N, K), K, N)


def test_tc_dequant_recipe_matches_oracle_bf16_edge_blocks():
    # Extreme headers: largest and smallest normal fp16 d, a subnormal d,
    # dmin 0 and dmin = d, every 6-bit scale and min at 0 and at 63, all codes.
    q = [e % 16 for e in range(256)]
    heads = [(0x7BFF, 0x7BFF, 63, 63), (0x0400, 0x0400, 63, 63), (0x0001, 0x0000, 63, 0),
             (0x3C00, 0x0000, 1, 0), (0x2E66, 0x2E66, 0, 63), (0x1E00, 0x2000, 37, 11)]
    blocks = [oracle.q4k_pack_block(db, mb, [s] * 8, [m] * 8, q) for db, mb, s, m in heads]
    W = np.concatenate(blocks).reshape(len(heads), 144)
    _check_tc_blocks(W, 256, len(heads))


def _split(xb: np.ndarray):
    """n and s_b of one 256-value block, as the one-token kernel forms them."""
    amax = F32(np.abs(xb).max())
    if amax == 0:
        ex = 0
    else:
        ebits = int((np.array([amax * F32(1.0 / 127.0)], F32).view(np.uint32)[0] >> 23) & 0xFF)
        ex = max(ebits - 126, -112)
    n = np.rint(xb.astype(np.float64) * np.exp2(15 - ex))  # exact product, nearest-even
    return n, np.exp2(ex), float(amax)


def test_one_token_split_error_bound():
    g = synth.rng(12)
    cases = [g.standard_normal(256).astype(F32) for _ in range(200)]
    cases += [(g.standard_normal(256) * 10.0 ** g.integers(-30, 30)).astype(F32) for _ in range(200)]
    spike = g.uniform(-1, 1, 256).astype(F32)
    spike[17] = F32(1000.0)
    cases += [spike, np.zeros(256, F32), np.full(256, F32(-3.0)), g.integers(-8, 9, 256).astype(F32)]
    for xb in cases:
        n, sb, amax = _split(xb)
        assert np.abs(n).max() < 2 ** 22
        # Three digits: n = 65536·p2 + 256·p1 + p0, p0 and p1 in [0, 255], p2 a signed byte.
        p0, p1, p2 = n % 256, (n // 256) % 256, n // 65536
        assert p2.min() >= -128 and p2.max() <= 127
        assert np.array_equal(65536 * p2 + 256 * p1 + p0, n)
        err = np.abs(xb.astype(np.float64) - sb * 2.0 ** -15 * n).max()
        assert err <= 2.0 ** -15 * amax / 127, (err, amax)


def test_one_token_split_exact_on_short_values():
    # Integers below 2^21 and values with at most 21 significant bits below
    # the leading bit of their block maximum come through the split unchanged.
    g = synth.rng(13)
    for _ in range(100):
        xb = g.integers(-(1 << 21), 1 << 21, 256).astype(F32)
        n, sb, _ = _split(xb)
        assert np.array_equal(sb * 2.0 ** -15 * n, xb.astype(np.float64))
    for lead in (1.0, 1.5, 1.984, 1.99, 1.9999):  # step 2^-21 below 127/64, 2^-20 above
        for e in (-30, -3, 0, 1, 17):
            xb = g.integers(-(1 << 20), 1 << 20, 256).astype(np.float64) * 2.0 ** (e - 20)
            xb[0] = np.round(lead * 2.0 ** 20) * 2.0 ** (e - 20)  # the maximum, on the same grid
            xb = xb.astype(F32)
            assert np.array_equal(xb.astype(np.float64), np.round(xb.astype(np.float64) * 2.0 ** (20 - e)) * 2.0 ** (e - 20))
            n, sb, _ = _split(xb)
            assert np.array_equal(sb * 2.0 ** -15 * n, xb.astype(np.float64)), (lead, e)


def test_one_token_split_step_at_most_2_to_minus_20():
    # The largest grid step occurs when the block maximum's mantissa is just
    # below 2: then a value 2^-21 of the leading power of two away from a
    # grid point is not exact, which is why the claim stops at 21 bits.
    xb = np.zeros(256, F32)
    xb[0] = F32(1.9999)
    xb[1] = F32(2.0 ** -21)
    n, sb, _ = _split(xb)
    assert sb * 2.0 ** -15 == 2.0 ** -20
    assert sb * 2.0 ** -15 * n[1] != float(xb[1])
