"""CPU checks of three arithmetic recipes the CUDA kernels rely on, restated in
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

2. One-token GEMV, activation split.  Each 32-value group of x is rounded to
   n = rint(x·2^23 / s_g) with s_g = 2^e the power of two just above
   max|x_g| / 255 (its exponent read from the float's exponent field of the
   fp32 product max·(1/255)), so n fits 31 bits and splits into three
   unsigned byte digits and one signed one.  The claims: |x − s_g·2^-23·n| ≤
   max(2^-23·max|x_g|/255, 2^-127) for every value (s_g is below
   2·max|x_g|/255, and at least 2^-103), values
   of magnitude at least s_g are exact, and a large activation in one group
   leaves every other group's representation unchanged.  Together with exact
   integer code-dots this keeps a row within 1e-4 of the oracle even when an
   activation of 1e5 sits on weights that are zero.

3. FP32 register-tile GEMV (3-8 tokens), dequantized weight: one rounding of
   the offset and one of the weight (see below), zero sub-blocks exactly zero.
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


def _split(xg: np.ndarray):
    """n and s_g of one 32-value group, as the one-token kernel forms them."""
    amax = F32(np.abs(xg).max())
    if amax == 0:
        ex = 0
    else:
        ebits = int((np.array([amax * F32(1.0 / 255.0)], F32).view(np.uint32)[0] >> 23) & 0xFF)
        ex = max(ebits - 126, -103)
    n = np.rint(xg.astype(np.float64) * np.exp2(23 - ex))  # exact product, nearest-even
    return n, np.exp2(ex), float(amax)


def _split_row(x: np.ndarray) -> np.ndarray:
    """The activations as the kernel represents them: s_g·2^-23·n, group by group."""
    out = np.empty(x.shape, np.float64)
    for g0 in range(0, x.size, 32):
        n, sg, _ = _split(x[g0:g0 + 32])
        out[g0:g0 + 32] = sg * 2.0 ** -23 * n
    return out


def test_one_token_split_error_bound():
    g = synth.rng(12)
    cases = [g.standard_normal(32).astype(F32) for _ in range(400)]
    cases += [(g.standard_normal(32) * 10.0 ** g.integers(-30, 30)).astype(F32) for _ in range(400)]
    spike = g.uniform(-1, 1, 32).astype(F32)
    spike[17] = F32(1e5)
    tiny = (g.standard_normal(32) * F32(1e-36)).astype(F32)
    cases += [spike, tiny, np.zeros(32, F32), np.full(32, F32(-3.0)), g.integers(-8, 9, 32).astype(F32),
              np.full(32, F32(3.0e38))]
    for xg in cases:
        n, sg, amax = _split(xg)
        assert np.abs(n).max() < 2 ** 31
        # Four digits: n = 2^24·p3 + 2^16·p2 + 2^8·p1 + p0, p0..p2 in [0, 255], p3 a signed byte.
        p0, p1, p2, p3 = n % 256, (n // 256) % 256, (n // 65536) % 256, n // 2 ** 24
        assert p3.min() >= -128 and p3.max() <= 127
        assert np.array_equal(2 ** 24 * p3 + 65536 * p2 + 256 * p1 + p0, n)
        err = np.abs(xg.astype(np.float64) - sg * 2.0 ** -23 * n).max()
        # Groups below 255·2^-103 keep the step 2^-126 (the scale's lower bound).
        assert err <= max(2.0 ** -23 * amax / 255, 2.0 ** -127), (err, amax)
        assert sg < 2 * amax / 255 or amax == 0 or sg == 2.0 ** -103


def test_one_token_split_exact_at_or_above_the_group_scale():
    # Every value of magnitude at least s_g is a multiple of the step
    # s_g·2^-23, so it comes through unchanged; integers below 2^23 in
    # groups whose maximum is below 2^23 are too.
    g = synth.rng(13)
    for _ in range(200):
        xg = (g.standard_normal(32) * 10.0 ** g.integers(-20, 20)).astype(F32)
        n, sg, _ = _split(xg)
        big = np.abs(xg) >= sg
        assert np.array_equal((sg * 2.0 ** -23 * n)[big], xg.astype(np.float64)[big])
    for _ in range(100):
        xg = g.integers(-(1 << 23) + 1, 1 << 23, 32).astype(F32)
        n, sg, _ = _split(xg)
        assert np.array_equal(sg * 2.0 ** -23 * n, xg.astype(np.float64))


def test_one_token_split_groups_are_independent():
    # A spike changes only its own group's scale.
    g = synth.rng(14)
    x = g.standard_normal(256).astype(F32)
    y = x.copy()
    y[77] = F32(1e5)
    a, b = _split_row(x), _split_row(y)
    same = np.ones(256, bool)
    same[64:96] = False
    assert np.array_equal(a[same], b[same])


def _row_error_with_spike(K, spike, zero_kind, seed):
    """Max per-row relative error of the split recipe (exact code-dots, the
    represented activations times the oracle's fp32 weights, summed in
    double) against the oracle, with one activation of size `spike` on
    weights that are zero in every row."""
    g = synth.rng(seed)
    N = 64
    W = synth.q4k_weights(g, N, K).reshape(N, K // 256, 144).copy()
    b, sub, e = 3, 5, 7            # block 3, sub-block 5, element 7 of it
    pos = 256 * b + 32 * sub + e
    for r in range(N):
        blk = W[r, b]
        d, dmin, sc, m = _header_scales(blk)
        sc, m = [int(v) for v in sc], [int(v) for v in m]
        q = []
        qs = blk[16:144]
        for k in range(256):
            jj, l = k // 64, k % 64    # slab jj: low nibbles are l < 32, high nibbles l >= 32
            byte = qs[32 * jj + (l % 32)]
            q.append(int(byte & 15) if l < 32 else int(byte >> 4))
        if zero_kind == "subblock":
            sc[sub], m[sub] = 0, 0
        else:
            m[sub] = 0
            q[32 * sub + e] = 0
        dbits = int(np.frombuffer(blk[0:2].tobytes(), "<u2")[0])
        mbits = int(np.frombuffer(blk[2:4].tobytes(), "<u2")[0])
        W[r, b] = oracle.q4k_pack_block(dbits, mbits, sc, m, q)
    W = W.reshape(-1)
    x = synth.activations(g, 1, K).reshape(-1)
    x[pos] = F32(spike)
    w32 = oracle.q4k_dequant(W, K, N).astype(np.float64)
    assert np.all(w32[:, pos] == 0.0)
    ref = oracle.q4k_matmul(x.reshape(1, K), W, K, N)[0]
    got = w32 @ _split_row(x)
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def test_one_token_split_spike_on_zero_weights_stays_within_1e_4():
    # The verdict's scenario: activations of 1e4 and 1e5 on a position whose
    # weights are zero, by sc = m = 0 for the whole sub-block or by q = 0 with
    # m = 0 at that element.  The grid of every other group is untouched and
    # the spike's own group keeps ~2^-30 of its maximum.
    for K in (4096, 11008):
        for spike in (1e4, 1e5, -1e5):
            for kind in ("subblock", "element"):
                err = _row_error_with_spike(K, spike, kind, seed=21)
                assert err < 1e-5, (K, spike, kind, err)


# 3. The FP32 register-tile kernel (3-8 tokens, the 8-token chunks above),
#    dequantized weight.  Per sub-block s' = 256·d·sc (exact: an 11-bit
#    mantissa times a 6-bit integer, scaled by a power of two) and
#    o' = fma(dmin, m, s'/2) (one rounding); a code q becomes the float
#    0.5 + q/256 (exact, built by one byte permute) and the weight is
#    w' = fma(0.5 + q/256, s', −o') (one rounding).  So w' − w, with
#    w = d·sc·q − dmin·m exact, is the rounding of o' plus the rounding of
#    w', at most 2^-24·(|o'| + |w'|), and a sub-block whose scale and min are
#    zero gives weights that are exactly zero.

def _multi_recipe(d: F32, dmin: F32, sc: int, m: int, q: np.ndarray) -> np.ndarray:
    s = F32(F32(256.0) * d) * F32(sc)                                       # exact
    o = F32(np.float64(dmin) * np.float64(m) + 0.5 * np.float64(s))          # fma, one rounding
    nib = (0.5 + q.astype(np.float64) / 256.0).astype(F32)                  # exact
    return (nib.astype(np.float64) * np.float64(s) - np.float64(o)).astype(F32), o  # fma, one rounding


def _multi_weights(W: np.ndarray, K: int, N: int):
    """The recipe's weights and the per-weight bound 2^-24·(|o'| + |w'|)."""
    blocks = W.reshape(N, K // 256, 144)
    w = np.empty((N, K), F32)
    bound = np.empty((N, K), np.float64)
    for r in range(N):
        for b in range(K // 256):
            blk = blocks[r, b]
            d, dmin, sc, m = _header_scales(blk)
            qs = blk[16:144].astype(np.uint32)
            for sub in range(8):
                slab = qs[32 * (sub // 2):32 * (sub // 2) + 32]
                q = slab & 15 if sub % 2 == 0 else slab >> 4
                ws, o = _multi_recipe(d, dmin, int(sc[sub]), int(m[sub]), q)
                k0 = 256 * b + 32 * sub
                w[r, k0:k0 + 32] = ws
                bound[r, k0:k0 + 32] = 2.0 ** -24 * (abs(np.float64(o)) + np.abs(ws.astype(np.float64)))
    return w, bound


def _exact_weights(W: np.ndarray, K: int, N: int) -> np.ndarray:
    blocks = W.reshape(N, K // 256, 144)
    w = np.empty((N, K), np.float64)
    for r in range(N):
        for b in range(K // 256):
            d, dmin, sc, m = _header_scales(blocks[r, b])
            qs = blocks[r, b, 16:144].astype(np.uint32)
            for sub in range(8):
                slab = qs[32 * (sub // 2):32 * (sub // 2) + 32]
                q = (slab & 15 if sub % 2 == 0 else slab >> 4).astype(np.float64)
                k0 = 256 * b + 32 * sub
                w[r, k0:k0 + 32] = np.float64(d) * sc[sub] * q - np.float64(dmin) * m[sub]
    return w


def test_multi_dequant_recipe_within_two_roundings():
    g = synth.rng(12)
    K, N = 1024, 48
    W = synth.q4k_weights(g, N, K)
    w, bound = _multi_weights(W, K, N)
    exact = _exact_weights(W, K, N)
    # 2^-24·|w'| of slack for the double rounding of the fp64 emulation.
    assert np.all(np.abs(w.astype(np.float64) - exact) <= bound + 2.0 ** -24 * np.abs(w.astype(np.float64)))
    # The exact weight is also the oracle's (before its one fp32 rounding).
    assert np.array_equal(exact.astype(F32), oracle.q4k_dequant(W, K, N))


def test_multi_dequant_recipe_zero_sub_blocks_are_exactly_zero_and_rows_meet_1e_4():
    # Sub-blocks with scale and min 0 (valid Q4_K) dequantize to exact zeros,
    # so an activation of 1e5 there adds nothing; the recipe's rows stay
    # within the 1e-4 contract of the oracle with such spikes.
    g = synth.rng(13)
    K, N = 1024, 32
    W = synth.q4k_weights(g, N, K).reshape(N, K // 256, 144).copy()
    q = [e % 16 for e in range(256)]
    zero = oracle.q4k_pack_block(0x2E66, 0x2E66, [0] * 8, [0] * 8, q)
    W[:, 1] = np.frombuffer(zero.tobytes(), np.uint8)
    W = W.reshape(-1)
    w, _ = _multi_weights(W, K, N)
    assert np.all(w[:, 256:512] == 0)
    x = synth.activations(g, 2, K).astype(np.float64)
    x[:, 300] = 1e5
    x[1, 511] = -1e5
    y = x @ w.astype(np.float64).T
    ref = oracle.q4k_matmul(x.astype(F32), W, K, N)
    for t in range(2):
        assert np.abs(y[t] - ref[t]).max() <= 1e-4 * np.abs(ref[t]).max()
