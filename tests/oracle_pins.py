"""Pins for the CPU oracle: checks against facts other than the oracle itself.

Each pin takes a loaded oracle library (so the planted-mistake tests can run
the same pins against a deliberately broken copy) and raises AssertionError
when the oracle disagrees with the fact it pins.

Sources of the facts:
  * hand-worked fixtures in tests/golden/ (worked out by hand, cited there);
  * IEEE 754 binary16 and bfloat16 definitions, checked against numpy / torch;
  * closed forms and special cases of w = d·sc·q − dmin·m (SKaiNET PR #562,
    section "Pipeline");
  * the lazy-dmin identity of the same section, as an invariant between two
    differently ordered computations;
  * integer counts for the ternary code-dot (SKaiNET issue #1138, section
    "Tests": exact equality on the code-dot for integer activations);
  * an exact-rational brute force (tests/fraction_reference.py);
  * for Q4_0 (SKaiNET PR #562, section "Out of scope"): a hand-worked block,
    nibble positions, and equality with the Q4_K oracle on blocks that both
    formats can express;
  * for the one-time relayout of Q4_K for the tensor cores (SKaiNET docs
    "Eager execution: backends and kernels", relayout-once paragraph): a
    hand-worked relayout of the hand-worked block, the canonical
    dequantization (itself pinned above) bit for bit, and code positions.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

import oracle
import synth
import fraction_reference as fr
from golden import fixtures


def _hand_block(lib):
    fx = fixtures.read("q4k_handworked_block.txt")
    sc = fixtures.ints(fx["sc"])
    m = fixtures.ints(fx["m"])
    q = [(e // 32 + e % 32) % 16 for e in range(256)]
    blk = oracle.q4k_pack_block(int(fx["d_bits"], 16), int(fx["dmin_bits"], 16), sc, m, q, lib=lib)
    return fx, blk


def pin_fp16_decode(lib):
    # IEEE 754 binary16 closed forms.
    cases = {0x3C00: 1.0, 0x3800: 0.5, 0x3400: 0.25, 0xC000: -2.0, 0x7BFF: 65504.0,
             0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24, 0x0400: 2.0 ** -14, 0x0000: 0.0}
    for bits, v in cases.items():
        got = oracle.fp16_to_double(bits, lib=lib)
        assert got == v, (hex(bits), got, v)
    # Every finite pattern against numpy's binary16 conversion.
    allbits = np.arange(65536, dtype=np.uint16)
    ref = allbits.view("<f2").astype(np.float64)
    finite = np.isfinite(ref)
    got = np.array([oracle.fp16_to_double(int(b), lib=lib) for b in allbits[finite][::37]])
    assert np.array_equal(got, ref[finite][::37])


def pin_bf16_round(lib):
    import torch
    g = np.random.default_rng(7)
    vals = np.concatenate([g.standard_normal(2000).astype(np.float32),
                           (g.standard_normal(500) * 1e-30).astype(np.float32),
                           np.array([1.0, 1.00390625, 1.005859375, 255.5, -3.0e38], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle.round_bf16(float(v), lib=lib) for v in vals], np.float32)
    assert np.array_equal(got, ref)


def pin_handworked_pack(lib):
    fx, blk = _hand_block(lib)
    assert list(blk[4:16]) == fixtures.hexbytes(fx["packed_scales"])
    assert list(blk[16:20]) == fixtures.hexbytes(fx["qs_0_3"])
    assert list(blk[48:52]) == fixtures.hexbytes(fx["qs_32_35"])


def pin_handworked_values(lib):
    fx, blk = _hand_block(lib)
    w = oracle.q4k_dequant(blk, 256, 1, lib=lib)[0]
    for e in (0, 31, 32, 255):
        assert w[e] == float(fx[f"w_{e}"]), (e, w[e])
    ones = np.ones((1, 256), np.float32)
    assert oracle.q4k_matmul(ones, blk, 256, 1, lib=lib)[0, 0] == float(fx["sum_w"])
    x = np.array([[(e % 7) - 3 for e in range(256)]], np.float32)
    want = float(fx["y_x_mod7"])
    assert oracle.q4k_matmul(x, blk, 256, 1, lib=lib)[0, 0] == want
    assert oracle.q4k_matmul_lazy(x, blk, 256, 1, lib=lib)[0, 0] == want


def pin_nibble_positions(lib):
    # One nonzero qs byte at a time: byte 32j+l = 0xAB puts code 11 at element
    # 64j+l (low nibble) and code 10 at element 64j+32+l (high nibble); with
    # d = 1, every sc = 1 and dmin = 0 those are the only nonzero values.
    sc = [1] * 8
    m = [0] * 8
    for j in range(4):
        for l in (0, 7, 16, 31):
            q = [0] * 256
            q[64 * j + l] = 0xB
            q[64 * j + 32 + l] = 0xA
            blk = oracle.q4k_pack_block(0x3C00, 0x0000, sc, m, q, lib=lib)
            assert blk[16 + 32 * j + l] == 0xAB
            blk2 = np.zeros(144, np.uint8)
            blk2[:16] = blk[:16]
            blk2[16 + 32 * j + l] = 0xAB
            w = oracle.q4k_dequant(blk2, 256, 1, lib=lib)[0]
            want = np.zeros(256, np.float32)
            want[64 * j + l] = 11
            want[64 * j + 32 + l] = 10
            assert np.array_equal(w, want), (j, l)


def pin_scale_positions(lib):
    # Distinct scales per sub-block, all codes 1, dmin = 0: each
    # sub-block's 32 values equal its own scale.  Then mins alone (codes 0,
    # d = 0, dmin = 1): each sub-block's values equal minus its own min.
    sc = [1, 2, 4, 8, 16, 32, 3, 63]
    m = [5, 7, 9, 11, 17, 33, 48, 63]
    q = [1] * 256
    blk = oracle.q4k_pack_block(0x3C00, 0x0000, sc, m, q, lib=lib)
    w = oracle.q4k_dequant(blk, 256, 1, lib=lib)[0]
    assert np.array_equal(w, np.repeat(np.array(sc, np.float32), 32))
    blk = oracle.q4k_pack_block(0x0000, 0x3C00, sc, m, [0] * 256, lib=lib)
    w = oracle.q4k_dequant(blk, 256, 1, lib=lib)[0]
    assert np.array_equal(w, -np.repeat(np.array(m, np.float32), 32))


def pin_special_cases(lib):
    g = np.random.default_rng(3)
    K, N, T = 512, 3, 2
    x = g.standard_normal((T, K)).astype(np.float32)
    # All codes 0 and all mins 0: y = 0.
    W = synth.q4k_weights(g, N, K)
    W3 = W.reshape(N, K // 256, 144).copy()
    W3[:, :, 16:] = 0
    W3[:, :, 4:16] = 0
    assert np.all(oracle.q4k_matmul(x, W3, K, N, lib=lib) == 0.0)
    # d = 0, dmin = 1, every m = 1: y = −Σx.
    W3 = W.reshape(N, K // 256, 144).copy()
    W3[:, :, 0:2] = [0x00, 0x00]
    W3[:, :, 2:4] = [0x00, 0x3C]
    W3[:, :, 4:16] = [0, 0, 0, 0, 1, 1, 1, 1, 0x10, 0x10, 0x10, 0x10]
    y = oracle.q4k_matmul(x, W3, K, N, lib=lib)
    want = -x.astype(np.float64).sum(axis=1)
    assert np.allclose(y, want[:, None], rtol=0, atol=1e-9)


def pin_one_hot_rows(lib):
    # x = e_k picks out w[o][k]; rows of x go to rows of y (no transposition).
    K, N = 512, 5
    g = np.random.default_rng(11)
    W = synth.q4k_weights(g, N, K)
    w = oracle.q4k_dequant(W, K, N, lib=lib)
    ks = [0, 1, 31, 32, 63, 64, 255, 256, 300, 511]
    x = np.zeros((len(ks), K), np.float32)
    for t, k in enumerate(ks):
        x[t, k] = 1.0
    y = oracle.q4k_matmul(x, W, K, N, lib=lib)
    for t, k in enumerate(ks):
        assert np.array_equal(y[t], w[:, k].astype(np.float64)), k


def pin_lazy_equals_direct(lib):
    x, W, K, N, T = synth.q4k_case((1024, 64, 3), seed=5)
    yd = oracle.q4k_matmul(x, W, K, N, lib=lib)
    yl = oracle.q4k_matmul_lazy(x, W, K, N, lib=lib)
    # The direct form rounds each dequantized weight to fp32 once (relative
    # error ≤ 2^-24); the lazy form keeps every value exact in double.  So the
    # two may differ by at most 2^-24·Σ_k |x_k·w_k| plus double round-off.
    w = oracle.q4k_dequant(W, K, N, lib=lib).astype(np.float64)
    bound = 2.0 ** -24 * (np.abs(x.astype(np.float64)) @ np.abs(w).T) * (1 + 1e-6)
    bound += 1e-12 * np.abs(yd).max()
    assert np.all(np.abs(yd - yl) <= bound)


def pin_fraction_bruteforce(lib):
    for (K, N, T), seed in (((256, 2, 2), 1), ((512, 3, 1), 2), ((256, 4, 3), 4)):
        x, W, K, N, T = synth.q4k_case((K, N, T), seed=seed)
        y = oracle.q4k_matmul(x, W, K, N, lib=lib)
        exact = fr.q4k_matmul(x.tolist(), [bytes(r) for r in W], K)
        for t in range(T):
            for o in range(N):
                e = exact[t][o]
                assert abs(Fraction(y[t, o]) - e) <= Fraction(1, 10 ** 9) * (1 + abs(e)), (t, o)


def pin_ternary_handworked(lib):
    fx = fixtures.read("ternary_handworked.txt")
    codes = fixtures.ints(fx["codes"])
    packed = oracle.ternary_pack(codes, lib=lib)
    assert list(packed) == fixtures.hexbytes(fx["bytes"])
    x = np.array([fixtures.ints(fx["x"])], np.float32)
    dot, y = oracle.ternary_gemv(x, packed, float(fx["scale"]), 8, 1, lib=lib)
    assert dot[0, 0] == float(fx["dot"])
    assert y[0, 0] == np.float32(fx["y"])


def pin_ternary_integer_count(lib):
    # On integer activations the code-dot is an integer: the sum of x over the
    # +1 codes minus the sum over the −1 codes, counted in Python integers.
    g = np.random.default_rng(9)
    K, N, T = 2560, 7, 3
    codes = g.integers(-1, 2, size=(N, K))
    W = np.stack([oracle.ternary_pack(c, lib=lib) for c in codes])
    x = g.integers(-8, 9, size=(T, K))
    dot, _ = oracle.ternary_gemv(x.astype(np.float32), W, 1.0, K, N, lib=lib)
    for t in range(T):
        for o in range(N):
            plus = int(x[t][codes[o] == 1].sum())
            minus = int(x[t][codes[o] == -1].sum())
            assert dot[t, o] == plus - minus, (t, o)
    # All-ones activation: count of +1 codes minus count of −1 codes.
    dot1, _ = oracle.ternary_gemv(np.ones((1, K), np.float32), W, 1.0, K, N, lib=lib)
    assert np.array_equal(dot1[0], (codes == 1).sum(1) - (codes == -1).sum(1))
    # Bytes read back through the brute-force decoder give the same codes.
    for o in range(N):
        assert fr.ternary_codes(bytes(W[o]), K) == codes[o].tolist()


def pin_ternary_scale(lib):
    # The scale multiplies the fp32 code-dot once, after the dot product.
    x, W, scale, K, N, T = synth.ternary_case((256, 9, 2), seed=13, xkind="int")
    dot, y = oracle.ternary_gemv(x, W, scale, K, N, lib=lib)
    dot1, y1 = oracle.ternary_gemv(x, W, 1.0, K, N, lib=lib)
    assert np.array_equal(dot, dot1)
    assert np.array_equal(y1, dot.astype(np.float32))
    assert np.array_equal(y, (dot.astype(np.float32).astype(np.float64) * np.float64(scale)).astype(np.float32))


def pin_bf16_variant(lib):
    # With bf16-exact operands (d = 1, dmin = 0, sc·q ≤ 225, small integer x)
    # the bf16 variant equals the direct form; otherwise it equals the direct
    # form applied to bf16-rounded operands (rounded by torch here).
    import torch
    K, N = 256, 4
    g = np.random.default_rng(17)
    W = np.stack([oracle.q4k_pack_block(0x3C00, 0, g.integers(0, 16, 8), [0] * 8,
                                        g.integers(0, 16, 256), lib=lib) for _ in range(N)])
    x = g.integers(-4, 5, size=(2, K)).astype(np.float32)
    assert np.array_equal(oracle.q4k_matmul_bf16(x, W, K, N, lib=lib),
                          oracle.q4k_matmul(x, W, K, N, lib=lib))
    x, W, K, N, T = synth.q4k_case((512, 6, 2), seed=19)
    w = oracle.q4k_dequant(W, K, N, lib=lib)
    wb = torch.from_numpy(w).to(torch.bfloat16).double().numpy()
    xb = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    want = xb @ wb.T
    got = oracle.q4k_matmul_bf16(x, W, K, N, lib=lib)
    assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()


def pin_q4_0_handworked(lib):
    fx = fixtures.read("q4_0_handworked_block.txt")
    q = list(range(16)) + [(7 + l) % 16 for l in range(16)]
    blk = oracle.q4_0_pack_block(int(fx["d_bits"], 16), q, lib=lib)
    assert list(blk[2:6]) == fixtures.hexbytes(fx["qs_0_3"])
    assert blk[17] == fixtures.hexbytes(fx["qs_15"])[0]
    w = oracle.q4_0_dequant(blk, 32, 1, lib=lib)[0]
    for e in (0, 15, 16, 31):
        assert w[e] == float(fx[f"w_{e}"]), (e, w[e])
    ones = np.ones((1, 32), np.float32)
    assert oracle.q4_0_matmul(ones, blk, 32, 1, lib=lib)[0, 0] == float(fx["sum_w"])
    x = np.array([[(e % 3) - 1 for e in range(32)]], np.float32)
    assert oracle.q4_0_matmul(x, blk, 32, 1, lib=lib)[0, 0] == float(fx["y_x_mod3"])


def pin_q4_0_nibble_positions(lib):
    # Byte l = 0xAB with every other byte 0x88 (code 8, value 0) and d = 1:
    # element l is 11 − 8 = 3 and element 16 + l is 10 − 8 = 2, the rest 0.
    for l in (0, 5, 15):
        blk = np.full(18, 0x88, np.uint8)
        blk[0:2] = [0x00, 0x3C]
        blk[2 + l] = 0xAB
        w = oracle.q4_0_dequant(blk, 32, 1, lib=lib)[0]
        want = np.zeros(32, np.float32)
        want[l], want[16 + l] = 3.0, 2.0
        assert np.array_equal(w, want), l


def pin_q4_0_as_q4k(lib):
    # Eight Q4_0 blocks sharing one d are the Q4_K block with that d, every
    # scale 1, dmin = d and every min 8 (w = d·q − d·8), the codes in the
    # same element order: an independent check against the Q4_K oracle,
    # itself pinned by the hand-worked Q4_K block above.
    g = np.random.default_rng(23)
    N, K = 3, 512
    rows40, rowsk = [], []
    for _ in range(N):
        r40, rk = [], []
        for b in range(K // 256):
            d_bits = int(g.integers(0x1C00, 0x2C00))
            codes = g.integers(0, 16, 256)
            for i in range(8):
                r40.append(oracle.q4_0_pack_block(d_bits, codes[32 * i:32 * i + 32], lib=lib))
            rk.append(oracle.q4k_pack_block(d_bits, d_bits, [1] * 8, [8] * 8, codes, lib=lib))
        rows40.append(np.concatenate(r40))
        rowsk.append(np.concatenate(rk))
    W40, Wk = np.stack(rows40), np.stack(rowsk)
    assert np.array_equal(oracle.q4_0_dequant(W40, K, N, lib=lib), oracle.q4k_dequant(Wk, K, N, lib=lib))
    x = g.standard_normal((2, K)).astype(np.float32)
    assert np.array_equal(oracle.q4_0_matmul(x, W40, K, N, lib=lib), oracle.q4k_matmul(x, Wk, K, N, lib=lib))


def pin_q4_0_fraction_bruteforce(lib):
    g = np.random.default_rng(29)
    for K, N, T in ((32, 2, 2), (96, 3, 1)):
        W = np.stack([np.concatenate([oracle.q4_0_pack_block(int(g.integers(0x1800, 0x3000)),
                                                             g.integers(0, 16, 32), lib=lib)
                                      for _ in range(K // 32)]) for _ in range(N)])
        x = g.standard_normal((T, K)).astype(np.float32)
        y = oracle.q4_0_matmul(x, W, K, N, lib=lib)
        exact = fr.q4_0_matmul(x.tolist(), [bytes(r) for r in W], K)
        for t in range(T):
            for o in range(N):
                e = exact[t][o]
                assert abs(Fraction(y[t, o]) - e) <= Fraction(1, 10 ** 9) * (1 + abs(e)), (t, o)


def pin_swiglu(lib):
    # silu(z) = z / (1 + e^-z): closed values, then h = silu(g)·u where g and
    # u come from one-hot activations (x = e_k gives the weights' column k),
    # so every g and u is a known dequantized weight.
    K, N = 256, 6
    g_ = np.random.default_rng(37)
    Wg = synth.q4k_weights(g_, N, K)
    Wu = synth.q4k_weights(g_, N, K)
    wg = oracle.q4k_dequant(Wg, K, N, lib=lib).astype(np.float64)
    wu = oracle.q4k_dequant(Wu, K, N, lib=lib).astype(np.float64)
    ks = [0, 77, 255]
    x = np.zeros((len(ks), K), np.float32)
    for t, k in enumerate(ks):
        x[t, k] = 1.0
    g, u, h = oracle.q4k_ffn_swiglu(x, Wg, Wu, K, N, lib=lib)
    for t, k in enumerate(ks):
        assert np.array_equal(g[t], wg[:, k]) and np.array_equal(u[t], wu[:, k])
        sig = 1.0 / (1.0 + np.exp(-wg[:, k]))
        assert np.allclose(h[t], wg[:, k] * sig * wu[:, k], rtol=1e-15, atol=0)
    # Closed values of silu through a one-row weight: w = d·q with d = 1,
    # dmin = 0, sc = 1 gives g = q exactly; u = 1 via the same construction.
    q = [0] * 256
    q[0], q[1], q[2] = 0, 1, 15
    Wg1 = oracle.q4k_pack_block(0x3C00, 0, [1] * 8, [0] * 8, q, lib=lib)
    qu = [1] * 256
    Wu1 = oracle.q4k_pack_block(0x3C00, 0, [1] * 8, [0] * 8, qu, lib=lib)
    x = np.zeros((3, K), np.float32)
    for t in range(3):
        x[t, t] = 1.0
    _, _, h = oracle.q4k_ffn_swiglu(x, Wg1, Wu1, K, 1, lib=lib)
    assert h[0, 0] == 0.0
    assert abs(h[1, 0] - 0.7310585786300049) < 1e-15      # 1 / (1 + e^-1)
    assert abs(h[2, 0] - 14.999995411466594) < 1e-13      # 15 / (1 + e^-15)


def _q6k_sub(v):
    return 8 * (v // 128) + 2 * ((v % 128) // 32) + (v % 32) // 16


def pin_q6k_handworked(lib):
    fx = fixtures.read("q6k_handworked_block.txt")
    sc = [s - 8 for s in range(16)]
    q = [(5 * v + 3) % 64 for v in range(256)]
    blk = oracle.q6k_pack_block(int(fx["d_bits"], 16), sc, q, lib=lib)
    assert list(blk[0:4]) == fixtures.hexbytes(fx["ql_0_3"])
    assert blk[128] == fixtures.hexbytes(fx["qh_0"])[0]
    assert list(blk[192:196]) == fixtures.hexbytes(fx["scales_0_3"])
    w = oracle.q6k_dequant(blk, 256, 1, lib=lib)[0]
    for v in (0, 17, 100, 255):
        assert w[v] == float(fx[f"w_{v}"]), (v, w[v])
    assert oracle.q6k_matmul(np.ones((1, 256), np.float32), blk, 256, 1, lib=lib)[0, 0] == float(fx["sum_w"])
    x = np.array([[(v % 5) - 2 for v in range(256)]], np.float32)
    assert oracle.q6k_matmul(x, blk, 256, 1, lib=lib)[0, 0] == float(fx["y_x_mod5"])


def pin_q6k_code_positions(lib):
    # d = 1, every scale 1, every code 32 (value 0) except code 63 at one
    # value: exactly that value is 31.  Each group, both halves, both
    # sub-blocks of a group.
    for v in (0, 15, 16, 31, 32, 47, 63, 64, 95, 96, 127, 128, 160, 200, 255):
        q = [32] * 256
        q[v] = 63
        blk = oracle.q6k_pack_block(0x3C00, [1] * 16, q, lib=lib)
        w = oracle.q6k_dequant(blk, 256, 1, lib=lib)[0]
        want = np.zeros(256, np.float32)
        want[v] = 31.0
        assert np.array_equal(w, want), v
        # The same code written straight into the bytes (independent of the
        # packer): ql nibble 15 and qh bits 3 at the computed places.
        raw = oracle.q6k_pack_block(0x3C00, [1] * 16, [32] * 256, lib=lib)
        n, g, l = v // 128, (v % 128) // 32, v % 32
        ql = 64 * n + (32 if g % 2 else 0) + l
        raw[ql] |= 0xF0 if g >= 2 else 0x0F
        raw[128 + 32 * n + l] |= 3 << (2 * g)
        assert np.array_equal(oracle.q6k_dequant(raw, 256, 1, lib=lib)[0], want), v


def pin_q6k_scale_positions(lib):
    # Every code 33 (value +1 before scaling), distinct signed scales: each
    # value is its sub-block's scale.
    sc = [-128, -3, 1, 2, 5, 7, 11, 13, 17, 19, 23, 29, 31, 64, 100, 127]
    blk = oracle.q6k_pack_block(0x3C00, sc, [33] * 256, lib=lib)
    w = oracle.q6k_dequant(blk, 256, 1, lib=lib)[0]
    assert np.array_equal(w, np.array([sc[_q6k_sub(v)] for v in range(256)], np.float32))


def pin_q6k_fraction_bruteforce(lib):
    g = np.random.default_rng(41)
    for K, N, T in ((256, 2, 2), (512, 2, 1)):
        W = np.stack([np.concatenate([oracle.q6k_pack_block(int(g.integers(0x1400, 0x2400)),
                                                            g.integers(-128, 128, 16), g.integers(0, 64, 256),
                                                            lib=lib)
                                      for _ in range(K // 256)]) for _ in range(N)])
        x = g.standard_normal((T, K)).astype(np.float32)
        y = oracle.q6k_matmul(x, W, K, N, lib=lib)
        exact = fr.q6k_matmul(x.tolist(), [bytes(r) for r in W], K)
        for t in range(T):
            for o in range(N):
                e = exact[t][o]
                assert abs(Fraction(y[t, o]) - e) <= Fraction(1, 10 ** 9) * (1 + abs(e)), (t, o)


def _tc_chunk(R, K, o, c):
    """The 48 bytes of chunk c of row o in the tile-major relayout."""
    t, r = divmod(o, 256)
    off = ((t * (K // 64) + c) * 256 + r) * 48
    return R[off:off + 48]


def pin_tc_relayout_handworked(lib):
    # The relayout of the hand-worked block against bytes worked out by hand,
    # and its values against the block's own hand-worked values.
    fx, blk = _hand_block(lib)
    tx = fixtures.read("q4k_tc_relayout_handworked.txt")
    R = oracle.q4k_tc_relayout(blk, 256, 1, lib=lib)
    assert R.size == int(tx["bytes"])
    for j in range(4):
        ch = _tc_chunk(R, 256, 0, j)
        assert int(tx[f"chunk_{j}_offset"]) == ch.ctypes.data - R.ctypes.data
        words = ch[:16].copy().view("<u4")
        assert [int(v) for v in words] == [int(v, 16) for v in tx[f"chunk_{j}_words"].split()], j
    assert list(_tc_chunk(R, 256, 0, 0)[16:20]) == fixtures.hexbytes(tx["chunk_0_qs_0_3"])
    assert list(_tc_chunk(R, 256, 0, 1)[16:20]) == fixtures.hexbytes(tx["chunk_1_qs_0_3"])
    # Rows 1..255 of the tile are padding.
    mask = np.ones(R.size, bool)
    for j in range(4):
        mask[j * 256 * 48:j * 256 * 48 + 48] = False
    assert not R[mask].any()
    w = oracle.q4k_tc_dequant(R, 256, 1, lib=lib)[0]
    for e in (0, 31, 32, 255):
        assert w[e] == float(fx[f"w_{e}"]), (e, w[e])


def pin_tc_relayout_round_trip(lib):
    # The relayouted weight is the same matrix: its dequantization equals the
    # canonical block's bit for bit, over random blocks, rows in two tiles,
    # and the extremes of the fp16 factors (subnormal, largest finite, zero)
    # and of the 6-bit fields (0 and 63).
    g = np.random.default_rng(13)
    K, N = 768, 300
    W = synth.q4k_weights(g, N, K).reshape(N, K // 256, 144).copy()
    heads = [(0x0001, 0x7BFF), (0x7BFF, 0x0001), (0x0000, 0x3C00), (0x3C00, 0x0000), (0x03FF, 0x0400)]
    for i, (d, dm) in enumerate(heads):
        o, b = divmod(i, K // 256)
        W[o + 255, b, 0:4] = [d & 255, d >> 8, dm & 255, dm >> 8]
    W[4, 0, 4:16] = 0xFF   # every sc and m = 63
    W[4, 1, 4:16] = 0x00   # every sc and m = 0
    W = W.reshape(-1)
    R = oracle.q4k_tc_relayout(W, K, N, lib=lib)
    assert R.size == 512 * K // 64 * 48
    a = oracle.q4k_tc_dequant(R, K, N, lib=lib)
    b = oracle.q4k_dequant(W, K, N, lib=lib)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def pin_tc_chunk_positions(lib):
    # One nonzero code byte at row o, block b, slab j, byte l lands in chunk
    # 4b + j of row o: tile o // 256, run (tile·K/64 + 4b + j), row o mod 256
    # of the run, byte 16 + l; nowhere else.
    K, N = 512, 300
    base = np.zeros((N, K // 256, 144), np.uint8)
    base[:, :, 0:2] = [0x00, 0x3C]
    for (o, b, j, l) in ((0, 0, 0, 0), (1, 1, 3, 31), (255, 0, 2, 7), (256, 1, 1, 16), (299, 0, 3, 5)):
        W = base.copy()
        W[o, b, 16 + 32 * j + l] = 0xAB
        R = oracle.q4k_tc_relayout(W.reshape(-1), K, N, lib=lib)
        hit = np.flatnonzero(R.reshape(-1, 48)[:, 16:])
        t, r = divmod(o, 256)
        want = (((t * (K // 64) + 4 * b + j) * 256 + r) * 32) + l
        assert hit.tolist() == [want], (o, b, j, l, hit.tolist(), want)


ALL_PINS = [
    pin_fp16_decode, pin_bf16_round, pin_handworked_pack, pin_handworked_values,
    pin_nibble_positions, pin_scale_positions, pin_special_cases, pin_one_hot_rows,
    pin_lazy_equals_direct, pin_fraction_bruteforce, pin_ternary_handworked,
    pin_ternary_integer_count, pin_ternary_scale, pin_bf16_variant,
    pin_q4_0_handworked, pin_q4_0_nibble_positions, pin_q4_0_as_q4k, pin_q4_0_fraction_bruteforce,
    pin_swiglu, pin_q6k_handworked, pin_q6k_code_positions, pin_q6k_scale_positions,
    pin_q6k_fraction_bruteforce, pin_tc_relayout_handworked, pin_tc_relayout_round_trip,
    pin_tc_chunk_positions,
]
