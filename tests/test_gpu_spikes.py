"""Large activations on weights that are zero: the one-token kernel's
precision bound must hold on valid inputs with a wide dynamic range.

The Q4_K format allows sc = 0, m = 0 and q = 0 (w = d·sc·q − dmin·m,
SKaiNET PR #562 "feat(kernel): SIMD-fused Q4_K matmul kernel +
Q4KMatmulKernel SPI", section "Pipeline"), so a position can carry a zero
weight in every row while the activation there is 1e4 or 1e5 times the
others, as outlier channels of LLM hidden states are.  The product's bound
(section "Test plan": 1e-4 relative to the gold reference, per token row
against max|ref|) must hold there too.  Each case puts one spike on such a
position, made zero in two ways — the whole 32-value sub-block (sc = m = 0)
or the single element (q = 0 with m = 0) — at inputDim 4096 and 11008, and
runs it through every route of the one-token kernel: Q4_K at 1 to 4 tokens
(the spike in one token), Q4_0 (q = 8, or d = 0 for the block), Q6_K
(q = 32, or a zero 16-value sub-block scale), the fused gate+up SwiGLU, and
the ternary payload (code 0 at the spike), plus the FP32 3-8 token kernel.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_rows_close, ffn, gemv, ternary

pytestmark = pytest.mark.gpu
REL = 1e-4
SPIKES = [1e4, 1e5, -1e5]
KS = [4096, 11008]
# The spike's position: block 3, sub-block 5, element 7 of it.
BLK, SUB, ELEM = 3, 5, 7
POS = 256 * BLK + 32 * SUB + ELEM


def _fp16_bits(v: float) -> int:
    return int(np.array([v], "<f2").view("<u2")[0])


def _q4k_with_zero(g, N, K, kind):
    """Random Q4_K rows whose weight at POS is zero in every row."""
    W = synth.q4k_weights(g, N, K).reshape(N, K // 256, 144)
    for r in range(N):
        sc = g.integers(0, 64, 8)
        m = g.integers(0, 64, 8)
        q = g.integers(0, 16, 256)
        if kind == "subblock":
            sc[SUB] = 0
            m[SUB] = 0
        else:
            m[SUB] = 0
            q[32 * SUB + ELEM] = 0
        W[r, BLK] = oracle.q4k_pack_block(_fp16_bits(g.uniform(1e-3, 1e-2)), _fp16_bits(g.uniform(0, 1e-2)),
                                          sc, m, q)
    W = W.reshape(N, -1)
    assert np.all(oracle.q4k_dequant(W, K, N)[:, POS] == 0.0)
    return W


def _x_with_spike(g, T, K, spike, tok):
    x = synth.activations(g, T, K)
    x[tok, POS] = np.float32(spike)
    return x


@pytest.mark.parametrize("kind", ["subblock", "element"])
@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_q4k_spike_on_zero_weights(K, T, kind):
    N = 160
    g = synth.rng(K + 10 * T + (kind == "element"))
    W = _q4k_with_zero(g, N, K, kind)
    for spike in SPIKES:
        x = _x_with_spike(g, T, K, spike, tok=T // 2)
        y = gemv("q4k_matmul", x, W, K, N)
        assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL, f"K{K} T{T} {kind} spike {spike:g}")


@pytest.mark.parametrize("kind", ["block", "element"])
@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("T", [1, 3])
def test_q4_0_spike_on_zero_weights(K, T, kind):
    N = 96
    g = synth.rng(2 * K + T)
    W = synth.q4_0_weights(g, N, K).reshape(N, K // 32, 18)
    b32 = POS // 32
    for r in range(N):
        q = g.integers(0, 16, 32)
        d = g.uniform(1e-3, 1e-2)
        if kind == "block":
            d = 0.0
        else:
            q[POS % 32] = 8
        W[r, b32] = oracle.q4_0_pack_block(_fp16_bits(d), q)
    W = W.reshape(N, -1)
    assert np.all(oracle.q4_0_dequant(W, K, N)[:, POS] == 0.0)
    for spike in SPIKES:
        x = _x_with_spike(g, T, K, spike, tok=T - 1)
        y = gemv("q4_0_gemv", x, W, K, N)
        assert_rows_close(y, oracle.q4_0_matmul(x, W, K, N), REL, f"Q4_0 K{K} {kind} spike {spike:g}")


@pytest.mark.parametrize("kind", ["subblock", "element"])
@pytest.mark.parametrize("K", KS)
def test_q6k_spike_on_zero_weights(K, kind):
    N = 96
    g = synth.rng(3 * K + 1)
    W = synth.q6k_weights(g, N, K).reshape(N, K // 256, 210)
    for r in range(N):
        sc = g.integers(-128, 128, 16)
        q = g.integers(0, 64, 256)
        e = POS % 256
        if kind == "subblock":
            sc[e // 16] = 0
        else:
            q[e] = 32
        W[r, BLK] = oracle.q6k_pack_block(_fp16_bits(g.uniform(1e-3, 1e-2)), sc, q)
    W = W.reshape(N, -1)
    assert np.all(oracle.q6k_dequant(W, K, N)[:, POS] == 0.0)
    for spike in SPIKES:
        x = _x_with_spike(g, 1, K, spike, tok=0)
        y = gemv("q6k_gemv", x, W, K, N)
        assert_rows_close(y, oracle.q6k_matmul(x, W, K, N), REL, f"Q6_K K{K} {kind} spike {spike:g}")


@pytest.mark.parametrize("K", [4096])
def test_ffn_swiglu_spike_on_zero_weights(K):
    N = 128
    g = synth.rng(K + 5)
    Wg = _q4k_with_zero(g, N, K, "subblock")
    Wu = _q4k_with_zero(g, N, K, "element")
    for spike in SPIKES:
        x = _x_with_spike(g, 1, K, spike, tok=0)
        h = ffn(x, Wg, Wu, K, N)
        gg, u, ref = oracle.q4k_ffn_swiglu(x, Wg, Wu, K, N)
        silu = 0.5 * gg[0] * (1.0 + np.tanh(0.5 * gg[0]))  # g·sigmoid(g), no overflow
        bound = 1e-4 * np.abs(u[0]).max() * (1.1 * np.abs(gg[0]).max() + np.abs(silu).max())
        bound += 1e-6 * np.abs(ref[0]).max()
        err = np.abs(h[0].astype(np.float64) - ref[0]).max()
        assert err <= bound, (spike, err, bound)


@pytest.mark.parametrize("T", [1, 3])
def test_ternary_spike_on_zero_code(T):
    # 2560 -> 6912 shape family (K a multiple of 256: the byte-plane kernel).
    K, N = 2560, 200
    g = synth.rng(77 + T)
    codes = g.integers(-1, 2, size=(N, K))
    codes[:, POS] = 0
    W = np.stack([oracle.ternary_pack(codes[r]) for r in range(N)])
    scale = 1.25
    for spike in SPIKES:
        x = _x_with_spike(g, T, K, spike, tok=0)
        y = ternary(x, W, scale, K, N)
        dot, _ = oracle.ternary_gemv(x, W, scale, K, N)
        assert_rows_close(y, scale * dot, REL, f"ternary T{T} spike {spike:g}")
