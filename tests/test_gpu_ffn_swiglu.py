"""GPU parity of the fused Llama FFN input side (q4k_ffn_swiglu):
h = silu(x·W_gateᵀ) ⊙ (x·W_upᵀ), both weights Q4_K, against the CPU oracle.

The pages name this operation only as the llama.cpp benchmark "ffn_swiglu"
(PR #37 "ggml-cpu: cache-aware tiling in ggml_compute_forward_mul_mat",
section "Measured impact"); the formula is the standard Llama FFN.  g and u
are each held to the Q4_K one-token bound (1e-4 of their row maximum, SKaiNET
PR #562 section "Test plan"); silu is 1.1-Lipschitz, so per token
    max_o |h − h_ref| <= 1e-4 · max|u| · (1.1·max|g| + max|silu(g)|)
plus fp32 rounding of the product (1e-6 of max|h| here).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import GUARD, GUARD_VALUE, dev

pytestmark = pytest.mark.gpu


def ffn(x, Wg, Wu, K, N):
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf = torch.full((2 * GUARD + T * N,), float(GUARD_VALUE), dtype=torch.float32, device="cuda")
    out = buf[GUARD:GUARD + T * N]
    q.q4k_ffn_swiglu(dev(x), dev(Wg.reshape(-1)), dev(Wu.reshape(-1)), N=N, out=out)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD] == GUARD_VALUE) and np.all(b[GUARD + T * N:] == GUARD_VALUE), "write outside h"
    q.device_status()
    return out.view(T, N).cpu().numpy()


def check(h, x, Wg, Wu, K, N, what):
    g, u, ref = oracle.q4k_ffn_swiglu(x, Wg, Wu, K, N)
    assert np.all(np.isfinite(h)), what
    for t in range(ref.shape[0]):
        silu = 0.5 * g[t] * (1.0 + np.tanh(0.5 * g[t]))  # g·sigmoid(g), no overflow
        bound = 1e-4 * np.abs(u[t]).max() * (1.1 * np.abs(g[t]).max() + np.abs(silu).max())
        bound += 1e-6 * np.abs(ref[t]).max()
        err = np.abs(h[t].astype(np.float64) - ref[t]).max()
        assert err <= bound, f"{what}: token {t}: err {err:.3e} > {bound:.3e}"


def case(K, N, T, seed):
    g = synth.rng(seed)
    Wg = synth.q4k_weights(g, N, K)
    Wu = synth.q4k_weights(g, N, K)
    x = synth.activations(g, T, K)
    return x, Wg, Wu


SHAPES = [(256, 1), (256, 37), (1024, 300), (4096, 1000), (4096, 11008), (11008, 4096), (8192, 33), (32768, 5)]


@pytest.mark.parametrize("K,N", SHAPES, ids=[f"K{k}_N{n}" for k, n in SHAPES])
def test_shapes(K, N):
    x, Wg, Wu = case(K, N, 1, seed=K + N)
    check(ffn(x, Wg, Wu, K, N), x, Wg, Wu, K, N, f"K{K} N{N}")


TOKENS = [(1024, 513, 2), (1024, 513, 3), (256, 37, 6), (1024, 300, 5), (4096, 11008, 4), (4096, 11008, 8),
          (4096, 1000, 12), (11008, 4096, 7)]


@pytest.mark.parametrize("K,N,T", TOKENS, ids=[f"K{k}_N{n}_T{t}" for k, n, t in TOKENS])
def test_several_tokens(K, N, T):
    # 2 tokens: one-token launches; 3 and more: the register-tile kernel over
    # both weights, 8 tokens per pass (pairs over K up to 4 tokens).
    x, Wg, Wu = case(K, N, T, seed=9 + K + N + T)
    check(ffn(x, Wg, Wu, K, N), x, Wg, Wu, K, N, f"K{K} N{N} T{T}")


def test_same_buffer_for_gate_and_up():
    # W_gate = W_up: h = silu(g)·g.
    x, Wg, _ = case(4096, 700, 1, seed=12)
    check(ffn(x, Wg, Wg, 4096, 700), x, Wg, Wg, 4096, 700, "shared weight")


def test_gate_rows_and_up_rows_not_mixed():
    # Up rows all zero codes and mins: u = 0 exactly, so h = 0 exactly on
    # every row whatever the gate; then gate zero: silu(0)·u = 0.
    K, N = 4096, 300
    x, Wg, Wu = case(K, N, 1, seed=13)
    Wz = Wu.reshape(N, K // 256, 144).copy()
    Wz[:, :, 4:] = 0
    Wz = Wz.reshape(N, -1)
    assert np.all(ffn(x, Wg, Wz, K, N) == 0.0)
    assert np.all(ffn(x, Wz, Wu, K, N) == 0.0)


def test_run_to_run_bit_identity():
    x, Wg, Wu = case(4096, 11008, 1, seed=14)
    assert ffn(x, Wg, Wu, 4096, 11008).tobytes() == ffn(x, Wg, Wu, 4096, 11008).tobytes()
