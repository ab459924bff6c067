"""GPU parity of the Q4_K FP32 path (q4k_matmul) against the CPU oracle.

Tolerance (SKaiNET PR #562, section "Test plan": 1e-4 relative against the
gold dequantize-then-matmul reference), read per token row t as
max_o |gpu − oracle| <= 1e-4 · max_o |oracle|.  Cases: the hand-worked block
(exact), one-hot activations (element order), the workloads' shapes (full
outputs where the oracle is quick, sampled rows at the largest sizes), an
odd-shape sweep over the kernels (1–2 tokens, 3–8 tokens, 8-token chunks and 64-token tiles above),
ragged row counts, and run-to-run bit identity.
"""
import numpy as np
import pytest

import oracle
import synth
from golden import fixtures
from gpu_helpers import assert_rows_close, q4k

pytestmark = pytest.mark.gpu
REL = 1e-4


def _hand_block():
    fx = fixtures.read("q4k_handworked_block.txt")
    q = [(e // 32 + e % 32) % 16 for e in range(256)]
    blk = oracle.q4k_pack_block(int(fx["d_bits"], 16), int(fx["dmin_bits"], 16),
                                fixtures.ints(fx["sc"]), fixtures.ints(fx["m"]), q)
    return fx, blk


@pytest.mark.parametrize("T", [1, 2, 3, 8, 9, 64])
def test_handworked_block_exact(T):
    fx, blk = _hand_block()
    xm = np.array([(e % 7) - 3 for e in range(256)], np.float32)
    x = np.stack([xm if t % 2 == 0 else np.ones(256, np.float32) for t in range(T)])
    y = q4k(x, blk, 256, 1)
    for t in range(T):
        want = float(fx["y_x_mod7"]) if t % 2 == 0 else float(fx["sum_w"])
        assert y[t, 0] == want, (t, y[t, 0], want)


@pytest.mark.parametrize("T", [1, 5])
def test_one_hot_reproduces_weights(T):
    # Pins the element order inside the kernels: x = e_k must return w[:, k].
    K, N = 512, 37
    g = synth.rng(21)
    W = synth.q4k_weights(g, N, K)
    w = oracle.q4k_dequant(W, K, N)
    ks = [0, 5, 31, 32, 40, 63, 64, 100, 127, 128, 191, 192, 255, 256, 300, 383, 384, 511]
    for i in range(0, len(ks), T):
        chunk = ks[i:i + T]
        x = np.zeros((len(chunk), K), np.float32)
        for t, k in enumerate(chunk):
            x[t, k] = 1.0
        y = q4k(x, W, K, N)
        for t, k in enumerate(chunk):
            ref = w[:, k].astype(np.float64)
            assert np.abs(y[t] - ref).max() <= 1e-6 * np.abs(w).max(), k


@pytest.mark.parametrize("name", ["q4k_gemv_1024x1024_t1", "q4k_gemv_4096x1024_t1",
                                  "q4k_gemv_4096x4096_t1"])
def test_decode_workloads_full(name):
    x, W, K, N, T = synth.q4k_case(name)
    y = q4k(x, W, K, N)
    assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL, name)


SWEEP = [
    (256, 1, 1), (256, 3, 2), (256, 33, 7), (256, 1000, 9), (512, 3, 8), (512, 33, 16),
    (512, 1000, 1), (768, 5, 3), (1280, 33, 1), (2048, 17, 4), (4096, 33, 63), (4096, 65, 64),
    (4096, 7, 65), (11008, 33, 1), (11008, 3, 8), (11008, 9, 9), (8192, 31, 1), (16384, 5, 1),
    (24576, 3, 1), (24576, 3, 2), (65536, 2, 1), (3072, 1001, 1), (3072, 1001, 2),
    # 2 tokens on the byte-plane kernel (one token per compute warp).
    (11008, 40, 2), (4096, 77, 2),
    # 3-8 tokens on the FP32 register-tile kernel (3, 4, 6 and 8 token
    # tiles, the 3 and 6 token ones padded in the row butterfly).
    (4096, 300, 3), (4096, 1000, 4), (1024, 77, 4), (256, 9, 3), (2048, 99, 3),
    (4096, 301, 5), (768, 13, 6), (11008, 21, 5), (4096, 129, 7),
]


@pytest.mark.parametrize("K,N,T", SWEEP, ids=[f"K{k}_N{n}_T{t}" for k, n, t in SWEEP])
def test_shape_sweep(K, N, T):
    x, W, K, N, T = synth.q4k_case((K, N, T), seed=K + N + T)
    y = q4k(x, W, K, N)
    assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL, f"K{K} N{N} T{T}")


def _sampled(K, N, T, seed, nsample=192):
    x, W, K, N, T = synth.q4k_case((K, N, T), seed=seed)
    y = q4k(x, W, K, N)
    g = np.random.default_rng(seed + 1)
    rows = np.unique(np.concatenate([[0, N - 1], g.choice(N, nsample, replace=False)]))
    ref = oracle.q4k_matmul(x, W[rows], K, len(rows))
    assert_rows_close(y[:, rows], ref, REL, f"K{K} N{N} T{T} sampled")
    assert np.all(np.isfinite(y))


def test_prefill_workload_sampled():
    # 64 tokens × 4096 → 11008, FP32 variant, sampled output rows.
    _sampled(4096, 11008, 64, seed=0)


@pytest.mark.parametrize("K,N,T", [(4096, 4096, 16), (11008, 4096, 24), (4096, 11008, 32), (4096, 4096, 70),
                                   (4096, 11008, 40), (4096, 8192, 33)],
                         ids=["chunks_4096_t16", "chunks_11008_t24", "chunks_11008rows_t32", "chunks_4096_t70",
                              "tiles_11008rows_t40", "tiles_8192rows_t33"])
def test_many_tokens_sampled(K, N, T):
    # More than 8 tokens: 8-token chunks of the register-tile kernel (up to
    # 32 tokens, or an output too narrow to fill the SMs with 64-token
    # tiles; the last chunk ragged) and the 64-token FP32 tile kernel
    # (ragged token tiles), sampled output rows.
    _sampled(K, N, T, seed=K + N + T)


@pytest.mark.parametrize("K,N", [(8192, 8192), (16384, 16384), (14336, 4096)])
def test_large_one_token_sampled(K, N):
    # One-token GEMVs above 4096²: the 8192² and 16384² bench matrices and a
    # 14336-wide row (Llama-3-8B down projection), sampled output rows.
    _sampled(K, N, 1, seed=K + N)


@pytest.mark.parametrize("K,N,T", [(14336, 4096, 8), (16384, 4096, 5), (13056, 4096, 3)])
def test_multi_token_wide_rows_full(K, N, T):
    # 3-8 token kernel with rows so wide that fewer ring slots than compute
    # warps fit in shared memory (13056 values and up), and more row groups
    # per CTA than slots, so every slot is reused: all outputs checked.
    x, W, K, N, T = synth.q4k_case((K, N, T), seed=K + T)
    y = q4k(x, W, K, N)
    assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL, f"K{K} N{N} T{T}")


@pytest.mark.parametrize("K,N", synth.LLAMA7B_LAYER[3:7])
@pytest.mark.parametrize("T", [1, 8])
def test_llama7b_layer_shapes_sampled(K, N, T):
    _sampled(K, N, T, seed=7 * K + N + T)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_run_to_run_bit_identity(T):
    x, W, K, N, T = synth.q4k_case((4096, 4096, T), seed=3)
    a = q4k(x, W, K, N)
    b = q4k(x, W, K, N)
    assert a.tobytes() == b.tobytes()


def test_special_case_min_only():
    # d = 0, dmin = 1, every m = 1: y = −Σx on every row.
    K, N, T = 1024, 9, 3
    g = synth.rng(5)
    W = synth.q4k_weights(g, N, K).reshape(N, K // 256, 144)
    W[:, :, 0:4] = [0x00, 0x00, 0x00, 0x3C]
    W[:, :, 4:16] = [0, 0, 0, 0, 1, 1, 1, 1, 0x10, 0x10, 0x10, 0x10]
    x = synth.activations(g, T, K)
    for TT in (1, T):
        y = q4k(x[:TT], W, K, N)
        want = -x[:TT].astype(np.float64).sum(1)
        assert np.abs(y - want[:, None]).max() <= 1e-5 * np.abs(x).sum()


@pytest.mark.parametrize("K", [1024, 4096, 11008])
def test_one_token_wide_dynamic_range(K):
    # One value per 256-value block 1000 times larger than the others.  The
    # small activations still carry about 1% of each output, so the one-token
    # kernel's rounding of x relative to each block's maximum must stay far
    # below 1e-4 of the output scale (a split to 2^-14 of the block maximum
    # would already miss the bound; dropping the small values misses it 100x).
    N = 96
    g = synth.rng(K + 1)
    W = synth.q4k_weights(g, N, K)
    x = g.uniform(-1.0, 1.0, size=(1, K)).astype(np.float32)
    spikes = g.integers(0, 256, size=K // 256) + 256 * np.arange(K // 256)
    x[0, spikes] = np.float32(1000.0) * np.sign(g.uniform(-1, 1, size=spikes.size)).astype(np.float32)
    y = q4k(x, W, K, N)
    assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL, f"K{K} spikes")


def test_one_token_integer_activations_near_exact():
    # Integer activations up to 2^21 in magnitude are represented exactly by
    # the one-token split, so the only error left is fp32 rounding of the
    # scaled sums: far below the 1e-4 bound.
    K, N = 4096, 128
    g = synth.rng(77)
    W = synth.q4k_weights(g, N, K)
    x = g.integers(-(1 << 21), 1 << 21, size=(1, K)).astype(np.float32)
    ref = oracle.q4k_matmul(x, W, K, N)
    y = q4k(x, W, K, N)
    assert_rows_close(y, ref, 2e-6, "integer activations")
