"""GPU parity of the tensor-core Q4_K path (q4k_matmul_tc) against the oracle.

The product is the one defined by SKaiNET PR #562 "feat(kernel): SIMD-fused
Q4_K matmul kernel + Q4KMatmulKernel SPI" (sections "Pipeline" and "Test
plan"), with both operands rounded to bfloat16 before the multiply and the
products accumulated in FP32.  Two tolerances, per token row t:
  * against the bf16-rounded oracle (w rounded to bf16 after the fp32
    dequantization, x rounded to bf16, exact products, double sum):
    max_o |gpu − ref| <= 1e-4 · max_o |ref|;
  * against the exact fp64 oracle: max_o |gpu − ref| <= 1e-2 · max_o |ref|
    (bf16 keeps 8 significant bits, so each operand carries up to 2^-9
    relative rounding; over a long random sum that is a few 1e-3 of the row's
    largest output).  This second bound is statistical: it describes the
    operand rounding, not the kernel, and is checked only where a token row
    has enough outputs (N >= 128) for its maximum to be representative.
Cases whose bf16 products and partial sums are exact in fp32 are compared
bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from golden import fixtures
from gpu_helpers import assert_rows_close, max_rel_err, q4k

pytestmark = pytest.mark.gpu
REL_BF16 = 1e-4
REL_EXACT = 1e-2


def _tc(x, W, K, N):
    return q4k(x, W, K, N, tc=True)


def _hand_block():
    fx = fixtures.read("q4k_handworked_block.txt")
    q = [(e // 32 + e % 32) % 16 for e in range(256)]
    return oracle.q4k_pack_block(int(fx["d_bits"], 16), int(fx["dmin_bits"], 16),
                                 fixtures.ints(fx["sc"]), fixtures.ints(fx["m"]), q)


@pytest.mark.parametrize("T", [1, 16, 17, 64, 65, 130])
def test_handworked_block_bit_exact(T):
    # Small-integer activations: every bf16 product and partial sum is exact
    # in fp32, so the tensor cores must return the bf16 oracle bit for bit.
    blk = _hand_block()
    xm = np.array([(e % 7) - 3 for e in range(256)], np.float32)
    x = np.stack([np.roll(xm, t) for t in range(T)])
    y = _tc(x, blk, 256, 1)
    ref = oracle.q4k_matmul_bf16(x, blk, 256, 1).astype(np.float32)
    assert y.tobytes() == ref.tobytes()


@pytest.mark.parametrize("N", [37, 300])
def test_one_hot_reproduces_bf16_weights(N):
    # x = e_k returns bf16(w[:, k]) exactly: pins the element order of the
    # dequantized tile, the 128-byte swizzle, the K steps inside a chunk and
    # the row order across CTAs.
    K = 512
    g = synth.rng(23)
    W = synth.q4k_weights(g, N, K)
    ks = [0, 5, 7, 8, 15, 16, 31, 32, 40, 63, 64, 100, 127, 128, 191, 192, 255, 256, 300, 383,
          384, 447, 448, 511]
    x = np.zeros((len(ks), K), np.float32)
    for t, k in enumerate(ks):
        x[t, k] = 1.0
    y = _tc(x, W, K, N)
    ref = oracle.q4k_matmul_bf16(x, W, K, N).astype(np.float32)
    assert y.tobytes() == ref.tobytes()


SWEEP = [
    (256, 1, 1), (256, 128, 16), (256, 129, 17), (512, 300, 33), (768, 5, 3), (1024, 1000, 48),
    (2048, 130, 128), (4096, 257, 64), (4096, 65, 65), (4096, 300, 200), (11008, 33, 64),
    (16384, 9, 20), (65536, 2, 16),
]


@pytest.mark.parametrize("K,N,T", SWEEP, ids=[f"K{k}_N{n}_T{t}" for k, n, t in SWEEP])
def test_shape_sweep(K, N, T):
    x, W, K, N, T = synth.q4k_case((K, N, T), seed=K + N + T + 1)
    y = _tc(x, W, K, N)
    assert_rows_close(y, oracle.q4k_matmul_bf16(x, W, K, N), REL_BF16, f"bf16 K{K} N{N} T{T}")
    if N >= 128:
        assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL_EXACT, f"exact K{K} N{N} T{T}")


def test_prefill_workload_sampled(capsys):
    # 64 tokens × 4096 → 11008: every output computed on the GPU, a sample of
    # rows (including the first and last CTA's) by the oracle.
    x, W, K, N, T = synth.q4k_case("q4k_prefill_4096x11008_t64")
    y = _tc(x, W, K, N)
    g = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], g.choice(N, 256, replace=False)]))
    Ws = W.reshape(N, -1)[rows]
    ref_b = oracle.q4k_matmul_bf16(x, Ws, K, len(rows))
    ref_x = oracle.q4k_matmul(x, Ws, K, len(rows))
    assert_rows_close(y[:, rows], ref_b, REL_BF16, "prefill vs bf16 oracle")
    assert_rows_close(y[:, rows], ref_x, REL_EXACT, "prefill vs exact oracle")
    with capsys.disabled():
        print(f"\n[q4k_matmul_tc 64x4096x11008] max row-relative error: "
              f"vs bf16 oracle {max_rel_err(y[:, rows], ref_b):.3e}, "
              f"vs exact oracle {max_rel_err(y[:, rows], ref_x):.3e}")


def test_run_to_run_bit_identity():
    x, W, K, N, T = synth.q4k_case((4096, 1000, 64), seed=4)
    assert _tc(x, W, K, N).tobytes() == _tc(x, W, K, N).tobytes()


def test_special_case_min_only():
    # d = 0, dmin = 1, every m = 1: w = −1 exactly, so y = −Σ bf16(x).
    K, N, T = 1024, 130, 20
    g = synth.rng(5)
    W = synth.q4k_weights(g, N, K).reshape(N, K // 256, 144)
    W[:, :, 0:4] = [0x00, 0x00, 0x00, 0x3C]
    W[:, :, 4:16] = [0, 0, 0, 0, 1, 1, 1, 1, 0x10, 0x10, 0x10, 0x10]
    x = synth.activations(g, T, K)
    y = _tc(x, W, K, N)
    xb = np.vectorize(oracle.round_bf16, otypes=[np.float64])(x)
    want = -xb.sum(1)
    assert np.abs(y - want[:, None]).max() <= 1e-5 * np.abs(xb).sum(1).max()
