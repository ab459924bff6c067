"""GPU parity of ternary_gemv against the CPU oracle.

SKaiNET issue #1138, section "Tests": exact equality on the code-dot, a
tolerance only for summation order.  With integer activations the fp32
code-dot is exact in any order, so the GPU must match the oracle bit for bit,
including the single rounding of the scale multiply; with N(0,1) activations
the per-row bound is 1e-4 · max|oracle|.
"""
import numpy as np
import pytest

import oracle
import synth
from golden import fixtures
from gpu_helpers import assert_rows_close, ternary

pytestmark = pytest.mark.gpu
REL = 1e-4


def test_handworked_example():
    fx = fixtures.read("ternary_handworked.txt")
    W = np.array(fixtures.hexbytes(fx["bytes"]), np.uint8)
    x = np.array([fixtures.ints(fx["x"])], np.float32)
    assert ternary(x, W, 1.0, 8, 1)[0, 0] == float(fx["dot"])
    assert ternary(x, W, float(fx["scale"]), 8, 1)[0, 0] == np.float32(fx["y"])


@pytest.mark.parametrize("T", [1, 16])
def test_workload_integer_bit_exact(T):
    x, W, scale, K, N, T = synth.ternary_case((2560, 6912, T), xkind="int")
    dot, y_ref = oracle.ternary_gemv(x, W, scale, K, N)
    y1 = ternary(x, W, 1.0, K, N)
    assert np.array_equal(y1.astype(np.float64), dot), "code-dot not exact"
    y = ternary(x, W, scale, K, N)
    assert y.tobytes() == y_ref.tobytes(), "scaled output not bit-exact"


@pytest.mark.parametrize("T", [1, 16])
def test_workload_normal(T):
    x, W, scale, K, N, T = synth.ternary_case((2560, 6912, T))
    dot, _ = oracle.ternary_gemv(x, W, scale, K, N)
    y = ternary(x, W, scale, K, N)
    assert_rows_close(y, dot * np.float64(scale), REL, f"ternary T{T}")


ODD = [(4, 1, 1), (8, 3, 2), (12, 5, 1), (100, 33, 3), (2564, 7, 1), (4100, 9, 9), (64, 1000, 1),
       (8192, 65, 17), (6000, 13, 8), (16, 2, 4)]
# Shapes for the streamed kernels (K % 64 == 0, 16-byte aligned weights):
# K % 256 == 0 with up to 3 tokens runs on the shared byte-plane kernel,
# everything else on the float one-token kernel (one token) and the
# register-tile kernel (2..8-token tiles, several K chunks); K = 65536 is
# beyond the shared kernel's geometry.
STREAMED = [(64, 1, 1), (128, 48, 2), (2560, 100, 3), (6400, 37, 5), (7680, 20, 1), (7744, 3, 1),
            (2560, 6913, 1), (1024, 4097, 16), (256, 1, 8), (65536, 2, 1), (65536, 3, 9),
            (4096, 300, 12), (512, 152 * 8 + 5, 1), (2560, 49, 7)]


@pytest.mark.parametrize("K,N,T", ODD, ids=[f"K{k}_N{n}_T{t}" for k, n, t in ODD])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_odd_shapes_and_unaligned_weights(K, N, T, offset):
    x, W, scale, K, N, T = synth.ternary_case((K, N, T), seed=K + N + T, xkind="int")
    _, y_ref = oracle.ternary_gemv(x, W, scale, K, N)
    y = ternary(x, W, scale, K, N, weight_offset=offset)
    assert y.tobytes() == y_ref.tobytes()


@pytest.mark.parametrize("K,N,T", STREAMED, ids=[f"K{k}_N{n}_T{t}" for k, n, t in STREAMED])
def test_streamed_shapes_integer_bit_exact(K, N, T):
    x, W, scale, K, N, T = synth.ternary_case((K, N, T), seed=3 * K + N + T, xkind="int")
    dot, y_ref = oracle.ternary_gemv(x, W, scale, K, N)
    assert np.array_equal(ternary(x, W, 1.0, K, N).astype(np.float64), dot)
    assert ternary(x, W, scale, K, N).tobytes() == y_ref.tobytes()


@pytest.mark.parametrize("K,N,T", STREAMED[:8], ids=[f"K{k}_N{n}_T{t}" for k, n, t in STREAMED[:8]])
def test_streamed_shapes_normal(K, N, T):
    x, W, scale, K, N, T = synth.ternary_case((K, N, T), seed=5 * K + N + T)
    dot, _ = oracle.ternary_gemv(x, W, scale, K, N)
    assert_rows_close(ternary(x, W, scale, K, N), dot * np.float64(scale), REL, f"K{K} N{N} T{T}")


def test_field_value_three_decodes_to_plus_two():
    # The literal formula maps bits 11 to +2; both sides decode it that way.
    K, N = 64, 3
    W = np.full((N, K // 4), 0xFF, np.uint8)
    W[1] = 0xAA  # all fields 2 → +1
    W[2] = 0x00  # all fields 0 → −1
    for T in (1, 2, 9):  # the one-token, tile and fallback kernels
        x = synth.activations(synth.rng(1), T, K, "int")
        dot, y_ref = oracle.ternary_gemv(x, W, 1.0, K, N)
        y = ternary(x, W, 1.0, K, N)
        assert y.tobytes() == y_ref.tobytes()
        assert np.array_equal(dot[:, 0], 2 * x.astype(np.float64).sum(1))


@pytest.mark.parametrize("T", [1, 16])
def test_run_to_run_bit_identity(T):
    x, W, scale, K, N, T = synth.ternary_case((2560, 6912, T))
    a = ternary(x, W, scale, K, N)
    b = ternary(x, W, scale, K, N)
    assert a.tobytes() == b.tobytes()


def test_bench_shape_sixteen_tokens_normal():
    # The 16-token bench workload's shape with N(0,1) activations.
    x, W, scale, K, N, T = synth.ternary_case("ternary_gemv_2560x6912_t16")
    dot, _ = oracle.ternary_gemv(x, W, scale, K, N)
    assert_rows_close(ternary(x, W, scale, K, N), dot * np.float64(scale), REL, "2560x6912 T16")
