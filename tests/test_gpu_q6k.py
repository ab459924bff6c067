"""GPU parity of the Q6_K GEMV (q6k_gemv) against the CPU oracle.

The block is the second follow-up format named by SKaiNET PR #562
"feat(kernel): SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI" (section
"Out of scope": ql + qh with four codes per qh byte, half-interleaved), read
with ggml's byte layout (210-byte blocks, w = d·scale·(q − 32)).  Tolerance as
for Q4_K (section "Test plan"): per token row t,
max_o |gpu − oracle| <= 1e-4 · max_o |oracle|.  Rows are 210·K/256 bytes, so
most rows and blocks start off the 16-byte grid; the cases cover row counts
that are not multiples of 8 (the last stage ends off the grid), one-hot
activations (element order), the hand-worked block, several tokens, the bench
shape, and run-to-run bit identity.
"""
import numpy as np
import pytest

import oracle
import synth
from golden import fixtures
from gpu_helpers import GUARD, GUARD_VALUE, assert_rows_close, dev

pytestmark = pytest.mark.gpu
REL = 1e-4


def q6k(x, W, K, N):
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf = torch.full((2 * GUARD + T * N,), float(GUARD_VALUE), dtype=torch.float32, device="cuda")
    out = buf[GUARD:GUARD + T * N]
    q.q6k_gemv(dev(x), dev(np.ascontiguousarray(W, np.uint8).reshape(-1)), N=N, out=out)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD] == GUARD_VALUE) and np.all(b[GUARD + T * N:] == GUARD_VALUE), "write outside y"
    q.device_status()
    return out.view(T, N).cpu().numpy()


def test_handworked_block_exact():
    fx = fixtures.read("q6k_handworked_block.txt")
    blk = oracle.q6k_pack_block(int(fx["d_bits"], 16), [s - 8 for s in range(16)],
                                [(5 * v + 3) % 64 for v in range(256)])
    x = np.stack([np.array([(v % 5) - 2 for v in range(256)], np.float32), np.ones(256, np.float32)])
    y = q6k(x, blk[None, :], 256, 1)
    assert y[0, 0] == float(fx["y_x_mod5"])
    assert y[1, 0] == float(fx["sum_w"])


def test_one_hot_reproduces_weights():
    K, N = 512, 37
    g = synth.rng(61)
    W = synth.q6k_weights(g, N, K)
    w = oracle.q6k_dequant(W, K, N)
    for k in (0, 15, 16, 31, 32, 63, 64, 95, 96, 127, 128, 200, 255, 256, 300, 383, 384, 511):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y = q6k(x, W, K, N)
        assert np.abs(y[0] - w[:, k]).max() <= 1e-6 * np.abs(w).max(), k


SWEEP = [(256, 1), (256, 7), (256, 37), (512, 1000), (768, 9), (1024, 1024), (2048, 17), (4096, 33),
         (4096, 4096), (4096, 4093), (11008, 33), (14336, 9), (32768, 5)]


@pytest.mark.parametrize("K,N", SWEEP, ids=[f"K{k}_N{n}" for k, n in SWEEP])
def test_shape_sweep(K, N):
    x, W, K, N, T = synth.q6k_case((K, N, 1), seed=K + 5 * N)
    assert_rows_close(q6k(x, W, K, N), oracle.q6k_matmul(x, W, K, N), REL, f"K{K} N{N}")


@pytest.mark.parametrize("T", [2, 3])
def test_several_tokens(T):
    x, W, K, N, T = synth.q6k_case((1024, 301, T), seed=70 + T)
    assert_rows_close(q6k(x, W, K, N), oracle.q6k_matmul(x, W, K, N), REL, f"T{T}")


def test_bench_workload_full():
    x, W, K, N, T = synth.q6k_case("q6k_gemv_4096x4096_t1")
    assert_rows_close(q6k(x, W, K, N), oracle.q6k_matmul(x, W, K, N), REL, "4096x4096")


def test_run_to_run_bit_identity():
    x, W, K, N, T = synth.q6k_case((4096, 1000, 1), seed=9)
    assert q6k(x, W, K, N).tobytes() == q6k(x, W, K, N).tobytes()
