"""GPU parity of the Q4_0 GEMV (q4_0_gemv) against the CPU oracle.

The block is the follow-up format named by SKaiNET PR #562 "feat(kernel):
SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI" (section "Out of scope":
32 values in 18 bytes, same algorithm), read with ggml's byte layout (fp16 d,
then 16 bytes of nibbles: low nibbles elements 0..15, high nibbles 16..31;
w = d·(q − 8)).  Tolerance as for Q4_K (section "Test plan"): per token row t,
max_o |gpu − oracle| <= 1e-4 · max_o |oracle|.  Cases: the hand-worked block
(exact), one-hot activations (element order), a shape sweep with ragged row
counts up to the largest inputDim, several tokens, the bench workload's shape,
wide dynamic range inside a block, and run-to-run bit identity.
"""
import numpy as np
import pytest

import oracle
import synth
from golden import fixtures
from gpu_helpers import GUARD, GUARD_VALUE, assert_rows_close, dev

pytestmark = pytest.mark.gpu
REL = 1e-4


def q4_0(x, W, K, N):
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf = torch.full((2 * GUARD + T * N,), float(GUARD_VALUE), dtype=torch.float32, device="cuda")
    out = buf[GUARD:GUARD + T * N]
    q.q4_0_gemv(dev(x), dev(np.ascontiguousarray(W, np.uint8).reshape(-1)), N=N, out=out)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD] == GUARD_VALUE) and np.all(b[GUARD + T * N:] == GUARD_VALUE), "write outside y"
    q.device_status()
    return out.view(T, N).cpu().numpy()


def test_handworked_block_exact():
    # The fixture's block repeated over a 256-value row (eight blocks), so the
    # row's result is eight times the block's, exactly.
    fx = fixtures.read("q4_0_handworked_block.txt")
    q = list(range(16)) + [(7 + l) % 16 for l in range(16)]
    blk = oracle.q4_0_pack_block(int(fx["d_bits"], 16), q)
    W = np.tile(blk, 8)[None, :]
    xb = np.array([(e % 3) - 1 for e in range(32)], np.float32)
    x = np.stack([np.tile(xb, 8), np.ones(256, np.float32)])
    y = q4_0(x, W, 256, 1)
    assert y[0, 0] == 8 * float(fx["y_x_mod3"])
    assert y[1, 0] == 8 * float(fx["sum_w"])


def test_one_hot_reproduces_weights():
    K, N = 512, 37
    g = synth.rng(31)
    W = synth.q4_0_weights(g, N, K)
    w = oracle.q4_0_dequant(W, K, N)
    for k in (0, 1, 15, 16, 17, 31, 32, 63, 64, 100, 255, 256, 300, 511):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y = q4_0(x, W, K, N)
        assert np.abs(y[0] - w[:, k]).max() <= 1e-6 * np.abs(w).max(), k


SWEEP = [(256, 1), (256, 37), (512, 1000), (768, 5), (1024, 1024), (2048, 17), (4096, 33),
         (4096, 4096), (11008, 33), (14336, 9), (16384, 5), (32768, 3)]


@pytest.mark.parametrize("K,N", SWEEP, ids=[f"K{k}_N{n}" for k, n in SWEEP])
def test_shape_sweep(K, N):
    x, W, K, N, T = synth.q4_0_case((K, N, 1), seed=K + 3 * N)
    assert_rows_close(q4_0(x, W, K, N), oracle.q4_0_matmul(x, W, K, N), REL, f"K{K} N{N}")


@pytest.mark.parametrize("T", [2, 3])
def test_several_tokens(T):
    x, W, K, N, T = synth.q4_0_case((1024, 300, T), seed=40 + T)
    assert_rows_close(q4_0(x, W, K, N), oracle.q4_0_matmul(x, W, K, N), REL, f"T{T}")


def test_bench_workload_full():
    x, W, K, N, T = synth.q4_0_case("q4_0_gemv_4096x4096_t1")
    assert_rows_close(q4_0(x, W, K, N), oracle.q4_0_matmul(x, W, K, N), REL, "4096x4096")


def test_wide_dynamic_range():
    # One value per 256-value group 1000 times larger than the others (as in
    # the Q4_K test): the small activations must still count.
    K, N = 4096, 96
    g = synth.rng(55)
    W = synth.q4_0_weights(g, N, K)
    x = g.uniform(-1.0, 1.0, size=(1, K)).astype(np.float32)
    spikes = g.integers(0, 256, size=K // 256) + 256 * np.arange(K // 256)
    x[0, spikes] = np.float32(1000.0) * np.sign(g.uniform(-1, 1, size=spikes.size)).astype(np.float32)
    assert_rows_close(q4_0(x, W, K, N), oracle.q4_0_matmul(x, W, K, N), REL, "spikes")


def test_run_to_run_bit_identity():
    x, W, K, N, T = synth.q4_0_case((4096, 1000, 1), seed=8)
    assert q4_0(x, W, K, N).tobytes() == q4_0(x, W, K, N).tobytes()
