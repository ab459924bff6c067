"""Failure detection on the GPU without a fault: a bounded in-kernel wait
that runs out sets the device status word, the kernel exits cleanly, the
host reads Q4MM_ERR_TIMEOUT from q4mm_device_status, and the context stays
usable — the next ordinary call is right.

The wait is made to run out through the library's test hook
(q4mm_test_fail_next_wait): the next call never issues the copy of one
weight stage and bounds its waits by about a millisecond.  Nothing is left
in flight, nothing traps or waits without a bound.  Covered: the one-token
kernel (a ring that holds every stage, and one that is reused), a Q6_K
row format whose stages start off the 16-byte grid, the fused gate+up FFN
(1, 4 and 8 tokens), the 3-8 token kernel (single warps and pairs) and the
tensor-core prefill on canonical and relayouted weights and above 128
tokens (clusters of CTAs that still meet at their cluster barriers and
release tensor memory).
"""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_rows_close, dev, gemv

pytestmark = pytest.mark.gpu
LIMIT = 2_000_000   # SM cycles, about a millisecond
TIMEOUT = -5
REL = 1e-4


def _fail_once(call):
    """Arm the hook, run `call` once, and check that it reports a time-out
    within a second; the status word is cleared afterwards."""
    import torch
    import quantized_matmul_q4_gb300 as q
    torch.cuda.synchronize()
    q.device_status()
    q.arm_wait_failure(0, LIMIT)
    t0 = time.perf_counter()
    call()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    with pytest.raises(q.Q4mmError) as e:
        q.device_status()
    assert e.value.code == TIMEOUT
    assert elapsed < 1.0, elapsed
    q.device_status()  # cleared by the read above


def _q4k_case(K, N, T, seed):
    g = synth.rng(seed)
    return synth.q4k_weights(g, N, K), synth.activations(g, T, K)


@pytest.mark.parametrize("K,N,T", [(4096, 4096, 1), (4096, 11008, 1), (4096, 512, 6), (4096, 4096, 4),
                                   (11008, 4096, 3)],
                         ids=["one_token_whole_ring", "one_token_reused_ring", "multi_token", "multi_token_pairs",
                              "multi_token_pairs_wide_rows"])
def test_q4k_wait_runs_out_then_next_call_is_right(K, N, T):
    import torch
    import quantized_matmul_q4_gb300 as q
    W, x = _q4k_case(K, N, T, seed=K + N + T)
    wd, xd = dev(W.reshape(-1)), dev(x)
    junk = torch.empty((T, N), dtype=torch.float32, device="cuda")
    _fail_once(lambda: q.q4k_matmul(xd, wd, N=N, out=junk))
    y = gemv("q4k_matmul", x, W, K, N)
    assert_rows_close(y, oracle.q4k_matmul(x, W, K, N), REL, "after a time-out")


def test_q6k_wait_runs_out_then_next_call_is_right():
    import torch
    import quantized_matmul_q4_gb300 as q
    K, N = 4352, 3000  # 17 blocks: rows of 3570 bytes, stages off the 16-byte grid
    g = synth.rng(31)
    W, x = synth.q6k_weights(g, N, K), synth.activations(g, 1, K)
    junk = torch.empty((1, N), dtype=torch.float32, device="cuda")
    wd, xd = dev(W.reshape(-1)), dev(x)
    _fail_once(lambda: q.q6k_gemv(xd, wd, N=N, out=junk))
    y = gemv("q6k_gemv", x, W, K, N)
    assert_rows_close(y, oracle.q6k_matmul(x, W, K, N), REL, "after a time-out")


def test_tensor_core_wait_runs_out_then_next_call_is_right():
    import torch
    import quantized_matmul_q4_gb300 as q
    K, N, T = 4096, 512, 64
    W, x = _q4k_case(K, N, T, seed=77)
    wd, xd = dev(W.reshape(-1)), dev(x)
    junk = torch.empty((T, N), dtype=torch.float32, device="cuda")
    _fail_once(lambda: q.q4k_matmul_tc(xd, wd, N=N, out=junk))
    y = q.q4k_matmul_tc(xd, wd, N=N).cpu().numpy()
    q.device_status()
    assert_rows_close(y, oracle.q4k_matmul_bf16(x, W, K, N), REL, "after a time-out")


def test_tensor_core_relayouted_and_wide_tile_waits_run_out():
    # The relayouted weight (one bulk copy per chunk), and a 200-token call
    # (the bf16 pre-pass, then tiles whose activations come by TMA).
    import torch
    import quantized_matmul_q4_gb300 as q
    for K, N, T, relay in ((4096, 512, 64, True), (2048, 300, 200, False)):
        W, x = _q4k_case(K, N, T, seed=K + T)
        wd, xd = dev(W.reshape(-1)), dev(x)
        wr = q.q4k_relayout_tc(wd, K, N=N) if relay else None
        junk = torch.empty((T, N), dtype=torch.float32, device="cuda")
        if relay:
            _fail_once(lambda: q.q4k_matmul_tc_relayouted(xd, wr, N=N, out=junk))
            y = q.q4k_matmul_tc_relayouted(xd, wr, N=N).cpu().numpy()
        else:
            _fail_once(lambda: q.q4k_matmul_tc(xd, wd, N=N, out=junk))
            y = q.q4k_matmul_tc(xd, wd, N=N).cpu().numpy()
        q.device_status()
        assert_rows_close(y, oracle.q4k_matmul_bf16(x, W, K, N), REL, f"after a time-out, relay={relay}")


@pytest.mark.parametrize("T", [1, 4, 8], ids=["one_token", "pairs", "eight_tokens"])
def test_fused_ffn_wait_runs_out_then_next_call_is_right(T):
    import torch
    import quantized_matmul_q4_gb300 as q
    K, N = 4096, 11008
    g = synth.rng(41)
    Wg, Wu, x = synth.q4k_weights(g, N, K), synth.q4k_weights(g, N, K), synth.activations(g, T, K)
    gd, ud, xd = dev(Wg.reshape(-1)), dev(Wu.reshape(-1)), dev(x)
    junk = torch.empty((T, N), dtype=torch.float32, device="cuda")
    _fail_once(lambda: q.q4k_ffn_swiglu(xd, gd, ud, N=N, out=junk))
    h = q.q4k_ffn_swiglu(xd, gd, ud, N=N).cpu().numpy()
    q.device_status()
    g_ref, u_ref, h_ref = oracle.q4k_ffn_swiglu(x, Wg, Wu, K, N)
    silu = 0.5 * g_ref * (1.0 + np.tanh(0.5 * g_ref))  # g·sigmoid(g), no overflow
    # The fused FFN's bound (1e-4 on g and u, silu 1.1-Lipschitz), per token.
    bound = 1e-4 * np.abs(u_ref).max() * (1.1 * np.abs(g_ref).max() + np.abs(silu).max()) + 1e-6 * np.abs(h_ref).max()
    assert np.abs(h - h_ref).max() <= bound, "after a time-out"
