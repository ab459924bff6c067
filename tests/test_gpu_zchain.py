"""GPU parity of chained launches, in the launch configuration the benchmark
times: consecutive calls on one stream (each kernel may start before the
previous one ends and waits for it before touching activations or outputs),
replayed from a CUDA graph, and the same chain as plain stream launches.

Every launch reads the previous launch's output as its activations
(x_{i+1} = y_i, square matrices), so a kernel that read x or wrote y before
its predecessor had finished would see the NaN the outputs are filled with
beforehand, or a half-written vector.  Each link is checked against the
oracle on the activations the GPU actually used, on sampled output rows,
with the tolerance of its path (1e-4 per token row against max|ref|; the
tensor-core path against the oracle's bf16-operand variant).  The weights'
block scales are smaller than the workloads' generator draws so that the
values stay far inside fp32 range along the chain.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_rows_close

pytestmark = pytest.mark.gpu
REL = 1e-4
LINKS = 6


def _weights(kind, g, K, N):
    if kind == "q4_0":
        return synth.q4_0_weights(g, N, K, d_range=(2e-4, 2e-3))
    if kind == "q6k":
        return synth.q6k_weights(g, N, K, d_range=(2e-5, 2e-4))
    if kind == "ternary":
        return synth.ternary_weights(g, N, K)
    return synth.q4k_weights(g, N, K, d_range=(2e-5, 2e-4), dmin_range=(0.0, 2e-4))


def _entry(kind, tc):
    import quantized_matmul_q4_gb300 as q
    if kind == "q4_0":
        return q.q4_0_gemv_ptr
    if kind == "q6k":
        return q.q6k_gemv_ptr
    if kind == "ternary":
        return None
    return q.q4k_matmul_tc_ptr if tc else q.q4k_matmul_ptr


def _reference(kind, tc, x, W, rows, K, scale):
    Wr = np.ascontiguousarray(W[rows])
    n = len(rows)
    if kind == "q4_0":
        return oracle.q4_0_matmul(x, Wr, K, n)
    if kind == "q6k":
        return oracle.q6k_matmul(x, Wr, K, n)
    if kind == "ternary":
        dot, _ = oracle.ternary_gemv(x, Wr, scale, K, n)
        return dot * np.float64(scale)
    return oracle.q4k_matmul_bf16(x, Wr, K, n) if tc else oracle.q4k_matmul(x, Wr, K, n)


def _run_chain(kind, tc, K, T, Ws, x0, scale, graph):
    import torch
    import quantized_matmul_q4_gb300 as q
    dev = torch.device("cuda")
    wd = [torch.from_numpy(np.ascontiguousarray(W).reshape(-1)).to(dev) for W in Ws]
    bufs = [torch.from_numpy(np.ascontiguousarray(x0)).to(dev)]
    bufs += [torch.empty((T, K), dtype=torch.float32, device=dev) for _ in Ws]
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    entry = _entry(kind, tc)

    def step():
        for i, w in enumerate(wd):
            if kind == "ternary":
                q.ternary_gemv_ptr(bufs[i].data_ptr(), w.data_ptr(), scale, bufs[i + 1].data_ptr(), K, K, T, sp)
            else:
                entry(bufs[i].data_ptr(), w.data_ptr(), bufs[i + 1].data_ptr(), K, K, T, sp)

    def poison():
        torch.cuda.synchronize()
        for b in bufs[1:]:
            b.fill_(float("nan"))
        torch.cuda.synchronize()

    if graph:
        # Library set-up (device query, kernel attributes) outside capture.
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            step()
        poison()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
    else:
        poison()
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
    q.device_status()
    return [b.cpu().numpy() for b in bufs]


CASES = [("q4k", False, 4096, 1), ("q4k", False, 4096, 8), ("q4k", False, 4096, 64), ("q4k", True, 4096, 64),
         ("q4_0", False, 4096, 1), ("q6k", False, 4096, 1), ("ternary", False, 2560, 1)]


@pytest.mark.parametrize("graph", [True, False], ids=["graph", "stream"])
@pytest.mark.parametrize("kind,tc,K,T", CASES, ids=[f"{k}{'_tc' if tc else ''}_K{K}_T{T}" for k, tc, K, T in CASES])
def test_chained_launches(kind, tc, K, T, graph):
    g = synth.rng(K + T + (100 if tc else 0) + len(kind))
    Ws = [_weights(kind, g, K, K) for _ in range(LINKS)]
    scale = float(synth.ternary_scale(g)) * 0.05 if kind == "ternary" else 1.0
    x0 = synth.activations(g, T, K)
    bufs = _run_chain(kind, tc, K, T, Ws, x0, scale, graph)
    rows = np.unique(np.concatenate([[0, K - 1], g.choice(K, 62, replace=False)]))
    for i, W in enumerate(Ws):
        x, y = bufs[i], bufs[i + 1]
        assert np.all(np.isfinite(y)), f"link {i}: non-finite output"
        ref = _reference(kind, tc, x, W, rows, K, scale)
        assert_rows_close(y[:, rows], ref, REL, f"{kind} link {i}")
