"""q4k_matmul_tc_noalloc: the tensor-core Q4_K product with its scratch in a
fixed device array inside the library, for callers that cannot allocate
device memory during a call (a host framework whose allocator owns the whole
device budget, a set-up without stream-ordered memory pools, a serving loop
that keeps allocator calls off its hot path).

It must give exactly what q4k_matmul_tc gives (the same kernels run, only
the scratch differs), on calls in a row: the first two use the array (more
than 128 tokens), the second smaller than the first, so it runs over a
scratch array that still holds the first call's data; the third needs no
scratch.  Two calls issued back to back on one stream, with no
synchronisation between them and different activations, must both be
right: the second call's rounding of x into the array waits for the first
call's kernels, which still read it.  A call that needs more scratch than
the array holds is refused before anything is launched.

This file is collected last on purpose (pytest orders files by name)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
REL = 1e-4
FIXED_BYTES = 16 << 20
DIM = -1


def _run(entry, x, W, K, N):
    """Call a raw-pointer entry point (the C ABI) on device copies of x and W;
    returns y as numpy.  y starts as NaN so that unwritten outputs show."""
    import torch
    T = x.shape[0]
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    wd = torch.from_numpy(np.ascontiguousarray(W, np.uint8).reshape(-1)).cuda()
    yd = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    entry(xd.data_ptr(), wd.data_ptr(), yd.data_ptr(), K, N, T, stream)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def _assert_rows_close(got, ref, what):
    assert np.all(np.isfinite(got)), f"{what}: unwritten or non-finite output"
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    for t in range(ref.shape[0]):
        err = np.abs(got[t] - ref[t]).max()
        scale = np.abs(ref[t]).max()
        assert err <= REL * scale, f"{what}: token {t}: max err {err:.3e} > {REL:g} x {scale:.3e}"


def test_two_calls_in_a_row_match_the_allocating_entry_point():
    import quantized_matmul_q4_gb300 as q
    # (tokens, inputDim, outputDim, seed).  Above 128 tokens the bf16 copy of
    # x goes into the array; the second of those calls is the smaller one.
    cases = [(200, 4096, 1000, 11), (150, 1024, 300, 12), (64, 4096, 1000, 13)]
    for T, K, N, seed in cases:
        g = synth.rng(seed)
        W = synth.q4k_weights(g, N, K)
        x = synth.activations(g, T, K)
        ref = _run(q.q4k_matmul_tc_ptr, x, W, K, N)
        got = _run(q.q4k_matmul_tc_noalloc_ptr, x, W, K, N)
        assert np.all(np.isfinite(got)), f"T={T}: unwritten or non-finite output"
        assert got.tobytes() == ref.tobytes(), f"T={T} K={K} N={N}: differs from q4k_matmul_tc"
    q.device_status()


def test_back_to_back_on_one_stream_without_sync():
    import torch
    import oracle
    import quantized_matmul_q4_gb300 as q
    # Two calls of 200 and 180 tokens with different x, issued one after the
    # other on the same stream, both through the shared array, then checked
    # against the bf16-operand oracle and bit for bit against q4k_matmul_tc.
    K, N = 2048, 300
    g = synth.rng(17)
    W = synth.q4k_weights(g, N, K)
    xs = [synth.activations(g, 200, K), synth.activations(g, 180, K)]
    wd = torch.from_numpy(np.ascontiguousarray(W).reshape(-1)).cuda()
    xd = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in xs]
    yd = [torch.full((x.shape[0], N), float("nan"), dtype=torch.float32, device="cuda") for x in xs]
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    for x, y in zip(xd, yd):
        q.q4k_matmul_tc_noalloc_ptr(x.data_ptr(), wd.data_ptr(), y.data_ptr(), K, N, x.shape[0], stream)
    torch.cuda.synchronize()
    q.device_status()
    for x, y in zip(xs, yd):
        got = y.cpu().numpy()
        _assert_rows_close(got, oracle.q4k_matmul_bf16(x, W, K, N), f"T={x.shape[0]} back to back")
        ref = _run(q.q4k_matmul_tc_ptr, x, W, K, N)
        assert got.tobytes() == ref.tobytes(), f"T={x.shape[0]}: back-to-back result differs from q4k_matmul_tc"


def test_oversize_call_is_refused_before_launch():
    import torch
    import quantized_matmul_q4_gb300 as q
    # 1040 tokens of an 8192 -> 256 layer: 16.25 MiB of bf16 activations.
    T, K, N = 1040, 8192, 256
    need = (T * K * 2 + 255) // 256 * 256
    assert need > FIXED_BYTES
    x = torch.zeros(T * K, dtype=torch.float32, device="cuda")
    w = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    y = torch.full((T * N,), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(q.Q4mmError) as e:
        q.q4k_matmul_tc_noalloc_ptr(x.data_ptr(), w.data_ptr(), y.data_ptr(), K, N, T,
                                    torch.cuda.current_stream().cuda_stream)
    assert e.value.code == DIM
    assert "scratch" in q.last_error()
    torch.cuda.synchronize()
    assert bool(torch.all(y == 7.0)), "a refused call must leave y untouched"
