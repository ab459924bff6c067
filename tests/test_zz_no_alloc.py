"""q4k_matmul_tc_noalloc: the tensor-core Q4_K product with its scratch in a
fixed device array inside the library, for callers that cannot allocate
device memory during a call (a host framework whose allocator owns the whole
device budget, a set-up without stream-ordered memory pools, a serving loop
that keeps allocator calls off its hot path).

It must give what q4k_matmul_tc gives, within the tensor-core tests'
tolerance (1e-4 of each token row's largest output), on calls in a row: the
first two use the array (more than 128 tokens), the second smaller than the
first, so it runs over a scratch array that still holds the first call's
data; the third needs no scratch.  A call that needs more scratch than
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
        _assert_rows_close(got, ref, f"T={T} K={K} N={N}")
    q.device_status()


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
