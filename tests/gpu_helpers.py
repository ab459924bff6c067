"""Helpers for the GPU parity tests: move seeded inputs to the device, call the
C ABI through the binding, and compare with the oracle per token row."""
from __future__ import annotations

import numpy as np

GUARD = 64  # guard elements on each side of every output buffer
GUARD_VALUE = np.float32(-12345.678)


def dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _guarded_out(T, N):
    import torch
    buf = torch.full((2 * GUARD + T * N,), float(GUARD_VALUE), dtype=torch.float32, device="cuda")
    return buf, buf[GUARD:GUARD + T * N]


def _check_guards(buf, T, N):
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD] == GUARD_VALUE), "write before the output buffer"
    assert np.all(b[GUARD + T * N:] == GUARD_VALUE), "write past the output buffer"


def q4k(x: np.ndarray, W: np.ndarray, K: int, N: int, tc: bool = False) -> np.ndarray:
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf, out = _guarded_out(T, N)
    fn = q.q4k_matmul_tc if tc else q.q4k_matmul
    fn(dev(x), dev(W.reshape(-1)), N=N, out=out)
    torch.cuda.synchronize()
    _check_guards(buf, T, N)
    q.device_status()
    return out.view(T, N).cpu().numpy()


def ternary(x: np.ndarray, W: np.ndarray, scale: float, K: int, N: int,
            weight_offset: int = 0) -> np.ndarray:
    """weight_offset > 0 places the packed weight at an odd byte address."""
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf, out = _guarded_out(T, N)
    wflat = np.ascontiguousarray(W, np.uint8).reshape(-1)
    wdev = dev(np.concatenate([np.zeros(weight_offset, np.uint8), wflat]))
    wview = wdev[weight_offset:]
    q.ternary_gemv(dev(x), wview, scale, N=N, out=out)
    torch.cuda.synchronize()
    _check_guards(buf, T, N)
    q.device_status()
    return out.view(T, N).cpu().numpy()


def assert_rows_close(got: np.ndarray, ref: np.ndarray, rel: float, what: str = ""):
    """Per token row t: max_o |got − ref| <= rel · max_o |ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    for t in range(ref.shape[0]):
        err = np.abs(got[t] - ref[t]).max()
        scale = np.abs(ref[t]).max()
        assert err <= rel * scale, f"{what}: token {t}: max err {err:.3e} > {rel:g} x {scale:.3e}"


def max_rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return max(float(np.abs(got[t] - ref[t]).max() / max(np.abs(ref[t]).max(), 1e-300))
               for t in range(ref.shape[0]))


def gemv(fn_name: str, x: np.ndarray, W: np.ndarray, K: int, N: int) -> np.ndarray:
    """Call the tensor entry point `fn_name` (q4k_matmul, q4_0_gemv, q6k_gemv)
    on device copies of x and W with a guarded output; returns y [T, N]."""
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf, out = _guarded_out(T, N)
    getattr(q, fn_name)(dev(x), dev(np.ascontiguousarray(W, np.uint8).reshape(-1)), N=N, out=out)
    torch.cuda.synchronize()
    _check_guards(buf, T, N)
    q.device_status()
    return out.view(T, N).cpu().numpy()


def ffn(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, K: int, N: int) -> np.ndarray:
    """q4k_ffn_swiglu on device copies, guarded output; returns h [T, N]."""
    import torch
    import quantized_matmul_q4_gb300 as q
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf, out = _guarded_out(T, N)
    q.q4k_ffn_swiglu(dev(x), dev(Wg.reshape(-1)), dev(Wu.reshape(-1)), N=N, out=out)
    torch.cuda.synchronize()
    _check_guards(buf, T, N)
    q.device_status()
    return out.view(T, N).cpu().numpy()
