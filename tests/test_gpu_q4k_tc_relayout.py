"""GPU parity of the one-time relayout (q4k_relayout_tc) and of the
tensor-core prefill on relayouted weights (q4k_matmul_tc_relayouted).

The relayout follows SKaiNET docs "Eager execution: backends and kernels"
(weights relayouted once when registered, not on every call); the target
layout is the library's own (48 bytes per row and 64-value chunk: fp32
d·sc and dmin·m of the chunk's two sub-blocks, then its 32 code bytes;
tile-major, each chunk of a 256-row tile one contiguous run, zero rows
padding the last tile).
Bars:
  * the relayouted bytes equal the oracle's relayout byte for byte (byte
    work), over random blocks and extreme block headers;
  * the relayouted product equals q4k_matmul_tc on the canonical weight bit
    for bit (the same fp32 dequantized values enter the same MMAs in the
    same order), and stays within the bf16 tolerance of the oracle
    (per token row, max_o |gpu − ref| <= 1e-4 · max_o |ref| against the
    bf16-rounded oracle on the canonical weight).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import GUARD, assert_rows_close, dev, q4k

pytestmark = pytest.mark.gpu
REL_BF16 = 1e-4
GUARD_BYTE = 0xA5


def _relayout_gpu(W, K, N):
    import torch
    import quantized_matmul_q4_gb300 as q
    nbytes = q.tc_relayout_bytes(K, N)
    assert nbytes == oracle.q4k_tc_bytes(K, N)
    buf = torch.full((2 * GUARD * 16 + nbytes,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
    out = buf[GUARD * 16:GUARD * 16 + nbytes]
    q.q4k_relayout_tc(dev(np.ascontiguousarray(W, np.uint8).reshape(-1)), K, N=N, out=out)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:GUARD * 16] == GUARD_BYTE), "write before the relayout buffer"
    assert np.all(b[GUARD * 16 + nbytes:] == GUARD_BYTE), "write past the relayout buffer"
    return b[GUARD * 16:GUARD * 16 + nbytes]


def _mm_relayouted(x, R, K, N):
    import torch
    import quantized_matmul_q4_gb300 as q
    from gpu_helpers import _check_guards, _guarded_out
    x = np.ascontiguousarray(x, np.float32).reshape(-1, K)
    T = x.shape[0]
    buf, out = _guarded_out(T, N)
    q.q4k_matmul_tc_relayouted(dev(x), dev(R), N=N, out=out)
    torch.cuda.synchronize()
    _check_guards(buf, T, N)
    q.device_status()
    return out.view(T, N).cpu().numpy()


def _extreme_headers(W, K, N):
    # Subnormal and largest finite fp16 factors, zero factors, and the 6-bit
    # fields all 0 and all 63, on the first rows.
    W = W.reshape(N, K // 256, 144).copy()
    heads = [(0x0001, 0x7BFF), (0x7BFF, 0x0001), (0x0000, 0x3C00), (0x3C00, 0x0000), (0x03FF, 0x0400)]
    for i, (d, dm) in enumerate(heads):
        o, b = divmod(i, K // 256)
        if o < N:
            W[o, b, 0:4] = [d & 255, d >> 8, dm & 255, dm >> 8]
    W[0, 0, 4:16] = 0xFF
    if K >= 512:
        W[0, 1, 4:16] = 0x00
    return W.reshape(-1)


SHAPES = [(256, 1), (512, 300), (768, 5), (4096, 257), (11008, 33), (4096, 11008), (65536, 2)]


@pytest.mark.parametrize("K,N", SHAPES, ids=[f"K{k}_N{n}" for k, n in SHAPES])
def test_relayout_bytes_bit_exact(K, N):
    g = synth.rng(K + N)
    W = _extreme_headers(synth.q4k_weights(g, N, K), K, N)
    got = _relayout_gpu(W, K, N)
    want = oracle.q4k_tc_relayout(W, K, N)
    assert got.tobytes() == want.tobytes()


CASES = [(256, 1, 1), (256, 129, 16), (512, 300, 17), (1024, 1000, 48), (4096, 257, 64), (4096, 65, 65),
         (2048, 130, 128), (4096, 300, 200), (11008, 33, 64), (16384, 9, 20), (65536, 2, 16)]


@pytest.mark.parametrize("K,N,T", CASES, ids=[f"K{k}_N{n}_T{t}" for k, n, t in CASES])
def test_relayouted_product_equals_canonical(K, N, T):
    x, W, K, N, T = synth.q4k_case((K, N, T), seed=3 * K + N + T)
    W = _extreme_headers(W, K, N)
    R = _relayout_gpu(W, K, N)
    y_r = _mm_relayouted(x, R, K, N)
    y_c = q4k(x, W, K, N, tc=True)
    assert y_r.tobytes() == y_c.tobytes()
    assert_rows_close(y_r, oracle.q4k_matmul_bf16(x, W, K, N), REL_BF16, f"relayouted K{K} N{N} T{T}")


def test_one_hot_reproduces_bf16_weights():
    # x = e_k returns bf16(w[:, k]) exactly through the relayouted path:
    # pins the chunk order, the sub-block scales of each half and the rows.
    K, N = 1024, 300
    g = synth.rng(29)
    W = synth.q4k_weights(g, N, K)
    R = oracle.q4k_tc_relayout(W, K, N)
    ks = [0, 31, 32, 63, 64, 95, 96, 127, 255, 256, 511, 512, 767, 800, 1023]
    x = np.zeros((len(ks), K), np.float32)
    for t, k in enumerate(ks):
        x[t, k] = 1.0
    y = _mm_relayouted(x, R, K, N)
    ref = oracle.q4k_matmul_bf16(x, W, K, N).astype(np.float32)
    assert y.tobytes() == ref.tobytes()


def test_prefill_workload_sampled():
    # 64 tokens × 4096 → 11008 on the relayouted weight: equal to the
    # canonical path everywhere, and to the oracle on sampled rows.
    x, W, K, N, T = synth.q4k_case("q4k_prefill_4096x11008_t64")
    R = _relayout_gpu(W, K, N)
    y_r = _mm_relayouted(x, R, K, N)
    y_c = q4k(x, W, K, N, tc=True)
    assert y_r.tobytes() == y_c.tobytes()
    g = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, 255, 256, N - 1], g.choice(N, 128, replace=False)]))
    ref = oracle.q4k_matmul_bf16(x, W.reshape(N, -1)[rows], K, len(rows))
    assert_rows_close(y_r[:, rows], ref, REL_BF16, "relayouted prefill vs bf16 oracle")
