"""Launch geometry of the one-token and the 3-8 token GEMV kernels, checked
on the CPU.

The library's own host headers (csrc/t1_geometry.h, csrc/multi_geometry.h)
are compiled into a small shim and called over many shapes; the invariants
are re-derived here: every row belongs to one CTA, the ring fits shared
memory, and every wait on a reused ring slot follows the waiting warp's own
consumption of the slot's previous contents (the kernels wait on slot
barriers by phase parity, which names the awaited stage only if the previous
phase is known to be complete).
"""
import ctypes
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
FIELDS = ["ok", "wide", "wc", "pass_rows", "rg", "ncw", "stage_rows", "rows_per_cta", "grid",
          "x_staged", "nslots", "pre_stages", "xs_bytes", "part_bytes", "slot_bytes", "smem", "cw",
          "slot_rows"]
SMS, SMEM = 152, 232448  # GB300: SMs and opt-in shared memory per block


_LIB = []


def _shim(tmp_path_factory):
    if not _LIB:
        out = str(tmp_path_factory.mktemp("geo") / "libgeo.so")
        subprocess.run(["g++", "-std=c++17", "-O1", "-shared", "-fPIC", "-o", out,
                        os.path.join(HERE, "launch_geometry_shim.cpp")], check=True)
        lib = ctypes.CDLL(out)
        lib.t1_plan.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_longlong)]
        lib.multi_plan.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_longlong)]
        _LIB.append(lib)
    return _LIB[0]


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    lib = _shim(tmp_path_factory)

    def call(group_bytes, K, N, T, vrow_mult=1):
        buf = (ctypes.c_longlong * len(FIELDS))()
        sums = 1 if group_bytes == 144 else 0   # the Q4_K geometry (Q4_0 shares its row size, without sums)
        lib.t1_plan(group_bytes, sums, K, N, T, vrow_mult, SMS, SMEM, buf)
        return dict(zip(FIELDS, buf))
    return call


FORMATS = {"q4k": (144, (1, 2, 3, 4)), "q4_0": (144, (1, 2, 8)), "q6k": (210, (1, 2, 8)),
           "ternary": (64, (1, 2, 3))}


@pytest.mark.parametrize("fmt", sorted(FORMATS))
def test_geometry_invariants(plan, fmt):
    gb, Ts = FORMATS[fmt]
    checked = 0
    for K in range(256, 32768 + 1, 256):
        for T in Ts:
            for N in (1, 256, 4096, 11008, 32000):
                for vm in ((1, 2) if fmt == "q4k" and T == 1 else (1,)):
                    g = plan(gb, K, N, T, vm)
                    if not g["ok"]:
                        continue
                    checked += 1
                    rows, grid = g["rows_per_cta"], g["grid"]
                    assert grid * rows >= N and (grid - 1) * rows < N, (K, N, T)
                    assert 1 <= grid <= SMS
                    # A slot holds its stage from the 16-byte boundary below it.
                    row_bytes = (K // 256) * gb
                    pad = 16 if row_bytes % 16 else 0
                    assert g["slot_bytes"] % 16 == 0 and g["slot_bytes"] >= g["stage_rows"] * row_bytes + (pad and 15)
                    assert g["smem"] <= SMEM
                    assert g["smem"] == g["xs_bytes"] + g["nslots"] * g["slot_bytes"] + \
                        16 * g["nslots"] + g["part_bytes"]
                    assert g["ncw"] == T * g["wc"] * g["rg"] <= g["cw"]
                    stages = -(-vm * rows // g["stage_rows"])
                    assert g["cw"] == 16 and 1 <= g["nslots"] <= 16
                    # One slot only for a single stage, or where two do not fit
                    # (its stages then go in turn).
                    assert g["nslots"] > 1 or stages == 1 or \
                        g["xs_bytes"] + 2 * g["slot_bytes"] + g["part_bytes"] + 32 > SMEM
                    # A pass (4 or 2 rows per row slot) never straddles two stages.
                    assert g["slot_rows"] in (4, 2)
                    assert g["stage_rows"] % g["pass_rows"] == 0 and g["pass_rows"] % g["slot_rows"] == 0
                    # Stages are the fewest whole passes of at least 16 KB (or
                    # every row of the CTA), or, where that leaves a streaming
                    # ring under 4 slots, the same of a pass of every row
                    # group.  Consumers wait on a slot's stage tag before its
                    # parity, so any ring depth is sound.
                    def stage_of(sq):
                        want = sq * max(1, -(-16384 // (sq * row_bytes)))
                        return min(want, sq * -(-vm * rows // sq))
                    assert g["stage_rows"] in (stage_of(g["pass_rows"]), stage_of(g["pass_rows"] * g["rg"])), \
                        (fmt, K, N, T, vm, g)
                    if g["stage_rows"] != stage_of(g["pass_rows"]):
                        assert g["nslots"] < 4 or g["stage_rows"] == stage_of(g["pass_rows"] * g["rg"])
    assert checked > 500


def test_known_geometries(plan):
    # 4096²: 147 CTAs (4 SMs spare) of 28 rows, eight row groups of two
    # warps for seven 4-row passes; four 8-row stages, no reuse.
    g = plan(144, 4096, 4096, 1)
    assert (g["grid"], g["rows_per_cta"], g["rg"], g["stage_rows"], g["nslots"]) == (147, 28, 8, 8, 4)
    # 16384²: a long launch keeps every SM; two row groups of eight warps;
    # staged x (64 KB) would leave room for only two 4-row stages, so the
    # threads load x themselves and four 4-row stages (36.9 KB) are in
    # flight.
    g = plan(144, 16384, 16384, 1)
    assert (g["grid"], g["rg"], g["stage_rows"], g["nslots"], g["x_staged"]) == (152, 2, 4, 4, 0)
    # 14336²: the same trade (x would leave three slots).
    g = plan(144, 14336, 14336, 1)
    assert (g["stage_rows"], g["nslots"], g["x_staged"]) == (4, 5, 0)
    # 12288²: x staged still leaves four 4-row slots, so it stays staged.
    g = plan(144, 12288, 12288, 1)
    assert (g["stage_rows"], g["nslots"], g["x_staged"]) == (4, 4, 1)
    # 8192²: x staged, eight 4-row stages of 18.4 KB in flight.
    g = plan(144, 8192, 8192, 1)
    assert (g["stage_rows"], g["nslots"], g["x_staged"]) == (4, 8, 1)
    # 32768-wide rows take all 16 warps; odd-width Q6_K rows that wide fall
    # back to 2-row passes.
    g = plan(144, 32768, 1024, 1)
    assert g["ok"] and g["wc"] == 16
    g = plan(210, 31488, 4096, 1)
    assert g["ok"] and g["slot_rows"] == 2
    # Rows too wide for 16 compute warps, or too many tokens for the row width.
    assert not plan(144, 33024, 64, 1)["ok"]
    assert not plan(144, 11008, 64, 3)["ok"]


def test_streaming_launches_keep_stages_in_flight(plan):
    # A CTA whose rows all fit the ring holds them all; a streaming CTA keeps
    # at least four pass-sized stages in flight, or two stages of a pass of
    # every row group.
    for K, N in ((4096, 4096), (4096, 11008)):
        g = plan(144, K, N, 1)
        assert g["nslots"] * g["stage_rows"] >= g["rows_per_cta"], (K, N, g)
    for K, N in ((8192, 8192), (11008, 4096), (16384, 16384)):
        g = plan(144, K, N, 1)
        assert g["nslots"] * g["stage_rows"] < g["rows_per_cta"], (K, N, g)
        assert g["nslots"] >= 4 or g["stage_rows"] % (g["pass_rows"] * g["rg"]) == 0, (K, N, g)


MULTI = ["ok", "grid", "rows_per_cta", "nslots", "consumers", "smem", "x_staged"]


@pytest.fixture(scope="module")
def multi(tmp_path_factory):
    lib = _shim(tmp_path_factory)

    def call(K, N, ring_bytes=200 * 1024, T=0, vrow_mult=1):
        buf = (ctypes.c_longlong * len(MULTI))()
        lib.multi_plan(K, N, SMS, SMEM, ring_bytes, T, vrow_mult, buf)
        return dict(zip(MULTI, buf))
    return call


def test_multi_token_ring_slots_have_one_consumer(multi):
    # Compute warp c takes groups c, c + n, … (n consumers); the group in
    # slot s is always taken by warp s mod n, and a warp meets its slot again
    # exactly one ring lap later, so it has consumed the slot's previous
    # group itself before it waits on the next.
    checked = 0
    for ring, vm in ((200 * 1024, 1), (128 * 1024, 1), (64 * 1024, 1), (8192, 1), (200 * 1024, 2)):
        for K in range(256, 32768 + 1, 256):
            for N in (1, 5, 100, 4096, 11008, 32000):
                g = multi(K, N, ring, 0, vm)
                if not g["ok"]:
                    continue
                checked += 1
                n, c = g["nslots"], g["consumers"]
                rows, grid = g["rows_per_cta"], g["grid"]
                assert rows % 4 == 0 and grid * rows >= N and (grid - 1) * rows < N
                assert g["smem"] <= SMEM and n >= 1
                assert c == min(7, n) and n % c == 0
                groups = rows // 4
                owner, last = {}, {}
                for grp in range(groups):
                    slot, warp = grp % n, grp % c
                    assert owner.setdefault(slot, warp) == warp, (K, N, ring, n)
                    if slot in last:
                        assert grp - last[slot] == n
                    last[slot] = grp
    assert checked > 1000


def _pair_order_safe(groups, L):
    """The pair protocol's happens-before order for one pair's groups
    0..groups-1, L = the pair's groups between two uses of one ring slot.
    Events: S2(k) the second warp starts group k, W2(k) it writes buffer
    k mod 2 and arrives on that buffer's barrier, R1(k) the first warp reads
    it, E1(k) / E2(k) the warps release the slot (E2 before W2, E1 after
    R1).  S2(k) needs the slot refilled: E1(k - L) and E2(k - L).  True if
    every W2(k) comes after R1(k - 2) (the buffer and barrier are free)."""
    import functools

    @functools.lru_cache(maxsize=None)
    def before(a, b):  # is event a ordered before event b?
        if a == b:
            return True
        kind, k = b
        preds = []
        if kind == "S2" and k >= L:
            preds += [("E1", k - L), ("E2", k - L)]
        if kind in ("S2",) and k >= 1:
            preds.append(("W2", k - 1))  # the second warp's program order
        if kind == "E2":
            preds.append(("S2", k))
        if kind == "W2":
            preds.append(("E2", k))
        if kind == "R1":
            preds.append(("W2", k))
            if k >= 1:
                preds.append(("E1", k - 1))  # the first warp's program order
        if kind == "E1":
            preds.append(("R1", k))
        return any(before(a, p) for p in preds)

    return all(before(("R1", k - 2), ("W2", k)) for k in range(2, groups))


def test_multi_token_pairs_reuse_buffers_in_order(multi):
    # Up to 4 tokens a pair of warps takes each group (the first over half of
    # the blocks, the second over the rest), the second handing its sums to
    # the first through one of two buffers chosen by the group's parity, and
    # the first releasing the ring slot only after reading them.  That keeps
    # the second at most one group ahead only while a slot comes back to the
    # pair every one or two of its groups (nslots <= 2 pairs): checked for
    # every geometry, with the order derived from the barriers.
    assert _pair_order_safe(8, 1) and _pair_order_safe(8, 2) and not _pair_order_safe(8, 3)
    checked = 0
    for T, vm in ((1, 1), (2, 1), (3, 1), (4, 1), (3, 2), (4, 2)):
        for K in range(256, 32768 + 1, 512):
            for N in (1, 5, 100, 4096, 11008, 32000):
                g = multi(K, N, 200 * 1024, T, vm)
                if not g["ok"]:
                    continue
                checked += 1
                n, c = g["nslots"], g["consumers"]
                groups = -(-(g["rows_per_cta"] // 4) // c)  # a pair's groups, at most
                assert n % c == 0 and _pair_order_safe(groups, n // c), (K, N, T, n, c)
    assert checked > 500


def test_multi_token_known_geometries(multi):
    # 14336-wide rows: six 32 KB slots fit, so six consumer warps, one each.
    g = multi(14336, 4096)
    assert (g["nslots"], g["consumers"]) == (6, 6)
    # 4096 -> 11008: 19 groups per CTA, 16 slots would fit; 14 keep two per warp.
    g = multi(4096, 11008)
    assert (g["nslots"], g["consumers"]) == (14, 7)


def test_multi_token_x_staged_where_it_fits(multi):
    # x (T·K fp32) goes into shared memory when it fits beside one ring slot
    # per consumer warp; the slot rule (one consumer per slot, slots a
    # multiple of the consumers) holds either way.
    for K in range(256, 32768 + 1, 256):
        for T in (2, 4, 5, 8):
            for N in (100, 4096, 11008):
                g = multi(K, N, 200 * 1024, T)
                if not g["ok"]:
                    continue
                n, c = g["nslots"], g["consumers"]
                assert g["smem"] <= SMEM and c == min(7, n) and n % c == 0
                row_bytes = (K // 256) * 144
                if g["x_staged"]:
                    assert g["smem"] >= T * K * 4 + n * 4 * row_bytes
    assert multi(4096, 4096, 200 * 1024, 8)["x_staged"] == 1
    assert multi(4096, 11008, 200 * 1024, 8)["x_staged"] == 1
    assert multi(11008, 4096, 200 * 1024, 8)["x_staged"] == 0
    # The fused gate+up at 8 tokens on 4096 -> 11008: slots of both weights'
    # rows (18.4 KB) leave no room for 128 KB of staged x beside seven of
    # them, so x is loaded by the threads and every consumer warp has a slot.
    g = multi(4096, 11008, 200 * 1024, 8, 2)
    assert (g["nslots"], g["consumers"], g["x_staged"]) == (7, 7, 0) and g["smem"] <= SMEM
    # 32768-wide rows: two slots of both weights' rows (147 KB each) do not
    # fit, so the fused FFN falls back to one-token launches.
    assert multi(32768, 4096, 200 * 1024, 4, 2)["ok"] == 0 and multi(32768, 4096, 200 * 1024, 4, 1)["ok"] == 1


def test_q4k_matmul_kernel_choice(tmp_path_factory):
    # q4k_matmul's kernel per token count (csrc/dispatch.h): the byte-plane
    # kernel for 1-2 tokens, the register-tile kernel for 3-8, its 8-token
    # chunks up to 32 tokens or when 64-token tiles (3 CTAs per 128 rows)
    # would leave SMs without a CTA, else the FP32 tile kernel.
    lib = _shim(tmp_path_factory)
    lib.q4k_path.argtypes = [ctypes.c_int] * 3
    ONE, TILE, CHUNKS, FP32 = 0, 1, 2, 3
    cases = [((1, 4096), ONE), ((2, 11008), ONE), ((3, 4096), TILE), ((8, 11008), TILE), ((9, 4096), CHUNKS),
             ((32, 11008), CHUNKS), ((33, 11008), FP32), ((64, 11008), FP32), ((64, 4096), CHUNKS),
             ((500, 4096), CHUNKS), ((64, 6400), CHUNKS), ((64, 6528), FP32), ((1000, 32000), FP32)]
    for (T, N), want in cases:
        assert lib.q4k_path(T, N, SMS) == want, (T, N)
