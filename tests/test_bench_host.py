"""Host-side checks of bench.py: the multi-rank timing aggregation over gloo
(world size 2, CPU), the reference arm's JSON line, and the traffic record's
invalidation when the kernel sources change."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world, use_cuda=False)
    bench.barrier(dist)
    got = bench.max_over_ranks(values[rank], dist)
    out.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [3.25, 7.5]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == {0: 7.5, 1: 7.5}


def test_reference_arm_json_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "scaling", "dtype", "config",
                "cpu_baseline", "e2e"):
        assert key in line
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_nonzero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT, env=env)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_warmup_minimum():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_traffic_record_tracks_kernel_sources(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    w = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    rec = tmp_path / "summary.md"
    rec.write_text(f"kernel_source_sha256: {bench.kernel_source_hash(w)}\n"
                   "dram_bytes_per_launch: 9500000\n")
    assert bench.profiled_traffic(w, str(rec))[0] == 9500000
    rec.write_text("kernel_source_sha256: 0000\ndram_bytes_per_launch: 9500000\n")
    assert bench.profiled_traffic(w, str(rec))[0] is None


def test_workload_plans():
    # Every workload's step is larger than the 129 MB L2, and its byte and
    # flop counts follow the formats' sizes.
    sys.path.insert(0, ROOT)
    import bench
    for name, w in bench.WORKLOADS.items():
        plan = bench.Plan(w, w.layers)
        assert plan.weight_bytes > 2 * 129e6, name
        assert len(plan.launches) == w.layers * len(w.mats)
        for K, N, wo, xo, yo, m in plan.launches:
            assert wo % 256 == 0 and (K, N) == w.mats[m]
    w = bench.WORKLOADS["q4k_gemv_4096x4096_t1"]
    plan = bench.Plan(w, 64)
    assert plan.weight_bytes == 64 * 9437184
    assert plan.alg_bytes == 64 * (9437184 + 4 * 4096 + 4 * 4096)
    t = bench.Plan(bench.WORKLOADS["ternary_gemv_2560x6912_t16"], 1)
    assert t.weight_bytes == 6912 * 640 and t.flops == 2.0 * 2560 * 6912 * 16
    llama = bench.Plan(bench.WORKLOADS["llama7b_decode_t1"], 32)
    assert llama.weight_bytes == 32 * 113836032
    # 16 tokens: two 8-token kernels per call, the weights counted once.
    w16 = bench.WORKLOADS["llama7b_decode_t16"]
    assert w16.kernels_per_call == 2 and bench.Plan(w16, 32).weight_bytes == llama.weight_bytes
    assert bench.Plan(w16, 1).flops == 16 * bench.Plan(bench.WORKLOADS["llama7b_decode_t1"], 1).flops
    # The fused gate+up at 8 tokens: both weights per call, one kernel.
    ffn8 = bench.Plan(bench.WORKLOADS["llama7b_ffn_swiglu_t8"], 1)
    assert ffn8.weight_bytes == 2 * 11008 * 16 * 144 and bench.WORKLOADS["llama7b_ffn_swiglu_t8"].kernels_per_call == 1
    # Every other workload launches one kernel per call.
    assert all(w.kernels_per_call == 1 for n, w in bench.WORKLOADS.items() if n != "llama7b_decode_t16")


@pytest.mark.parametrize("workload", ["ternary_gemv_2560x6912_t16", "q4k_prefill_tc_4096x11008_t64"])
def test_reference_arm_other_workloads(workload):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["config"]["workload"] == workload and line["value"] > 0
    assert line["unit"] == bench_unit(workload)


def bench_unit(workload):
    sys.path.insert(0, ROOT)
    import bench
    return bench.WORKLOADS[workload].unit
