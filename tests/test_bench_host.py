"""Host logic of the benchmark on CPU: the multi-process plumbing (gloo, world size 2) and
the reference arm's JSON line.

The layer has no exchange step, so N GPUs run N independent replicas: the only
cross-rank traffic is the barrier around the timed region and the max of the
per-rank step times.  These tests run that plumbing as two gloo ranks on the
host, with no GPU."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, ms_of_rank, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_setup(world)
    try:
        bench.barrier(w)
        ms = bench.max_over_ranks(ms_of_rank[r], w)
        q.put((r, w, local, dist.get_backend(), ms, bench.job_rate(8192, w, ms)))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_sum_the_units():
    world, port = 2, _free_port()
    ms_of_rank = [0.61, 0.67]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms_of_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(world))
    for r, (rank, w, local, backend, ms, rate) in enumerate(got):
        assert (rank, w, local, backend) == (r, world, r, "gloo")
        assert ms == max(ms_of_rank)  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 8192 / 0.67e-3)  # units of both replicas / slowest time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_rate(8192, 1, 0.5) == pytest.approx(8192 / 0.5e-3)


def test_reference_arm_on_a_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line_on_cpu():
    # the oracle arm runs on host cores only: one step on a 2-token sample
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--cpu-tokens", "2"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env={k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and "2 tokens" in d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    sys.path.insert(0, ROOT)
    import bench
    from bit_grouped_expert_top_gb300.inputs import CONFIGS
    assert d["config"] == bench.workload_config(CONFIGS["prefill_t8192"], 1)  # the GPU arm's config
