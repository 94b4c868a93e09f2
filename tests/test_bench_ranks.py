"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1
run the same reduction and rate helpers the GPU ranks run (the path shards
by independent heads, so the only cross-rank steps are a barrier and the
max of the elapsed times), and the reference arm prints from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        # rank r measured (1.5 + r) ms for the step and (10 - r) ms end to end
        step_ms, e2e_ms = bench.max_over_ranks([1.5 + rank, 10.0 - rank], dist, "cpu")
        rate = bench.whole_job_rate(3.0e9, world, step_ms)
        out.put((rank, step_ms, e2e_ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(world))
    for rank, step_ms, e2e_ms, rate in res:
        assert step_ms == 2.5          # the slower rank's step time
        assert e2e_ms == 10.0          # the slower rank's end-to-end time
        assert rate == pytest.approx(3.0e9 * 2 / 2.5e-3)  # both ranks' work over that time


def test_world_size_one_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    bench.barrier(None)
    assert bench.max_over_ranks([1.25, 7], None, "cpu") == [1.25, 7.0]
    assert bench.whole_job_rate(1e9, 1, 2.0) == pytest.approx(5e11)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_from_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "c1", "--steps", "1", "--warmup", "3", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if rank == 0:
        assert len(lines) == 1
        res = json.loads(lines[0])
        assert res["impl"] == "reference" and res["value"] > 0
        assert res["cpu_baseline"]["kind"] == "oracle"
        assert res["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []


@pytest.mark.parametrize("workload", ["c1", "s1", "d1"])
def test_reference_arm_line_format(workload):
    """One process, N = 1: the reference arm's single JSON line carries the
    contract's keys for the attention, row-softmax and decode workloads."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        workload, "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    res = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in res, key
    assert res["impl"] == "reference" and res["n_gpus"] == 1 and res["steps"] == 1 and res["warmup"] == 3
    assert res["value"] > 0 and res["ms_per_step"] > 0 and res["higher_is_better"] is True
    assert res["config"]["workload"].startswith(workload)
    cb = res["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == res["value"]
    assert res["e2e"] == {"value": res["value"], "unit": res["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
