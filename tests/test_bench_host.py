"""Host side of the benchmark (no GPU): how ranks combine their timings, and the
CPU reference arm's launch and JSON line.

The N > 1 path runs one process per GPU with no collective on the data path; the
only cross-rank step is the timing: the job's time is its slowest rank's, and its
work is world times one rank's.  Two gloo ranks on the CPU run that same code."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_job_rate_one_process():
    ms, rate = bench.job_rate(None, "cpu", 20.0, 1e12, 2)
    assert ms == 20.0
    assert rate == pytest.approx(2 * 1e12 / 0.020 / 1e12)     # 100 TFLOP/s


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_per_rank, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.job_rate(dist, "cpu", ms_per_rank[rank], 1e12, 2)))
    finally:
        dist.destroy_process_group()


def test_job_rate_two_gloo_ranks():
    """Rank 1 is twice as slow: both ranks report its time, and the job's rate is
    two ranks' work over that time."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ms = [10.0, 20.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = dict(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    for r in range(2):
        ms_job, rate = res[r]
        assert ms_job == 20.0
        assert rate == pytest.approx(2 * 2 * 1e12 / 0.020 / 1e12)   # 200 TFLOP/s


def _run_bench(args, env_extra, timeout):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, 120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_json_line():
    """One short step of the oracle on the default workload: one JSON line with the
    contract's keys, the reference marked and its CPU sample described."""
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"],
                   {"RANK": "0", "WORLD_SIZE": "1"}, 600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "7b_prefill"
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
