"""bench.py's replica path with two ranks on CPU (gloo, world size 2): the
job's step time is its slowest rank's, the value is every rank's tokens over
that time, and the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, step_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(step_ms[rank], torch.device("cpu"), world)
        q.put((rank, got, bench.job_tokens_per_s(32, world, got)))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_report_the_slowest_step_and_the_whole_job_tokens():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    step_ms = [2.0, 2.5]  # rank 1 is the slower one
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]  # both ranks agree on the max
    assert res[0][2] == pytest.approx(2 * 32 / 2.5e-3)  # 64 tokens per 2.5 ms step


def test_one_rank_is_the_identity():
    assert bench.max_over_ranks(1.75, torch.device("cpu"), 1) == 1.75
    assert bench.job_tokens_per_s(32, 1, 2.0) == pytest.approx(16000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "1", "--cpu-sample", "2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
    # rank 0 of the same job prints the line, with the job's rank count
    env0 = dict(env, RANK="0", LOCAL_RANK="0")
    r0 = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                         "--steps", "1", "--warmup", "1", "--cpu-sample", "2"],
                        capture_output=True, text=True, timeout=300, cwd=ROOT, env=env0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    d = json.loads(r0.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
