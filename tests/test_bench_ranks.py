"""The multi-process side of bench.py, on CPU with the gloo backend.

The path does not shard (each GPU runs its own replica), so the only
cross-rank logic is the timing: every time is the maximum over ranks and the
whole-job value is all ranks' work over that time.  The reference arm runs on
rank 0 only; the other ranks exit 0 without work."""
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


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r is slow on entry r: each maximum comes from a different rank
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        q.put((rank, bench.max_over_ranks(mine, world)))
    finally:
        dist.destroy_process_group()


def test_times_are_the_maximum_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 5.0, 0.5]


def test_whole_job_value_counts_every_rank_over_the_slowest():
    sys.path.insert(0, ROOT)
    import bench
    flop = 2.0 * 65536 * 1024 * 2048
    assert bench.whole_job_tflops(flop, 1, 1e-3) == pytest.approx(flop / 1e-3 / 1e12)
    assert bench.whole_job_tflops(flop, 4, 2e-3) == pytest.approx(2 * flop / 1e-3 / 1e12)
    assert bench.max_over_ranks([3.0, 1.0], 1) == [3.0, 1.0]


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                           "--workload", "probe", "--gpus", str(world)],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run_reference(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference(0, 2)
    assert r0.returncode == 0, r0.stderr
    lines = [l for l in r0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
