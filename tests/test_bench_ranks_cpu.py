"""bench.py's multi-process logic on the CPU: world-size-2 gloo ranks (replicas; the only
cross-rank step is the max of the timings) and the reference arm's non-zero ranks."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench as b
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = b.max_over_ranks([10.0 + rank, 5.0 - rank, 7.5], torch.device("cpu"))
        torch.distributed.barrier()
        queue.put((rank, b.dist_env(), got))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = {}
        for _ in procs:
            rank, env, got = queue.get(timeout=120)
            res[rank] = (env, got)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # every rank ends with the slowest rank's time of each measurement
    assert res[0][1] == res[1][1] == [11.0, 5.0, 7.5]
    assert res[0][0] == (2, 0, 0) and res[1][0] == (2, 1, 1)


def test_max_over_ranks_without_a_group_is_the_identity():
    assert bench.max_over_ranks([3, 4.5], torch.device("cpu")) == [3.0, 4.5]


def test_whole_job_gbs_counts_every_rank_over_the_slowest_time():
    # 2 ranks x 1000 calls x 134,217,728 B in 23.5 ms
    assert bench.whole_job_gbs(2, 1000, 134217728, 23.5) == pytest.approx(2 * 1000 * 134217728 / 0.0235 / 1e9)
    assert bench.whole_job_gbs(1, 10, 10**9, 1000.0) == pytest.approx(10.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT="29999")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
