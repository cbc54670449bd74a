"""The bench's multi-rank path on the host: two gloo ranks (no GPU) agree on the
slowest rank's time, meet at the barrier, and count the whole job's tokens; under a
launcher only rank 0 runs the reference arm."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(world, backend="gloo")
    try:
        bench.barrier(w)
        t = bench.max_over_ranks(10.0 + 5.0 * r, w, device="cpu")   # rank 1 is the slow one
        out.put((r, w, local, t, bench.job_throughput(w, 32768, 4, t)))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=10) for _ in range(2))
    assert [(r, w, local) for r, w, local, _, _ in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(t == 15.0 for _, _, _, t, _ in res)
    # two replicas of 32768 tokens, 4 steps, in the slowest rank's 15 s
    assert all(v == pytest.approx(2 * 32768 * 4 / 15.0) for *_, v in res)


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.job_throughput(1, 100, 2, 4.0) == 50.0


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
