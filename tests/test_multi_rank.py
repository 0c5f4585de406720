"""The N > 1 host logic of bench.py on CPU: two gloo ranks agree on the
slowest rank's time and on the whole-job value, and only rank 0 of the
reference arm does any work or prints."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, step_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.slowest_rank_ms(step_ms[rank], world, "cpu")
        out.put((rank, bench._dist(), slow, bench.job_tflops(world, 4.0e9, slow)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    step_ms = [0.150, 0.175]
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, step_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, dist_env, slow, value) in enumerate(got):
        assert r == rank and dist_env == (2, rank, rank)
        assert slow == pytest.approx(0.175, rel=0, abs=1e-15)
        # both ranks' work over the slower rank's step: 2 * 4 GFLOP / 0.175 ms
        assert value == pytest.approx(2 * 4.0e9 / 0.175e-3 / 1e12, rel=1e-12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.slowest_rank_ms(0.2, 1, "cpu") == 0.2
    assert bench.job_tflops(1, 2.0e9, 0.5) == pytest.approx(4.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
