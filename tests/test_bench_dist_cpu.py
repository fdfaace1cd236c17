"""The multi-rank path of bench.py on the CPU: world size 2 over gloo.

On a multi-GPU node every rank times its own replica (weak scaling, no
data-path collective); the job's time is the slowest rank's, and the job's
rate counts every rank's tokens. Here two processes on 127.0.0.1 run the
same helpers bench.py uses, and the reference arm's non-zero ranks are
checked to leave at once without work."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_info()
        slowest = bench.max_over_ranks(times[rank], torch.device("cpu"))
        rate = bench.job_rate(w, 1000, slowest)
        dist.barrier()
        out.put((r, w, local, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    times = [2.5, 4.0]  # ms per step of rank 0 and rank 1
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get() for _ in range(2))
    for r, (rank, world, local, slowest, rate) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert slowest == 4.0
        # 2 ranks x 1000 tokens in 4 ms = 0.5 Mtokens/s
        assert rate == pytest.approx(0.5)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, torch.device("cpu")) == 3.25
    assert bench.job_rate(1, 2_000_000, 1000.0) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_fp32", "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
