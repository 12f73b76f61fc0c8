"""The replica bookkeeping of bench.py under torchrun, checked on CPU.

With N ranks every rank is an independent replica of the step. The timed
region of the job is the slowest rank's, taken by one MAX all-reduce, and the
whole-job throughput counts the bytes of every rank in that time. Only rank 0
prints. The reference arm (the CPU oracle) runs on rank 0 alone, and the other
ranks exit 0 without work."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench as b

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, b.max_over_ranks(times[rank], world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    times = [4.0, 6.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert got == {0: 6.5, 1: 6.5}


def test_whole_job_value_counts_every_replica():
    one = bench.whole_job_gbs(3.3e9, 1, 10.0)  # 3.3 GB in 10 ms
    assert abs(one - 330.0) < 1e-9
    assert abs(bench.whole_job_gbs(3.3e9, 2, 10.0) - 2 * one) < 1e-9
    assert bench.max_over_ranks(7.0, 1) == 7.0  # one rank: no collective


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
