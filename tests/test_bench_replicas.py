"""Host logic of the multi-GPU path (replicas, no collective on the data path),
run as two gloo ranks on the CPU: each rank gets its own batch, the timed
region's length is the slowest rank's, and the job's throughput counts every
rank's tokens."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(elapsed[rank], dist, "cpu")
        tput = bench.job_throughput(64, world, 20, slowest)
        out.put((rank, slowest, tput, bench.replica_seeds(5, rank)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    elapsed = [0.8, 1.25]  # seconds each rank spent on its timed steps
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, elapsed, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, tput, _ in res:
        assert slowest == 1.25
        assert tput == 64 * 2 * 20 / 1.25
    seeds = [r[3] for r in res]
    # every seed of the replica differs between the ranks, rank 0 keeps the one-GPU run's
    assert all(seeds[0][k] != seeds[1][k] for k in seeds[0])
    assert seeds[0] == __import__("bench").replica_seeds(5, 0)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_throughput(64, 1, 20, 2.0) == 640.0


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_other_ranks_exit_quietly(rank):
    # under torchrun only rank 0 runs and prints the reference arm; the others exit 0 without work
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""

