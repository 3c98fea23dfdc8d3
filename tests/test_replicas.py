"""bench.py's multi-GPU mode: independent replicas, no collective on the data path.  The host
logic that turns per-rank timings into the whole-job number runs here on two gloo ranks (CPU),
and the reference arm's non-zero ranks exit without work."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as tdist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mor = bench.make_max_over_ranks(world, torch.device("cpu"))
        # rank r processed 100 units in (r + 1) seconds
        value, slowest = bench.replica_throughput(100, float(rank + 1), world, mor)
        out.put((rank, value, slowest))
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks: 2 x 100 units over the slowest rank's 2 s
    assert res == [(0, 100.0, 2.0), (1, 100.0, 2.0)]


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.replica_throughput(50, 0.5, 1, bench.make_max_over_ranks(1, None)) == (100.0, 0.5)


def test_reference_arm_nonzero_rank_exits_without_output():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
