"""The N>1 host logic of bench.py on CPU: two gloo ranks (world_size 2).

Vectors are independent, so ranks shard the work with no collective on the data
path; the only cross-rank operations are the barrier around the timed region
and the max-over-ranks of the elapsed time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    r, local, w = bench.dist_env()
    elapsed = 10.0 * (rank + 1)  # rank 1 is the slow one
    bench.barrier()
    m = bench.dist_max(elapsed)
    bench.barrier()
    q.put((r, local, w, m, bench.rank_seed(4, r)))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_shards():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1]
    assert all(o[2] == world for o in out)
    assert all(o[3] == 20.0 for o in out), "every rank must see the max over ranks"
    assert out[0][4] == 4 and out[1][4] != 4, "rank 0 draws the specified seed, others their own"


def test_single_process_helpers(monkeypatch):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.dist_max(3.5) == 3.5


def test_reference_arm_only_on_rank0(monkeypatch, capsys):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""
