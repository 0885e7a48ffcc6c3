"""The benchmark's N>1 bookkeeping on CPU: two gloo ranks, each with its own
batch (weak scaling), whole-job throughput = all ranks' pairs over the slowest
rank's time. No GPU and no data-path collective: the path shards by query."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seconds = 1.0 + rank            # rank 1 is the slower one
    pairs = 1000 * (rank + 1)
    value, tmax = bench.whole_job(pairs, 10, seconds, dist, "cpu")
    out[rank] = (value, tmax, bench.rank_seed("batched_decode", rank))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_whole_job_value():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of a process that already runs threads
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # (1000 + 2000) pairs x 10 steps over the slowest rank's 2 s
    for r in range(world):
        assert res[r][0] == pytest.approx(3000 * 10 / 2.0)
        assert res[r][1] == pytest.approx(2.0)
    assert res[0][2] != res[1][2]   # distinct batches per rank


def test_single_rank_whole_job_value():
    import bench
    assert bench.whole_job(500, 4, 2.0) == (1000.0, 2.0)
