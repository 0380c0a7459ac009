"""The N > 1 bench path on CPU: world_size-2 gloo ranks (no GPU).  Each rank runs an
independent replica; the job's throughput is all ranks' units over the slowest rank's
time, taken with a max all-reduce."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LORA_BENCH_BACKEND="gloo")
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    elapsed_local = 1.0 + rank          # rank 1 is the slow one
    value, elapsed = bench.aggregate_throughput(64, 10, w, elapsed_local)
    out[rank] = (value, elapsed)
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        value, elapsed = res[rank]
        assert elapsed == 2.0
        assert value == pytest.approx(64 * 10 * 2 / 2.0)
