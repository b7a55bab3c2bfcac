"""bench.py's multi-rank bookkeeping on CPU (gloo, world size 2): max-over-ranks
timing and the whole-job aggregate of independent per-rank replicas."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    t = 1.0 + rank  # rank 1 is the slow one
    tmax = bench.max_over_ranks(t, ws)
    agg = bench.aggregate_line(16, ws, tmax)
    bench.barrier(ws)
    out[rank] = (tmax, agg)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ws = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn")
    assert out[0] == out[1] == (2.0, 16.0)
