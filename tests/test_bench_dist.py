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


def test_class_roofline_bound_and_fraction():
    """The per-class roofline: the roof is whichever of flops at the tensor
    rate and bytes at the copy rate takes longer, achieved = work / measured
    time; a class with neither a byte nor a flop model reports no fraction."""
    import types
    import bench
    peaks = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "_source": "test"}
    w = types.SimpleNamespace(name="none")
    # 1.6 TFLOP and 1 GB in 2 ms: 1 ms at 1600 TFLOP/s against 0.125 ms at 8 TB/s -> tensor
    r = bench.class_roofline("gemm", {"launches": 4, "ms": 2.0, "flops": 1.6e12, "bytes": 1e9}, w, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(800.0) and r["frac"] == pytest.approx(0.5)
    assert r["avg_launch_us"] == pytest.approx(500.0) and r["algorithmic_flops_per_launch"] == pytest.approx(4e11)
    # 8 GB and 1 TFLOP in 2 ms: 1 ms at 8 TB/s against 0.625 ms at 1600 TFLOP/s -> hbm
    r = bench.class_roofline("attention", {"launches": 2, "ms": 2.0, "flops": 1e12, "bytes": 8e9}, w, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(4000.0) and r["frac"] == pytest.approx(0.5)
    r = bench.class_roofline("select", {"launches": 3, "ms": 0.03, "flops": 0.0, "bytes": 0.0}, w, peaks)
    assert r["frac"] is None and r["bound"] is None and r["avg_launch_us"] == pytest.approx(10.0)
    assert bench.class_roofline("rows", {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0}, w, peaks) is None
