"""The multi-rank logic of bench.py: with two gloo ranks on the CPU, the job
time is the slowest rank's; independent replicas count every rank's tokens,
a token-sharded batch (--token-parallel) counts the batch's tokens once."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    bench.barrier(ws)
    ms_max, value = bench.aggregate(ws, 16384, 10.0 * (rank + 1))
    # --token-parallel: one batch of 16384 tokens split over the ranks
    ms_sh, value_sh = bench.aggregate_sharded(ws, 16384, 10.0 * (rank + 1))
    out[rank] = (ms_max, value, ms_sh, value_sh)
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms_max, value, ms_sh, value_sh = out[r]
        assert ms_max == pytest.approx(20.0)
        assert value == pytest.approx(2 * 16384 / 0.020)
        # a sharded batch counts its tokens once, over the slowest rank
        assert ms_sh == pytest.approx(20.0)
        assert value_sh == pytest.approx(16384 / 0.020)


def test_single_rank_aggregation():
    import bench
    assert bench.aggregate(1, 1000, 5.0) == (5.0, pytest.approx(200000.0))
