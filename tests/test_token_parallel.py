"""The exchange of token data parallelism on the CPU: two gloo ranks split a
batch's tokens, run linear_cross_entropy_token_gb300.token_parallel's
collectives around a stand-in for the library's per-rank steps, and must
together give the fp64 oracle's loss, dx and dW of the whole batch.

The stand-in computes one shard with the oracle on that shard alone (its own
n_valid as divisor) and rescales by n_local / n_total, which is what dividing
by the batch's total means; the wrapper's job is to get n_total, the dW sum
and the loss sum right across ranks, and that is what the whole-batch oracle
checks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads


class OracleShard:
    """The two per-rank steps of the library, on the CPU, in float64."""

    def count_valid(self, t, ignore_index=-100):
        return torch.tensor(int((t != ignore_index).sum()), dtype=torch.int32)

    def forward_backward_shard(self, x, W, t, n_valid_total, ignore_index=-100, chunk=0, dx=None,
                               dW=None):
        r = oracle.flce_reference(x.numpy(), W.numpy(), t.numpy(), ignore_index)
        n_total = int(n_valid_total)
        f = r.n_valid / n_total if n_total else 0.0
        return (torch.tensor(r.loss * f, dtype=torch.float64), torch.from_numpy(r.dx * f),
                torch.from_numpy(r.dW * f))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, case, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    from linear_cross_entropy_token_gb300.token_parallel import (shard_bounds,
                                                                 token_parallel_forward_backward)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    x, W, t = (torch.from_numpy(a) for a in case)
    a, b = shard_bounds(len(t), ws, rank)
    loss, dx, dW = token_parallel_forward_backward(OracleShard(), x[a:b].contiguous(), W,
                                                   t[a:b].contiguous())
    out[rank] = (float(loss), dx.numpy(), dW.numpy(), a, b)
    dist.destroy_process_group()


def _batch(N, H, V, ignore_frac, seed, all_ignored_prefix=0):
    w = workloads.generate(workloads.custom(N, H, V, "fp32", ignore_frac=ignore_frac, seed=seed))
    t = w.t.copy()
    t[:all_ignored_prefix] = -100
    return w.x_f64(), w.W_f64(), t


CASES = {
    # uneven shards (N odd) with 20% of the targets ignored
    "ragged": dict(N=37, H=16, V=53, ignore_frac=0.2, seed=5),
    # rank 0's tokens are all ignored: its loss share and dW term are zero,
    # yet its count enters every rank's divisor
    "rank0_ignored": dict(N=24, H=8, V=31, ignore_frac=0.0, seed=6, all_ignored_prefix=12),
    # every token ignored: loss, dx and dW are all zero
    "all_ignored": dict(N=10, H=8, V=17, ignore_frac=0.0, seed=7, all_ignored_prefix=10),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_two_gloo_ranks_match_the_whole_batch(name):
    x, W, t = _batch(**CASES[name])
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, (x, W, t), out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    ref = oracle.flce_reference(x, W, t)
    dx = np.zeros_like(ref.dx)
    for r in range(2):
        loss, dx_r, dW_r, a, b = out[r]
        assert loss == pytest.approx(ref.loss, rel=1e-12, abs=1e-15)
        np.testing.assert_allclose(dW_r, ref.dW, rtol=1e-10, atol=1e-15)
        dx[a:b] = dx_r
    np.testing.assert_allclose(dx, ref.dx, rtol=1e-10, atol=1e-15)
    assert out[0][4] == out[1][3]  # the shards tile the batch
    if name == "all_ignored":
        assert ref.loss == 0.0 and not ref.dW.any()


def test_shard_bounds_tile_the_batch():
    from linear_cross_entropy_token_gb300.token_parallel import shard_bounds
    for N in (0, 1, 7, 16, 1001):
        for ws in (1, 2, 3, 8):
            spans = [shard_bounds(N, ws, r) for r in range(ws)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            assert all(spans[i][1] == spans[i + 1][0] for i in range(ws - 1))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_bounds(10, 2, 2)
