"""Token data parallelism: one batch's tokens split over the ranks of a
torch.distributed group, each rank holding a replica of W.

The mean loss divides by the whole batch's non-ignored tokens and dW sums
over all of its tokens ("Fused Linear Cross-Entropy: LLM 학습 logits 메모리
병목 없애기", section "FLCE의 핵심 아이디어": per-chunk dlogits, dx and dW, the
sums divided by the token count at the end). Token chunks are independent
except for those two sums, so splitting the tokens over ranks, the way
"Transformer Math 101", section "3D 병렬화", splits a batch over model
replicas, takes three collectives per step:

1. all-reduce (sum) of each rank's non-ignored token count, a scalar, so that
   every rank divides by the batch's total;
2. the rank's fused forward + backward with that divisor;
3. all-reduce (sum) of dW and of the rank's share of the loss.

dx needs no exchange: its rows are the rank's own tokens. The per-rank steps
run in the library's kernels (flce_count_valid, flce_forward_backward_shard);
this module only orders them around the collectives. On GPUs the group is
NCCL and every tensor stays on the device: the step never synchronises the
host. The handle argument is anything with the two methods of
linear_cross_entropy_token_gb300.FLCE used below.
"""
from __future__ import annotations

from typing import Optional


def token_parallel_forward_backward(handle, x, W, t, ignore_index: int = -100, chunk: int = 0,
                                    group=None, dx=None, dW=None):
    """One rank's part of a token-sharded fused linear cross-entropy step.

    x (N_r, H) and t (N_r,) are this rank's tokens; W (V, H) is the replica,
    the same on every rank. Returns (loss, dx, dW): loss, a 0-dim float32
    tensor holding the batch's mean loss (the same on every rank); dx, this
    rank's rows of the batch gradient; dW, the batch's dW (the same on every
    rank). Every rank of `group` must call this with the same W shape and
    ignore_index.
    """
    import torch.distributed as dist
    n_total = handle.count_valid(t, ignore_index)
    dist.all_reduce(n_total, op=dist.ReduceOp.SUM, group=group)
    loss, dx, dW = handle.forward_backward_shard(x, W, t, n_total, ignore_index=ignore_index,
                                                 chunk=chunk, dx=dx, dW=dW)
    dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(loss, op=dist.ReduceOp.SUM, group=group)
    return loss, dx, dW


def shard_bounds(N: int, world_size: int, rank: int) -> tuple:
    """Rows [start, stop) of an N-token batch that rank `rank` of
    `world_size` takes: contiguous blocks, the first N % world_size ranks one
    token longer."""
    if world_size < 1 or not 0 <= rank < world_size or N < 0:
        raise ValueError("need world_size >= 1, 0 <= rank < world_size, N >= 0")
    base, extra = divmod(N, world_size)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def check_status(handle, loss) -> Optional[float]:
    """Host value of the step's loss after the handle's device-side status
    check (raises FlceError if a shard recorded an error). Synchronises."""
    handle.async_status()
    return float(loss.item())
