"""Token data parallelism on the GPU, through the C ABI: a batch split into
shards, each shard's fused call dividing by the batch's total n_valid
(flce_count_valid, flce_forward_backward_shard), the loss shares and dW terms
summed and the dx rows concatenated, against the fp64 oracle on the whole
batch. Two shards run in one process on one GPU (no collective); the
torch.distributed wrapper runs over a one-rank NCCL group, so its
collectives are exercised on the device tensors it really passes."""
import socket

import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import GRAD_RTOL, LOSS_RTOL, device_inputs, rel_fro, to_np64

pytestmark = pytest.mark.gpu


def _shards(N, k):
    from linear_cross_entropy_token_gb300.token_parallel import shard_bounds
    return [shard_bounds(N, k, r) for r in range(k)]


def _sharded(h, x, W, t, spans, chunk=0):
    """Per-shard counts summed on the device, then each shard's call."""
    counts = [h.count_valid(t[a:b]) for a, b in spans]
    total = torch.stack(counts).sum().to(torch.int32)
    loss = torch.zeros((), dtype=torch.float64, device=x.device)
    dW = None
    dx = torch.empty_like(x)
    for a, b in spans:
        l_s, dx_s, dW_s = h.forward_backward_shard(x[a:b], W, t[a:b], total, chunk=chunk,
                                                   dx=dx[a:b])
        loss += l_s.double()
        dW = dW_s.double() if dW is None else dW + dW_s.double()
    h.async_status()
    return loss.item(), dx, dW, [int(c) for c in counts], int(total)


@pytest.mark.parametrize("dtype,N,H,V,ign,chunk,k", [
    ("bf16", 1000, 256, 5003, 0.1, 0, 2),      # two shards, odd V, 10% ignored
    ("bf16", 777, 128, 4099, 0.3, 128, 3),     # three ragged shards, several chunks each
    ("fp32", 300, 64, 1000, 0.2, 64, 2),       # the fp32 path at its 1e-5 tolerance
])
def test_shards_sum_to_the_whole_batch(dtype, N, H, V, ign, chunk, k):
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(N, H, V, dtype, targets="zipf", ignore_frac=ign,
                                            seed=N + k))
    x, W, t = device_inputs(w)
    h = FLCE(dtype, 0)
    try:
        loss, dx, dW, counts, total = _sharded(h, x, W, t, _shards(N, k), chunk)
    finally:
        h.close()
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
    assert total == ref.n_valid and sum(counts) == ref.n_valid
    assert abs(loss - ref.loss) / ref.loss <= LOSS_RTOL
    assert rel_fro(to_np64(dx), ref.dx) <= GRAD_RTOL[dtype]
    assert rel_fro(dW.cpu().numpy(), ref.dW) <= GRAD_RTOL[dtype]


@pytest.mark.parametrize("mode,budget", [("slabs", 4 << 20), ("recompute", 48 << 20)])
def test_shards_in_the_other_dlogits_modes(mode, budget):
    """The batch's divisor reaches the dlogits epilogue of the recomputing
    GEMM too (slab walk: several slabs per chunk)."""
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(900, 128, 20011, "bf16", ignore_frac=0.1, seed=31))
    x, W, t = device_inputs(w)
    h = FLCE("bf16", 0, dlogits_mode=mode, hbm_budget_bytes=budget)   # slabs: four of 6656
    try:
        loss, dx, dW, counts, total = _sharded(h, x, W, t, _shards(900, 2), chunk=256)
        if mode == "slabs":
            assert h.last_plan()["vocab_slab"] < w.V
    finally:
        h.close()
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
    assert total == ref.n_valid
    assert abs(loss - ref.loss) / ref.loss <= LOSS_RTOL
    assert rel_fro(to_np64(dx), ref.dx) <= 1e-2
    assert rel_fro(dW.cpu().numpy(), ref.dW) <= 1e-2


def test_shard_with_every_token_ignored():
    """A shard with no valid token adds nothing but still counts; a batch
    with none at all gives zeros."""
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(512, 128, 3001, "bf16", seed=3))
    w.t[:256] = -100
    x, W, t = device_inputs(w)
    h = FLCE("bf16", 0)
    try:
        loss, dx, dW, counts, total = _sharded(h, x, W, t, _shards(512, 2))
        assert counts == [0, 256] and total == 256
        ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
        assert abs(loss - ref.loss) / ref.loss <= LOSS_RTOL
        assert not dx[:256].float().abs().sum().item()
        assert rel_fro(to_np64(dx), ref.dx) <= 1e-2
        assert rel_fro(dW.cpu().numpy(), ref.dW) <= 1e-2
        t_all = torch.full_like(t, -100)
        loss0, dx0, dW0, counts0, total0 = _sharded(h, x, W, t_all, _shards(512, 2))
        assert total0 == 0 and loss0 == 0.0
        assert not dx0.float().abs().sum().item() and not dW0.abs().sum().item()
    finally:
        h.close()


def test_divisor_below_the_local_count_is_refused():
    from linear_cross_entropy_token_gb300 import FLCE, FlceError
    w = workloads.generate(workloads.custom(256, 64, 1000, "bf16", seed=4))
    x, W, t = device_inputs(w)
    h = FLCE("bf16", 0)
    try:
        too_small = torch.tensor(10, dtype=torch.int32, device="cuda")
        loss, _, _ = h.forward_backward_shard(x, W, t, too_small)
        with pytest.raises(FlceError) as e:
            h.async_status()
        assert e.value.status_name == "FLCE_ERR_INVALID_ARG"
        assert np.isnan(loss.item())
        # the handle works afterwards
        ok = h.count_valid(t)
        loss, _, _ = h.forward_backward_shard(x, W, t, ok)
        h.async_status()
        assert np.isfinite(loss.item())
    finally:
        h.close()


def test_wrapper_over_a_one_rank_nccl_group():
    import torch.distributed as dist

    from linear_cross_entropy_token_gb300 import FLCE
    from linear_cross_entropy_token_gb300.token_parallel import (check_status,
                                                                 token_parallel_forward_backward)
    w = workloads.generate(workloads.custom(640, 256, 8191, "bf16", targets="zipf", ignore_frac=0.05,
                                            seed=8))
    x, W, t = device_inputs(w)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    h = FLCE("bf16", 0)
    try:
        loss, dx, dW = token_parallel_forward_backward(h, x, W, t)
        loss_v = check_status(h, loss)
    finally:
        h.close()
        dist.destroy_process_group()
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
    assert abs(loss_v - ref.loss) / ref.loss <= LOSS_RTOL
    assert rel_fro(to_np64(dx), ref.dx) <= 1e-2
    assert rel_fro(to_np64(dW), ref.dW) <= 1e-2
