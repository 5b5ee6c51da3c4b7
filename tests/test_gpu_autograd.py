"""The autograd wrapper: loss.backward() through the fused call gives the
oracle's gradients; the incoming gradient scales them; reduction='sum'; the
sync-free mode agrees and runs inside a captured CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import device_inputs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sync_free", [False, True])
@pytest.mark.parametrize("dtype,tol", [("bf16", 1e-2), ("fp32", 1e-5)])
def test_backward_matches_oracle(dtype, tol, sync_free):
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    w = workloads.generate(workloads.custom(600, 128, 3000, dtype, ignore_frac=0.1, seed=41))
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t)
    x, W, t = device_inputs(w)
    x.requires_grad_()
    W.requires_grad_()
    loss = linear_cross_entropy(x, W, t, chunk=256, sync_free=sync_free)
    loss.backward()
    assert abs(loss.item() - ref.loss) / ref.loss <= 1e-3
    assert rel_fro(x.grad.double().cpu().numpy(), ref.dx) <= tol
    assert rel_fro(W.grad.double().cpu().numpy(), ref.dW) <= tol


@pytest.mark.parametrize("sync_free", [False, True])
def test_grad_output_scaling_and_sum_reduction(sync_free):
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    w = workloads.generate(workloads.custom(500, 64, 2000, "bf16", ignore_frac=0.2, seed=42))
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t)
    x, W, t = device_inputs(w)
    x.requires_grad_()
    W.requires_grad_()
    (3.0 * linear_cross_entropy(x, W, t, sync_free=sync_free)).backward()
    assert rel_fro(x.grad.double().cpu().numpy(), 3.0 * ref.dx) <= 1e-2
    x.grad = None
    W.grad = None
    s = linear_cross_entropy(x, W, t, reduction="sum", sync_free=sync_free)
    s.backward()
    nv = ref.n_valid
    assert abs(s.item() - ref.loss * nv) / (ref.loss * nv) <= 1e-3
    assert rel_fro(W.grad.double().cpu().numpy(), nv * ref.dW) <= 1e-2


def test_sync_free_step_in_a_cuda_graph():
    """A whole training step of the loss (forward, backward into static
    gradient buffers) captured once and replayed on new inputs written into
    the same tensors gives the oracle's loss and gradients for those inputs."""
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    ws = [workloads.generate(workloads.custom(512, 128, 3000, "bf16", ignore_frac=0.1, seed=s))
          for s in (43, 44)]
    x, W, t = device_inputs(ws[0])
    x.requires_grad_()
    W.requires_grad_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):   # warm-up outside capture: workspace and autograd state
            x.grad = None
            W.grad = None
            linear_cross_entropy(x, W, t, sync_free=True).backward()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    x.grad = None
    W.grad = None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loss = linear_cross_entropy(x, W, t, sync_free=True)
        loss.backward()
    for w in ws:
        x2, W2, t2 = device_inputs(w)
        with torch.no_grad():
            x.copy_(x2)
            W.copy_(W2)
        t.copy_(t2)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t)
        assert abs(loss.item() - ref.loss) / ref.loss <= 1e-3
        assert rel_fro(x.grad.double().cpu().numpy(), ref.dx) <= 1e-2
        assert rel_fro(W.grad.double().cpu().numpy(), ref.dW) <= 1e-2
