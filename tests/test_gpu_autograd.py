"""The autograd wrapper: loss.backward() through the fused call gives the
oracle's gradients; the incoming gradient scales them; reduction='sum'."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import device_inputs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,tol", [("bf16", 1e-2), ("fp32", 1e-5)])
def test_backward_matches_oracle(dtype, tol):
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    w = workloads.generate(workloads.custom(600, 128, 3000, dtype, ignore_frac=0.1, seed=41))
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t)
    x, W, t = device_inputs(w)
    x.requires_grad_()
    W.requires_grad_()
    loss = linear_cross_entropy(x, W, t, chunk=256)
    loss.backward()
    assert abs(loss.item() - ref.loss) / ref.loss <= 1e-3
    assert rel_fro(x.grad.double().cpu().numpy(), ref.dx) <= tol
    assert rel_fro(W.grad.double().cpu().numpy(), ref.dW) <= tol


def test_grad_output_scaling_and_sum_reduction():
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    w = workloads.generate(workloads.custom(500, 64, 2000, "bf16", ignore_frac=0.2, seed=42))
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t)
    x, W, t = device_inputs(w)
    x.requires_grad_()
    W.requires_grad_()
    (3.0 * linear_cross_entropy(x, W, t)).backward()
    assert rel_fro(x.grad.double().cpu().numpy(), 3.0 * ref.dx) <= 1e-2
    x.grad = None
    W.grad = None
    s = linear_cross_entropy(x, W, t, reduction="sum")
    s.backward()
    nv = ref.n_valid
    assert abs(s.item() - ref.loss * nv) / (ref.loss * nv) <= 1e-3
    assert rel_fro(W.grad.double().cpu().numpy(), nv * ref.dW) <= 1e-2
