"""Randomised pins for the fp64 oracle: on shapes, scales, ignore patterns and
chunk sizes drawn by hypothesis, the oracle agrees with the library routine
torch.nn.functional.cross_entropy + autograd in float64, and its chunked
schedule equals the unchunked result."""
import numpy as np
import pytest
import torch

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import assume, given, settings, strategies as st  # noqa: E402


@settings(max_examples=80, deadline=None)
@given(N=st.integers(1, 40), H=st.integers(1, 16), V=st.integers(1, 60),
       seed=st.integers(0, 2**31 - 1), scale=st.sampled_from([0.05, 1.0, 8.0]),
       ignore_p=st.floats(0.0, 0.9), chunk=st.integers(1, 48))
def test_random_cases_match_torch_fp64(N, H, V, seed, scale, ignore_p, chunk):
    g = np.random.default_rng(seed)
    x = scale * g.standard_normal((N, H))
    W = scale * g.standard_normal((V, H))
    t = g.integers(0, V, size=N)
    t[g.random(N) < ignore_p] = oracle.IGNORE_INDEX
    assume((t != oracle.IGNORE_INDEX).any())   # torch's mean over no tokens is NaN
    xt = torch.tensor(x, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(xt @ Wt.T, torch.tensor(t), ignore_index=-100)
    loss.backward()
    r = oracle.flce_reference(x, W, t)
    assert r.loss == pytest.approx(loss.item(), rel=1e-10, abs=1e-12)
    gx, gW = xt.grad.numpy(), Wt.grad.numpy()
    # dx = d·W and dW = dᵀ·x sum terms of both signs (each row of d sums to
    # zero), so their rounding error scales with |d|·|W| and |d|ᵀ·|x|, not
    # with the result: |d| <= (softmax + onehot) / n_valid bounds |d|
    z = x @ W.T
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    keep = t != oracle.IGNORE_INDEX
    d_abs = p.copy()
    d_abs[np.flatnonzero(keep), t[keep]] += 1.0
    d_abs[~keep] = 0.0
    d_abs /= keep.sum()
    fx = np.linalg.norm(d_abs @ np.abs(W))
    fW = np.linalg.norm(d_abs.T @ np.abs(x))
    assert np.linalg.norm(r.dx - gx) <= 1e-10 * (np.linalg.norm(gx) + fx) + 1e-300
    assert np.linalg.norm(r.dW - gW) <= 1e-10 * (np.linalg.norm(gW) + fW) + 1e-300
    rc = oracle.flce_reference(x, W, t, chunk=chunk)
    assert rc.loss == pytest.approx(r.loss, rel=1e-12, abs=1e-14)
    np.testing.assert_allclose(rc.dx, r.dx, rtol=0, atol=1e-12 * (1 + np.abs(r.dx).max()))
    np.testing.assert_allclose(rc.dW, r.dW, rtol=0, atol=1e-12 * (1 + np.abs(r.dW).max()))
