"""Pins for the fp64 oracle, against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas. Each checks the oracle
against something independent of it: hand-derived closed forms, the W = 0
closed form, invariants of softmax cross-entropy, central finite differences
of the loss, chunk-order independence of the FLCE schedule, and the library
routine torch.nn.functional.cross_entropy with autograd in float64.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"ln": math.log}))


def _mat(rows):
    return np.array([[_ev(v) for v in r] for r in rows], dtype=np.float64)


def _rand(N, H, V, seed=0, ignore=(), w_std=0.5):
    g = np.random.default_rng(seed)
    x = g.standard_normal((N, H))
    W = w_std * g.standard_normal((V, H))
    t = g.integers(0, V, size=N)
    for i in ignore:
        t[i] = oracle.IGNORE_INDEX
    return x, W, t


# ------------------------------------------------------------ golden cases

@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "hand_worked.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    x, W = _mat(case["x"]), _mat(case["W"])
    t = np.array(case["t"], dtype=np.int64)
    for chunk in (None, 1, 2):
        r = oracle.flce_reference(x, W, t, case["ignore_index"], chunk=chunk)
        assert r.loss == pytest.approx(_ev(case["loss"]), abs=1e-14)
        np.testing.assert_allclose(r.token_loss, [_ev(v) for v in case["token_loss"]], atol=1e-14)
        np.testing.assert_allclose(r.dx, _mat(case["dx"]), atol=1e-14)
        np.testing.assert_allclose(r.dW, _mat(case["dW"]), atol=1e-14)


def test_page_printed_sizes_match_workloads():
    items = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))["items"]
    for it in items:
        s = workloads.CONFIGS[it["config"]]
        if it["quantity"] == "logit_elements":
            assert s.N * s.V == it["value"]
        elif it["quantity"] == "logit_bytes_bf16_gb":
            assert abs(s.N * s.V * 2 / 1e9 - it["value"]) <= it["tolerance"]
        elif it["quantity"] == "hidden_bytes_bf16_gb":
            assert abs(s.N * s.H * 2 / 1e9 - it["value"]) <= it["tolerance"]
        else:
            raise AssertionError(it["quantity"])


# ------------------------------------------------------- closed form W = 0

def test_closed_form_zero_weight():
    N, H, V = 13, 5, 17
    g = np.random.default_rng(1)
    x = g.standard_normal((N, H))
    t = g.integers(0, V, size=N)
    t[[2, 7]] = -100
    W = np.zeros((V, H))
    r = oracle.flce_reference(x, W, t, return_dlogits=True)
    valid = t != -100
    nv = valid.sum()
    assert r.loss == pytest.approx(math.log(V), abs=1e-14)
    np.testing.assert_array_equal(r.dx, 0.0)
    onehot = np.zeros((N, V))
    onehot[np.flatnonzero(valid), t[valid]] = 1.0
    d_expect = valid[:, None] * (1.0 / V - onehot) / nv
    np.testing.assert_allclose(r.dlogits, d_expect, atol=1e-15)
    dW_expect = np.zeros((V, H))
    xs = x[valid].sum(axis=0) / V
    for j in range(V):
        dW_expect[j] = (xs - x[valid & (t == j)].sum(axis=0)) / nv
    np.testing.assert_allclose(r.dW, dW_expect, atol=1e-14)


# -------------------------------------------------------------- invariants

def test_dlogit_rows_and_dW_columns_sum_to_zero():
    x, W, t = _rand(40, 9, 31, seed=2, ignore=(3, 4))
    r = oracle.flce_reference(x, W, t, return_dlogits=True)
    np.testing.assert_allclose(r.dlogits.sum(axis=1), 0.0, atol=1e-15)
    np.testing.assert_allclose(r.dW.sum(axis=0), 0.0, atol=1e-14)
    # ignored rows carry no gradient at all
    np.testing.assert_array_equal(r.dlogits[[3, 4]], 0.0)
    np.testing.assert_array_equal(r.dx[[3, 4]], 0.0)


def test_shift_invariance_and_stability():
    """W -> W + 1·uᵀ adds x_i·u to every logit of row i: loss and gradients
    do not change. |z| ~ 1e4 would overflow exp without the max shift."""
    x, W, t = _rand(24, 6, 19, seed=3, ignore=(0,))
    u = np.full(6, 3.0e3) * np.sign(np.random.default_rng(4).standard_normal(6))
    r0 = oracle.flce_reference(x, W, t)
    r1 = oracle.flce_reference(x, W + u[None, :], t)
    assert np.isfinite(r1.loss)
    assert r1.loss == pytest.approx(r0.loss, rel=1e-9)
    np.testing.assert_allclose(r1.dW, r0.dW, atol=1e-10)
    np.testing.assert_allclose(r1.dx, r0.dx, atol=1e-8)


def test_dx_dW_inner_product_identity():
    """<dW, W>_F = sum_ij d_ij z_ij = <dx, x>_F."""
    x, W, t = _rand(30, 8, 23, seed=5, ignore=(1,))
    r = oracle.flce_reference(x, W, t)
    assert np.sum(r.dW * W) == pytest.approx(np.sum(r.dx * x), rel=1e-12)


# --------------------------------------------------- finite differences

def _loss(x, W, t):
    return oracle.flce_reference(x, W, t).loss


def test_central_finite_differences():
    N, H, V = 6, 5, 11
    x, W, t = _rand(N, H, V, seed=6, ignore=(4,), w_std=0.7)
    r = oracle.flce_reference(x, W, t)
    h = 1e-6
    fd_x = np.zeros_like(x)
    for i in range(N):
        for k in range(H):
            xp, xm = x.copy(), x.copy()
            xp[i, k] += h
            xm[i, k] -= h
            fd_x[i, k] = (_loss(xp, W, t) - _loss(xm, W, t)) / (2 * h)
    fd_W = np.zeros_like(W)
    for j in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, k] += h
            Wm[j, k] -= h
            fd_W[j, k] = (_loss(x, Wp, t) - _loss(x, Wm, t)) / (2 * h)
    np.testing.assert_allclose(r.dx, fd_x, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(r.dW, fd_W, rtol=1e-6, atol=1e-9)
    # the ignored token's hidden state has no influence on the loss
    np.testing.assert_allclose(fd_x[4], 0.0, atol=1e-9)


# ------------------------------------------------------- chunk invariance

@pytest.mark.parametrize("chunk", [1, 7, 64, 100])
def test_chunked_schedule_equals_unchunked(chunk):
    x, W, t = _rand(100, 12, 37, seed=7, ignore=(0, 50, 99))
    r0 = oracle.flce_reference(x, W, t)
    r1 = oracle.flce_reference(x, W, t, chunk=chunk)
    assert r1.loss == pytest.approx(r0.loss, rel=1e-12)
    np.testing.assert_allclose(r1.dx, r0.dx, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r1.dW, r0.dW, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r1.token_loss, r0.token_loss, atol=1e-12)


# ---------------------------------------------------- library routine pin

@pytest.mark.parametrize("shape,ignore", [((16, 8, 50), (3,)), ((64, 32, 300), (0, 5, 63))])
def test_matches_torch_cross_entropy_autograd_fp64(shape, ignore):
    N, H, V = shape
    x, W, t = _rand(N, H, V, seed=8, ignore=ignore)
    xt = torch.tensor(x, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(xt @ Wt.T, torch.tensor(t), ignore_index=-100)
    loss.backward()
    r = oracle.flce_reference(x, W, t)
    assert r.loss == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(r.dx, xt.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r.dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-14)
    per_tok = torch.nn.functional.cross_entropy(xt.detach() @ Wt.detach().T, torch.tensor(t),
                                                ignore_index=-100, reduction="none")
    np.testing.assert_allclose(r.token_loss, per_tok.numpy(), rtol=1e-12, atol=1e-14)


def test_other_ignore_index_value():
    x, W, t = _rand(20, 4, 9, seed=9)
    t[[1, 2]] = 7            # treat class 7 as the ignore marker
    r = oracle.flce_reference(x, W, t, ignore_index=7)
    xt = torch.tensor(x, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(xt @ Wt.T, torch.tensor(t), ignore_index=7)
    loss.backward()
    assert r.n_valid == 20 - int((t == 7).sum())
    assert r.loss == pytest.approx(loss.item(), rel=1e-12)
    np.testing.assert_allclose(r.dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-14)


# --------------------------------------------------------------- edge cases

def test_all_tokens_ignored_gives_zeros():
    x, W, t = _rand(5, 3, 7, seed=10)
    t[:] = -100
    for chunk in (None, 2):
        r = oracle.flce_reference(x, W, t, chunk=chunk)
        assert r.loss == 0.0 and r.n_valid == 0
        np.testing.assert_array_equal(r.dx, 0.0)
        np.testing.assert_array_equal(r.dW, 0.0)


def test_empty_batch():
    r = oracle.flce_reference(np.zeros((0, 4)), np.ones((5, 4)), np.zeros(0, np.int64))
    assert r.loss == 0.0 and r.dx.shape == (0, 4)
    np.testing.assert_array_equal(r.dW, 0.0)


@pytest.mark.parametrize("bad", [-1, 7, 100, -101])
def test_out_of_range_target_raises(bad):
    x, W, t = _rand(4, 3, 7, seed=11)
    t[2] = bad
    with pytest.raises(ValueError):
        oracle.flce_reference(x, W, t)


# ----------------------------------------- one-by-one outputs vs the whole

def test_sampled_outputs_equal_full_result():
    x, W, t = _rand(70, 10, 45, seed=12, ignore=(2, 3, 69))
    r = oracle.flce_reference(x, W, t)
    rows = np.array([0, 2, 5, 33, 69])
    np.testing.assert_allclose(oracle.token_loss_rows(x, W, t, rows), r.token_loss[rows], atol=1e-13)
    np.testing.assert_allclose(oracle.dx_rows(x, W, t, rows, r.n_valid), r.dx[rows], atol=1e-14)
    lse = oracle.lse_rows(x, W, np.arange(70), block=16)
    np.testing.assert_allclose(lse, r.lse, atol=1e-13)
    J = np.array([0, 4, 44, 17])
    np.testing.assert_allclose(oracle.dW_rows(x, W, t, J, lse, r.n_valid, block=9), r.dW[J],
                               atol=1e-14)


def test_one_by_one_outputs_on_bf16_rows():
    """The one-by-one functions take a lazily widened bf16 matrix and refuse
    raw bit patterns."""
    w = workloads.generate(workloads.custom(60, 16, 50, "bf16", ignore_frac=0.1, seed=13))
    r = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t)
    xr = workloads.F64Rows(w.x)
    rows = np.array([1, 7, 59])
    np.testing.assert_allclose(oracle.dx_rows(xr, w.W_f64(), w.t, rows, r.n_valid), r.dx[rows],
                               atol=1e-14)
    lse = oracle.lse_rows(xr, w.W_f64(), np.arange(60))
    np.testing.assert_allclose(oracle.dW_rows(xr, w.W_f64(), w.t, [0, 49], lse, r.n_valid),
                               r.dW[[0, 49]], atol=1e-14)
    with pytest.raises(TypeError):
        oracle.token_loss_rows(w.x, w.W_f64(), w.t, rows)
    with pytest.raises(TypeError):
        oracle.flce_reference(w.x, w.W, w.t)


# --------------------------------------- planted mistakes fail the pins

def _fd_mismatch(monkeypatch_target, replacement, monkeypatch):
    monkeypatch.setattr(oracle.flce_oracle, monkeypatch_target, replacement)
    try:
        test_central_finite_differences()
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    """A dropped term, a wrong sign or a transposed operand in the oracle's
    steps makes a pin fail: here, the finite-difference pin."""
    f = oracle.flce_oracle
    good_smo = f.softmax_minus_onehot
    good_lse = f.logsumexp_rows

    def wrong_sign(z, lse, t, valid):
        return -good_smo(z, lse, t, valid)

    def dropped_onehot(z, lse, t, valid):
        g = np.exp(z - lse[:, None])
        g[~valid] = 0.0
        return g

    def lse_without_log(z):
        return good_lse(z) + 0.1

    assert _fd_mismatch("softmax_minus_onehot", wrong_sign, monkeypatch)
    monkeypatch.setattr(f, "softmax_minus_onehot", good_smo)
    assert _fd_mismatch("softmax_minus_onehot", dropped_onehot, monkeypatch)
    monkeypatch.setattr(f, "softmax_minus_onehot", good_smo)
    assert _fd_mismatch("logsumexp_rows", lse_without_log, monkeypatch)
