"""Parity at the full workload sizes, in the launch configuration bench.py
times (default HBM budget, planned chunk), on outputs the fp64 oracle computes
one by one: the loss (from every token's log-sum-exp), sampled token losses,
sampled rows of dx, sampled rows of dW; plus properties that hold at any
size. The Qwen3-shaped batch runs its default-budget plan (C = 4096, the
backward GEMMs in one launch), the same budget with separate backward
launches (C = 3328, a ragged last chunk) and the chunk sweep
C in {1024, 2048, 4096, 8192}. The
131,072-token batch has a module of its own (test_zy_long_context.py)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import LOSS_RTOL, device_inputs, rel_fro

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

GiB = 1 << 30


def _sample_rows(w, n=48, seed=0):
    g = np.random.default_rng(seed)
    rows = set(g.choice(w.N, n, replace=False).tolist())
    rows |= {0, w.N - 1}
    ign = np.flatnonzero(w.t == -100)
    if len(ign):
        rows.add(int(ign[0]))
    return np.array(sorted(rows))


def _sample_vocab(w, n=40, seed=1):
    g = np.random.default_rng(seed)
    J = set(range(8)) | {w.V - 1, w.V - 3, w.V // 2}
    J |= set(g.choice(w.V, n, replace=False).tolist())
    J |= set(np.unique(w.t[w.t >= 0])[:4].tolist())
    return np.array(sorted(J))


class Ref:
    """Oracle values for one workload, computed once."""

    def __init__(self, w, full_lse=True):
        self.w = w
        x = workloads.F64Rows(w.x)
        self.Wd = w.W_f64()
        self.valid = oracle.valid_mask(w.t, w.ignore_index)
        self.n_valid = int(self.valid.sum())
        self.rows = _sample_rows(w)
        self.J = _sample_vocab(w)
        self.tok = oracle.token_loss_rows(x, self.Wd, w.t, self.rows)
        self.dx = oracle.dx_rows(x, self.Wd, w.t, self.rows, self.n_valid)
        self.lse = None
        if full_lse:
            self.lse = oracle.lse_rows(x, self.Wd, np.arange(w.N), block=512)
            zt = np.zeros(w.N)
            vi = np.flatnonzero(self.valid)
            for s in range(0, len(vi), 4096):
                r = vi[s:s + 4096]
                zt[r] = np.einsum("ij,ij->i", w.x_f64(r), self.Wd[w.t[r]])
            self.loss = float(np.sum((self.lse - zt)[self.valid])) / self.n_valid
            self.dW = oracle.dW_rows(x, self.Wd, w.t, self.J, self.lse, self.n_valid)


def _check(handle, w, ref, chunk=0):
    x, W, t = device_inputs(w)
    loss, dx, dW = handle.forward_backward(x, W, t, chunk=chunk)
    tl = handle.token_losses(w.N)
    torch.cuda.synchronize()
    plan = handle.last_plan()
    # loss
    if ref.lse is not None:
        assert abs(loss - ref.loss) / abs(ref.loss) <= LOSS_RTOL, (loss, ref.loss)
    # the loss is the mean of the token losses (consistency at any size)
    tl64 = tl.double()
    assert abs(tl64.sum().item() / ref.n_valid - loss) <= 1e-5 * abs(loss)
    # sampled token losses and dx rows
    got_tok = tl[torch.from_numpy(ref.rows).cuda()].double().cpu().numpy()
    assert rel_fro(got_tok, ref.tok) <= LOSS_RTOL
    got_dx = dx[torch.from_numpy(ref.rows).cuda()].double().cpu().numpy()
    assert rel_fro(got_dx, ref.dx) <= 1e-2
    # sampled dW rows
    if ref.lse is not None:
        got_dw = dW[torch.from_numpy(ref.J).cuda()].double().cpu().numpy()
        assert rel_fro(got_dw, ref.dW) <= 1e-2
    # properties: dW's column sums vanish; <dW, W> = <dx, x>
    colsum = dW.double().sum(0)
    assert (colsum.norm() / dW.double().norm()).item() <= 1e-2
    a = (dW.double() * W.double()).sum().item()
    b = (dx.double() * x.double()).sum().item()
    assert abs(a - b) <= 1e-2 * abs(b)
    return plan


@pytest.fixture(scope="module")
def llama3():
    w = workloads.make("llama3_bf16")
    return w, Ref(w)


def test_llama3_bench_configuration(llama3):
    from linear_cross_entropy_token_gb300 import FLCE
    w, ref = llama3
    h = FLCE("bf16", 0)
    try:
        plan = _check(h, w, ref)
        assert plan["chunk"] == 4096 and plan["num_chunks"] == 4
    finally:
        h.close()


@pytest.fixture(scope="module")
def qwen3():
    w = workloads.make("qwen3_bf16")
    return w, Ref(w)


@pytest.mark.parametrize("chunk", workloads.QWEN3_CHUNKS)
def test_qwen3_chunk_sweep(qwen3, chunk):
    from linear_cross_entropy_token_gb300 import FLCE
    w, ref = qwen3
    h = FLCE("bf16", 0, hbm_budget_bytes=4 * GiB)
    try:
        plan = _check(h, w, ref, chunk=chunk)
        assert plan["chunk"] == chunk
    finally:
        h.close()


def test_qwen3_bench_configuration(qwen3):
    """The default HBM budget, as bench.py runs it: the dx and dW GEMMs share
    one launch with an unsplit dx reduction, which leaves room for C = 4096,
    four chunks."""
    from linear_cross_entropy_token_gb300 import FLCE
    w, ref = qwen3
    h = FLCE("bf16", 0)
    try:
        plan = _check(h, w, ref)
    finally:
        h.close()
    assert (plan["chunk"], plan["num_chunks"], plan["dx_splits"]) == (4096, 4, 1)
    assert plan["backward_one_launch"] == 1


def test_qwen3_separate_backward_launches(qwen3):
    """The default budget with the dx and dW GEMMs in launches of their own:
    five dx splits leave room for C = 3328, five chunks, the last one ragged
    (3072 tokens)."""
    from linear_cross_entropy_token_gb300 import FLCE
    w, ref = qwen3
    h = FLCE("bf16", 0, backward="separate")
    try:
        plan = _check(h, w, ref)
    finally:
        h.close()
    assert (plan["chunk"], plan["num_chunks"], plan["backward_one_launch"]) == (3328, 5, 0)
    assert w.N - 4 * plan["chunk"] == 3072


def test_qwen3_slab_backward(qwen3):
    """The vocabulary-slab backward on the Qwen3-shaped batch (6 slabs of
    29184 columns per chunk, the last ragged), on the same sampled outputs."""
    from linear_cross_entropy_token_gb300 import FLCE
    w, ref = qwen3
    h = FLCE("bf16", 0, dlogits_mode="slabs")
    try:
        plan = _check(h, w, ref)
    finally:
        h.close()
    assert (plan["chunk"], plan["vocab_slab"]) == (4096, 29184)
    assert plan["workspace_bytes"] < 0.35e9


@pytest.mark.parametrize("N,H,V,budget_gib", [
    # the largest chunk the planner takes (32768 tokens) over a 262k-entry
    # vocabulary in one chunk: the chunk buffer holds 8.6e9 logits, so every
    # offset into it needs 64 bits
    (32768, 512, 262147, 24),
    # a 16384-wide hidden state: 256 k-blocks per logits tile, 64 hidden
    # tiles across dx and dW
    (4096, 16384, 50257, 0),
])
def test_maximum_sizes(N, H, V, budget_gib):
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(N, H, V, "bf16", targets="zipf", ignore_frac=0.05,
                                            seed=N + H))
    ref = Ref(w)
    h = FLCE("bf16", 0, hbm_budget_bytes=budget_gib * GiB)
    try:
        plan = _check(h, w, ref)
        if budget_gib:
            assert plan["chunk"] == N and plan["num_chunks"] == 1
            assert plan["chunk"] * plan["ldv"] > (1 << 33)
    finally:
        h.close()
