"""The vocabulary-slab backward (FLCE_DLOGITS_SLABS): its workspace does not
grow with V, and it reaches the oracle's result like the other two modes.
The handles get a 48 MiB budget, so that at these sizes the planned slab is
narrower than V (several slabs, the last one ragged) as well as wider (one
slab), on every tile shape; the full-size Llama-3-shaped batch is checked on
sampled outputs with the default budget and with a 64 MiB one."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import assert_parity, rel_fro, run

pytestmark = pytest.mark.gpu

BUDGET = 48 << 20


@pytest.fixture(scope="module", params=["wide", "pair", "single"])
def slabs(request):
    from linear_cross_entropy_token_gb300 import FLCE
    h = FLCE("bf16", 0, dlogits_mode="slabs", cta=request.param, hbm_budget_bytes=BUDGET)
    yield h
    h.close()


def _oracle(w, chunk=512):
    return oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index, chunk=chunk)


def _slab_count(res, V):
    return math.ceil(V / res["plan"]["vocab_slab"])


def test_small_bf16_config(slabs):
    w = workloads.make("small_bf16")
    res = run(slabs, w)
    assert _slab_count(res, w.V) == 4       # 2048 tokens: slabs of 9728 columns
    assert_parity(res, _oracle(w), "bf16", token_rtol=1e-3)


@pytest.mark.parametrize("N,H,V,chunk,ign,targets,min_slabs", [
    (2048, 64, 70001, 0, 0.1, "uniform", 4),     # several slabs, the last ragged; odd V
    (4096, 128, 20000, 0, 0.05, "zipf", 2),      # targets crowd the first slab
    (3000, 72, 33333, 1500, 0.1, "uniform", 2),  # ragged chunks, a K tail, C % 256 != 0
    (1000, 256, 4099, 300, 0.1, "uniform", 1),   # one slab wider than V
    (130, 64, 300, 0, 0.0, "uniform", 1),        # smaller than one tile along every axis
    (200, 64, 1, 0, 0.1, "uniform", 1),          # one class: every loss and gradient is 0
])
def test_shapes(slabs, N, H, V, chunk, ign, targets, min_slabs):
    w = workloads.generate(workloads.custom(N, H, V, "bf16", targets=targets, ignore_frac=ign,
                                            seed=N + 7 * V))
    res = run(slabs, w, chunk=chunk)
    assert _slab_count(res, V) >= min_slabs
    assert_parity(res, _oracle(w), "bf16", token_rtol=1e-3)


def test_matches_inplace_mode():
    """Same inputs, the in-place mode: equal loss, and gradients within the
    bf16 rounding of dlogits."""
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(4096, 256, 30000, "bf16", ignore_frac=0.1, seed=12))
    a_h, b_h = FLCE("bf16", 0), FLCE("bf16", 0, dlogits_mode="slabs", hbm_budget_bytes=BUDGET)
    try:
        a = run(a_h, w, chunk=4096)
        b = run(b_h, w, chunk=4096)
    finally:
        a_h.close()
        b_h.close()
    assert _slab_count(b, w.V) >= 3
    assert b["plan"]["workspace_bytes"] < a["plan"]["workspace_bytes"]
    assert abs(a["loss"] - b["loss"]) <= 1e-6 * abs(a["loss"])
    assert rel_fro(b["dx"], a["dx"]) <= 5e-3 and rel_fro(b["dW"], a["dW"]) <= 5e-3


def test_all_tokens_ignored(slabs):
    w = workloads.generate(workloads.custom(2048, 64, 40000, "bf16", seed=13))
    w.t[:] = -100
    res = run(slabs, w)
    assert res["loss"] == 0.0
    assert np.all(res["dx"] == 0.0) and np.all(res["dW"] == 0.0)


def test_zero_weight_closed_form(slabs):
    """W = 0 over several slabs: loss = ln V, dx = 0 exactly, and
    dW_j = (1/n_v)(sum_valid x_i / V - sum_{valid, t_i = j} x_i)."""
    V = 40000
    w = workloads.generate(workloads.custom(2048, 64, V, "bf16", ignore_frac=0.1, seed=14))
    w.W[:] = 0
    res = run(slabs, w)
    assert _slab_count(res, V) >= 2
    assert abs(res["loss"] - math.log(V)) <= 2e-6 * math.log(V)
    assert np.all(res["dx"] == 0.0)
    x = w.x_f64()
    valid = w.t != -100
    dW = np.tile(x[valid].sum(0) / V, (V, 1))
    np.subtract.at(dW, w.t[valid], x[valid])
    dW /= valid.sum()
    assert rel_fro(res["dW"], dW) <= 1e-2


def test_repeatable_bit_for_bit(slabs):
    """dx accumulates over the slabs in slab order: no atomics race."""
    w = workloads.generate(workloads.custom(2048, 128, 40000, "bf16", ignore_frac=0.1, seed=15))
    a = run(slabs, w)
    b = run(slabs, w)
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["dx"], b["dx"]) and np.array_equal(a["dW"], b["dW"])


@pytest.fixture(scope="module")
def llama3():
    from test_gpu_fullsize import Ref
    w = workloads.make("llama3_bf16")
    return w, Ref(w)


@pytest.mark.slow
@pytest.mark.parametrize("budget,chunk,slab", [(0, 4096, 29184), (64 << 20, 1920, 9216)])
def test_llama3_sampled_and_memory(llama3, budget, chunk, slab):
    """The 16,384-token, 128,256-vocabulary batch: sampled outputs against
    the oracle, and an extra HBM footprint far below one chunk of logits
    (1.05 GB at C = 4096), with the default budget (5 slabs) and with a
    64 MiB one (14 slabs of 1664-token chunks)."""
    from test_gpu_fullsize import _check
    from linear_cross_entropy_token_gb300 import FLCE
    w, ref = llama3
    h = FLCE("bf16", 0, dlogits_mode="slabs", hbm_budget_bytes=budget)
    try:
        plan = _check(h, w, ref)
    finally:
        h.close()
    assert (plan["chunk"], plan["vocab_slab"]) == (chunk, slab)
    assert plan["workspace_bytes"] <= (budget or 0.33e9) < 4096 * w.V * 2


def test_graph_capture_with_side_stream(slabs):
    """The slab backward forks each slab's dW GEMM onto a second stream and
    joins it before the call ends: captured in a CUDA graph and replayed on
    new inputs, it gives the oracle's results on those inputs."""
    from flce_testing import device_inputs, to_np64
    ws = [workloads.generate(workloads.custom(2048, 64, 40000, "bf16", ignore_frac=0.1, seed=s))
          for s in (50, 51)]
    x, W, t = device_inputs(ws[0])
    dx = torch.empty_like(x)
    dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    nv = torch.empty((), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # outside capture: allocates the workspace
        slabs.forward_backward_async(x, W, t, loss=loss, n_valid=nv, dx=dx, dW=dW)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert math.ceil(40000 / slabs.last_plan()["vocab_slab"]) >= 2
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        slabs.forward_backward_async(x, W, t, loss=loss, n_valid=nv, dx=dx, dW=dW)
    for w in ws[::-1]:
        x2, W2, t2 = device_inputs(w)
        x.copy_(x2)
        W.copy_(W2)
        t.copy_(t2)
        g.replay()
        torch.cuda.synchronize()
        assert_parity({"loss": loss.item(), "dx": to_np64(dx), "dW": to_np64(dW)}, _oracle(w), "bf16")
        assert nv.item() == int((w.t != -100).sum())
    slabs.async_status()


@pytest.mark.slow
def test_long_context_sampled_and_memory():
    """The 131,072-token batch: 32 chunks of 5 slabs, sampled outputs
    against the oracle, and the measured drop in free HBM within the plan's
    workspace (0.32 GB, against 33.6 GB of full logits)."""
    from test_gpu_fullsize import Ref, _check
    from flce_testing import device_inputs
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.make("long_bf16")
    ref = Ref(w, full_lse=False)
    h = FLCE("bf16", 0, dlogits_mode="slabs")
    try:
        x, W, t = device_inputs(w)
        dx = torch.empty_like(x)
        dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        h.forward_backward(x, W, t, dx=dx, dW=dW)
        free1, _ = torch.cuda.mem_get_info()
        plan = h.last_plan()
        assert (plan["chunk"], plan["num_chunks"], plan["vocab_slab"]) == (4096, 32, 29184)
        assert free0 - free1 <= plan["workspace_bytes"] + (64 << 20)
        assert plan["workspace_bytes"] * 100 < w.N * w.V * 2
        del x, W, t, dx, dW
        torch.cuda.empty_cache()
        _check(h, w, ref)
    finally:
        h.close()


def test_autograd_slab_mode_without_a_handle():
    """linear_cross_entropy(..., dlogits_mode="slabs", hbm_budget_bytes=...)
    keeps its own slab handle."""
    from flce_testing import device_inputs
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    w = workloads.generate(workloads.custom(2048, 128, 40000, "bf16", ignore_frac=0.1, seed=17))
    x, W, t = device_inputs(w)
    x.requires_grad_(True)
    W.requires_grad_(True)
    loss = linear_cross_entropy(x, W, t, dlogits_mode="slabs", hbm_budget_bytes=BUDGET)
    loss.backward()
    res = {"loss": loss.item(), "dx": x.grad.double().cpu().numpy(), "dW": W.grad.double().cpu().numpy()}
    assert_parity(res, _oracle(w), "bf16")


def test_autograd_with_a_slab_handle():
    """The autograd wrapper takes a handle: a slab handle gives the
    oracle's loss and gradients through loss.backward()."""
    from flce_testing import device_inputs
    from linear_cross_entropy_token_gb300 import FLCE
    from linear_cross_entropy_token_gb300.autograd import linear_cross_entropy
    w = workloads.generate(workloads.custom(2048, 128, 40000, "bf16", ignore_frac=0.1, seed=16))
    h = FLCE("bf16", 0, dlogits_mode="slabs", hbm_budget_bytes=BUDGET)
    try:
        x, W, t = device_inputs(w)
        x.requires_grad_(True)
        W.requires_grad_(True)
        loss = linear_cross_entropy(x, W, t, handle=h)
        loss.backward()
        assert math.ceil(w.V / h.last_plan()["vocab_slab"]) >= 2
        res = {"loss": loss.item(), "dx": x.grad.double().cpu().numpy(),
               "dW": W.grad.double().cpu().numpy()}
        assert_parity(res, _oracle(w), "bf16")
    finally:
        h.close()


@pytest.mark.parametrize("N,H,V,chunk,budget,min_slabs", [
    (256, 128, 4096, 64, 0, 1),            # the tiny fp32 config: one slab
    (256, 128, 4096, 64, 300 << 10, 4),    # four slabs of 1024
    (300, 100, 2999, 128, 320 << 10, 6),   # ragged chunks, a ragged last slab, odd H
])
def test_fp32_slabs(N, H, V, chunk, budget, min_slabs):
    """The slab walk on the fp32 CUDA-core path, at the fp32 tolerance."""
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(N, H, V, "fp32", ignore_frac=0.1, seed=N + V))
    h = FLCE("fp32", 0, dlogits_mode="slabs", hbm_budget_bytes=budget)
    try:
        res = run(h, w, chunk=chunk)
    finally:
        h.close()
    assert _slab_count(res, V) >= min_slabs
    assert_parity(res, oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index), "fp32",
                  token_rtol=1e-5)


def test_caller_workspace_and_pipelined_host_calls(slabs):
    """The slab backward in caller-owned workspace, and through the
    pipelined host-buffer entry with two calls in flight."""
    from flce_testing import to_np64
    from linear_cross_entropy_token_gb300 import FlceError
    ws = [workloads.generate(workloads.custom(2048, 64, 40000, "bf16", ignore_frac=0.1, seed=30 + i))
          for i in range(2)]
    buf = torch.empty(slabs.workspace_bytes(2048, 64, 40000) + 4096, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 1024
    slabs.set_workspace(buf[off:off + slabs.workspace_bytes(2048, 64, 40000)])
    try:
        assert_parity(run(slabs, ws[0]), _oracle(ws[0]), "bf16")
        assert slabs.last_plan()["vocab_slab"] < 40000
        host = [(torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16).pin_memory(),
                 torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16).pin_memory(),
                 torch.from_numpy(w.t).pin_memory()) for w in ws]
        outs = [(torch.empty(2048, 64, dtype=torch.bfloat16, device="cuda"),
                 torch.empty(40000, 64, dtype=torch.float32, device="cuda")) for _ in ws]
        t0, _, _ = slabs.submit_host(*host[0], dx=outs[0][0], dW=outs[0][1])
        t1, _, _ = slabs.submit_host(*host[1], dx=outs[1][0], dW=outs[1][1])
        losses = [slabs.wait(t0), slabs.wait(t1)]
        for w, loss, (dx, dW) in zip(ws, losses, outs):
            assert_parity({"loss": loss, "dx": to_np64(dx), "dW": to_np64(dW)}, _oracle(w), "bf16")
        slabs.set_workspace(buf[off:off + 1024])
        with pytest.raises(FlceError) as e:
            run(slabs, ws[0])
        assert e.value.status_name == "FLCE_ERR_BUDGET"
    finally:
        slabs.set_workspace(None)


def test_other_ignore_index_and_bad_target(slabs):
    from flce_testing import device_inputs
    from linear_cross_entropy_token_gb300 import FlceError
    w = workloads.generate(workloads.custom(2048, 64, 40000, "bf16", seed=32))
    w.t[::5] = 3                     # class 3 marks the ignored tokens
    res = run(slabs, w, ignore_index=3)
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, ignore_index=3, chunk=512)
    assert_parity(res, ref, "bf16", token_rtol=1e-3)
    w.t[17] = 40000
    x, W, t = device_inputs(w)
    with pytest.raises(FlceError) as e:
        slabs.forward_backward(x, W, t, ignore_index=3)
    assert e.value.status_name == "FLCE_ERR_BAD_TARGET"


def test_empty_batch_and_single_token(slabs):
    x = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    W = torch.randn(3000, 64, device="cuda").to(torch.bfloat16)
    t = torch.empty(0, device="cuda", dtype=torch.int64)
    dW = torch.full((3000, 64), 7.0, device="cuda")
    loss, dx, dW = slabs.forward_backward(x, W, t, dW=dW)
    assert loss == 0.0 and dx.shape == (0, 64) and torch.all(dW == 0)
    w = workloads.generate(workloads.custom(1, 64, 40000, "bf16", seed=33))
    assert_parity(run(slabs, w), _oracle(w), "bf16")
