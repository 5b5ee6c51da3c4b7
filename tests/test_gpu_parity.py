"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element
by element, on the seeded workloads, at sizes the oracle finishes in seconds
that still span several tiles and ragged tails, plus the edge cases."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import assert_parity, device_inputs, rel_fro, run, to_np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["single", "pair", "pair-one_launch", "wide", "wide-one_launch",
                                        "auto", "auto-one_launch"])
def bf16(request):
    """Every GEMM tile shape: one CTA per 128 x 256 tile; CTA pairs per
    256 x 256 tile and per 256 x 512 tile, each with the dx and dW GEMMs in
    one dynamically scheduled launch or in two launches; and the default,
    which picks wide or pair tiles per GEMM (one launch then runs on the dx
    GEMM's tile shape)."""
    from linear_cross_entropy_token_gb300 import FLCE
    cta, _, sep = request.param.partition("-")
    h = FLCE("bf16", 0, hbm_budget_bytes=4 << 30, cta=cta,
             backward=sep or "auto")
    yield h
    h.close()


@pytest.fixture(scope="module")
def bf16_recompute():
    from linear_cross_entropy_token_gb300 import FLCE
    h = FLCE("bf16", 0, dlogits_mode="recompute")
    yield h
    h.close()


@pytest.fixture(scope="module")
def fp32():
    from linear_cross_entropy_token_gb300 import FLCE
    h = FLCE("fp32", 0)
    yield h
    h.close()


def _oracle(w, chunk=None):
    return oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index, chunk=chunk)


def test_tiny_fp32_config(fp32):
    w = workloads.make("tiny_fp32")
    res = run(fp32, w, chunk=w.spec.chunk)
    assert res["plan"]["chunk"] == 64 and res["plan"]["num_chunks"] == 4
    assert_parity(res, _oracle(w), "fp32", token_rtol=1e-5)


def test_small_bf16_config(bf16):
    w = workloads.make("small_bf16")
    res = run(bf16, w)
    assert res["plan"]["num_chunks"] == 1
    assert_parity(res, _oracle(w), "bf16", token_rtol=1e-3)


def test_small_bf16_config_recompute(bf16_recompute):
    w = workloads.make("small_bf16")
    res = run(bf16_recompute, w)
    assert_parity(res, _oracle(w), "bf16", token_rtol=1e-3)


@pytest.fixture(scope="module", params=["inplace", "recompute"])
def bf16_pair(request):
    from linear_cross_entropy_token_gb300 import FLCE
    h = FLCE("bf16", 0, hbm_budget_bytes=4 << 30, dlogits_mode=request.param, cta="pair")
    yield h
    h.close()


@pytest.mark.parametrize("N,H,V,chunk,ign", [
    (2048, 1024, 32000, 0, 0.1),     # the small bf16 config's shape
    (1000, 256, 4099, 300, 0.1),     # odd V, N % C != 0, C % 256 != 0
    (256, 128, 4096, 64, 0.0),       # C < 128: the pair's second CTA holds no rows
    (777, 136, 1000, 384, 0.2),      # K tail, ragged 256-row pair tiles
    (1536, 256, 8192, 512, 0.05),
])
def test_cta_pair_tiles(bf16_pair, N, H, V, chunk, ign):
    """The same parity on 256 x 256 tiles computed by CTA pairs."""
    w = workloads.generate(workloads.custom(N, H, V, "bf16", ignore_frac=ign, seed=N + 3 * V))
    assert_parity(run(bf16_pair, w, chunk=chunk), _oracle(w), "bf16", token_rtol=1e-3)


def test_cta_pair_matches_single(bf16_pair):
    """Both tile shapes accumulate each output in the same k order: results
    agree to rounding of the fp32 accumulation order within a k-block."""
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(1024, 512, 6000, "bf16", ignore_frac=0.1, seed=31))
    single = FLCE("bf16", 0, cta="single")
    try:
        a = run(single, w, chunk=512)
    finally:
        single.close()
    b = run(bf16_pair, w, chunk=512)
    assert abs(a["loss"] - b["loss"]) <= 1e-5 * abs(a["loss"])
    assert rel_fro(b["dW"], a["dW"]) <= 1e-2 and rel_fro(b["dx"], a["dx"]) <= 1e-2


@pytest.mark.parametrize("N,H,V,chunk,ign", [
    (1000, 256, 4099, 300, 0.1),     # odd V: last vocab tile holds 3 columns; N % C != 0, C % 128 != 0
    (512, 512, 50257, 0, 0.05),      # GPT-2-sized vocabulary
    (256, 128, 4096, 64, 0.0),       # C < 128 in bf16
    (777, 136, 1000, 256, 0.2),      # H not a multiple of 64 (K tail), V < one 1024-column span
    (130, 64, 300, 0, 0.0),          # everything smaller than one tile along some axis
    (1, 64, 500, 0, 0.0),            # a single token
    (300, 8, 1000, 0, 0.1),          # the narrowest hidden size a bf16 row allows (16 bytes)
    (257, 24, 2000, 128, 0.1),       # H inside the first k-block, N one past a tile
    (129, 72, 513, 0, 0.0),          # one k-block and a tail; V two past a multiple of 256
    (200, 64, 1, 0, 0.1),            # one class: every loss and gradient is exactly 0
    (200, 64, 2, 0, 0.0),            # two classes
])
def test_ragged_shapes(bf16, N, H, V, chunk, ign):
    w = workloads.generate(workloads.custom(N, H, V, "bf16", ignore_frac=ign, seed=N + V))
    res = run(bf16, w, chunk=chunk)
    assert_parity(res, _oracle(w), "bf16", token_rtol=1e-3)


@pytest.mark.parametrize("N,H,V,chunk", [(1000, 256, 4099, 300), (256, 128, 4096, 64)])
def test_ragged_shapes_recompute(bf16_recompute, N, H, V, chunk):
    w = workloads.generate(workloads.custom(N, H, V, "bf16", ignore_frac=0.1, seed=5))
    assert_parity(run(bf16_recompute, w, chunk=chunk), _oracle(w), "bf16", token_rtol=1e-3)


@pytest.mark.parametrize("N,H,V,chunk", [(300, 100, 999, 128), (64, 7, 33, 0)])
def test_fp32_ragged(fp32, N, H, V, chunk):
    w = workloads.generate(workloads.custom(N, H, V, "fp32", ignore_frac=0.1, seed=9))
    assert_parity(run(fp32, w, chunk=chunk), _oracle(w), "fp32", token_rtol=1e-5)


def test_chunk_sizes_agree(bf16):
    """Chunking is exact: every C gives the oracle's result."""
    w = workloads.generate(workloads.custom(1536, 256, 8192, "bf16", ignore_frac=0.05, seed=2))
    ref = _oracle(w)
    for c in (128, 384, 512, 1536, 0):
        assert_parity(run(bf16, w, chunk=c), ref, "bf16", token_rtol=1e-3)


# ------------------------------------------------------------ edge cases

def test_all_tokens_ignored(bf16, fp32):
    for h, dt in ((bf16, "bf16"), (fp32, "fp32")):
        w = workloads.generate(workloads.custom(300, 64, 500, dt, seed=3))
        w.t[:] = -100
        res = run(h, w, chunk=128)
        assert res["loss"] == 0.0
        assert np.all(res["dx"] == 0.0) and np.all(res["dW"] == 0.0)
        assert np.all(res["token_loss"] == 0.0)


def test_empty_batch(bf16):
    W = torch.randn(100, 64, device="cuda").to(torch.bfloat16)
    x = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    t = torch.empty(0, device="cuda", dtype=torch.int64)
    dW = torch.full((100, 64), 7.0, device="cuda")
    loss, dx, dW = bf16.forward_backward(x, W, t, dW=dW)
    assert loss == 0.0 and dx.shape == (0, 64) and torch.all(dW == 0)


def test_zero_weight_closed_form(bf16):
    """W = 0: every logit is 0, loss = ln V, dx = 0 exactly,
    dW_j = (1/n_v)(sum_valid x_i / V - sum_{valid, t_i = j} x_i)."""
    w = workloads.generate(workloads.custom(700, 128, 3000, "bf16", ignore_frac=0.1, seed=4))
    w.W[:] = 0
    res = run(bf16, w, chunk=256)
    assert abs(res["loss"] - math.log(3000)) <= 2e-6 * math.log(3000)
    assert np.all(res["dx"] == 0.0)
    x = w.x_f64()
    valid = w.t != -100
    nv = valid.sum()
    dW = np.tile(x[valid].sum(0) / 3000, (3000, 1))
    np.subtract.at(dW, w.t[valid], x[valid])
    dW /= nv
    assert rel_fro(res["dW"], dW) <= 1e-2


def test_bad_target_reports_status(bf16):
    from linear_cross_entropy_token_gb300 import FlceError
    w = workloads.generate(workloads.custom(200, 64, 500, "bf16", seed=6))
    for bad in (500, -5):
        w.t[17] = bad
        x, W, t = device_inputs(w)
        with pytest.raises(FlceError) as e:
            bf16.forward_backward(x, W, t)
        assert e.value.status_name == "FLCE_ERR_BAD_TARGET"


def test_other_ignore_index(bf16):
    w = workloads.generate(workloads.custom(400, 64, 700, "bf16", seed=7))
    w.t[::5] = 3                     # class 3 marks the ignored tokens
    res = run(bf16, w, chunk=128, ignore_index=3)
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, ignore_index=3)
    assert_parity(res, ref, "bf16", token_rtol=1e-3)


def test_large_logits_stability(bf16):
    """W -> W + 1·uᵀ shifts every logit of token i by x_i·u (|z| ~ 100..200,
    beyond exp's fp32 range): loss and gradients stay finite and match the
    oracle on the same (rounded) inputs."""
    w = workloads.generate(workloads.custom(512, 128, 2000, "bf16", ignore_frac=0.05, seed=8))
    u = np.float32(4.0) * np.sign(np.random.default_rng(0).standard_normal(128)).astype(np.float32)
    Wf = workloads.bf16_bits_to_f32(w.W) + u[None, :]
    workloads.round_f32_to_bf16_bits(Wf.astype(np.float32), w.W)
    ref = _oracle(w)
    assert np.abs(w.x_f64() @ w.W_f64()[:1].T).max() > 90
    res = run(bf16, w, chunk=256)
    assert np.isfinite(res["loss"])
    assert_parity(res, ref, "bf16", token_rtol=1e-3)


def test_repeatable_bit_for_bit(bf16):
    w = workloads.generate(workloads.custom(1024, 256, 5000, "bf16", ignore_frac=0.1, seed=10))
    a = run(bf16, w, chunk=384)
    b = run(bf16, w, chunk=384)
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["dx"], b["dx"]) and np.array_equal(a["dW"], b["dW"])


def test_host_buffer_entry_point(bf16):
    w = workloads.generate(workloads.custom(600, 128, 3000, "bf16", ignore_frac=0.1, seed=11))
    xh = torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    Wh = torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16).pin_memory()
    th = torch.from_numpy(w.t).pin_memory()
    loss, dx, dW = bf16.forward_backward_host(xh, Wh, th, chunk=256)
    res = {"loss": loss, "dx": to_np64(dx), "dW": to_np64(dW)}
    assert_parity(res, _oracle(w), "bf16")
    # with profiling on, the copies are timed and counted, and launch no kernel
    bf16.set_profiling(True)
    bf16.profile_reset()
    launches = bf16.launch_count()
    bf16.forward_backward_host(xh, Wh, th, chunk=256)
    prof = bf16.profile()
    bf16.set_profiling(False)
    bf16.profile_reset()
    copy = prof["h2d_copy"]
    assert copy["launches"] == 1 and copy["total_ms"] > 0
    assert copy["bytes"] == (600 * 128 + 3000 * 128) * 2 + 600 * 8
    assert bf16.launch_count() - launches == sum(v["launches"] for k, v in prof.items() if k != "h2d_copy")


def test_workspace_bytes_matches_the_call(bf16):
    """flce_workspace_bytes on a handle predicts the workspace of the plan the
    next call runs with, and reports a budget that cannot hold one chunk."""
    from linear_cross_entropy_token_gb300 import FLCE, FlceError
    w = workloads.generate(workloads.custom(1000, 256, 4099, "bf16", ignore_frac=0.1, seed=13))
    for chunk in (0, 300):
        n = bf16.workspace_bytes(1000, 256, 4099, chunk)
        run(bf16, w, chunk=chunk)
        assert n == bf16.last_plan()["workspace_bytes"]
    tiny = FLCE("bf16", 0, hbm_budget_bytes=1 << 20)
    try:
        with pytest.raises(FlceError) as e:
            tiny.workspace_bytes(16384, 4096, 128256)
        assert e.value.status_name == "FLCE_ERR_BUDGET"
    finally:
        tiny.close()


def test_pipelined_host_submissions(bf16):
    """submit/wait with two calls in flight: each call's loss and outputs
    match the oracle on its own inputs. A third submission while two are
    outstanding, and a wait on a ticket that is not outstanding, are refused."""
    from linear_cross_entropy_token_gb300 import FlceError
    ws = [workloads.generate(workloads.custom(600, 128, 3000, "bf16", ignore_frac=0.1, seed=20 + i))
          for i in range(3)]
    host = [(torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16).pin_memory(),
             torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16).pin_memory(),
             torch.from_numpy(w.t).pin_memory()) for w in ws]
    outs = [(torch.empty(600, 128, dtype=torch.bfloat16, device="cuda"),
             torch.empty(3000, 128, dtype=torch.float32, device="cuda")) for _ in ws]
    t0, _, _ = bf16.submit_host(*host[0], chunk=256, dx=outs[0][0], dW=outs[0][1])
    t1, _, _ = bf16.submit_host(*host[1], chunk=256, dx=outs[1][0], dW=outs[1][1])
    with pytest.raises(FlceError) as e:
        bf16.submit_host(*host[2], chunk=256, dx=outs[2][0], dW=outs[2][1])
    assert e.value.status_name == "FLCE_ERR_INVALID_ARG"
    losses = [bf16.wait(t0)]
    t2, _, _ = bf16.submit_host(*host[2], chunk=256, dx=outs[2][0], dW=outs[2][1])
    losses += [bf16.wait(t1), bf16.wait(t2)]
    with pytest.raises(FlceError):
        bf16.wait(t2)
    for w, loss, (dx, dW) in zip(ws, losses, outs):
        assert_parity({"loss": loss, "dx": to_np64(dx), "dW": to_np64(dW)}, _oracle(w), "bf16")


def test_device_result_entry_and_graph_capture(bf16):
    """flce_forward_backward_async leaves loss and n_valid in device memory
    without a host sync. Captured in a CUDA graph and replayed after new
    inputs are written into the same buffers, it gives the oracle's results
    on those inputs."""
    ws = [workloads.generate(workloads.custom(1000, 256, 4099, "bf16", ignore_frac=0.1, seed=s))
          for s in (40, 41)]
    x, W, t = device_inputs(ws[0])
    dx = torch.empty_like(x)
    dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    nv = torch.empty((), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # outside capture: allocates the workspace
        bf16.forward_backward_async(x, W, t, chunk=300, loss=loss, n_valid=nv, dx=dx, dW=dW)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert_parity({"loss": loss.item(), "dx": to_np64(dx), "dW": to_np64(dW)}, _oracle(ws[0]), "bf16")
    assert nv.item() == int((ws[0].t != -100).sum())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bf16.forward_backward_async(x, W, t, chunk=300, loss=loss, n_valid=nv, dx=dx, dW=dW)
    for w in ws[::-1]:
        x2, W2, t2 = device_inputs(w)
        x.copy_(x2)
        W.copy_(W2)
        t.copy_(t2)
        g.replay()
        torch.cuda.synchronize()
        assert_parity({"loss": loss.item(), "dx": to_np64(dx), "dW": to_np64(dW)}, _oracle(w), "bf16")
        assert nv.item() == int((w.t != -100).sum())
    bf16.async_status()


def test_device_result_reports_errors_late(bf16):
    """An out-of-range target in a sync-free call: the device loss is NaN and
    the error comes out of flce_async_status once, then the handle is clean."""
    from linear_cross_entropy_token_gb300 import FlceError
    w = workloads.generate(workloads.custom(200, 64, 500, "bf16", seed=42))
    w.t[5] = 600
    x, W, t = device_inputs(w)
    loss, _, _, _ = bf16.forward_backward_async(x, W, t)
    torch.cuda.synchronize()
    assert math.isnan(loss.item())
    with pytest.raises(FlceError) as e:
        bf16.async_status()
    assert e.value.status_name == "FLCE_ERR_BAD_TARGET"
    bf16.async_status()
    w.t[5] = 3
    x, W, t = device_inputs(w)
    loss, _, _, _ = bf16.forward_backward_async(x, W, t)
    bf16.async_status()
    assert abs(loss.item() - _oracle(w).loss) <= 1e-3 * _oracle(w).loss


def test_misaligned_or_mismatched_arguments_are_refused(bf16):
    """The C ABI refuses pointers its vector loads and TMA maps cannot take
    (before any launch), and the binding refuses tensors whose shapes do not
    fit together."""
    import ctypes
    w = workloads.generate(workloads.custom(64, 64, 300, "bf16", seed=14))
    x, W, t = device_inputs(w)
    dx = torch.empty_like(x)
    dW = torch.empty(W.shape, dtype=torch.float32, device="cuda")
    raw = torch.zeros(64 * 8 + 16, dtype=torch.uint8, device="cuda")
    loss = ctypes.c_float()
    s = torch.cuda.current_stream().cuda_stream
    fb = bf16.lib.flce_forward_backward
    assert fb(bf16.h, x.data_ptr(), W.data_ptr(), raw.data_ptr() + 4, 64, 64, 300, -100, 0,
              ctypes.byref(loss), dx.data_ptr(), dW.data_ptr(), s) == 1
    assert fb(bf16.h, x.data_ptr() + 8, W.data_ptr(), t.data_ptr(), 63, 64, 300, -100, 0,
              ctypes.byref(loss), dx.data_ptr(), dW.data_ptr(), s) == 1
    assert fb(bf16.h, x.data_ptr(), W.data_ptr(), t.data_ptr(), 64, 60, 300, -100, 0,
              ctypes.byref(loss), dx.data_ptr(), dW.data_ptr(), s) == 1   # H % 8 != 0
    with pytest.raises(ValueError):
        bf16.forward_backward(x, W[:, :32].contiguous(), t)
    with pytest.raises(ValueError):
        bf16.forward_backward(x, W, t[:63])
    with pytest.raises(ValueError):
        bf16.forward_backward(x, W, t, dW=torch.empty(299, 64, device="cuda"))
    # the handle still works afterwards
    assert_parity(run(bf16, w), _oracle(w), "bf16")


def test_two_handles_on_two_streams():
    """Two handles driven on two streams at once (each call only waits for its
    own stream) give the same results as the same calls made one at a time."""
    from linear_cross_entropy_token_gb300 import FLCE
    ws = [workloads.generate(workloads.custom(1500, 256, 7000, "bf16", ignore_frac=0.1, seed=s))
          for s in (50, 51)]
    hs = [FLCE("bf16", 0, cta="pair"), FLCE("bf16", 0, cta="pair")]
    try:
        inputs = [device_inputs(w) for w in ws]
        alone = []
        for h, (x, W, t) in zip(hs, inputs):
            loss, dx, dW = h.forward_backward(x, W, t, chunk=512)
            alone.append((loss, dx.clone(), dW.clone()))
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        outs = [None, None]
        torch.cuda.synchronize()
        for rep in range(3):
            for i in (0, 1):
                with torch.cuda.stream(streams[i]):
                    loss, n_valid, dx, dW = hs[i].forward_backward_async(*inputs[i], chunk=512)
                    outs[i] = (loss, dx, dW)
            torch.cuda.synchronize()
            for i in (0, 1):
                assert outs[i][0].item() == alone[i][0]
                assert torch.equal(outs[i][1], alone[i][1]) and torch.equal(outs[i][2], alone[i][2])
        for h in hs:
            h.async_status()
    finally:
        for h in hs:
            h.close()


def test_workspace_allocation_failure_is_reported():
    """A plan whose workspace the device cannot hold (a 328 GB chunk buffer
    under a 1 TB budget) fails in cudaMalloc before any launch: the call
    reports FLCE_ERR_BUDGET and the handle still works afterwards."""
    from linear_cross_entropy_token_gb300 import FLCE, FlceError
    N, H, V = 32768, 8, 5_000_000
    h = FLCE("bf16", 0, hbm_budget_bytes=1 << 40)
    try:
        assert h.workspace_bytes(N, H, V) > 300e9
        x = torch.zeros(N, H, dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(V, H, dtype=torch.bfloat16, device="cuda")
        t = torch.zeros(N, dtype=torch.int64, device="cuda")
        with pytest.raises(FlceError) as e:
            h.forward_backward(x, W, t)
        assert e.value.status_name == "FLCE_ERR_BUDGET"
        del x, W, t
        torch.cuda.empty_cache()
        w = workloads.generate(workloads.custom(500, 64, 1000, "bf16", seed=15))
        assert_parity(run(h, w), _oracle(w), "bf16")
    finally:
        h.close()


def test_caller_workspace(bf16):
    from linear_cross_entropy_token_gb300 import FLCE, FlceError, plan
    w = workloads.generate(workloads.custom(500, 64, 1000, "bf16", seed=12))
    p = plan(500, 64, 1000, "bf16", chunk=256)
    h = FLCE("bf16", 0)
    try:
        buf = torch.empty(p["workspace_bytes"] + 4096, dtype=torch.uint8, device="cuda")
        off = (-buf.data_ptr()) % 1024
        h.set_workspace(buf[off:off + p["workspace_bytes"]])
        assert_parity(run(h, w, chunk=256), _oracle(w), "bf16")
        small = buf[off:off + 1024]
        h.set_workspace(small)
        with pytest.raises(FlceError) as e:
            run(h, w, chunk=256)
        assert e.value.status_name == "FLCE_ERR_BUDGET"
    finally:
        h.close()


@pytest.mark.parametrize("V,fused", [(262083, True), (262211, False)])
def test_combine_and_dlogits_launches_by_row_width(V, fused):
    """In-place mode runs the log-sum-exp combine and the dlogits pass as one
    launch, a block per token row, for chunk rows of at most 262144 columns
    (the buffer's row is V rounded up to 64), and as two launches beyond
    that; both forms match the oracle."""
    from linear_cross_entropy_token_gb300 import FLCE
    w = workloads.generate(workloads.custom(200, 64, V, "bf16", ignore_frac=0.1, seed=31))
    h = FLCE("bf16", 0)
    try:
        h.set_profiling(True)
        h.profile_reset()
        res = run(h, w)
        prof = h.profile()
    finally:
        h.close()
    assert ("combine_dlogits" in prof) == fused
    assert ("lse_combine" in prof) == (not fused) and ("dlogits_inplace" in prof) == (not fused)
    assert_parity(res, _oracle(w), "bf16", token_rtol=1e-3)
