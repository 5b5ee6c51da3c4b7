"""flce_loss_static, the loss-only entry point that allocates no device memory.

It serves callers that cannot let a library call cudaMalloc: a framework
whose pool allocator must account for every byte of device memory, a runtime
on a fixed memory plan, or code that must not pay the device-wide
synchronisation of cudaFree. Its scratch is a static device array inside the
library, so this test checks three things through the C ABI. Its loss and
per-token losses match those of the handle-based flce_forward_backward, on
two calls in a row with different shapes (the shared scratch keeps the
previous call's contents). A repeated call takes no device memory. Sizes
beyond the scratch are refused.

This file is collected last on purpose: a run that stops at its first failure
has then already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from flce_testing import LOSS_RTOL, device_inputs, rel_fro

pytestmark = pytest.mark.gpu


def test_loss_static_matches_forward_backward_on_two_calls():
    from linear_cross_entropy_token_gb300 import FLCE, flce
    h = FLCE("bf16", 0)
    cases = [(1000, 256, 4099, 0.1, 21), (3000, 512, 50257, 0.05, 22)]
    try:
        for i, (N, H, V, ign, seed) in enumerate(cases):
            w = workloads.generate(workloads.custom(N, H, V, "bf16", ignore_frac=ign, seed=seed))
            x, W, t = device_inputs(w)
            loss_ref, _, _ = h.forward_backward(x, W, t)
            tl_ref = h.token_losses(N).double().cpu().numpy()
            out = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            free0, _ = torch.cuda.mem_get_info()
            loss, tl = flce.loss_static(x, W, t, token_loss=out)
            torch.cuda.synchronize()
            free1, _ = torch.cuda.mem_get_info()
            if i > 0:
                # the first call on a device may load the library's module that
                # holds the static array; a later call takes nothing
                assert free1 == free0
            assert abs(loss - loss_ref) / abs(loss_ref) <= LOSS_RTOL, (loss, loss_ref)
            assert rel_fro(tl.double().cpu().numpy(), tl_ref) <= LOSS_RTOL
            assert np.isfinite(tl.cpu().numpy()).all()
    finally:
        h.close()


def test_loss_static_refuses_sizes_beyond_its_scratch():
    from linear_cross_entropy_token_gb300 import flce
    lib = flce.load()
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(1, dtype=torch.int64, device="cuda")
    tl = torch.zeros(1, dtype=torch.float32, device="cuda")
    loss = ctypes.c_float()
    # V = 20 million needs 128 x 78125 x 8 bytes = 80 MB of scratch for one
    # 128-token chunk, beyond the 64 MiB array: refused before any launch
    st = lib.flce_loss_static(buf.data_ptr(), buf.data_ptr(), t.data_ptr(), 1, 8, 20_000_000, -100,
                              ctypes.byref(loss), tl.data_ptr(), None)
    assert st == 1  # FLCE_ERR_INVALID_ARG
