"""flce_loss_static, the loss-only entry point that allocates no device memory.

It serves callers that cannot let a library call cudaMalloc: a framework
whose pool allocator must account for every byte of device memory, a runtime
on a fixed memory plan, or code that must not pay the device-wide
synchronisation of cudaFree. Its scratch is a static device array inside the
library, so this test checks, through the C ABI, on several calls in a row
with different shapes (the shared scratch keeps the previous call's
contents):

* its loss and per-token losses against the fp64 oracle, and against those
  of the handle-based flce_forward_backward, within the loss tolerance of
  the other tests;
* batches of one chunk, of several chunks with a ragged last one, and a
  vocabulary so large that the scratch bound shortens the chunk below 4096
  tokens;
* that a repeated call takes no device memory, and that sizes beyond the
  scratch are refused.

This file is collected last on purpose: a run that stops at its first failure
has then already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from flce_testing import LOSS_RTOL, device_inputs, rel_fro

pytestmark = pytest.mark.gpu

# (N, H, V, ignored fraction, seed)
CASES = [
    (1000, 256, 4099, 0.1, 21),        # one chunk, odd V
    (3000, 512, 50257, 0.05, 22),      # one chunk, GPT-2-sized vocabulary
    (9000, 512, 32000, 0.1, 23),       # three 4096-token chunks, the last 808 tokens
    (1500, 64, 2_000_000, 0.1, 24),    # the scratch holds 256-token chunks: six, the last 220
]


def _oracle_token_losses(w, block=32):
    """Per-token losses from the oracle's definition, a few rows at a time
    (the 2,000,000-entry vocabulary's logits do not fit host memory whole)."""
    xr = workloads.F64Rows(w.x)
    Wd = w.W_f64()
    out = np.empty(w.N)
    for s in range(0, w.N, block):
        r = np.arange(s, min(w.N, s + block))
        out[r] = oracle.token_loss_rows(xr, Wd, w.t, r, w.ignore_index)
    n_valid = int(oracle.valid_mask(w.t, w.ignore_index).sum())
    return out, float(out.sum()) / n_valid


def test_loss_static_matches_the_oracle_and_forward_backward_on_calls_in_a_row():
    from linear_cross_entropy_token_gb300 import FLCE, flce
    h = FLCE("bf16", 0)
    try:
        for i, (N, H, V, ign, seed) in enumerate(CASES):
            w = workloads.generate(workloads.custom(N, H, V, "bf16", ignore_frac=ign, seed=seed))
            x, W, t = device_inputs(w)
            loss_fb, _, _ = h.forward_backward(x, W, t)
            tl_fb = h.token_losses(N).double().cpu().numpy()
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
            got = tl.double().cpu().numpy()
            assert np.isfinite(got).all()
            ref_tl, ref_loss = _oracle_token_losses(w)
            assert abs(loss - ref_loss) / ref_loss <= LOSS_RTOL, (N, V, loss, ref_loss)
            assert rel_fro(got, ref_tl) <= LOSS_RTOL, (N, V)
            assert not got[w.t == -100].any()
            assert abs(loss - loss_fb) / abs(loss_fb) <= LOSS_RTOL, (loss, loss_fb)
            assert rel_fro(got, tl_fb) <= LOSS_RTOL
            del x, W, t, out
    finally:
        h.close()


def test_loss_static_refuses_sizes_beyond_its_scratch():
    from linear_cross_entropy_token_gb300 import flce
    lib = flce.load()
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(1, dtype=torch.int64, device="cuda")
    tl = torch.zeros(1, dtype=torch.float32, device="cuda")
    loss = ctypes.c_float()
    # V = 20 million needs 128 x 312500 x 8 bytes = 320 MB of scratch for one
    # 128-token chunk (a partial per 64 vocabulary columns), beyond the 64 MiB
    # array: refused before any launch
    st = lib.flce_loss_static(buf.data_ptr(), buf.data_ptr(), t.data_ptr(), 1, 8, 20_000_000, -100,
                              ctypes.byref(loss), tl.data_ptr(), None)
    assert st == 1  # FLCE_ERR_INVALID_ARG
