"""Helpers for the GPU tests: move a workload to the device, run the library
through its C ABI, and compare with the oracle in float64 on the host."""
import numpy as np
import torch


def device_inputs(w, device="cuda"):
    """x, W, t of a workload as device tensors (bf16 bits reinterpreted)."""
    if w.x.dtype == np.uint16:
        x = torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16)
        W = torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16)
    else:
        x = torch.from_numpy(w.x)
        W = torch.from_numpy(w.W)
    t = torch.from_numpy(w.t)
    return x.to(device), W.to(device), t.to(device)


def to_np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(a - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def run(handle, w, chunk=0, ignore_index=-100):
    x, W, t = device_inputs(w)
    loss, dx, dW = handle.forward_backward(x, W, t, ignore_index=ignore_index, chunk=chunk)
    torch.cuda.synchronize()
    tl = handle.token_losses(w.N) if w.N else torch.zeros(0)
    return {"loss": loss, "dx": to_np64(dx), "dW": to_np64(dW), "token_loss": to_np64(tl),
            "plan": handle.last_plan()}


# tolerances stated for the method: loss relative error, dx/dW relative
# Frobenius error (bf16 inputs with fp32 accumulation / fp32 inputs)
LOSS_RTOL = 1e-3
GRAD_RTOL = {"bf16": 1e-2, "fp32": 1e-5}


def assert_parity(res, ref, dtype, token_rtol=None):
    tol = GRAD_RTOL[dtype]
    if ref.loss == 0.0:
        assert res["loss"] == 0.0
    else:
        assert abs(res["loss"] - ref.loss) / abs(ref.loss) <= LOSS_RTOL, (res["loss"], ref.loss)
    edx = rel_fro(res["dx"], ref.dx)
    edw = rel_fro(res["dW"], ref.dW)
    assert edx <= tol, f"dx relative Frobenius error {edx:.3e} > {tol}"
    assert edw <= tol, f"dW relative Frobenius error {edw:.3e} > {tol}"
    if token_rtol is not None and len(ref.token_loss):
        et = rel_fro(res["token_loss"], ref.token_loss)
        assert et <= token_rtol, f"token loss relative error {et:.3e}"
    return edx, edw
