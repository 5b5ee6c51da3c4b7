"""Host-side checks of the Python binding: the C ABI takes bare pointers and
sizes, so every shape, dtype, device and layout mismatch must be refused
before a call reaches it. CPU tensors stand in for device tensors here."""
import pytest
import torch

from linear_cross_entropy_token_gb300.flce import check_call_tensors

CPU = torch.device("cpu")
OTHER = torch.device("meta")


def _ok(N=6, H=8, V=10, dtype=torch.bfloat16):
    x = torch.zeros(N, H, dtype=dtype)
    W = torch.zeros(V, H, dtype=dtype)
    t = torch.zeros(N, dtype=torch.int64)
    dx = torch.zeros(N, H, dtype=dtype)
    dW = torch.zeros(V, H, dtype=torch.float32)
    return x, W, t, dx, dW


def test_consistent_call_passes():
    x, W, t, dx, dW = _ok()
    check_call_tensors(x, W, t, dx, dW, torch.bfloat16, CPU, CPU)
    check_call_tensors(x, W, t, None, None, torch.bfloat16, CPU, CPU)


@pytest.mark.parametrize("case", [
    "W_columns", "t_length", "x_1d", "t_2d", "x_dtype", "W_dtype", "t_dtype", "x_strided",
    "W_device", "dx_shape", "dx_dtype", "dW_shape", "dW_dtype", "dW_strided", "dx_device",
])
def test_mismatch_is_refused(case):
    x, W, t, dx, dW = _ok()
    if case == "W_columns":
        W = torch.zeros(10, 16, dtype=torch.bfloat16)
    elif case == "t_length":
        t = torch.zeros(5, dtype=torch.int64)
    elif case == "x_1d":
        x = torch.zeros(48, dtype=torch.bfloat16)
    elif case == "t_2d":
        t = torch.zeros(6, 1, dtype=torch.int64)
    elif case == "x_dtype":
        x = x.float()
    elif case == "W_dtype":
        W = W.half()
    elif case == "t_dtype":
        t = t.int()
    elif case == "x_strided":
        x = torch.zeros(8, 6, dtype=torch.bfloat16).T
    elif case == "W_device":
        W = W.to(OTHER)
    elif case == "dx_shape":
        dx = torch.zeros(6, 4, dtype=torch.bfloat16)
    elif case == "dx_dtype":
        dx = dx.float()
    elif case == "dW_shape":
        dW = torch.zeros(9, 8)
    elif case == "dW_dtype":
        dW = dW.bfloat16()
    elif case == "dW_strided":
        dW = torch.zeros(8, 10).T
    elif case == "dx_device":
        dx = dx.to(OTHER)
    with pytest.raises(ValueError):
        check_call_tensors(x, W, t, dx, dW, torch.bfloat16, CPU, CPU)
