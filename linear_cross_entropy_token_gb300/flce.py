"""ctypes binding of libflce.so (include/flce.h), using torch tensors for
device memory and torch's current CUDA stream.

The binding only marshals arguments. Every step of the computation runs in
the library's kernels; there is no other code path. If libflce.so is missing,
loading raises: build it with ``linear_cross_entropy_token_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libflce.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "flce.h")

FLCE_OK = 0
STATUS = {0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_UNSUPPORTED", 3: "FLCE_ERR_BUDGET",
          4: "FLCE_ERR_BAD_TARGET", 5: "FLCE_ERR_TIMEOUT", 6: "FLCE_ERR_CUDA"}
DTYPE_BF16, DTYPE_FP32 = 0, 1
DLOGITS = {"auto": 0, "inplace": 1, "recompute": 2, "slabs": 3}
DLOGITS_NAMES = {v: k for k, v in DLOGITS.items()}
CTA = {"auto": 0, "single": 1, "pair": 2, "wide": 4}
BACKWARD = {"auto": 0, "separate": 1, "one_launch": 2}
KERNEL_KINDS = ["count_valid", "gemm_logits_lse", "lse_combine", "dlogits_inplace",
                "gemm_dlogits_recompute", "gemm_dx", "dx_split_reduce", "gemm_dw",
                "loss_finalize", "simt_gemm_f32", "simt_tile_stats_f32", "gemm_dx_dw",
                "device_result", "combine_dlogits", "h2d_copy"]


class FlceError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class Config(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("device", ctypes.c_int32),
                ("hbm_budget_bytes", ctypes.c_uint64), ("dlogits_mode", ctypes.c_int32),
                ("timeout_ms", ctypes.c_int32), ("cta_pair", ctypes.c_int32),
                ("backward_launch", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int64), ("num_chunks", ctypes.c_int64),
                ("vocab_tiles", ctypes.c_int64), ("ldv", ctypes.c_int64),
                ("dx_splits", ctypes.c_int64), ("workspace_bytes", ctypes.c_uint64),
                ("logits_bytes", ctypes.c_uint64), ("tile_m", ctypes.c_int64),
                ("tile_n", ctypes.c_int64), ("vocab_slab", ctypes.c_int64),
                ("dlogits_mode", ctypes.c_int64), ("tile_n_dx", ctypes.c_int64),
                ("tile_n_dw", ctypes.c_int64), ("dw_beside_dx", ctypes.c_int64),
                ("backward_one_launch", ctypes.c_int64)]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["dlogits"] = DLOGITS_NAMES.get(d["dlogits_mode"], str(d["dlogits_mode"]))
        return d


class KernelProfile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("total_ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libflce.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: the CUDA library must be built "
                           "(linear_cross_entropy_token_gb300.build.build())")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
    sigs = {
        "flce_abi_version": (i32, []),
        "flce_status_string": (ctypes.c_char_p, [i32]),
        "flce_make_plan": (i32, [ctypes.POINTER(Config), i64, i64, i64, i64, i32, ctypes.POINTER(Plan)]),
        "flce_create": (i32, [ctypes.POINTER(vp), ctypes.POINTER(Config)]),
        "flce_destroy": (None, [vp]),
        "flce_set_workspace": (i32, [vp, vp, u64]),
        "flce_forward_backward": (i32, [vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                        ctypes.POINTER(ctypes.c_float), vp, vp, vp]),
        "flce_forward_backward_host": (i32, [vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                             ctypes.POINTER(ctypes.c_float), vp, vp, vp]),
        "flce_forward_backward_async": (i32, [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp,
                                              vp, vp]),
        "flce_async_status": (i32, [vp, vp]),
        "flce_count_valid": (i32, [vp, vp, i64, i64, vp, vp]),
        "flce_forward_backward_shard": (i32, [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp,
                                              vp, vp]),
        "flce_submit_host": (i32, [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp,
                                   ctypes.POINTER(u64)]),
        "flce_wait": (i32, [vp, u64, ctypes.POINTER(ctypes.c_float)]),
        "flce_token_losses": (i32, [vp, vp, i64, vp]),
        "flce_last_plan": (i32, [vp, ctypes.POINTER(Plan)]),
        "flce_set_profiling": (i32, [vp, i32]),
        "flce_profile_read": (i32, [vp, i32, ctypes.POINTER(KernelProfile)]),
        "flce_profile_reset": (None, [vp]),
        "flce_kernel_name": (ctypes.c_char_p, [i32]),
        "flce_launch_count": (i64, [vp]),
        "flce_workspace_bytes": (u64, [vp, i64, i64, i64, i64]),
        "flce_last_error": (ctypes.c_char_p, [vp]),
        "flce_check_gemm": (i32, [vp, i32, i32, vp, vp, vp, i64, i64, i64, vp]),
        "flce_check_wait_timeout": (i32, [vp, u32, vp]),
        "flce_loss_static": (i32, [vp, vp, vp, i64, i64, i64, i64, ctypes.POINTER(ctypes.c_float),
                                   vp, vp]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def header_functions() -> list:
    """Names of the functions include/flce.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_0-9]+)\s*\(", txt)))


def make_config(dtype: str = "bf16", device: int = 0, hbm_budget_bytes: int = 0,
                dlogits_mode: str = "auto", timeout_ms: int = 0, cta: str = "auto",
                backward: str = "auto") -> Config:
    return Config(DTYPE_BF16 if dtype == "bf16" else DTYPE_FP32, device, hbm_budget_bytes,
                  DLOGITS[dlogits_mode], timeout_ms, CTA[cta], BACKWARD[backward])


def plan(N: int, H: int, V: int, dtype: str = "bf16", chunk: int = 0, hbm_budget_bytes: int = 0,
         num_sms: int = 0, cta: str = "auto", dlogits_mode: str = "auto",
         backward: str = "auto") -> dict:
    """The token-chunk plan for one call (host only; no device needed)."""
    lib = load()
    cfg = make_config(dtype, 0, hbm_budget_bytes, dlogits_mode, cta=cta, backward=backward)
    p = Plan()
    st = lib.flce_make_plan(ctypes.byref(cfg), N, H, V, chunk, num_sms, ctypes.byref(p))
    if st != FLCE_OK:
        raise FlceError(st, "flce_make_plan")
    return p.as_dict()


def check_call_tensors(x, W, t, dx, dW, dtype, in_device, out_device) -> None:
    """Shapes, dtypes, devices and contiguity of one call's tensors. The C ABI
    takes bare pointers and sizes, so a mismatch left unchecked here would
    become an out-of-bounds access there. x (N, H) and W (V, H) of `dtype` and
    t (N,) int64 on in_device; dx (N, H) of `dtype` and dW (V, H) float32 on
    out_device, when given. Raises ValueError."""
    import torch
    if x.dim() != 2 or W.dim() != 2 or t.dim() != 1:
        raise ValueError("x and W must be 2-D, t 1-D")
    N, H = x.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError(f"W has {W.shape[1]} columns, x has {H}")
    if t.shape[0] != N:
        raise ValueError(f"t has {t.shape[0]} entries, x has {N} rows")
    if x.dtype != dtype or W.dtype != dtype or t.dtype != torch.int64:
        raise ValueError(f"x and W must be {dtype}, t must be int64")
    for name, ten in (("x", x), ("W", W), ("t", t)):
        if ten.device != in_device or not ten.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor on {in_device}")
    for name, ten, shape, dt in (("dx", dx, (N, H), dtype), ("dW", dW, (V, H), torch.float32)):
        if ten is None:
            continue
        if tuple(ten.shape) != shape or ten.dtype != dt:
            raise ValueError(f"{name} must be {dt} of shape {shape}")
        if ten.device != out_device or not ten.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor on {out_device}")


def _stream_ptr(device) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


class FLCE:
    """One library handle on one device, for one input dtype ("bf16" or "fp32")."""

    def __init__(self, dtype: str = "bf16", device: int = 0, hbm_budget_bytes: int = 0,
                 dlogits_mode: str = "auto", timeout_ms: int = 0, cta: str = "auto",
                 backward: str = "auto"):
        self.lib = load()
        self.dtype = dtype
        self.device = device
        self.cfg = make_config(dtype, device, hbm_budget_bytes, dlogits_mode, timeout_ms, cta,
                               backward)
        h = ctypes.c_void_p()
        st = self.lib.flce_create(ctypes.byref(h), ctypes.byref(self.cfg))
        if st != FLCE_OK:
            raise FlceError(st, "flce_create (needs a compute capability 10.3 GPU)")
        self.h = h

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.flce_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st: int, what: str) -> None:
        if st != FLCE_OK:
            msg = self.lib.flce_last_error(self.h)
            raise FlceError(st, f"{what}: {msg.decode() if msg else ''}")

    def _torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def forward_backward(self, x, W, t, ignore_index: int = -100, chunk: int = 0,
                         dx=None, dW=None):
        """loss (float), dx (like x), dW (fp32, V x H) for device tensors x, W, t."""
        import torch
        dev = torch.device("cuda", self.device)
        check_call_tensors(x, W, t, dx, dW, self._torch_dtype(), dev, dev)
        N, H = x.shape
        V = W.shape[0]
        if dx is None:
            dx = torch.empty_like(x)
        if dW is None:
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
        loss = ctypes.c_float(0.0)
        st = self.lib.flce_forward_backward(self.h, x.data_ptr(), W.data_ptr(), t.data_ptr(), N, H, V,
                                            ignore_index, chunk, ctypes.byref(loss), dx.data_ptr(),
                                            dW.data_ptr(), _stream_ptr(dev))
        self._check(st, "flce_forward_backward")
        return loss.value, dx, dW

    def forward_backward_async(self, x, W, t, ignore_index: int = -100, chunk: int = 0,
                               loss=None, n_valid=None, dx=None, dW=None):
        """The fused call with no host synchronisation (capturable in a CUDA
        graph once the workspace exists): returns device tensors (loss, a
        0-dim float32, NaN after a device-side error; n_valid, a 0-dim
        int32; dx; dW), filled when the current stream gets there.
        async_status() reports device-side errors."""
        import torch
        dev = torch.device("cuda", self.device)
        check_call_tensors(x, W, t, dx, dW, self._torch_dtype(), dev, dev)
        N, H = x.shape
        V = W.shape[0]
        for name, ten, dt in (("loss", loss, torch.float32), ("n_valid", n_valid, torch.int32)):
            if ten is not None and (ten.numel() != 1 or ten.dtype != dt or ten.device != dev):
                raise ValueError(f"{name} must be one {dt} element on {dev}")
        if loss is None:
            loss = torch.empty((), dtype=torch.float32, device=dev)
        if n_valid is None:
            n_valid = torch.empty((), dtype=torch.int32, device=dev)
        if dx is None:
            dx = torch.empty_like(x)
        if dW is None:
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
        st = self.lib.flce_forward_backward_async(self.h, x.data_ptr(), W.data_ptr(), t.data_ptr(), N,
                                                  H, V, ignore_index, chunk, loss.data_ptr(),
                                                  n_valid.data_ptr(), dx.data_ptr(), dW.data_ptr(),
                                                  _stream_ptr(dev))
        self._check(st, "flce_forward_backward_async")
        return loss, n_valid, dx, dW

    def count_valid(self, t, ignore_index: int = -100, out=None):
        """This rank's non-ignored token count as a 0-dim int32 device tensor,
        written when the current stream gets there (no host sync)."""
        import torch
        dev = torch.device("cuda", self.device)
        if t.dim() != 1 or t.dtype != torch.int64 or t.device != dev or not t.is_contiguous():
            raise ValueError(f"t must be a contiguous 1-D int64 tensor on {dev}")
        if out is None:
            out = torch.empty((), dtype=torch.int32, device=dev)
        elif out.numel() != 1 or out.dtype != torch.int32 or out.device != dev:
            raise ValueError(f"out must be one int32 element on {dev}")
        st = self.lib.flce_count_valid(self.h, t.data_ptr(), t.shape[0], ignore_index,
                                       out.data_ptr(), _stream_ptr(dev))
        self._check(st, "flce_count_valid")
        return out

    def forward_backward_shard(self, x, W, t, n_valid_total, ignore_index: int = -100,
                               chunk: int = 0, loss=None, dx=None, dW=None):
        """One shard of a token-sharded batch: the fused call dividing by
        n_valid_total (a one-element int32 device tensor, the non-ignored
        tokens of every shard). Returns device tensors (loss, this shard's
        share of the batch mean; dx, this shard's rows; dW, this shard's
        term), with no host synchronisation; async_status() reports
        device-side errors."""
        import torch
        dev = torch.device("cuda", self.device)
        check_call_tensors(x, W, t, dx, dW, self._torch_dtype(), dev, dev)
        if (n_valid_total.numel() != 1 or n_valid_total.dtype != torch.int32
                or n_valid_total.device != dev):
            raise ValueError(f"n_valid_total must be one int32 element on {dev}")
        if loss is not None and (loss.numel() != 1 or loss.dtype != torch.float32 or loss.device != dev):
            raise ValueError(f"loss must be one float32 element on {dev}")
        N, H = x.shape
        V = W.shape[0]
        if loss is None:
            loss = torch.empty((), dtype=torch.float32, device=dev)
        if dx is None:
            dx = torch.empty_like(x)
        if dW is None:
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
        st = self.lib.flce_forward_backward_shard(self.h, x.data_ptr(), W.data_ptr(), t.data_ptr(), N,
                                                  H, V, ignore_index, chunk, n_valid_total.data_ptr(),
                                                  loss.data_ptr(), dx.data_ptr(), dW.data_ptr(),
                                                  _stream_ptr(dev))
        self._check(st, "flce_forward_backward_shard")
        return loss, dx, dW

    def async_status(self) -> None:
        """Wait for the current stream; raise FlceError for a device-side
        error recorded by forward_backward_async calls since the last check."""
        import torch
        st = self.lib.flce_async_status(self.h, _stream_ptr(torch.device("cuda", self.device)))
        self._check(st, "flce_async_status")

    def forward_backward_host(self, x_host, W_host, t_host, ignore_index: int = -100,
                              chunk: int = 0, dx=None, dW=None):
        """Same, with x, W, t in host memory (pinned for asynchronous copies)."""
        import torch
        dev = torch.device("cuda", self.device)
        check_call_tensors(x_host, W_host, t_host, dx, dW, self._torch_dtype(), torch.device("cpu"),
                           dev)
        N, H = x_host.shape
        V = W_host.shape[0]
        if dx is None:
            dx = torch.empty((N, H), dtype=self._torch_dtype(), device=dev)
        if dW is None:
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
        loss = ctypes.c_float(0.0)
        st = self.lib.flce_forward_backward_host(self.h, x_host.data_ptr(), W_host.data_ptr(),
                                                 t_host.data_ptr(), N, H, V, ignore_index, chunk,
                                                 ctypes.byref(loss), dx.data_ptr(), dW.data_ptr(),
                                                 _stream_ptr(dev))
        self._check(st, "flce_forward_backward_host")
        return loss.value, dx, dW

    def submit_host(self, x_host, W_host, t_host, ignore_index: int = -100, chunk: int = 0,
                    dx=None, dW=None):
        """Enqueue the host-buffer call and return (ticket, dx, dW) at once;
        the copies of this call overlap the compute of the previous one.
        wait(ticket) gives the loss. At most two may be outstanding."""
        import torch
        dev = torch.device("cuda", self.device)
        check_call_tensors(x_host, W_host, t_host, dx, dW, self._torch_dtype(), torch.device("cpu"),
                           dev)
        N, H = x_host.shape
        V = W_host.shape[0]
        if dx is None:
            dx = torch.empty((N, H), dtype=self._torch_dtype(), device=dev)
        if dW is None:
            dW = torch.empty((V, H), dtype=torch.float32, device=dev)
        ticket = ctypes.c_uint64(0)
        st = self.lib.flce_submit_host(self.h, x_host.data_ptr(), W_host.data_ptr(), t_host.data_ptr(),
                                       N, H, V, ignore_index, chunk, dx.data_ptr(), dW.data_ptr(),
                                       _stream_ptr(dev), ctypes.byref(ticket))
        self._check(st, "flce_submit_host")
        return ticket.value, dx, dW

    def wait(self, ticket: int) -> float:
        """Block until the submitted call `ticket` has finished; its loss."""
        loss = ctypes.c_float(0.0)
        self._check(self.lib.flce_wait(self.h, ticket, ctypes.byref(loss)), "flce_wait")
        return loss.value

    def token_losses(self, N: int):
        import torch
        out = torch.empty(N, dtype=torch.float32, device=torch.device("cuda", self.device))
        st = self.lib.flce_token_losses(self.h, out.data_ptr(), N, _stream_ptr(out.device))
        self._check(st, "flce_token_losses")
        return out

    def last_plan(self) -> dict:
        p = Plan()
        self._check(self.lib.flce_last_plan(self.h, ctypes.byref(p)), "flce_last_plan")
        return p.as_dict()

    def workspace_bytes(self, N: int, H: int, V: int, chunk: int = 0) -> int:
        """Device workspace a call of these sizes needs on this handle."""
        n = int(self.lib.flce_workspace_bytes(self.h, N, H, V, chunk))
        if n == 0:
            p = Plan()
            st = self.lib.flce_make_plan(ctypes.byref(self.cfg), N, H, V, chunk, 0, ctypes.byref(p))
            raise FlceError(st if st != FLCE_OK else 1, "flce_workspace_bytes: " +
                            self.lib.flce_last_error(self.h).decode())
        return n

    def set_workspace(self, buf) -> None:
        ptr = buf.data_ptr() if buf is not None else None
        n = buf.numel() * buf.element_size() if buf is not None else 0
        self._check(self.lib.flce_set_workspace(self.h, ptr, n), "flce_set_workspace")

    def set_profiling(self, enable: bool) -> None:
        self._check(self.lib.flce_set_profiling(self.h, int(enable)), "flce_set_profiling")

    def profile_reset(self) -> None:
        self.lib.flce_profile_reset(self.h)

    def profile(self) -> dict:
        out = {}
        for k, name in enumerate(KERNEL_KINDS):
            p = KernelProfile()
            self._check(self.lib.flce_profile_read(self.h, k, ctypes.byref(p)), "flce_profile_read")
            if p.launches:
                out[name] = {"launches": p.launches, "total_ms": p.total_ms, "flops": p.flops,
                             "bytes": p.bytes}
        return out

    def launch_count(self) -> int:
        return int(self.lib.flce_launch_count(self.h))

    def check_gemm(self, A, B, a_mn_major: bool, b_mn_major: bool, M: int, N: int, K: int):
        import torch
        if (A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or not A.is_contiguous()
                or not B.is_contiguous() or A.numel() != M * K or B.numel() != N * K
                or A.device != torch.device("cuda", self.device) or B.device != A.device):
            raise ValueError("A (M*K) and B (N*K) must be contiguous bf16 on the handle's device")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
        st = self.lib.flce_check_gemm(self.h, int(a_mn_major), int(b_mn_major), A.data_ptr(),
                                      B.data_ptr(), C.data_ptr(), M, N, K, _stream_ptr(A.device))
        self._check(st, "flce_check_gemm")
        return C

    def check_wait_timeout(self, timeout_us: int) -> int:
        import torch
        return int(self.lib.flce_check_wait_timeout(self.h, timeout_us,
                                                    _stream_ptr(torch.device("cuda", self.device))))


def loss_static(x, W, t, ignore_index: int = -100, token_loss=None):
    """Mean loss and per-token losses (no dx, dW) through flce_loss_static,
    which allocates no device memory: for callers whose device memory must
    all come from their own allocator. Returns (loss, token_loss)."""
    import torch
    lib = load()
    check_call_tensors(x, W, t, None, None, torch.bfloat16, x.device, x.device)
    N, H = x.shape
    V = W.shape[0]
    if token_loss is None:
        token_loss = torch.empty(N, dtype=torch.float32, device=x.device)
    elif (tuple(token_loss.shape) != (N,) or token_loss.dtype != torch.float32
          or token_loss.device != x.device or not token_loss.is_contiguous()):
        raise ValueError(f"token_loss must be contiguous float32 of shape ({N},) on {x.device}")
    loss = ctypes.c_float(0.0)
    with torch.cuda.device(x.device):
        st = lib.flce_loss_static(x.data_ptr(), W.data_ptr(), t.data_ptr(), N, H, V, ignore_index,
                                  ctypes.byref(loss), token_loss.data_ptr(), _stream_ptr(x.device))
    if st != FLCE_OK:
        raise FlceError(st, "flce_loss_static")
    return loss.value, token_loss


_handles = {}


def forward_backward(x, W, t, ignore_index: int = -100, chunk: int = 0):
    """Module-level call with a cached handle per (device, dtype)."""
    import torch
    dtype = "bf16" if x.dtype == torch.bfloat16 else "fp32"
    key = (x.device.index or 0, dtype)
    if key not in _handles:
        _handles[key] = FLCE(dtype, key[0])
    return _handles[key].forward_backward(x, W, t, ignore_index, chunk)
