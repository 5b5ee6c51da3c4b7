"""Fused linear cross-entropy (FLCE) on one GB300 (sm_103a).

The computation lives in libflce.so (C ABI: include/flce.h); this package is
its binding. ``FLCE`` wraps a handle; ``forward_backward`` returns the mean
cross-entropy of x·Wᵀ over non-ignored tokens with dx and dW, without ever
holding the N x V logits.
"""
from .flce import (FLCE, FlceError, KERNEL_KINDS, forward_backward, header_functions, load,
                   loss_static, plan)

__all__ = ["FLCE", "FlceError", "KERNEL_KINDS", "forward_backward", "header_functions", "load",
           "loss_static", "plan"]
