"""fp64 CPU oracle for fused linear cross-entropy. Test infrastructure only:
the tests, ``__graft_entry__.smoke()`` and the CPU baseline of ``bench.py``
use it; the CUDA path never does."""
from .flce_oracle import (IGNORE_INDEX, OracleResult, check_targets, dW_rows, dx_rows,
                          flce_reference, logsumexp_rows, lse_rows, project,
                          softmax_minus_onehot, target_logits, token_loss_rows,
                          token_losses, valid_mask)

__all__ = ["IGNORE_INDEX", "OracleResult", "check_targets", "dW_rows", "dx_rows",
           "flce_reference", "logsumexp_rows", "lse_rows", "project",
           "softmax_minus_onehot", "target_logits", "token_loss_rows", "token_losses",
           "valid_mask"]
