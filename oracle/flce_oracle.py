"""Plain fp64 CPU oracle for fused linear cross-entropy (FLCE).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run this module. The product path
never does, and this module imports nothing from the CUDA package.

What it computes, and where the pages define it. The pages are cited by
title and section:

* [FLCE] "Fused Linear Cross-Entropy: LLM 학습 logits 메모리 병목 없애기"
  (42jerrykim.github.io), section "FLCE의 핵심 아이디어: logits을 오래 들고
  있지 않는다": the four per-chunk steps (projection; CE forward with the
  gradient softmax - one_hot written over the logits buffer; dx = dlogits·W;
  dw += dlogits_chunkᵀ·x_chunk). Its PyTorch listing sums per-chunk losses
  and gradients and divides by the token count at the end.
* [CE-memory] "메모리 아끼면서 Cross Entropy Loss 계산하기 — 128K Context LLM
  학습 실전 가이드" (sigco.tistory.com), section "왜 Cross Entropy가 이렇게
  무거운가": logits = lm_head(hidden), then log_softmax and NLL.
* [Unsloth] "Unsloth 심층 아키텍처: 커스텀 Triton 커널과 수동 역전파(Manual
  Backprop)로 완성한 80% VRAM 절감과 5배 파인튜닝 가속" (techknowgenie.com),
  section "스트리밍 청크 기반 Fast CrossEntropy 손실 커널": per-token loss
  L = -z_y + log sum_j exp(z_j) and gradient dL/dz_i = softmax(z)_i - 1(i=y).
  The printed equations lost their LaTeX backslashes ("rac" is \\frac,
  "ight" is \\right, "ext" is \\text); this is the reading taken.

Readings where the pages are silent (each is listed with its reason in the
design notes of this repository):

* Mean over the non-ignored tokens. The [FLCE] listing divides by all tokens
  because it has no ignored ones; with ignored targets the mean runs over the
  n_valid = #{i : t_i != ignore_index} others, as in PyTorch's
  cross_entropy(reduction="mean") that the listing calls per chunk.
* n_valid = 0 (every token ignored): loss = 0, dx = 0, dW = 0.
* A target outside [0, V) that is not ignore_index is an error (ValueError).
* Inputs are taken exactly as given (the bf16-rounded values, upcast to fp64,
  for bf16 workloads).

Every function is a direct restatement of the definition in float64 numpy,
with the library matmul as its only building block.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

IGNORE_INDEX = -100


@dataclasses.dataclass
class OracleResult:
    loss: float                 # mean cross-entropy over non-ignored tokens
    dx: np.ndarray              # (N, H) d loss / d x
    dW: np.ndarray              # (V, H) d loss / d W
    token_loss: np.ndarray      # (N,) per-token loss, 0 for ignored tokens
    lse: np.ndarray             # (N,) log-sum-exp of each token's logits
    n_valid: int
    dlogits: Optional[np.ndarray] = None   # (N, V) when requested


# ---------------------------------------------------------------- the steps

def _values(a) -> np.ndarray:
    """Inputs as float64 values; integer arrays (such as raw bf16 bit
    patterns) are refused rather than read as numbers."""
    a = np.asarray(a)
    if a.dtype.kind in "iub":
        raise TypeError("the oracle takes real-valued inputs; widen bf16 bit patterns first")
    return a.astype(np.float64, copy=False)


def check_targets(t: np.ndarray, V: int, ignore_index: int) -> None:
    t = np.asarray(t)
    bad = (t != ignore_index) & ((t < 0) | (t >= V))
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise ValueError(f"target {int(t[i])} at token {i} is outside [0, {V}) "
                         f"and is not ignore_index={ignore_index}")


def valid_mask(t: np.ndarray, ignore_index: int) -> np.ndarray:
    """Tokens that take part in the mean (target != ignore_index)."""
    return np.asarray(t) != ignore_index


def project(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Step 1 of [FLCE] / [CE-memory]: logits z = x · Wᵀ, shape (rows, V)."""
    return x @ W.T


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """log sum_j exp(z_ij) per row, with the row max taken out first so that
    large logits do not overflow ([Unsloth]: the running max m and
    l = sum exp(z - m))."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def target_logits(z: np.ndarray, t: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """z_{i, t_i} for valid rows, 0 for ignored rows."""
    out = np.zeros(z.shape[0])
    rows = np.flatnonzero(valid)
    out[rows] = z[rows, t[rows]]
    return out


def token_losses(lse: np.ndarray, z_t: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """[Unsloth]: L_i = -z_{i,t_i} + log sum_j exp(z_ij); ignored rows give 0."""
    return np.where(valid, lse - z_t, 0.0)


def softmax_minus_onehot(z: np.ndarray, lse: np.ndarray, t: np.ndarray,
                         valid: np.ndarray) -> np.ndarray:
    """[Unsloth] / [FLCE] step 2: dL_i/dz_ij = softmax(z_i)_j - 1(j = t_i) for
    valid rows; ignored rows contribute nothing and get 0."""
    g = np.exp(z - lse[:, None])
    rows = np.flatnonzero(valid)
    g[rows, t[rows]] -= 1.0
    g[~valid] = 0.0
    return g


# ------------------------------------------------------------- whole method

def flce_reference(x: np.ndarray, W: np.ndarray, t: np.ndarray,
                   ignore_index: int = IGNORE_INDEX, chunk: Optional[int] = None,
                   return_dlogits: bool = False) -> OracleResult:
    """Mean cross-entropy of x·Wᵀ against t, with dx and dW, in float64.

    chunk=None evaluates the definition on the whole batch: logits, log-sum-
    exp, per-token loss, dlogits = (softmax - onehot)/n_valid, dx = dlogits·W,
    dW = dlogitsᵀ·x.

    chunk=C follows the [FLCE] control flow instead: for each block of C
    tokens, project, take the summed loss and the unscaled gradient
    softmax - onehot, produce that block's dx at once and add its
    dlogitsᵀ·x_chunk into dW; divide loss and gradients by the token count
    (n_valid) at the end. Both orders give the same result up to rounding.
    """
    x = _values(x)
    W = _values(W)
    t = np.asarray(t, dtype=np.int64)
    N, H = x.shape
    V, H2 = W.shape
    if H != H2 or t.shape != (N,):
        raise ValueError("shape mismatch: x (N,H), W (V,H), t (N,)")
    check_targets(t, V, ignore_index)
    valid = valid_mask(t, ignore_index)
    n_valid = int(valid.sum())

    if chunk is None:
        z = project(x, W)
        lse = logsumexp_rows(z)
        tl = token_losses(lse, target_logits(z, t, valid), valid)
        if n_valid == 0:
            d = np.zeros_like(z)
            loss = 0.0
        else:
            d = softmax_minus_onehot(z, lse, t, valid) / n_valid
            loss = float(tl.sum()) / n_valid
        dx = d @ W
        dW = d.T @ x
        return OracleResult(loss, dx, dW, tl, lse, n_valid,
                            d if return_dlogits else None)

    if chunk < 1:
        raise ValueError("chunk must be >= 1")
    dx = np.zeros((N, H))
    dW = np.zeros((V, H))
    lse = np.zeros(N)
    tl = np.zeros(N)
    d_all = np.zeros((N, V)) if return_dlogits else None
    loss_sum = 0.0
    for s in range(0, N, chunk):
        e = min(N, s + chunk)
        z = project(x[s:e], W)                                   # step 1
        lse[s:e] = logsumexp_rows(z)
        v = valid[s:e]
        tl[s:e] = token_losses(lse[s:e], target_logits(z, t[s:e], v), v)
        loss_sum += float(tl[s:e].sum())
        g = softmax_minus_onehot(z, lse[s:e], t[s:e], v)         # step 2
        dx[s:e] = g @ W                                          # step 3
        dW += g.T @ x[s:e]                                       # step 4
        if d_all is not None:
            d_all[s:e] = g
    if n_valid == 0:
        return OracleResult(0.0, dx * 0.0, dW * 0.0, tl, lse, 0,
                            d_all * 0.0 if d_all is not None else None)
    return OracleResult(loss_sum / n_valid, dx / n_valid, dW / n_valid, tl, lse,
                        n_valid, d_all / n_valid if d_all is not None else None)


# ------------------------------------------ one-by-one outputs at full size
#
# At sizes where the whole N x V logits do not fit a CPU budget, these give
# single outputs straight from the same definition: a token's loss, a row of
# dx, a row of dW. Each is exact given the inputs; nothing is approximated.

def lse_rows(x: np.ndarray, W: np.ndarray, rows: Sequence[int],
             block: int = 256) -> np.ndarray:
    """log-sum-exp of the logits of the given tokens (float64)."""
    rows = np.asarray(rows, dtype=np.int64)
    Wd = _values(W)
    out = np.empty(len(rows))
    for s in range(0, len(rows), block):
        r = rows[s:s + block]
        out[s:s + block] = logsumexp_rows(project(_values(x[r]), Wd))
    return out


def token_loss_rows(x, W, t, rows, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Per-token loss (0 for ignored tokens) of the given tokens."""
    rows = np.asarray(rows, dtype=np.int64)
    t = np.asarray(t, dtype=np.int64)
    Wd = _values(W)
    xr = _values(x[rows])
    z = project(xr, Wd)
    v = valid_mask(t[rows], ignore_index)
    return token_losses(logsumexp_rows(z), target_logits(z, t[rows], v), v)


def dx_rows(x, W, t, rows, n_valid: int, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Rows of dx = dlogits·W for the given tokens; needs only their own logits."""
    rows = np.asarray(rows, dtype=np.int64)
    t = np.asarray(t, dtype=np.int64)
    Wd = _values(W)
    z = project(_values(x[rows]), Wd)
    v = valid_mask(t[rows], ignore_index)
    if n_valid == 0:
        return np.zeros((len(rows), Wd.shape[1]))
    g = softmax_minus_onehot(z, logsumexp_rows(z), t[rows], v) / n_valid
    return g @ Wd


def dW_rows(x, W, t, vocab_rows, lse_all: np.ndarray, n_valid: int,
            ignore_index: int = IGNORE_INDEX, block: int = 4096) -> np.ndarray:
    """Rows j of dW = dlogitsᵀ·x for the given vocab entries. Each needs
    column j of dlogits for every token, hence the log-sum-exp of every
    token (lse_all, from lse_rows over all tokens)."""
    J = np.asarray(vocab_rows, dtype=np.int64)
    t = np.asarray(t, dtype=np.int64)
    WJ = _values(W[J])
    N = len(t)
    out = np.zeros((len(J), WJ.shape[1]))
    if n_valid == 0:
        return out
    for s in range(0, N, block):
        e = min(N, s + block)
        xb = _values(x[s:e])
        zJ = project(xb, WJ)                                  # (b, |J|)
        g = np.exp(zJ - lse_all[s:e, None])
        tb = t[s:e]
        onehot = tb[:, None] == J[None, :]
        g = g - onehot
        g[tb == ignore_index] = 0.0
        out += g.T @ xb
    return out / n_valid
