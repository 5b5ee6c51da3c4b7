"""Seeded synthetic inputs for fused linear cross-entropy (FLCE).

This module only draws random inputs. It holds none of the method's arithmetic,
and both the fp64 oracle and the CUDA path are fed from it.

Recipe (every config, unless a caller overrides a field):

* Generator: numpy PCG64. Each tensor gets its own seed sequence
  ``SeedSequence(entropy=seed, spawn_key=(tensor_id, block))`` with tensor ids
  x=0, W=1, targets=2, ignored positions=3. Large tensors are drawn in blocks
  of 2**24 elements in row-major order, one stream per block, so threads can
  fill blocks in parallel and the result does not depend on the thread count.
* x ~ N(0, 1) drawn in float32; W = float32(w_std) * N(0, 1) in float32,
  w_std = 0.02.
* bf16 configs round x and W once, on the host, to bfloat16 with
  round-to-nearest-even. Both sides then see the same rounded values: the
  CUDA path as bf16 bits, the oracle upcast exactly to float64.
* Targets: "uniform" draws integers in [0, V). "zipf" draws rank k in 1..V
  with P(k) proportional to k**-s (s = 1.1) by inverse CDF on a uniform
  draw; the token id is k - 1.
* Ignored tokens: exactly floor(p * N) positions, the first floor(p * N)
  entries of a seeded permutation of range(N), get ignore_index (-100).

The named configs are the workloads the FLCE pages reason about: a tiny fp32
case, a Llama-2-sized vocabulary, the Llama-3-shaped 4x4096-token batch whose
logits the Unsloth page sizes at 2,101,346,304 elements, the Qwen3-shaped
batch the FLCE page sizes at 4.97 GB of bf16 logits, and a 131,072-token
long-context batch.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from fractions import Fraction
from typing import Optional

import numpy as np

IGNORE_INDEX = -100
BLOCK = 1 << 24

_TENSOR_X, _TENSOR_W, _TENSOR_T, _TENSOR_IGN = 0, 1, 2, 3


@dataclasses.dataclass(frozen=True)
class ConfigSpec:
    name: str
    N: int
    H: int
    V: int
    dtype: str                 # "bf16" or "fp32": dtype of x, W and dx
    targets: str               # "uniform" or "zipf"
    ignore_frac: Fraction      # exact fraction of ignored tokens
    chunk: int = 0             # tokens per chunk; 0 lets the planner choose
    zipf_s: float = 1.1
    w_std: float = 0.02
    seed: int = 0


CONFIGS = {
    "tiny_fp32": ConfigSpec("tiny_fp32", 256, 128, 4096, "fp32", "uniform",
                            Fraction(0), chunk=64),
    "small_bf16": ConfigSpec("small_bf16", 2048, 1024, 32000, "bf16", "uniform",
                             Fraction(1, 10)),
    "llama3_bf16": ConfigSpec("llama3_bf16", 16384, 4096, 128256, "bf16", "zipf",
                              Fraction(1, 20)),
    "qwen3_bf16": ConfigSpec("qwen3_bf16", 16384, 4096, 151936, "bf16", "zipf",
                             Fraction(1, 20)),
    "long_bf16": ConfigSpec("long_bf16", 131072, 4096, 128256, "bf16", "uniform",
                            Fraction(0)),
    # one 4096-token chunk of the Llama-3-shaped batch against a 32768-entry
    # slice of the vocabulary: the same kernels at a size a profiler replays
    # quickly (W is 268 MB, above the 129 MB L2)
    "one_chunk_bf16": ConfigSpec("one_chunk_bf16", 4096, 4096, 32768, "bf16", "zipf",
                                 Fraction(1, 20)),
}

# chunk sizes swept on the Qwen3-shaped config
QWEN3_CHUNKS = (1024, 2048, 4096, 8192)


@dataclasses.dataclass
class Workload:
    spec: ConfigSpec
    x: np.ndarray   # (N, H): uint16 bf16 bits, or float32
    W: np.ndarray   # (V, H): uint16 bf16 bits, or float32
    t: np.ndarray   # (N,) int64, ignored positions hold IGNORE_INDEX

    @property
    def N(self) -> int:
        return self.spec.N

    @property
    def H(self) -> int:
        return self.spec.H

    @property
    def V(self) -> int:
        return self.spec.V

    @property
    def ignore_index(self) -> int:
        return IGNORE_INDEX

    def x_f64(self, rows: Optional[np.ndarray] = None) -> np.ndarray:
        return to_f64(self.x if rows is None else self.x[rows])

    def W_f64(self, rows: Optional[np.ndarray] = None) -> np.ndarray:
        return to_f64(self.W if rows is None else self.W[rows])


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


class F64Rows:
    """Rows of an input matrix (bf16 bits or float32), widened to float64 when
    indexed, so that a consumer never holds a full-size matrix in float64."""

    def __init__(self, a: np.ndarray):
        self.a = a
        self.shape = a.shape

    def __len__(self) -> int:
        return self.shape[0]

    def __getitem__(self, idx) -> np.ndarray:
        return to_f64(self.a[idx])


def round_f32_to_bf16_bits(f: np.ndarray, out: np.ndarray) -> None:
    """Round float32 values (finite) to bfloat16 bits, nearest-even, into out."""
    b = f.view(np.uint32)
    tmp = b >> np.uint32(16)
    tmp &= np.uint32(1)
    tmp += np.uint32(0x7FFF)
    tmp += b
    tmp >>= np.uint32(16)
    out[...] = tmp


def _stream(seed: int, tensor_id: int, block: int) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(tensor_id, block))
    return np.random.Generator(np.random.PCG64(ss))


def _normal_matrix(rows: int, cols: int, scale: float, seed: int, tensor_id: int,
                   dtype: str, threads: int) -> np.ndarray:
    total = rows * cols
    nblk = (total + BLOCK - 1) // BLOCK
    out = np.empty(total, np.uint16 if dtype == "bf16" else np.float32)

    def fill(b: int) -> None:
        lo, hi = b * BLOCK, min(total, (b + 1) * BLOCK)
        f = _stream(seed, tensor_id, b).standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            f *= np.float32(scale)
        if dtype == "bf16":
            round_f32_to_bf16_bits(f, out[lo:hi])
        else:
            out[lo:hi] = f

    if nblk == 1 or threads <= 1:
        for b in range(nblk):
            fill(b)
    else:
        with ThreadPoolExecutor(min(threads, nblk)) as ex:
            list(ex.map(fill, range(nblk)))
    return out.reshape(rows, cols)


def zipf_inverse_cdf(u: np.ndarray, V: int, s: float) -> np.ndarray:
    """Map uniforms in [0,1) to token ids k-1, P(k) proportional to k**-s."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, V - 1).astype(np.int64)


def make_targets(spec: ConfigSpec) -> np.ndarray:
    N, V = spec.N, spec.V
    g = _stream(spec.seed, _TENSOR_T, 0)
    if spec.targets == "uniform":
        t = g.integers(0, V, size=N, dtype=np.int64)
    elif spec.targets == "zipf":
        t = zipf_inverse_cdf(g.random(N), V, spec.zipf_s)
    else:
        raise ValueError(f"unknown target distribution {spec.targets!r}")
    n_ign = (N * spec.ignore_frac.numerator) // spec.ignore_frac.denominator
    if n_ign:
        perm = _stream(spec.seed, _TENSOR_IGN, 0).permutation(N)
        t[perm[:n_ign]] = IGNORE_INDEX
    return t


def spec(name: str, **overrides) -> ConfigSpec:
    base = CONFIGS[name]
    if "ignore_frac" in overrides:
        overrides["ignore_frac"] = Fraction(overrides["ignore_frac"]).limit_denominator(1 << 20)
    return dataclasses.replace(base, **overrides)


def custom(N: int, H: int, V: int, dtype: str = "bf16", targets: str = "uniform",
           ignore_frac=0, chunk: int = 0, seed: int = 0, name: str = "custom",
           w_std: float = 0.02) -> ConfigSpec:
    return ConfigSpec(name, N, H, V, dtype, targets,
                      Fraction(ignore_frac).limit_denominator(1 << 20),
                      chunk=chunk, seed=seed, w_std=w_std)


def generate(s: ConfigSpec, threads: Optional[int] = None) -> Workload:
    """Draw the workload for a spec (deterministic in the spec alone)."""
    if threads is None:
        threads = max(1, len(os.sched_getaffinity(0)))
    x = _normal_matrix(s.N, s.H, 1.0, s.seed, _TENSOR_X, s.dtype, threads)
    W = _normal_matrix(s.V, s.H, s.w_std, s.seed, _TENSOR_W, s.dtype, threads)
    t = make_targets(s)
    return Workload(s, x, W, t)


def make(name: str, threads: Optional[int] = None, **overrides) -> Workload:
    return generate(spec(name, **overrides), threads=threads)
