"""Seeded synthetic inputs for the W4A16 workloads.

This module only draws random numbers and casts them to the storage types; it
holds none of the quantization or matmul arithmetic.  The same host bytes feed
the CPU oracle and the CUDA library.

Recipe (per workload):
  rng = numpy.random.default_rng(seed)                       # PCG64
  W32 = rng.standard_normal((N, K), dtype=float32) * sigma
  if outliers: idx = rng.choice(N*K, size=round(0.001*N*K), replace=False)
               W32.flat[idx] *= 10                            # before the fp16 cast
  W   = W32.astype(float16)  (or kept fp32)
  A32 = rng.standard_normal((M, K), dtype=float32)           # drawn after W
  A   = bf16 round-to-nearest-even of A32, kept as uint16 bit patterns
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    K: int
    M: int
    sigma: float
    seed: int
    w_dtype: str          # "f16" or "f32"
    outliers: bool
    desc: str


# The five workloads: sizes, distributions and seeds.
WORKLOADS = {
    "tiny": Workload("tiny", 128, 256, 1, 0.02, 0, "f32", False,
                     "tiny correctness case: W fp32 [128,256] N(0,0.02), A bf16 [1,256]"),
    "llama7b_gemv": Workload("llama7b_gemv", 11008, 4096, 1, 0.02, 1, "f16", True,
                             "Llama-7B-shaped decode GEMV: W fp16 [11008,4096], A [1,4096]"),
    "skinny_m8": Workload("skinny_m8", 4096, 4096, 8, 0.02, 2, "f16", True,
                          "batched decode skinny GEMM: W fp16 [4096,4096], A [8,4096]"),
    "prefill_gemm": Workload("prefill_gemm", 14336, 4096, 2048, 0.02, 3, "f16", True,
                             "prefill GEMM: W fp16 [14336,4096], A [2048,4096]"),
    "mlp70b": Workload("mlp70b", 28672, 8192, 1, 0.015, 4, "f16", True,
                       "70B-scale MLP layer: W fp16 [28672,8192] N(0,0.015), A [1,8192]"),
}
WORKLOAD_ORDER = ["tiny", "llama7b_gemv", "skinny_m8", "prefill_gemm", "mlp70b"]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Input generation only (finite inputs): adds 0x7FFF plus the LSB of the kept
    half, then truncates."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def make_weights(N: int, K: int, sigma: float, seed: int, w_dtype: str = "f16",
                 outliers: bool = True, rng: np.random.Generator | None = None):
    """W[N,K] drawn as N(0, sigma^2), 0.1% of entries x10 (if outliers)."""
    if rng is None:
        rng = np.random.default_rng(seed)
    W32 = rng.standard_normal((N, K), dtype=np.float32)
    W32 *= np.float32(sigma)
    if outliers and N * K > 0:
        n_out = int(round(0.001 * N * K))
        if n_out:
            idx = rng.choice(N * K, size=n_out, replace=False)
            flat = W32.reshape(-1)
            flat[idx] *= np.float32(10.0)
    if w_dtype == "f16":
        return W32.astype(np.float16), rng
    if w_dtype == "f32":
        return W32, rng
    raise ValueError(w_dtype)


def make_activations(M: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """A[M,K] ~ N(0,1) as bf16 bit patterns (uint16)."""
    A32 = rng.standard_normal((M, K), dtype=np.float32)
    return f32_to_bf16_bits(A32)


def make_workload(name: str, M: int | None = None, N: int | None = None):
    """(W, A_bf16_bits) for a named workload; N and M may be overridden for
    down-scaled cases (the draw order and distributions are unchanged)."""
    w = WORKLOADS[name]
    n = w.N if N is None else N
    W, rng = make_weights(n, w.K, w.sigma, w.seed, w.w_dtype, w.outliers)
    A = make_activations(w.M if M is None else M, w.K, rng)
    return W, A


def make_random(N: int, K: int, M: int, seed: int, sigma: float = 0.02,
                w_dtype: str = "f16", outliers: bool = True):
    """Same recipe for arbitrary shapes (parity cases, edge tails)."""
    W, rng = make_weights(N, K, sigma, seed, w_dtype, outliers)
    A = make_activations(M, K, rng)
    return W, A
