"""Seeded synthetic inputs for the fused linear + cross-entropy path.

This module is shared by the fp64 oracle tests, the GPU parity tests and the
benchmark. It holds none of the method's arithmetic: it only draws random
numbers and rounds them to bf16.

Workloads. The shapes are the LM heads the pages use to illustrate the logit
blow-up ("Unsloth Architecture: Manual Triton Backpropagation, Fused
Cross-Entropy, and 80% VRAM Cut", section "The Un-Fused Cross-Entropy Logit
Disaster": vocabulary sizes per model family and the 16,384-token Llama-3
batch). No dataset is involved; the model names only fix N, D and V.

Recipe for workload k (seed k):
  rng = numpy.random.default_rng(k)
  H = rng.standard_normal((N, D), float32)            -> bf16 (round to nearest even)
  W = rng.standard_normal((V, D), float32) * 0.02     -> bf16
  y = uniform ints in [0, V)  or  truncated Zipf(s=1.1) on ids 0..V-1
  exactly round(frac * N) rows, chosen by rng.permutation(N), set to -100.
The draw order is fixed (H, W, labels, ignored rows) so every consumer sees
identical tensors.

Inputs of the final-RMSNorm path (make_norm_inputs, seed k): the pre-norm
hidden state X drawn like H and then scaled per row by exp(0.5 * z_i), z_i
standard normal (rows of different magnitude, as a residual stream has), and
the RMSNorm weight gamma = 1 + 0.1 * standard normal per channel; then W,
labels and ignored rows as above. Draw order: X, row scales, gamma, W, labels,
ignored rows.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    N: int
    D: int
    V: int
    labels: str           # "uniform" | "zipf"
    ignore_frac: float
    chunks: tuple         # chunk sizes this workload is run with

    @property
    def n_ignored(self) -> int:
        return int(round(self.ignore_frac * self.N))

    def flops_fwd_bwd(self) -> float:
        """Algorithmic FLOPs of one fused forward+backward: 6*N*D*V."""
        return 6.0 * self.N * self.D * self.V


WORKLOADS = {
    "tiny": Workload("tiny", 0, 256, 512, 32000, "uniform", 0.0, (1024,)),
    "llama2-7b": Workload("llama2-7b", 1, 4096, 4096, 32000, "uniform", 0.05, (1024,)),
    "mistral-7b": Workload("mistral-7b", 2, 8192, 4096, 32768, "zipf", 0.10, (1024,)),
    "llama3-8b": Workload("llama3-8b", 3, 16384, 4096, 128256, "uniform", 0.05, (1024,)),
    "qwen2.5-7b": Workload("qwen2.5-7b", 4, 16384, 3584, 152064, "zipf", 0.20, (512, 1024, 2048)),
}


def zipf_labels(rng: np.random.Generator, n: int, V: int, s: float = 1.1) -> np.ndarray:
    """Truncated Zipf on ranks 0..V-1 (p(k) proportional to (k+1)^-s), rank k = id k,
    sampled by inverse CDF from uniform draws."""
    w = (np.arange(1, V + 1, dtype=np.float64)) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int64)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """Round an fp32 array to bf16 (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def to_fp16(a: np.ndarray) -> torch.Tensor:
    """Round an fp32 array to fp16 (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float16)


def make_inputs(N: int, D: int, V: int, seed: int, labels: str = "uniform",
                n_ignored: int = 0, w_std: float = 0.02, h_std: float = 1.0, dtype: str = "bf16"):
    """Draw (H [N,D], W [V,D], y int64 [N]) on the CPU; H and W rounded to bf16
    (default) or fp16 from the same fp32 draws."""
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D), dtype=np.float32)
    if h_std != 1.0:
        H *= np.float32(h_std)
    W = rng.standard_normal((V, D), dtype=np.float32) * np.float32(w_std)
    if labels == "uniform":
        y = rng.integers(0, V, size=N, dtype=np.int64)
    elif labels == "zipf":
        y = zipf_labels(rng, N, V)
    else:
        raise ValueError(f"unknown label distribution {labels!r}")
    if n_ignored:
        y[rng.permutation(N)[:n_ignored]] = IGNORE_INDEX
    rnd = to_fp16 if dtype == "fp16" else to_bf16
    return rnd(H), rnd(W), torch.from_numpy(y)


def workload_inputs(w: Workload | str):
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_inputs(w.N, w.D, w.V, w.seed, w.labels, w.n_ignored)


def make_norm_inputs(N: int, D: int, V: int, seed: int, labels: str = "uniform",
                     n_ignored: int = 0, w_std: float = 0.02):
    """Draw (X bf16 [N,D], gamma bf16 [D], W bf16 [V,D], y int64 [N]) on the CPU."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, D), dtype=np.float32)
    X *= np.exp(0.5 * rng.standard_normal((N, 1))).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    W = rng.standard_normal((V, D), dtype=np.float32) * np.float32(w_std)
    if labels == "uniform":
        y = rng.integers(0, V, size=N, dtype=np.int64)
    elif labels == "zipf":
        y = zipf_labels(rng, N, V)
    else:
        raise ValueError(f"unknown label distribution {labels!r}")
    if n_ignored:
        y[rng.permutation(N)[:n_ignored]] = IGNORE_INDEX
    return to_bf16(X), to_bf16(gamma), to_bf16(W), torch.from_numpy(y)


def workload_norm_inputs(w: Workload | str):
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_norm_inputs(w.N, w.D, w.V, w.seed, w.labels, w.n_ignored)
