"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no quantization or GEMM arithmetic: it only draws random
matrices (numpy ``default_rng``) and rounds them to the input dtype.  Both the
CUDA path and the CPU oracle receive the identical bytes.

Recipes (shapes follow the workloads of the FP8 training scheme on the pages:
a 7168-wide hidden layer with an 18432-wide projection, MoE experts with
7168 x 4096 up-projections):

* tiny Fprop: A [128 x 512], W [512 x 256], fp32, N(0, 1), one generator seeded 0
  drawing A then W.
* layer Fprop: X [4096 x 7168] N(0, 1) with 0.1 % outliers (exactly
  round(0.001 * numel) positions, chosen without replacement, multiplied by
  100) then rounded to bf16, seed 0; W [7168 x 18432] N(0, 0.02) bf16, seed 1.
* backward of that layer: dY [4096 x 18432] N(0, 1e-3) bf16, seed 2 (the
  second parameter is read as a standard deviation, as for the weights).
* grouped MoE up-projection: 32 experts; 16384 routed rows, expert of each
  row drawn from a truncated Zipf law p_e ~ (e + 1)^-1.1, seed 3; every count
  padded up to a multiple of 128 with zero rows; activations N(0, 1) with
  0.1 % x100 outliers, bf16; W_e [7168 x 4096] N(0, 0.02) bf16.
* quantizer sweep: bf16 X [M x 7168] for M in {1024, 8192, 65536} with 0.1 %
  x100 outliers, seed 4; the layer's W for the 128x128 quantizer.
"""
from __future__ import annotations

import numpy as np
import torch

HIDDEN = 7168
FFN = 18432
TOKENS = 4096
EXPERTS = 32
EXPERT_N = 4096
ROUTED_ROWS = 16384
ZIPF_S = 1.1
OUTLIER_FRACTION = 0.001
OUTLIER_FACTOR = 100.0


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Round fp32 to bf16 (round-to-nearest-even, torch's CPU cast)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a bf16 tensor (the oracle's bf16 input)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def normal_with_outliers(rng: np.random.Generator, shape, std: float = 1.0,
                         fraction: float = OUTLIER_FRACTION,
                         factor: float = OUTLIER_FACTOR) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    n = x.size
    k = int(round(fraction * n))
    if k:
        pos = rng.choice(n, size=k, replace=False)
        x.reshape(-1)[pos] *= np.float32(factor)
    return x


def tiny_fprop():
    """(A fp32 [128 x 512], W fp32 [512 x 256])."""
    rng = np.random.default_rng(0)
    a = rng.standard_normal((128, 512), dtype=np.float32)
    w = rng.standard_normal((512, 256), dtype=np.float32)
    return a, w


def layer_activations(tokens: int = TOKENS, hidden: int = HIDDEN, seed: int = 0) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return to_bf16(normal_with_outliers(rng, (tokens, hidden)))


def layer_weight(k_in: int = HIDDEN, n_out: int = FFN, seed: int = 1) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return to_bf16(rng.standard_normal((k_in, n_out), dtype=np.float32) * np.float32(0.02))


def layer_grad_output(tokens: int = TOKENS, n_out: int = FFN, seed: int = 2) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return to_bf16(rng.standard_normal((tokens, n_out), dtype=np.float32) * np.float32(1e-3))


def zipf_expert_ids(experts: int = EXPERTS, rows: int = ROUTED_ROWS, s: float = ZIPF_S,
                    seed: int = 3) -> np.ndarray:
    """Expert of each routed token: a categorical over ranks 1..experts with
    p ~ rank^-s, seeded."""
    rng = np.random.default_rng(seed)
    p = (np.arange(1, experts + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    return rng.choice(experts, size=rows, p=p).astype(np.int64)


def zipf_counts(experts: int = EXPERTS, rows: int = ROUTED_ROWS, s: float = ZIPF_S,
                seed: int = 3) -> np.ndarray:
    choice = zipf_expert_ids(experts, rows, s, seed)
    return np.bincount(choice, minlength=experts).astype(np.int64)


def padded_offsets(counts: np.ndarray, multiple: int = 128) -> np.ndarray:
    padded = (counts + multiple - 1) // multiple * multiple
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


def grouped_moe(experts: int = EXPERTS, hidden: int = HIDDEN, n_out: int = EXPERT_N,
                rows: int = ROUTED_ROWS, seed: int = 3):
    """(counts, offsets, X bf16 [offsets[-1] x hidden] with zero padding rows,
    W bf16 [experts x hidden x n_out])."""
    counts = zipf_counts(experts, rows, seed=seed)
    offsets = padded_offsets(counts)
    rng = np.random.default_rng(seed + 100)
    x = np.zeros((int(offsets[-1]), hidden), np.float32)
    for e in range(experts):
        r0 = int(offsets[e])
        x[r0:r0 + int(counts[e])] = normal_with_outliers(rng, (int(counts[e]), hidden))
    w = rng.standard_normal((experts, hidden, n_out), dtype=np.float32) * np.float32(0.02)
    return counts, offsets, to_bf16(x), to_bf16(w)


def sweep_activations(m: int, hidden: int = HIDDEN, seed: int = 4) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return to_bf16(normal_with_outliers(rng, (m, hidden)))


def random_matrix(shape, seed: int, dtype=torch.bfloat16, std: float = 1.0,
                  outliers: bool = True) -> torch.Tensor:
    """General seeded test matrix (parity cases at small and ragged sizes)."""
    rng = np.random.default_rng(seed)
    x = normal_with_outliers(rng, shape, std=std) if outliers else \
        rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
    t = torch.from_numpy(x)
    return t.to(dtype) if dtype != torch.float32 else t
