"""Seeded synthetic inputs for the skinny BF16 decode projection.

Shared by the tests (oracle and CUDA path alike) and by ``bench.py``.  This
module only draws numbers; it holds none of the projection's arithmetic.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws W first, ``randn(N, K) * w_std`` rounded to bf16 (std 1/sqrt(K)
unless stated), then ``x_full = randn(64, K)`` rounded to bf16; a call with M
tokens uses ``x_full[:M]``, so one draw serves every M of a sweep.
"""
from __future__ import annotations

import math

import torch

MAX_TOKENS = 64


def weight(N: int, K: int, seed: int = 0, std: float | None = None) -> torch.Tensor:
    """W[N, K] bf16 ~ N(0, std^2), std = 1/sqrt(K) by default (CPU tensor)."""
    g = torch.Generator().manual_seed(seed)
    std = 1.0 / math.sqrt(K) if std is None else std
    return (torch.randn(N, K, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def case(N: int, K: int, seed: int = 0, std: float | None = None, max_tokens: int = MAX_TOKENS,
         dtype: torch.dtype = torch.bfloat16):
    """(W[N, K], x_full[max_tokens, K]) drawn in that order from one generator,
    rounded to `dtype` (bf16 or fp16)."""
    g = torch.Generator().manual_seed(seed)
    std = 1.0 / math.sqrt(K) if std is None else std
    w = (torch.randn(N, K, generator=g, dtype=torch.float32) * std).to(dtype)
    x = torch.randn(max_tokens, K, generator=g, dtype=torch.float32).to(dtype)
    return w, x


def small_integers(rows: int, cols: int, seed: int, lo: int = -8, hi: int = 8,
                   dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """Integers in [lo, hi] as bf16 or fp16 (exactly representable)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (rows, cols), generator=g).to(dtype)


def one_hot_rows(M: int, K: int, cols) -> torch.Tensor:
    """x[m, cols[m]] = 1, zero elsewhere (bf16)."""
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    for m, j in enumerate(cols):
        x[m, j] = 1.0
    return x


def identity_slice(N: int, K: int) -> torch.Tensor:
    """W[n, k] = 1 if n == k else 0 (bf16)."""
    w = torch.zeros(N, K, dtype=torch.bfloat16)
    d = min(N, K)
    w[torch.arange(d), torch.arange(d)] = 1.0
    return w
