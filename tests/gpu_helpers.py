"""Shared helpers for the GPU tests: oracle results cached per weight, and the
element-wise acceptance check with a readable failure report."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import projection_inputs as pin

DEV = "cuda:0"


@functools.lru_cache(maxsize=16)
def full_case(N: int, K: int, seed: int = 0):
    """(W, x_full[64], ref[64, N], s[64, N]) for the seeded workload; x_M = x_full[:M],
    so the oracle runs once per weight and serves every M."""
    w, x = pin.case(N, K, seed=seed)
    ref, s = oracle.projection(x, w)
    return w, x, ref, s


def to_f64(y: torch.Tensor) -> np.ndarray:
    return y.detach().float().cpu().double().numpy()


def assert_parity(y: torch.Tensor, ref: np.ndarray, s: np.ndarray, what: str) -> float:
    yv = to_f64(y)
    assert yv.shape == ref.shape, f"{what}: shape {yv.shape} vs {ref.shape}"
    ok = oracle.tolerance_ok(yv, ref, s)
    if not ok.all():
        bad = np.argwhere(~ok)
        m, n = bad[0]
        raise AssertionError(
            f"{what}: {len(bad)} of {ok.size} outputs outside |y-ref| <= 8e-3|ref| + 2e-3 s; "
            f"first at (m={m}, n={n}): y={yv[m, n]!r} ref={ref[m, n]!r} s={s[m, n]!r}; "
            f"rows hit {sorted(set(bad[:, 0].tolist()))[:8]} cols {sorted(set(bad[:, 1].tolist()))[:8]}")
    return oracle.tolerance_excess(yv, ref, s)


def run_proj(proj, x: torch.Tensor, out_dtype) -> torch.Tensor:
    out = torch.empty((x.shape[0], proj.N), dtype=out_dtype, device=x.device)
    proj.run(x, out)
    return out
