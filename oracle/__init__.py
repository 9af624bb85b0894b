"""CPU oracle for the skinny BF16 decode projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) may import
this package.  The product library never loads it and shares no code with it.

The arithmetic lives in ``ref.c`` (plain C, fp64; see the header there for the
definition and its sources).  This module builds that file with gcc and binds
it through ctypes; the only arithmetic written here is the acceptance bound,
which is the stated tolerance itself:

    |y - ref| <= 8e-3 * |ref| + 2e-3 * s,   s = sqrt(sum_k (x_k w_k)^2)

where y is the GPU result already rounded to its output dtype and widened to
float64, and ref is the unrounded fp64 sum.  (Reading: "after rounding to the
output dtype" applies to y; the oracle value stays unrounded.)

Every oracle function is pinned by ``tests/test_oracle.py`` against closed
forms, exact rational brute force and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref.c")
_BUILD_DIR = os.path.join(os.path.dirname(_HERE), "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

REL_TOL = 8e-3
ABS_TOL_SCALE = 2e-3

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``ref.c`` into ``_build/liboracle.so`` (OpenMP when available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
            "-std=c11", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No libgomp on this host: the serial loop computes the same values.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p_u16 = ctypes.POINTER(ctypes.c_uint16)
            p_f64 = ctypes.POINTER(ctypes.c_double)
            lib.oracle_projection.argtypes = [p_u16, ctypes.c_int64, p_u16, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                              p_f64, p_f64, ctypes.c_int]
            lib.oracle_projection.restype = None
            lib.oracle_projection_typed.argtypes = lib.oracle_projection.argtypes + [ctypes.c_int]
            lib.oracle_projection_typed.restype = None
            lib.oracle_fp16_to_f64.argtypes = [p_u16, ctypes.c_int64, p_f64]
            lib.oracle_fp16_to_f64.restype = None
            lib.oracle_bf16_to_f64.argtypes = [p_u16, ctypes.c_int64, p_f64]
            lib.oracle_bf16_to_f64.restype = None
            lib.oracle_round_bf16.argtypes = [p_f64, ctypes.c_int64, p_u16]
            lib.oracle_round_bf16.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_bits(a) -> np.ndarray:
    """Accept a numpy uint16 array or a CPU torch bf16/fp16 tensor; return uint16 bits."""
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("oracle inputs are 16-bit patterns (uint16)")
        return a
    import torch  # only for accepting torch CPU tensors as input containers
    if not isinstance(a, torch.Tensor) or a.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("oracle inputs are bf16/fp16 tensors or uint16 bit arrays")
    t = a.detach().cpu()
    return t.view(torch.int16).numpy().view(np.uint16)


def _input_type(x, w, dtype):
    """0 for bf16, 1 for fp16: explicit `dtype`, else the torch tensors' type."""
    if dtype is not None:
        return {"bf16": 0, "fp16": 1}[dtype]
    import torch
    kinds = {a.dtype for a in (x, w) if isinstance(a, torch.Tensor)}
    if len(kinds) > 1:
        raise TypeError("x and w must have the same 16-bit type")
    return 1 if kinds == {torch.float16} else 0


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def projection(x, w, *, with_scale: bool = True, threads: int = 0, dtype: str | None = None):
    """ref[M, N] = x[M, K] @ w[N, K]^T in fp64 (and s[M, N] for the bound).

    x, w: 2-D bf16 or fp16 (torch tensors, or uint16 bit arrays with dtype="bf16"
    or "fp16"; any row pitch with unit inner stride).  Returns (ref, s) as
    float64 arrays (s is None without scale).
    """
    kind = _input_type(x, w, dtype)
    xb, wb = _as_bits(x), _as_bits(w)
    if xb.ndim != 2 or wb.ndim != 2 or xb.shape[1] != wb.shape[1]:
        raise ValueError(f"shapes x{xb.shape} w{wb.shape}: need x[M,K], w[N,K]")
    if xb.strides[1] != 2 or wb.strides[1] != 2:
        xb, wb = np.ascontiguousarray(xb), np.ascontiguousarray(wb)
    M, K = xb.shape
    N = wb.shape[0]
    ref = np.empty((M, N), dtype=np.float64)
    s = np.empty((M, N), dtype=np.float64) if with_scale else None
    lib = _load()
    p_u16 = ctypes.POINTER(ctypes.c_uint16)
    p_f64 = ctypes.POINTER(ctypes.c_double)
    lib.oracle_projection_typed(
        xb.ctypes.data_as(p_u16), xb.strides[0] // 2,
        wb.ctypes.data_as(p_u16), wb.strides[0] // 2,
        M, N, K, ref.ctypes.data_as(p_f64),
        s.ctypes.data_as(p_f64) if s is not None else None, int(threads), kind)
    return ref, s


def projection_residual(x, w, residual, *, threads: int = 0):
    """(x @ w^T + residual, s): the projection with a residual added, in fp64.

    The residual [M, N] (torch bf16 / fp16 / fp32, or float64 array) is widened
    exactly and added to the fp64 sum once (page "vllm.models.kimi_k3.nvidia.
    low_latency_gemm", try_low_latency_gemm(x, weight, residual)).  s is the
    projection's own scale, unchanged by the residual.
    """
    ref, s = projection(x, w, threads=threads)
    if isinstance(residual, np.ndarray):
        r = residual.astype(np.float64)
    else:
        import torch
        r = residual.detach().cpu().to(torch.float64).numpy()  # exact widening
    if r.shape != ref.shape:
        raise ValueError(f"residual {r.shape} vs output {ref.shape}")
    return ref + r, s


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(_as_bits(bits))
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64(b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), b.size,
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def fp16_to_f64(bits) -> np.ndarray:
    """Exact widening of IEEE binary16 bit patterns to float64."""
    b = np.ascontiguousarray(_as_bits(bits))
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_fp16_to_f64(b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), b.size,
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def round_bf16(values) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even); returns uint16 bits."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_bf16(v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), v.size,
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    return out


def tolerance_ok(y, ref, s) -> np.ndarray:
    """Element-wise acceptance: |y - ref| <= 8e-3 |ref| + 2e-3 s."""
    y = np.asarray(y, dtype=np.float64)
    return np.abs(y - ref) <= REL_TOL * np.abs(ref) + ABS_TOL_SCALE * s


def tolerance_excess(y, ref, s) -> float:
    """max over elements of |y - ref| / (8e-3 |ref| + 2e-3 s); <= 1 passes."""
    y = np.asarray(y, dtype=np.float64)
    bound = REL_TOL * np.abs(ref) + ABS_TOL_SCALE * s
    err = np.abs(y - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                     np.where(err > 0, np.inf, 0.0))
    return float(r.max()) if r.size else 0.0


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))
