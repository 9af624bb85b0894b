"""GB300-native skinny BF16 decode projection: out[M, N] = x[M, K] @ W[N, K]^T.

Python front end of the C-ABI library (``libskinny_gemm.so``).  PyTorch is
used for device memory and streams only; this module passes pointers, sizes
and stream handles to the library, whose CUDA kernels do all of the work.
"""
from __future__ import annotations

import contextlib
import ctypes
from typing import Iterable, Sequence

import torch

from . import _native
from ._native import MAX_M, SkinnyGemmError

__all__ = ["Projection", "run_overlap", "tune_overlap", "SkinnyGemmError", "MAX_M", "library_path"]

_OUT_CODES = {torch.bfloat16: _native.SKG_BF16, torch.float16: _native.SKG_FP16,
              torch.float32: _native.SKG_FP32}
_IN_CODES = {torch.bfloat16: _native.SKG_BF16, torch.float16: _native.SKG_FP16}


def library_path() -> str:
    return _native.library_path()


_SAME_DEVICE = contextlib.nullcontext()


def _device_scope(index: int):
    """Make device `index` current for a call (a no-op when it already is)."""
    return _SAME_DEVICE if torch.cuda.current_device() == index else torch.cuda.device(index)


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _matrix(t: torch.Tensor, name: str) -> tuple[int, int]:
    """(data_ptr, row pitch in elements) of a 2-D tensor with unit inner stride."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got {tuple(t.shape)}")
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError(f"{name} needs a unit inner stride")
    return t.data_ptr(), (t.stride(0) if t.shape[0] > 1 else t.shape[1])


class Projection:
    """A prepared projection ``out = x @ weight.T`` for 1..256 tokens (decode: 1..64).

    ``weight`` [N, K] (bf16 or fp16, CUDA, unit inner stride) is borrowed: this
    object keeps a reference so it stays alive, and it must not be moved or
    resized.  ``out_dtype`` is torch.float32 or the weight's own dtype (default).
    ``deterministic=True`` keeps the autotuner to tactics with a fixed fp32
    summation order (SKG_PREPARE_DETERMINISTIC).
    """

    def __init__(self, weight: torch.Tensor, out_dtype: torch.dtype | None = None, *,
                 use_tactic_file: bool = True, pdl: bool = True, deterministic: bool = False):
        if out_dtype is None:
            out_dtype = weight.dtype
        if not weight.is_cuda:
            raise ValueError("weight must be a CUDA tensor")
        if weight.dtype not in _IN_CODES:
            raise ValueError(f"weight dtype {weight.dtype} unsupported")
        if out_dtype not in _OUT_CODES:
            raise ValueError(f"unsupported projection output dtype {out_dtype}")
        ptr, ldw = _matrix(weight, "weight")
        self._lib = _native.lib()
        with torch.cuda.device(weight.device):
            h = self._lib.skinny_gemm_prepare_ex(
                ptr, weight.shape[0], weight.shape[1], ldw, _IN_CODES[weight.dtype],
                _OUT_CODES[out_dtype],
                (0 if use_tactic_file else 1) | (0 if pdl else 2) | (4 if deterministic else 0))
        if not h:
            raise SkinnyGemmError(self._lib.skinny_gemm_last_status(), _native.last_error())
        self._h = ctypes.c_void_p(h)
        self.weight = weight
        self.N, self.K = weight.shape
        self.out_dtype = out_dtype
        self.device = weight.device
        self._dev_index = weight.device.index if weight.device.index is not None else \
            torch.cuda.current_device()

    # ---------------------------------------------------------------- running
    def run(self, x: torch.Tensor, out: torch.Tensor, stream=None,
            residual: torch.Tensor | None = None) -> torch.Tensor:
        """Write x @ W^T (+ residual) into the caller's ``out`` (no allocation);
        returns out.  ``residual`` has out's shape and dtype and may be out itself."""
        xp, ldx = _matrix(x, "x")
        op, ldo = _matrix(out, "out")
        if x.shape[1] != self.K or out.shape[1] != self.N or out.shape[0] != x.shape[0]:
            raise ValueError(f"shapes x{tuple(x.shape)} out{tuple(out.shape)} for W[{self.N}, {self.K}]")
        if x.dtype != self.weight.dtype or out.dtype != self.out_dtype:
            raise ValueError(f"dtypes x {x.dtype} / out {out.dtype}")
        if residual is None:
            _native.check(self._lib.skinny_gemm_run_strided(
                self._h, xp, ldx, x.shape[0], op, ldo, _stream_ptr(stream)))
            return out
        if residual.shape != out.shape or residual.dtype != out.dtype:
            raise ValueError(f"residual {tuple(residual.shape)} {residual.dtype} vs out")
        rp, ldr = _matrix(residual, "residual")
        _native.check(self._lib.skinny_gemm_run_residual(
            self._h, xp, ldx, x.shape[0], rp, ldr, op, ldo, _stream_ptr(stream)))
        return out

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((x.shape[0], self.N), dtype=self.out_dtype, device=x.device)
        return self.run(x, out, stream)

    def _check_host(self, x_host: torch.Tensor, out_host: torch.Tensor) -> None:
        if x_host.is_cuda or out_host.is_cuda:
            raise ValueError("run_host takes host tensors")
        if not (x_host.is_contiguous() and out_host.is_contiguous()):
            raise ValueError("run_host needs packed host buffers")
        if x_host.dim() != 2 or x_host.shape[1] != self.K or x_host.dtype != self.weight.dtype:
            raise ValueError(f"x_host must be [M, {self.K}] {self.weight.dtype}")
        if tuple(out_host.shape) != (x_host.shape[0], self.N) or out_host.dtype != self.out_dtype:
            raise ValueError(f"out_host must be [M, {self.N}] {self.out_dtype}")

    def run_host(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> torch.Tensor:
        """End-to-end call with host (ideally pinned) buffers; synchronizes the stream."""
        self._check_host(x_host, out_host)
        with _device_scope(self._dev_index):
            _native.check(self._lib.skinny_gemm_run_host(
                self._h, x_host.data_ptr(), x_host.shape[0], out_host.data_ptr(),
                _stream_ptr(stream)))
        return out_host

    def run_host_async(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> None:
        """Enqueue copy-in, projection and copy-out on the stream without waiting
        (pinned host buffers; synchronize the stream before reading out_host)."""
        self._check_host(x_host, out_host)
        with _device_scope(self._dev_index):
            _native.check(self._lib.skinny_gemm_run_host_async(
                self._h, x_host.data_ptr(), x_host.shape[0], out_host.data_ptr(),
                _stream_ptr(stream)))

    # ---------------------------------------------------------------- plan
    def autotune(self, Ms: Iterable[int], stream=None) -> None:
        ms = list(Ms)
        arr = (ctypes.c_int64 * len(ms))(*ms)
        with torch.cuda.device(self.device):
            _native.check(self._lib.skinny_gemm_autotune(self._h, arr, len(arr), _stream_ptr(stream)))

    def plan(self, M: int) -> str:
        buf = ctypes.create_string_buffer(128)
        _native.check(self._lib.skinny_gemm_plan_query(self._h, M, buf, 128))
        return buf.value.decode()

    def tactics(self, M: int) -> list[str]:
        buf = ctypes.create_string_buffer(1 << 16)
        n = self._lib.skinny_gemm_list_tactics(self._h, M, buf, 1 << 16)
        if n < 0:
            raise SkinnyGemmError(-n, _native.last_error())
        s = buf.value.decode()
        return s.split(";") if s else []

    def set_tactic(self, M: int, tactic: str) -> None:
        _native.check(self._lib.skinny_gemm_set_tactic(self._h, M, tactic.encode()))

    # ---------------------------------------------------------------- watchdog
    def check_status(self, stream=None) -> None:
        with torch.cuda.device(self.device):
            _native.check(self._lib.skinny_gemm_check_status(self._h, _stream_ptr(stream)))

    def inject_timeout(self, count: int, timeout_ns: int) -> None:
        _native.check(self._lib.skinny_gemm_debug_inject_timeout(self._h, count, timeout_ns))

    def inject_check(self, count: int) -> None:
        """Checked build only: the next `count` launches report one failed device check."""
        _native.check(self._lib.skinny_gemm_debug_inject_check(self._h, count))

    # ---------------------------------------------------------------- lifetime
    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.skinny_gemm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def run_overlap(main: Projection, fa: Projection, fb: Projection, x: torch.Tensor,
                out_main: torch.Tensor, fa_out: torch.Tensor, out_fb: torch.Tensor, *,
                chain: int = 1, aux_stream: torch.cuda.Stream,
                events: Sequence[torch.cuda.Event], stream=None) -> None:
    """Two-stream decode step: main GEMM on ``stream`` while the F_A -> F_B chain
    runs on ``aux_stream``, forked and joined with ``events`` (start, done).

    out_fb holds ``chain`` consecutive [M, N_fb] blocks, e.g. shape [chain, M, N_fb].
    """
    M = x.shape[0]
    if out_fb.numel() < chain * M * fb.N:
        raise ValueError("out_fb too small for the chain")
    for e in events:
        if e.cuda_event == 0:  # lazily created events: force creation on this device
            e.record(aux_stream)
    lib = _native.lib()
    _native.check(lib.skinny_gemm_run_overlap(
        main._h, fa._h, fb._h, chain, x.data_ptr(), M, out_main.data_ptr(), fa_out.data_ptr(),
        out_fb.data_ptr(), _stream_ptr(stream), _stream_ptr(aux_stream),
        ctypes.c_void_p(int(events[0].cuda_event)), ctypes.c_void_p(int(events[1].cuda_event))))


def tune_overlap(main: Projection, fa: Projection, fb: Projection, Ms: Iterable[int], *,
                 chain: int = 1, stream=None) -> None:
    """Pick fa's and main's tactics for each M by timing the whole two-stream
    step (see skinny_gemm_autotune_overlap); fb keeps its plan."""
    ms = list(Ms)
    arr = (ctypes.c_int64 * len(ms))(*ms)
    with torch.cuda.device(main.device):
        _native.check(_native.lib().skinny_gemm_autotune_overlap(
            main._h, fa._h, fb._h, chain, arr, len(ms), _stream_ptr(stream)))
