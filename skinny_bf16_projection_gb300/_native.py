"""ctypes binding of ``libskinny_gemm.so`` (the C ABI in include/skinny_gemm.h).

Argument marshalling only: every step of the projection runs in the library's
CUDA kernels.  Importing this module loads the library and fails loudly if it
has not been built; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libskinny_gemm.so")

# enum skinny_gemm_dtype / skinny_gemm_status (mirrors include/skinny_gemm.h)
SKG_BF16, SKG_FP16, SKG_FP32 = 0, 1, 2
SKG_OK, SKG_EINVAL, SKG_EALIGN, SKG_EUNSUPPORTED_M = 0, 1, 2, 3
SKG_EDEVICE, SKG_ECUDA, SKG_ECAPTURING, SKG_ETIMEOUT, SKG_ECHECK = 4, 5, 6, 7, 8
STATUS_NAMES = {0: "OK", 1: "EINVAL", 2: "EALIGN", 3: "EUNSUPPORTED_M", 4: "EDEVICE",
                5: "ECUDA", 6: "ECAPTURING", 7: "ETIMEOUT", 8: "ECHECK"}
MAX_M = 256

# (name, restype, argtypes) for every function the header declares.
_i64, _int, _vp, _cp, _u64, _sz = (ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_char_p, ctypes.c_uint64, ctypes.c_size_t)
SIGNATURES = [
    ("skinny_gemm_prepare", _vp, [_vp, _i64, _i64, _int, _int]),
    ("skinny_gemm_prepare_ex", _vp, [_vp, _i64, _i64, _i64, _int, _int, ctypes.c_uint]),
    ("skinny_gemm_run", _int, [_vp, _vp, _i64, _vp, _vp]),
    ("skinny_gemm_run_strided", _int, [_vp, _vp, _i64, _i64, _vp, _i64, _vp]),
    ("skinny_gemm_run_residual", _int, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp]),
    ("skinny_gemm_run_host", _int, [_vp, _vp, _i64, _vp, _vp]),
    ("skinny_gemm_run_host_async", _int, [_vp, _vp, _i64, _vp, _vp]),
    ("skinny_gemm_run_overlap", _int, [_vp, _vp, _vp, _int, _vp, _i64, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _vp]),
    ("skinny_gemm_autotune", _int, [_vp, ctypes.POINTER(_i64), _int, _vp]),
    ("skinny_gemm_autotune_overlap", _int, [_vp, _vp, _vp, _int, ctypes.POINTER(_i64), _int, _vp]),
    ("skinny_gemm_set_tactic", _int, [_vp, _i64, _cp]),
    ("skinny_gemm_tactic_normalize", _int, [_cp, _cp, _sz]),
    ("skinny_gemm_plan_query", _int, [_vp, _i64, _cp, _sz]),
    ("skinny_gemm_list_tactics", _int, [_vp, _i64, _cp, _sz]),
    ("skinny_gemm_check_status", _int, [_vp, _vp]),
    ("skinny_gemm_debug_inject_timeout", _int, [_vp, _int, _u64]),
    ("skinny_gemm_debug_inject_check", _int, [_vp, _int]),
    ("skinny_gemm_run_noalloc", _int, [_vp, _i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64,
                                       _vp]),
    ("skinny_gemm_destroy", None, [_vp]),
    ("skinny_gemm_last_error", _cp, []),
    ("skinny_gemm_last_status", _int, []),
    ("skinny_gemm_abi_version", _int, []),
]


class SkinnyGemmError(RuntimeError):
    """A C-ABI call returned an error code."""

    def __init__(self, code: int, message: str):
        super().__init__(f"[{STATUS_NAMES.get(code, code)}] {message}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def last_error() -> str:
    return lib().skinny_gemm_last_error().decode()


def check(code: int) -> None:
    if code != SKG_OK:
        raise SkinnyGemmError(code, last_error())
