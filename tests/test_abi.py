"""C-ABI boundary checks that need no GPU: the library builds for sm_103a,
loads, and exports every function include/skinny_gemm.h declares, with the
binding's table covering exactly the same set."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skinny_gemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(skinny_gemm_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    from skinny_bf16_projection_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("skinny_gemm_prepare", "skinny_gemm_run", "skinny_gemm_run_overlap",
                     "skinny_gemm_autotune", "skinny_gemm_plan_query", "skinny_gemm_destroy",
                     "skinny_gemm_check_status", "skinny_gemm_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_checked_library_exports_every_declared_symbol():
    """The checked build (device-side bounds checks) is the same ABI."""
    from skinny_bf16_projection_gb300 import build
    _, checked = build.build_all()
    lib = ctypes.CDLL(checked)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported by the checked build: {missing}"


def test_binding_covers_the_header(lib_path):
    from skinny_bf16_projection_gb300 import _native
    bound = sorted(name for name, _, _ in _native.SIGNATURES)
    assert bound == declared_functions()
    lib = _native.load(lib_path)
    assert lib.skinny_gemm_abi_version() == 1


def test_host_only_calls_without_a_gpu(lib_path):
    from skinny_bf16_projection_gb300 import _native
    lib = _native.load(lib_path)
    # No device work: argument validation answers before touching CUDA.
    assert lib.skinny_gemm_prepare(None, 16, 64, 0, 0) is None
    assert lib.skinny_gemm_last_status() == _native.SKG_EINVAL
    assert b"null weight" in lib.skinny_gemm_last_error()
    assert lib.skinny_gemm_prepare(ctypes.c_void_p(0x1000), 16, 64, 0, 1) is None  # FP16 out
    assert lib.skinny_gemm_last_status() == _native.SKG_EINVAL
    assert lib.skinny_gemm_prepare(ctypes.c_void_p(0x1000), 16, 60, 0, 0) is None  # K % 8
    assert lib.skinny_gemm_last_status() == _native.SKG_EALIGN
    assert lib.skinny_gemm_prepare(ctypes.c_void_p(0x1008), 16, 64, 0, 0) is None  # 8 B aligned
    assert lib.skinny_gemm_last_status() == _native.SKG_EALIGN
    assert lib.skinny_gemm_run(None, None, 1, None, None) == _native.SKG_EINVAL
    assert lib.skinny_gemm_plan_query(None, 1, None, 0) == _native.SKG_EINVAL
    lib.skinny_gemm_destroy(None)  # ignored


def test_kernel_sources_use_blackwell_primitives():
    csrc = os.path.join(ROOT, "skinny_bf16_projection_gb300", "csrc")
    text = "".join(open(os.path.join(csrc, f)).read() for f in os.listdir(csrc)
                   if f.endswith((".cu", ".cuh")))
    for needle in ("tcgen05.mma.cta_group::1.kind::f16", "tcgen05.alloc", "tcgen05.ld",
                   "cp.async.bulk.tensor.2d", "L2::evict_first", "griddepcontrol.wait",
                   "st.async.shared::cluster", "mapa.shared::cluster"):
        assert needle in text, needle


def test_tactic_grammar_without_a_gpu(lib_path):
    """The tactic strings accepted by skinny_gemm_set_tactic, parsed without a
    handle: canonical spellings round-trip, suffixes are order-free, and
    malformed strings are refused."""
    from skinny_bf16_projection_gb300 import _native
    lib = _native.load(lib_path)
    buf = ctypes.create_string_buffer(96)

    def norm(t):
        rc = lib.skinny_gemm_tactic_normalize(t.encode(), buf, 96)
        return buf.value.decode() if rc == _native.SKG_OK else rc

    for t in ("mma:r128:t8:b2:s3:c8", "mma:r64:t16:b1:s2:c16:d3", "tc:r128:t32:b2:s2:c8:d1",
              "tc:r64:t64:b2:s2:c4:d2:a", "tc:r128:t128:b1:s3:c4:a", "sk:r128:t16:b2:s3:p8",
              "sk:r128:t32:b1:s4:g2"):
        assert norm(t) == t
    assert norm("tc:r128:t64:b2:s2:c8:a:d1") == "tc:r128:t64:b2:s2:c8:d1:a"  # order-free
    assert norm("mma:r128:t8:b1:s2:c16:w:d3") == "mma:r128:t8:b1:s2:c16:d3:w"
    assert norm("tc:r128:t32:b2:s2:c8:w") == "tc:r128:t32:b2:s2:c8:w"
    assert norm("tc:r128:t64:b2:s2:c8:a:p1:d2") == "tc:r128:t64:b2:s2:c8:d2:p1:a"
    assert norm("mma:r64:t8:b4:s3:c4:p2") == "mma:r64:t8:b4:s3:c4:p2"
    assert norm("tc:r64:t64:b2:s2:c4:s:a:p2:d1") == "tc:r64:t64:b2:s2:c4:d1:p2:a:s"
    assert norm("tc:r128:t48:b1:s3:c8") == "tc:r128:t48:b1:s3:c8"
    for bad in ("bogus", "tc:r128:t32:b2:s2", "tc:r128:t32:b2:s2:c8:x", "tc:r128:t32:b2:s2:c8:d0",
                "tc:r128:t32:b2:s2:c8:d1:d2", "tc:r128:t32:b2:s2:c8:a:a", "mma:r128:t8:b2:s2:c8:a",
                "sk:r128:t16:b2:s3:p8:d1", "tc:r128:t32:b2:s2:g1", "mma:r128:t8:b2:s2:c8:ab",
                "sk:r128:t16:b2:s3:p8:w", "mma:r128:t8:b2:s2:c8:w:w", "tc:r128:t32:b2:s2:c8:wa",
                "mma:r64:t8:b4:s3:c4:p0", "mma:r64:t8:b4:s3:c4:p1:p2", "sk:r128:t16:b2:s3:g1:p1",
                "mma:r64:t8:b4:s3:c4:p1:w", "mma:r64:t8:b4:s3:c4:s", "tc:r64:t64:b2:s2:c4:s:s"):
        assert norm(bad) == _native.SKG_EINVAL, bad
