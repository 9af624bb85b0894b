"""The no-allocation entry point, skinny_gemm_run_noalloc, against the prepared one.

skinny_gemm_run_noalloc exists for callers that cannot allocate device memory
(a stream captured in global mode, an engine whose pool owns all of HBM, code
that must avoid cudaMalloc/cudaFree's implicit synchronization): it needs no
handle and keeps its only scratch, the watchdog status word, in a static
device array inside the library.  This test calls it through the C ABI twice
in a row per case (the array keeps the previous call's contents) and checks
each result against the CPU oracle with the bound the other tests use,
|y - ref| <= 8e-3 |ref| + 2e-3 s, and, since both entry points run the same
default tactic, bit for bit against the prepared entry point's output.

This file is collected last, so a run that stops at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def skg():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import skinny_bf16_projection_gb300 as m
    return m


@pytest.mark.parametrize("N,K,odt", [(1536, 128, torch.bfloat16), (3584, 7168, torch.bfloat16),
                                     (6288, 7168, torch.float32), (656, 1088, torch.bfloat16)])
def test_noalloc_matches_prepared_entry_point(skg, N, K, odt):
    lib = skg._native.lib()
    code = skg._native.SKG_FP32 if odt == torch.float32 else skg._native.SKG_BF16
    w, x = pin.case(N, K, seed=0)
    ref, s = oracle.projection(x, w)
    wd, xd = w.to(DEV), x.to(DEV)
    proj = skg.Projection(wd, odt, use_tactic_file=False)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for M in (1, 8, 33, 64):
        want = torch.empty((M, N), dtype=odt, device=DEV)
        proj.run(xd[:M], want)
        for call in range(2):
            got = torch.full((M, N), float("nan"), dtype=odt, device=DEV)
            rc = lib.skinny_gemm_run_noalloc(wd.data_ptr(), N, K, K, code, xd.data_ptr(), K, M,
                                             got.data_ptr(), N, stream)
            assert rc == 0, skg._native.last_error()
            torch.cuda.synchronize()
            y = got.float().cpu().double().numpy()
            ok = oracle.tolerance_ok(y, ref[:M], s[:M])
            assert ok.all(), (f"N={N} K={K} M={M} call {call}: {int((~ok).sum())} outputs outside "
                              f"|y - ref| <= 8e-3 |ref| + 2e-3 s of the oracle")
            assert torch.equal(got, want), (f"N={N} K={K} M={M} call {call}: differs from the "
                                            f"prepared entry point's default tactic {proj.plan(M)}")
    proj.close()


def test_noalloc_rejects_bad_requests(skg):
    lib = skg._native.lib()
    nat = skg._native
    w = torch.zeros((256, 1024), dtype=torch.bfloat16, device=DEV)
    x = torch.zeros((64, 1024), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros((64, 256), dtype=torch.bfloat16, device=DEV)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = lambda M, xp=x.data_ptr(), wp=w.data_ptr(): (wp, 256, 1024, 1024, nat.SKG_BF16, xp,
                                                       1024, M, out.data_ptr(), 256, st)
    assert lib.skinny_gemm_run_noalloc(*args(nat.MAX_M + 1)) == nat.SKG_EUNSUPPORTED_M
    assert lib.skinny_gemm_run_noalloc(*args(0)) == nat.SKG_EUNSUPPORTED_M
    assert lib.skinny_gemm_run_noalloc(*args(4, xp=x.data_ptr() + 2)) == nat.SKG_EALIGN
    assert lib.skinny_gemm_run_noalloc(*args(4, wp=w.data_ptr() + 2)) == nat.SKG_EALIGN
    assert lib.skinny_gemm_run_noalloc(w.data_ptr(), 256, 1024, 1024, 7, x.data_ptr(), 1024, 4,
                                       out.data_ptr(), 256, st) == nat.SKG_EINVAL
    assert lib.skinny_gemm_run_noalloc(*args(4)) == nat.SKG_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[:4]) == 0 and np.isfinite(out.float().cpu().numpy()).all()
