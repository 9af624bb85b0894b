"""The checked build (libskinny_gemm_checked.so, compiled with
SKG_DEVICE_CHECKS=1): every guarded shared-memory, TMEM, DSMEM and global access
is tested against its bounds before it is made, and a failed test is reported as
SKG_ECHECK by skinny_gemm_check_status.  compute-sanitizer is not available on
this GPU pool, so this build is the memory checker: the tests run the ragged
every-candidate case (mma.sync, tcgen05, stream-K, clusters 1-16), token counts
above one tile, fp32 / fp16 / residual outputs, full-size decode and packed
weights and the two-stream step through it, and require parity with the oracle
and no failed check."""
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, full_case, run_proj

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skg():
    import os
    import __graft_entry__
    __graft_entry__.build()
    import skinny_bf16_projection_gb300 as m
    from skinny_bf16_projection_gb300 import _native, build
    torch.cuda.set_device(0)
    _, path = build.build_all()
    saved = _native._lib
    saved_timeout = os.environ.get("SKINNY_GEMM_TIMEOUT_NS")
    # a skipped access leaves a barrier short of its bytes: its bounded wait then
    # expires after 0.2 s instead of the default 2 s
    os.environ["SKINNY_GEMM_TIMEOUT_NS"] = "200000000"
    _native._lib = _native.load(path)  # every handle made below runs the checked kernels
    try:
        yield m
    finally:
        _native._lib = saved
        if saved_timeout is None:
            os.environ.pop("SKINNY_GEMM_TIMEOUT_NS", None)
        else:
            os.environ["SKINNY_GEMM_TIMEOUT_NS"] = saved_timeout


def test_checked_library_is_the_one_in_use(skg):
    from skinny_bf16_projection_gb300 import _native
    assert _native.lib()._name.endswith("libskinny_gemm_checked.so"), _native.lib()._name


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_every_candidate_tactic_checked(skg, out_dtype):
    N, K = 656, 1088  # ragged row tiles and K blocks, as in the parity suite
    w, x, ref, s = full_case(N, K, seed=3)
    proj = skg.Projection(w.to(DEV), out_dtype, use_tactic_file=False)
    xd = x.to(DEV)
    n = 0
    for M in (1, 3, 8, 13, 16, 31, 48, 64):
        for t in proj.tactics(M):
            proj.set_tactic(M, t)
            y = run_proj(proj, xd[:M], out_dtype)
            assert_parity(y, ref[:M], s[:M], f"checked M={M} {t}")
            n += 1
        proj.check_status()  # raises SkinnyGemmError(ECHECK) if any access failed its test
    proj.close()
    assert n > 200, n


def test_large_token_counts_and_dtypes_checked(skg):
    N, K = 656, 1088
    w, x, ref, s = full_case(N, K, seed=3)
    wd = w.to(DEV)
    xl = pin.case(N, K, seed=5)[1]  # 64 rows; build 200 by stacking three seeds
    x200 = torch.cat([xl, pin.case(N, K, seed=6)[1], pin.case(N, K, seed=7)[1], xl[:8]])
    ref200, s200 = oracle.projection(x200, w)
    proj = skg.Projection(wd, use_tactic_file=False)
    for M in (65, 128, 200):
        for t in proj.tactics(M):
            proj.set_tactic(M, t)
            y = run_proj(proj, x200[:M].to(DEV), torch.bfloat16)
            assert_parity(y, ref200[:M], s200[:M], f"checked M={M} {t}")
    proj.check_status()
    proj.close()
    # fp16 operands
    w16, x16 = pin.case(N, K, seed=3, dtype=torch.float16)
    ref16, s16 = oracle.projection(x16, w16)
    p16 = skg.Projection(w16.to(DEV), use_tactic_file=False)
    for M in (1, 16, 48):
        for t in p16.tactics(M):
            p16.set_tactic(M, t)
            y = run_proj(p16, x16[:M].to(DEV), torch.float16)
            assert_parity(y, ref16[:M], s16[:M], f"checked fp16 M={M} {t}")
    p16.check_status()
    p16.close()
    # fused residual, in place
    pr = skg.Projection(wd, use_tactic_file=False)
    for M in (4, 32):
        r = (torch.randn(M, N, generator=torch.Generator().manual_seed(M)) / 4).to(torch.bfloat16)
        out = r.clone().to(DEV)
        pr.run(x[:M].to(DEV), out, residual=out)
        torch.cuda.synchronize()
        refr, sr = oracle.projection_residual(x[:M], w, r)
        assert_parity(out, refr, sr, f"checked residual M={M}")
    pr.check_status()
    pr.close()


@pytest.mark.parametrize("N", [3584, 6288])
def test_full_size_checked(skg, N):
    w, x, ref, s = full_case(N, 7168)
    proj = skg.Projection(w.to(DEV), use_tactic_file=False)
    xd = x.to(DEV)
    for M in (1, 8, 16, 32, 48, 64):
        y = run_proj(proj, xd[:M], torch.bfloat16)
        assert_parity(y, ref[:M], s[:M], f"checked N={N} M={M} {proj.plan(M)}")
    proj.check_status()
    proj.close()


def test_overlap_step_checked(skg):
    wp, x, ref, s = full_case(6288, 7168)
    wfb = pin.weight(1536, 128, seed=1)
    wp_d = wp.to(DEV)
    main = skg.Projection(wp_d, use_tactic_file=False)
    fa = skg.Projection(wp_d[:128], use_tactic_file=False)
    fb = skg.Projection(wfb.to(DEV), use_tactic_file=False)
    aux = torch.cuda.Stream(priority=-1)
    events = (torch.cuda.Event(), torch.cuda.Event())
    for M in (1, 32):
        out_main = torch.empty((M, 6288), dtype=torch.bfloat16, device=DEV)
        fa_out = torch.empty((M, 128), dtype=torch.bfloat16, device=DEV)
        out_fb = torch.empty((2, M, 1536), dtype=torch.bfloat16, device=DEV)
        skg.run_overlap(main, fa, fb, x[:M].to(DEV), out_main, fa_out, out_fb, chain=2,
                        aux_stream=aux, events=events)
        torch.cuda.synchronize()
        assert_parity(out_main, ref[:M], s[:M], f"checked overlap main M={M}")
        inp = fa_out
        for i in range(2):
            r, sb = oracle.projection(inp.cpu(), wfb)
            assert_parity(out_fb[i], r, sb, f"checked overlap F_B link {i} M={M}")
            inp = out_fb[i][:, :128]
    for p in (main, fa, fb):
        p.check_status()
        p.close()


def test_failed_check_is_reported_and_cleared(skg):
    """The reporting path: an injected failed check (the checked build's
    self-test, no access made) comes back from check_status as SKG_ECHECK naming
    the access; the status is cleared and the next launch is correct."""
    from skinny_bf16_projection_gb300 import _native
    w, x, ref, s = full_case(656, 1088, seed=3)
    proj = skg.Projection(w.to(DEV), use_tactic_file=False)
    xd = x.to(DEV)
    proj.inject_check(1)
    run_proj(proj, xd[:4], torch.bfloat16)
    with pytest.raises(skg.SkinnyGemmError) as e:
        proj.check_status()
    assert e.value.code == _native.SKG_ECHECK and "access 11" in str(e.value), str(e.value)
    y = run_proj(proj, xd[:4], torch.bfloat16)
    proj.check_status()
    assert_parity(y, ref[:4], s[:4], "after the injected check")
    proj.close()


def test_normal_library_refuses_check_injection():
    import __graft_entry__
    __graft_entry__.build()
    from skinny_bf16_projection_gb300 import _native, build
    import skinny_bf16_projection_gb300 as m
    lib = _native.load(build.LIB_PATH)
    w = pin.weight(256, 512, seed=5).to(DEV)
    h = lib.skinny_gemm_prepare(w.data_ptr(), 256, 512, _native.SKG_BF16, _native.SKG_BF16)
    assert h
    try:
        assert lib.skinny_gemm_debug_inject_check(h, 1) == _native.SKG_EINVAL
        assert b"not a checked build" in lib.skinny_gemm_last_error()
    finally:
        lib.skinny_gemm_destroy(h)
    del m
