"""Boundary promises of the C ABI that need a device: the tactic file written by
the autotuner and read back at prepare, the SKINNY_GEMM_TUNE modes, prepare's
refusal while a capture is visible, and the overlap step's argument checks,
which must refuse a bad step before anything is enqueued."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, run_proj

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def skg():
    import skinny_bf16_projection_gb300 as m
    return m


def read_lines(path):
    return [ln.split() for ln in open(path).read().splitlines() if ln.strip()] if path.exists() else []


def test_tactic_file_round_trip_and_tune_modes(tmp_path, monkeypatch):
    m = skg()
    path = tmp_path / "tactics.txt"
    monkeypatch.setenv("SKINNY_GEMM_TACTIC_FILE", str(path))
    monkeypatch.delenv("SKINNY_GEMM_TUNE", raising=False)
    monkeypatch.delenv("SKINNY_GEMM_FORCE_TACTIC", raising=False)
    N, K = 512, 1024
    w = pin.weight(N, K, seed=31).to(DEV)
    default = m.Projection(w, use_tactic_file=False)

    # the autotuner appends its pick, a later prepare ("cache", the default) reads it back
    p1 = m.Projection(w)
    p1.autotune([8])
    lines = read_lines(path)
    assert [ln[1:3] for ln in lines] == [["8", p1.plan(8)]]
    key = lines[0][0]
    assert m.Projection(w).plan(8) == p1.plan(8)

    # a hand-written entry for another token count is honoured as well
    cands = default.tactics(16)
    pick = next(t for t in reversed(cands) if t != default.plan(16))
    with open(path, "a") as f:
        f.write(f"{key} 16 {pick} 1.0\n")
        f.write(f"not-this-device 32 {cands[0]} 1.0\n")  # another key: ignored
    p3 = m.Projection(w)
    assert p3.plan(16) == pick and p3.plan(8) == p1.plan(8)
    assert p3.plan(32) == default.plan(32)

    # "off" ignores the file; an unknown mode is refused
    monkeypatch.setenv("SKINNY_GEMM_TUNE", "off")
    p4 = m.Projection(w)
    assert all(p4.plan(M) == default.plan(M) for M in (8, 16, 32, 64))
    monkeypatch.setenv("SKINNY_GEMM_TUNE", "bogus")
    with pytest.raises(m.SkinnyGemmError) as e:
        m.Projection(w)
    assert e.value.code == m._native.SKG_EINVAL

    # "full": only the decode token counts missing from the file are tuned (here 64)
    monkeypatch.setenv("SKINNY_GEMM_TUNE", "full")
    with open(path, "a") as f:
        for M in (1, 2, 4, 32, 48):
            f.write(f"{key} {M} {default.plan(M)} 1.0\n")
    before = len(read_lines(path))
    p5 = m.Projection(w)
    added = read_lines(path)[before:]
    assert [ln[1] for ln in added] == ["64"], added
    assert p5.plan(64) == added[0][2] and p5.plan(16) == pick

    x = pin.case(N, K, seed=32)[1]
    ref, s = oracle.projection(x, w.cpu())
    for M in (8, 16, 64):
        y = run_proj(p5, x[:M].to(DEV), torch.bfloat16)
        assert_parity(y, ref[:M], s[:M], f"plan from the tactic file, M={M} {p5.plan(M)}")
    for p in (default, p1, p3, p4, p5):
        p.close()


def test_prepare_refuses_while_capturing():
    """A capture on the per-thread default stream is visible to prepare, which
    then refuses before any allocation, leaving the capture intact."""
    m = skg()
    nat = m._native
    lib = nat.lib()
    cudart = ctypes.CDLL("libcudart.so.13")  # the runtime the library is linked against
    cudart.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
    cudart.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    cudart.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
    per_thread = ctypes.c_void_p(2)  # cudaStreamPerThread
    w = torch.randn(256, 1024, device=DEV).to(torch.bfloat16)
    torch.cuda.synchronize()
    assert cudart.cudaStreamBeginCapture(per_thread, 0) == 0  # global capture mode
    try:
        h = lib.skinny_gemm_prepare(w.data_ptr(), 256, 1024, nat.SKG_BF16, nat.SKG_BF16)
        code, msg = lib.skinny_gemm_last_status(), nat.last_error()
    finally:
        graph = ctypes.c_void_p()
        end = cudart.cudaStreamEndCapture(per_thread, ctypes.byref(graph))
        if graph.value:
            cudart.cudaGraphDestroy(graph)
    assert h is None and code == nat.SKG_ECAPTURING, msg
    assert end == 0, "the refused prepare must not invalidate the capture"
    p = m.Projection(w)  # outside the capture it prepares normally
    p.close()


def test_overlap_refuses_bad_buffers_before_forking():
    """Every buffer of the two-stream step is checked before the fork is
    recorded: a refused step leaves no unjoined aux stream in a capture."""
    m = skg()
    nat = m._native
    lib = nat.lib()
    wm = (torch.randn(512, 1024, device=DEV) / 32).to(torch.bfloat16)
    main = m.Projection(wm)
    fa = m.Projection(wm[:128])
    fb = m.Projection((torch.randn(256, 128, device=DEV) / 11).to(torch.bfloat16))
    fb_odd = m.Projection((torch.randn(132, 128, device=DEV) / 11).to(torch.bfloat16))  # 264 B rows
    M = 4
    x = torch.randn(M, 1024, device=DEV).to(torch.bfloat16)
    om = torch.empty(M, 512, device=DEV, dtype=torch.bfloat16)
    fo = torch.empty(M, 128, device=DEV, dtype=torch.bfloat16)
    fbo = torch.empty(2, M, 256, device=DEV, dtype=torch.bfloat16)
    fbo_odd = torch.empty(2, M, 132, device=DEV, dtype=torch.bfloat16)
    side, aux = torch.cuda.Stream(), torch.cuda.Stream()
    ev = [torch.cuda.Event(), torch.cuda.Event()]
    for e in ev:
        e.record(aux)
    torch.cuda.synchronize()

    def call(h_fb, chain, out_fb_ptr):
        return lib.skinny_gemm_run_overlap(
            main._h, fa._h, h_fb._h, chain, x.data_ptr(), M, om.data_ptr(), fo.data_ptr(),
            out_fb_ptr, ctypes.c_void_p(side.cuda_stream), ctypes.c_void_p(aux.cuda_stream),
            ctypes.c_void_p(ev[0].cuda_event), ctypes.c_void_p(ev[1].cuda_event))

    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    codes = []
    with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
        om.zero_()
        codes.append(call(fb, 1, None))                        # null out_fb
        codes.append(call(fb, 1, fbo.data_ptr() + 2))          # misaligned out_fb
        codes.append(call(fb_odd, 2, fbo_odd.data_ptr()))      # chain link pitch not 16 B
    assert codes == [nat.SKG_EINVAL, nat.SKG_EALIGN, nat.SKG_EALIGN], codes
    g.replay()
    torch.cuda.synchronize()
    # the well-formed step still runs, eager
    assert call(fb, 2, fbo.data_ptr()) == nat.SKG_OK
    torch.cuda.synchronize()
    ref, s = oracle.projection(x.cpu(), wm.cpu())
    assert_parity(om, ref, s, "overlap main after refused steps")
    for p in (main, fa, fb, fb_odd):
        p.close()
