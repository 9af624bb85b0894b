"""GPU parity of the fused residual epilogue, out = x @ W^T + residual, against
the oracle (projection in fp64 plus the residual widened exactly), under
|y - (ref + r)| <= 8e-3 |ref + r| + 2e-3 s, for every kernel family's store
path: direct stores, the cluster reduction and the stream-K fixup."""
import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, full_case, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skg():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import skinny_bf16_projection_gb300 as m
    return m


def residual_like(M, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(M, N, generator=g) * 3).to(dtype)


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float32])
def test_residual_full_size(skg, odt):
    w, x, _, _ = full_case(3584, 7168)
    proj = skg.Projection(w.to(DEV), odt, use_tactic_file=False)
    xd = x.to(DEV)
    for M in (1, 8, 32, 64):
        r = residual_like(M, 3584, odt, seed=M)
        ref, s = oracle.projection_residual(x[:M], w, r)
        out = torch.empty((M, 3584), dtype=odt, device=DEV)
        proj.run(xd[:M], out, residual=r.to(DEV))
        assert_parity(out, ref, s, f"residual M={M} {odt} {proj.plan(M)}")


def test_residual_every_candidate_tactic(skg):
    w, x, _, _ = full_case(656, 1088, seed=3)
    proj = skg.Projection(w.to(DEV), use_tactic_file=False)
    xd = x.to(DEV)
    kinds = set()
    for M in (1, 13, 48):
        r = residual_like(M, 656, torch.bfloat16, seed=100 + M)
        ref, s = oracle.projection_residual(x[:M], w, r)
        rd = r.to(DEV)
        for t in proj.tactics(M):
            proj.set_tactic(M, t)
            out = torch.empty((M, 656), dtype=torch.bfloat16, device=DEV)
            proj.run(xd[:M], out, residual=rd)
            assert_parity(out, ref, s, f"residual M={M} {t}")
            kinds.add(t.split(":")[0])
    assert {"tc", "mma", "sk"} <= kinds


def test_residual_in_place(skg):
    w, x, _, _ = full_case(3584, 7168)
    proj = skg.Projection(w.to(DEV), use_tactic_file=False)
    for M in (1, 16, 48):
        r = residual_like(M, 3584, torch.bfloat16, seed=7 * M)
        ref, s = oracle.projection_residual(x[:M], w, r)
        buf = r.to(DEV)
        proj.run(x[:M].to(DEV), buf, residual=buf)  # out += x @ W^T
        assert_parity(buf, ref, s, f"in place M={M} {proj.plan(M)}")


def test_residual_exact_integers_fp32(skg):
    w = pin.small_integers(320, 2048, seed=41)
    x = pin.small_integers(64, 2048, seed=42)
    proj = skg.Projection(w.to(DEV), torch.float32, use_tactic_file=False)
    for M in (1, 24, 64):
        r = pin.small_integers(M, 320, seed=43, lo=-5000, hi=5000).to(torch.float32)
        ref, _ = oracle.projection_residual(x[:M], w, r)
        for t in proj.tactics(M)[::4]:
            proj.set_tactic(M, t)
            out = torch.empty((M, 320), dtype=torch.float32, device=DEV)
            proj.run(x[:M].to(DEV), out, residual=r.to(DEV))
            assert np.array_equal(to_f64(out), ref), f"M={M} {t}"


def test_residual_partial_overlap_rejected(skg):
    proj = skg.Projection(torch.zeros(256, 1024, dtype=torch.bfloat16, device=DEV))
    buf = torch.zeros(9, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(skg.SkinnyGemmError):
        proj.run(torch.zeros(8, 1024, dtype=torch.bfloat16, device=DEV), buf[1:], residual=buf[:8])
