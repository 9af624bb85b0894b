"""GPU parity beyond the decode range: token tiles of 128 and 256 (tcgen05 with
N = 128 / 256, the accumulator read in 32-column chunks) and tiles of 64 / 128
tokens repeated over ceil(M / tile) token tiles (grid y), M = 65..256, against
the oracle under |y - ref| <= 8e-3 |ref| + 2e-3 s."""
import functools

import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, run_proj

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skg():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import skinny_bf16_projection_gb300 as m
    return m


@functools.lru_cache(maxsize=4)
def case256(N, K, seed=0):
    w, x = pin.case(N, K, seed=seed, max_tokens=256)
    ref, s = oracle.projection(x, w)
    return w, x, ref, s


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float32])
def test_large_token_counts_full_size(skg, odt):
    w, x, ref, s = case256(3584, 7168)
    proj = skg.Projection(w.to(DEV), odt, use_tactic_file=False)
    xd = x.to(DEV)
    for M in (65, 96, 128, 129, 200, 256):
        y = run_proj(proj, xd[:M], odt)
        assert_parity(y, ref[:M], s[:M], f"M={M} {odt} {proj.plan(M)}")
    assert proj.plan(100).split(":")[2] == "t128" and proj.plan(256).split(":")[2] == "t256"
    proj.check_status()


def test_large_token_counts_every_candidate(skg):
    w, x, ref, s = case256(656, 1088, seed=3)
    proj = skg.Projection(w.to(DEV), use_tactic_file=False)
    xd = x.to(DEV)
    for M in (65, 100, 200, 256):
        cands = proj.tactics(M)
        assert cands and all(t.startswith("tc:") for t in cands)
        assert any(":t64:" in t for t in cands)  # multi-tile candidates are offered
        for t in cands:
            proj.set_tactic(M, t)
            y = run_proj(proj, xd[:M], torch.bfloat16)
            assert_parity(y, ref[:M], s[:M], f"M={M} {t}")


@pytest.mark.parametrize("tactic", [None, "tc:r128:t64:b1:s3:c8", "tc:r128:t128:b1:s2:c4:d2"])
def test_large_m_rows_beyond_m_untouched(skg, tactic):
    w, x, ref, s = case256(3584, 7168)
    proj = skg.Projection(w.to(DEV), use_tactic_file=False)
    M = 130
    if tactic:
        proj.set_tactic(M, tactic)  # 3 or 2 token tiles, the last one ragged
    obuf = torch.full((M + 5, 3584), float("nan"), dtype=torch.bfloat16, device=DEV)
    xbuf = torch.full((256, 7168), float("nan"), dtype=torch.bfloat16, device=DEV)
    xbuf[:M] = x[:M].to(DEV)
    proj.run(xbuf[:M], obuf[:M])
    torch.cuda.synchronize()
    assert torch.isnan(obuf[M:]).all() and torch.isfinite(obuf[:M]).all()
    assert_parity(obuf[:M], ref[:M], s[:M], f"canary M=130 {proj.plan(M)}")
    proj.close()


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float32])
def test_token_tiles_full_size_with_residual(skg, odt):
    """Multi-tile tactics at full size, with the fused residual (in place) on
    the vectorized store path."""
    w, x, ref, s = case256(3584, 7168)
    proj = skg.Projection(w.to(DEV), odt, use_tactic_file=False)
    xd = x.to(DEV)
    for M, t in ((96, "tc:r128:t64:b1:s3:c8:d1"), (256, "tc:r128:t64:b1:s3:c8"),
                 (256, "tc:r128:t128:b2:s2:c4:d2"), (200, "tc:r128:t128:b1:s2:c8")):
        proj.set_tactic(M, t)
        y = run_proj(proj, xd[:M], odt)
        assert_parity(y, ref[:M], s[:M], f"M={M} {t}")
        res = torch.linspace(-2.0, 2.0, M * 3584).reshape(M, 3584).to(odt)
        want, ws = oracle.projection_residual(x[:M], w, res)
        out = res.to(DEV)
        proj.run(xd[:M], out, residual=out)
        torch.cuda.synchronize()
        assert_parity(out, want, ws, f"residual M={M} {t}")
    proj.close()
