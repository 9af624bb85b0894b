"""Seeded random shapes, pitches, token counts, output types and tactics through
the C ABI, each output checked element by element against the oracle under
|y - ref| <= 8e-3 |ref| + 2e-3 s.  Complements the fixed workloads: odd N, K
not a multiple of 64, padded row pitches, every kernel family."""
import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skg():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import skinny_bf16_projection_gb300 as m
    return m


def _cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        N = int(rng.integers(1, 2600))
        K = int(rng.integers(1, 520)) * 8          # bf16 rows stay 16-byte multiples
        M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 24, 32, 47, 64, 100, 200]))
        out_fp32 = bool(rng.integers(0, 2))
        pad_x = int(rng.integers(0, 3)) * 8        # x row pitch K + pad (16-byte multiple)
        pad_o = int(rng.integers(0, 5))            # any out pitch >= N
        pick = int(rng.integers(0, 1 << 30))
        out.append((i, N, K, M, out_fp32, pad_x, pad_o, pick))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"case{c[0]}")
def test_random_shape(skg, case):
    i, N, K, M, out_fp32, pad_x, pad_o, pick = case
    odt = torch.float32 if out_fp32 else torch.bfloat16
    w, x = pin.case(N, K, seed=100 + i, max_tokens=max(M, 1))
    ref, s = oracle.projection(x[:M], w)
    proj = skg.Projection(w.to(DEV), odt, use_tactic_file=False)
    cands = proj.tactics(M)
    if cands and pick % 3:  # two thirds of the cases force a random candidate tactic
        proj.set_tactic(M, cands[pick % len(cands)])
    xb = torch.full((M, K + pad_x), float("nan"), dtype=torch.bfloat16, device=DEV)
    xb[:, :K] = x[:M].to(DEV)
    ob = torch.full((M, N + pad_o), float("nan"), dtype=odt, device=DEV)
    proj.run(xb[:, :K], ob[:, :N])
    torch.cuda.synchronize()
    assert_parity(ob[:, :N], ref, s, f"N={N} K={K} M={M} {odt} ldx={K + pad_x} "
                                     f"ldo={N + pad_o} {proj.plan(M)}")
    if pad_o:
        assert torch.isnan(ob[:, N:]).all(), "columns beyond N were written"
    proj.check_status()
    proj.close()
