"""L2 prefetch of later weight stages before the PDL wait (tactic suffix
":p<k>"): the prefetch only changes where the weight bytes come from, never
what is computed, so every variant must match the oracle, and a dependent
chain of projections (each output the next input) launched with it must give
the bits of the same tactic launched without programmatic dependent launch."""
import re

import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, full_case, run_proj

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def skg():
    import skinny_bf16_projection_gb300 as m
    return m


def with_prefetch(tactics, ks=(1, 2, 4)):
    out = []
    for t in tactics:
        if t.startswith(("mma:", "tc:")):
            out += [f"{t}:p{k}" for k in ks]
    return out


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_prefetch_variants_on_ragged_shape(out_dtype):
    N, K = 656, 1088  # 17 K boxes: some CTAs have fewer refill stages than k
    w, x, ref, s = full_case(N, K, seed=3)
    proj = skg().Projection(w.to(DEV), out_dtype, use_tactic_file=False)
    xd = x.to(DEV)
    n = 0
    for M in (1, 13, 32, 64):
        for t in with_prefetch(proj.tactics(M)[::3]):
            proj.set_tactic(M, t)
            y = run_proj(proj, xd[:M], out_dtype)
            assert_parity(y, ref[:M], s[:M], f"M={M} {t}")
            n += 1
    proj.check_status()
    assert n >= 30, n


@pytest.mark.parametrize("N", [3584, 6288])
def test_prefetch_full_size(N):
    w, x, ref, s = full_case(N, 7168)
    proj = skg().Projection(w.to(DEV), use_tactic_file=False)
    xd = x.to(DEV)
    for M, t in ((1, "mma:r64:t8:b4:s3:c4:d3:p1"), (8, "mma:r128:t8:b1:s2:c16:d3:p2"),
                 (16, "mma:r64:t16:b2:s2:c8:d3:p1"), (32, "tc:r128:t32:b2:s2:c8:d1:p1"),
                 (64, "tc:r128:t64:b2:s2:c8:d2:p1:a")):
        proj.set_tactic(M, t)
        y = run_proj(proj, xd[:M], torch.bfloat16)
        assert_parity(y, ref[:M], s[:M], f"N={N} M={M} {t}")
    proj.check_status()


def test_prefetch_dependent_chain_matches_no_pdl():
    D = 4096
    w = pin.weight(D, D, seed=11, std=1.0 / np.sqrt(D))
    wd = w.to(DEV)
    x0 = pin.case(8, D, seed=12, max_tokens=32)[1]
    with_pdl = skg().Projection(wd, use_tactic_file=False)
    no_pdl = skg().Projection(wd, use_tactic_file=False, pdl=False)
    links = 6
    for M in (1, 16, 32):
        base = re.sub(r":p\d+", "", with_pdl.plan(M))  # the default plan may prefetch already
        no_pdl.set_tactic(M, base)
        ref = [x0[:M].to(DEV)] + [torch.empty((M, D), dtype=torch.bfloat16, device=DEV)
                                  for _ in range(links)]
        for i in range(links):
            no_pdl.run(ref[i], ref[i + 1])
        torch.cuda.synchronize()
        for k in (1, 2, 4):
            with_pdl.set_tactic(M, f"{base}:p{k}")
            bufs = [ref[0]] + [torch.full((M, D), float("nan"), dtype=torch.bfloat16, device=DEV)
                               for _ in range(links)]
            for i in range(links):
                with_pdl.run(bufs[i], bufs[i + 1])
            torch.cuda.synchronize()
            assert torch.equal(bufs[-1], ref[-1]), f"{base}:p{k} M={M}"
    ref_s, s_s = oracle.projection(ref[0].cpu(), w)
    assert_parity(ref[1], ref_s, s_s, "first link")
