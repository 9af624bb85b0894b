"""GPU parity for FP16 operands (both x and W fp16, fp32 accumulation, fp16 or
fp32 output) against the oracle's exact fp16 widening, under the same bound
|y - ref| <= 8e-3 |ref| + 2e-3 s as the bf16 path."""
import functools

import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, run_proj, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skg():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import skinny_bf16_projection_gb300 as m
    return m


@functools.lru_cache(maxsize=4)
def fp16_case(N, K, seed=0):
    w, x = pin.case(N, K, seed=seed, dtype=torch.float16)
    ref, s = oracle.projection(x, w)
    return w, x, ref, s


@pytest.mark.parametrize("odt", [torch.float16, torch.float32])
def test_fp16_full_size_every_token_tile(skg, odt):
    w, x, ref, s = fp16_case(3584, 7168)
    proj = skg.Projection(w.to(DEV), odt, use_tactic_file=False)
    xd = x.to(DEV)
    for M in (1, 2, 8, 16, 32, 48, 64):
        y = run_proj(proj, xd[:M], odt)
        assert_parity(y, ref[:M], s[:M], f"fp16 M={M} {odt} {proj.plan(M)}")
    proj.check_status()


def test_fp16_every_candidate_tactic_on_ragged_shape(skg):
    w, x, ref, s = fp16_case(656, 1088, seed=3)
    proj = skg.Projection(w.to(DEV), torch.float16, use_tactic_file=False)
    xd = x.to(DEV)
    kinds = set()
    for M in (1, 13, 48):
        for t in proj.tactics(M):
            proj.set_tactic(M, t)
            y = run_proj(proj, xd[:M], torch.float16)
            assert_parity(y, ref[:M], s[:M], f"fp16 M={M} {t}")
            kinds.add(t.split(":")[0])
    assert {"tc", "mma", "sk"} <= kinds


def test_fp16_small_integers_exact_in_fp32(skg):
    w = pin.small_integers(320, 2048, seed=31, dtype=torch.float16)
    x = pin.small_integers(64, 2048, seed=32, dtype=torch.float16)
    ref, _ = oracle.projection(x, w, with_scale=False)
    proj = skg.Projection(w.to(DEV), torch.float32, use_tactic_file=False)
    xd = x.to(DEV)
    for M in (1, 8, 64):
        for t in proj.tactics(M)[::3]:
            proj.set_tactic(M, t)
            y = run_proj(proj, xd[:M], torch.float32)
            assert np.array_equal(to_f64(y), ref[:M]), f"fp16 M={M} {t}"


def test_fp16_output_is_rounding_of_fp32_output(skg):
    w, x, _, _ = fp16_case(3584, 7168)
    wd, xd = w.to(DEV), x.to(DEV)
    p32 = skg.Projection(wd, torch.float32, use_tactic_file=False)
    p16 = skg.Projection(wd, torch.float16, use_tactic_file=False)
    for M in (1, 32):
        p16.set_tactic(M, p32.plan(M))
        assert torch.equal(run_proj(p32, xd[:M], torch.float32).to(torch.float16),
                           run_proj(p16, xd[:M], torch.float16))


def test_output_type_must_match_operands(skg):
    w16 = torch.zeros(256, 1024, dtype=torch.float16, device=DEV)
    wbf = torch.zeros(256, 1024, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(skg.SkinnyGemmError):
        skg.Projection(w16, torch.bfloat16)
    with pytest.raises(skg.SkinnyGemmError):
        skg.Projection(wbf, torch.float16)
    with pytest.raises(ValueError):  # x must have the weight's type
        skg.Projection(w16).run(torch.zeros(4, 1024, dtype=torch.bfloat16, device=DEV),
                                torch.empty(4, 256, dtype=torch.float16, device=DEV))
