"""Run-time K sharing within a cluster (tactic suffix ":w"): after its first
stages, whose K boxes are fixed, each CTA of a cluster takes the next boxes
from a counter in the cluster's first CTA.  Which CTA sums which box then
varies, so only the acceptance bound (and exact integer sums) can be checked,
never bits run to run; these tests cover every cluster candidate with ":w",
uneven K splits, full decode sizes, CUDA graphs and the deterministic flag."""
import numpy as np
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, full_case, run_proj, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def skg():
    import skinny_bf16_projection_gb300 as m
    return m


def shared_variants(tactics):
    """The candidates that can take ':w' (a cluster, no aliased receive buffer)."""
    out = []
    for t in tactics:
        f = t.split(":")
        if f[0] in ("mma", "tc") and int(f[5][1:]) > 1 and "a" not in f[6:]:
            out.append(t + ":w")
    return out


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_every_cluster_candidate_with_shared_k_on_ragged_shape(out_dtype):
    # 17 K boxes: the fixed first stages and the counter's hand-out split unevenly
    N, K = 656, 1088
    w, x, ref, s = full_case(N, K, seed=3)
    proj = skg().Projection(w.to(DEV), out_dtype, use_tactic_file=False)
    xd = x.to(DEV)
    n = 0
    for M in (1, 8, 13, 16, 31, 48, 64):
        for t in shared_variants(proj.tactics(M)):
            proj.set_tactic(M, t)
            assert proj.plan(M) == t
            for _ in range(2):
                y = run_proj(proj, xd[:M], out_dtype)
                assert_parity(y, ref[:M], s[:M], f"M={M} {t}")
            n += 1
    proj.check_status()
    assert n >= 20, n


def test_shared_k_exact_on_small_integers():
    """Integer inputs: every partial sum is exact, so whatever CTA sums which box
    the fp32 output equals the oracle bit for bit."""
    N, K = 320, 2048
    w = pin.small_integers(N, K, seed=21)
    x = pin.small_integers(64, K, seed=22)
    ref, _ = oracle.projection(x, w, with_scale=False)
    wd, xd = w.to(DEV), x.to(DEV)
    p32 = skg().Projection(wd, torch.float32, use_tactic_file=False)
    for M in (1, 8, 24, 64):
        for t in shared_variants(p32.tactics(M)):
            p32.set_tactic(M, t)
            y32 = run_proj(p32, xd[:M], torch.float32)
            assert np.array_equal(to_f64(y32), ref[:M]), f"fp32 not exact: M={M} {t}"


@pytest.mark.parametrize("N", [3584, 6288])
def test_shared_k_full_size_and_graph_replay(N):
    w, x, ref, s = full_case(N, 7168)
    proj = skg().Projection(w.to(DEV), use_tactic_file=False)
    xd = x.to(DEV)
    picks = {1: "mma:r128:t8:b1:s2:c16:d3:w", 8: "mma:r64:t8:b2:s2:c8:w",
             16: "mma:r64:t16:b2:s2:c8:d3:w", 32: "tc:r128:t32:b2:s2:c8:d1:w",
             64: "tc:r128:t64:b2:s2:c8:w"}
    outs = {}
    for M, t in picks.items():
        proj.set_tactic(M, t)
        outs[M] = run_proj(proj, xd[:M], torch.bfloat16)
        assert_parity(outs[M], ref[:M], s[:M], f"N={N} M={M} {t}")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for M in picks:
            proj.run(xd[:M], outs[M])
    for M in picks:
        outs[M].fill_(float("nan"))
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize()
    for M in picks:
        assert_parity(outs[M], ref[:M], s[:M], f"graph N={N} M={M} {picks[M]}")
    proj.check_status()


def test_deterministic_flag_keeps_fixed_order():
    w, x, ref, s = full_case(3584, 7168)
    proj = skg().Projection(w.to(DEV), use_tactic_file=False, deterministic=True)
    proj.autotune([1, 32])
    assert not proj.plan(1).endswith(":w") and not proj.plan(32).endswith(":w")
    xd = x.to(DEV)
    for M in (1, 32):
        a = run_proj(proj, xd[:M], torch.bfloat16)
        b = run_proj(proj, xd[:M], torch.bfloat16)
        assert torch.equal(a, b)
        assert_parity(a, ref[:M], s[:M], f"deterministic M={M} {proj.plan(M)}")
