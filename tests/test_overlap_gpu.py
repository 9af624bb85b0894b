"""GPU parity of the two-stream decode step: the packed W[6288, 7168] projection
on the main stream while the aux stream runs F_A (the packed weight's first 128
rows, prepared in place with its row pitch) and then a chain of F_B
W[1536, 128] projections, forked and joined by events, eager and captured in
one CUDA graph.  Each F_B link is checked against the oracle on the GPU's own
bf16 input, so a last-bit difference in one link does not compound."""
import pytest
import torch

import oracle
import projection_inputs as pin
from gpu_helpers import DEV, assert_parity, full_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    import __graft_entry__
    __graft_entry__.build()
    import skinny_bf16_projection_gb300 as skg
    torch.cuda.set_device(0)
    wp, x, ref, s = full_case(6288, 7168)
    wfb = pin.weight(1536, 128, seed=1)
    wp_d, wfb_d = wp.to(DEV), wfb.to(DEV)
    main = skg.Projection(wp_d)
    fa = skg.Projection(wp_d[:128])
    fb = skg.Projection(wfb_d)
    return dict(skg=skg, main=main, fa=fa, fb=fb, wfb=wfb, x=x.to(DEV), ref=ref, s=s)


def check_links(st, M, fa_out, out_fb, chain):
    assert_parity(fa_out, st["ref"][:M, :128], st["s"][:M, :128], f"F_A M={M}")
    inp = fa_out
    for i in range(chain):
        ref, s = oracle.projection(inp.cpu(), st["wfb"])
        assert_parity(out_fb[i], ref, s, f"F_B link {i} M={M}")
        inp = out_fb[i][:, :128]


@pytest.mark.parametrize("chain", [1, 4])
@pytest.mark.parametrize("M", [1, 4, 8, 16, 32])
def test_overlap_step_eager(setup, M, chain):
    st = setup
    aux = torch.cuda.Stream(priority=-1)
    events = (torch.cuda.Event(), torch.cuda.Event())
    out_main = torch.empty((M, 6288), dtype=torch.bfloat16, device=DEV)
    fa_out = torch.empty((M, 128), dtype=torch.bfloat16, device=DEV)
    out_fb = torch.empty((chain, M, 1536), dtype=torch.bfloat16, device=DEV)
    st["skg"].run_overlap(st["main"], st["fa"], st["fb"], st["x"][:M], out_main, fa_out, out_fb,
                          chain=chain, aux_stream=aux, events=events)
    torch.cuda.synchronize()
    assert_parity(out_main, st["ref"][:M], st["s"][:M], f"main M={M}")
    check_links(st, M, fa_out, out_fb, chain)


def test_overlap_step_captured_in_one_graph(setup):
    st = setup
    chain = 4
    aux = torch.cuda.Stream(priority=-1)
    events = (torch.cuda.Event(), torch.cuda.Event())
    graphs, bufs = [], []
    cap = torch.cuda.Stream()
    for M in (1, 8, 32):
        out_main = torch.zeros((M, 6288), dtype=torch.bfloat16, device=DEV)
        fa_out = torch.zeros((M, 128), dtype=torch.bfloat16, device=DEV)
        out_fb = torch.zeros((chain, M, 1536), dtype=torch.bfloat16, device=DEV)
        # eager once: creates the events outside capture
        st["skg"].run_overlap(st["main"], st["fa"], st["fb"], st["x"][:M], out_main, fa_out,
                              out_fb, chain=chain, aux_stream=aux, events=events)
        torch.cuda.synchronize()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            st["skg"].run_overlap(st["main"], st["fa"], st["fb"], st["x"][:M], out_main, fa_out,
                                  out_fb, chain=chain, aux_stream=aux, events=events)
        graphs.append(g)
        bufs.append((M, out_main, fa_out, out_fb))
    for (M, out_main, fa_out, out_fb) in bufs:
        out_main.zero_(); fa_out.zero_(); out_fb.zero_()
    torch.cuda.synchronize()
    for g in graphs:
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    for (M, out_main, fa_out, out_fb) in bufs:
        assert_parity(out_main, st["ref"][:M], st["s"][:M], f"graph main M={M}")
        check_links(st, M, fa_out, out_fb, chain)


def test_overlap_rejects_mismatched_handles(setup):
    st = setup
    skg = st["skg"]
    aux = torch.cuda.Stream()
    events = (torch.cuda.Event(), torch.cuda.Event())
    M = 4
    out_main = torch.empty((M, 6288), dtype=torch.bfloat16, device=DEV)
    fa_out = torch.empty((M, 128), dtype=torch.bfloat16, device=DEV)
    out_fb = torch.empty((1, M, 1536), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(skg.SkinnyGemmError):  # F_B's K (128) must equal F_A's N
        skg.run_overlap(st["main"], st["fb"], st["fb"], st["x"][:M], out_main, fa_out, out_fb,
                        aux_stream=aux, events=events)


def test_overlap_tuned_fa_plan_keeps_parity(setup):
    """skinny_gemm_autotune_overlap times F_A's and the main projection's
    candidates inside the whole step and installs the fastest; the step must
    stay correct with them, and the F_B plan must not change."""
    st = setup
    skg = st["skg"]
    fa = skg.Projection(st["main"].weight[:128], use_tactic_file=False)
    main = skg.Projection(st["main"].weight, use_tactic_file=False)
    chain = 4
    fb_before = [st["fb"].plan(M) for M in (1, 8, 32)]
    skg.tune_overlap(main, fa, st["fb"], [1, 8, 32], chain=chain)
    assert [st["fb"].plan(M) for M in (1, 8, 32)] == fb_before
    aux = torch.cuda.Stream(priority=-1)
    events = (torch.cuda.Event(), torch.cuda.Event())
    for M in (1, 5, 8, 32):
        out_main = torch.empty((M, 6288), dtype=torch.bfloat16, device=DEV)
        fa_out = torch.empty((M, 128), dtype=torch.bfloat16, device=DEV)
        out_fb = torch.empty((chain, M, 1536), dtype=torch.bfloat16, device=DEV)
        skg.run_overlap(main, fa, st["fb"], st["x"][:M], out_main, fa_out, out_fb,
                        chain=chain, aux_stream=aux, events=events)
        torch.cuda.synchronize()
        assert_parity(out_main, st["ref"][:M], st["s"][:M], f"tuned main M={M} {main.plan(M)}")
        check_links(st, M, fa_out, out_fb, chain)
    fa.close()
    main.close()
