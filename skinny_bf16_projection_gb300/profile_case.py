"""Run one projection configuration a few times, for profilers (ncu).

    python -m skinny_bf16_projection_gb300.profile_case --N 3584 --K 7168 --M 8 \
        [--out bf16|fp32] [--tactic tc:r128:t16:b2:s4:c8 | --use-tactic-file] \
        [--launches 4] [--copies 1]
    python -m skinny_bf16_projection_gb300.profile_case --overlap --M 1 \
        --tactic <main tactic> --fa-tactic <F_A tactic> [--launches 3]

Launches are plain stream launches (no graph), so each one is a separate
kernel for the profiler.  With --copies > 1 the launches rotate over that
many copies of the weight.  --use-tactic-file takes the plan from the file
named by SKINNY_GEMM_TACTIC_FILE (what the autotuner wrote there).
--overlap runs the two-stream decode step (packed W[6288, 7168] on the main
stream, F_A = its first 128 rows then F_B W[1536, 128] on an aux stream),
once per launch; per step the launch order is F_A, F_B, main.  Prints the
tactics used.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--N", type=int, default=3584)
    ap.add_argument("--K", type=int, default=7168)
    ap.add_argument("--M", type=int, default=8)
    ap.add_argument("--out", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--tactic", default=None)
    ap.add_argument("--use-tactic-file", action="store_true")
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--copies", type=int, default=1)
    ap.add_argument("--overlap", action="store_true")
    ap.add_argument("--fa-tactic", default=None)
    args = ap.parse_args()

    import projection_inputs as pin
    import skinny_bf16_projection_gb300 as skg
    from skinny_bf16_projection_gb300 import build
    build.build()

    dev = torch.device("cuda:0")
    odt = torch.bfloat16 if args.out == "bf16" else torch.float32
    if args.overlap:
        args.N = 6288
    w, x = pin.case(args.N, args.K, seed=0)
    wd = w.to(dev)
    ws = [wd] + [wd.clone() for _ in range(args.copies - 1)]
    projs = [skg.Projection(t, odt, use_tactic_file=args.use_tactic_file) for t in ws]
    if args.tactic:
        for p in projs:
            p.set_tactic(args.M, args.tactic)
    xd = x[:args.M].to(dev)
    out = torch.empty((args.M, args.N), dtype=odt, device=dev)
    torch.cuda.synchronize()
    if args.overlap:
        fa = skg.Projection(wd[:128], use_tactic_file=False)
        if args.fa_tactic:
            fa.set_tactic(args.M, args.fa_tactic)
        fb = skg.Projection(pin.weight(1536, 128, seed=1).to(dev), use_tactic_file=False)
        aux = torch.cuda.Stream(priority=-1)
        ev = (torch.cuda.Event(), torch.cuda.Event())
        fo = torch.empty((args.M, 128), dtype=torch.bfloat16, device=dev)
        fbo = torch.empty((1, args.M, 1536), dtype=torch.bfloat16, device=dev)
        for i in range(args.launches):
            skg.run_overlap(projs[i % len(projs)], fa, fb, xd, out, fo, fbo, chain=1,
                            aux_stream=aux, events=ev)
        torch.cuda.synchronize()
        print(f"profile_case overlap M={args.M} main={projs[0].plan(args.M)} "
              f"fa={fa.plan(args.M)} fb={fb.plan(args.M)} steps={args.launches}")
        return 0
    for i in range(args.launches):
        projs[i % len(projs)].run(xd, out)
    torch.cuda.synchronize()
    for p in projs:
        p.check_status()
    print(f"profile_case N={args.N} K={args.K} M={args.M} out={args.out} "
          f"tactic={projs[0].plan(args.M)} launches={args.launches}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
