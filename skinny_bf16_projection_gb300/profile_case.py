"""Run one projection configuration a few times, for profilers (ncu).

    python -m skinny_bf16_projection_gb300.profile_case --N 3584 --K 7168 --M 8 \
        [--out bf16|fp32] [--tactic tc:r128:t16:b2:s4:c8] [--launches 4] [--copies 1]

Launches are plain stream launches (no graph), so each one is a separate
kernel for the profiler.  With --copies > 1 the launches rotate over that
many copies of the weight.  Prints the tactic used.
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
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--copies", type=int, default=1)
    args = ap.parse_args()

    import projection_inputs as pin
    import skinny_bf16_projection_gb300 as skg
    from skinny_bf16_projection_gb300 import build
    build.build()

    dev = torch.device("cuda:0")
    odt = torch.bfloat16 if args.out == "bf16" else torch.float32
    w, x = pin.case(args.N, args.K, seed=0)
    wd = w.to(dev)
    ws = [wd] + [wd.clone() for _ in range(args.copies - 1)]
    projs = [skg.Projection(t, odt, use_tactic_file=False) for t in ws]
    if args.tactic:
        for p in projs:
            p.set_tactic(args.M, args.tactic)
    xd = x[:args.M].to(dev)
    out = torch.empty((args.M, args.N), dtype=odt, device=dev)
    torch.cuda.synchronize()
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
