"""Run the forward + backward a few times on one shape, for profiler captures.

    python -m exact_tiled_attention_24_gb300.profile_case --B 1 --H 32 --N 4096 --d 128 \
        --causal --iters 2

Inputs come from the seeded workload generator; nothing is checked or timed.
"""
from __future__ import annotations

import argparse


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--fwd-only", action="store_true")
    args = ap.parse_args()

    import torch

    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300 import build
    from exact_tiled_attention_24_gb300.workloads import make_inputs

    build.build()
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in make_inputs(args.B, args.H, args.N, args.d, seed=99))
    for _ in range(args.iters):
        o, lse = fa.fwd(q, k, v, causal=args.causal)
        if not args.fwd_only:
            fa.bwd(q, k, v, o, lse, do, causal=args.causal)
    torch.cuda.synchronize()
    if fa.last_device_error() != 0:
        raise SystemExit("device error")
    print("ok")


if __name__ == "__main__":
    main()
