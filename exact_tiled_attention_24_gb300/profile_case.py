"""Run the forward + backward a few times on one shape, for profiler captures.

    python -m exact_tiled_attention_24_gb300.profile_case --B 1 --H 32 --N 4096 --d 128 \
        --causal --iters 2 [--Hkv 8] [--fwd-only] [--q-std 4]
    python -m exact_tiled_attention_24_gb300.profile_case --softmax-rows 1216 --softmax-n 262144
    python -m exact_tiled_attention_24_gb300.profile_case --decode d1

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
    ap.add_argument("--q-std", type=float, default=1.0, help="standard deviation of q (c5 draws 4)")
    ap.add_argument("--Hkv", type=int, default=0, help="K/V heads (grouped-query); 0 = H")
    ap.add_argument("--softmax-rows", type=int, default=0, help="run the row softmax kernels instead")
    ap.add_argument("--softmax-n", type=int, default=262144)
    ap.add_argument("--decode", default="", help="run a decode workload (e.g. d1) instead")
    args = ap.parse_args()

    import torch

    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300 import build
    from exact_tiled_attention_24_gb300.workloads import DECODE_WORKLOADS, make_decode, make_inputs, make_rows

    build.build()
    dev = torch.device("cuda")
    if args.decode:
        dw = DECODE_WORKLOADS[args.decode]
        q, kc, vc, table, lens = make_decode(dw, dev)
        for _ in range(args.iters):
            fa.decode_paged(q, kc, vc, table, lens, n_splits=dw.n_splits)
        torch.cuda.synchronize()
        if fa.last_device_error() != 0:
            raise SystemExit("device error")
        print("ok")
        return
    if args.softmax_rows:
        x = make_rows(args.softmax_rows, args.softmax_n, seed=99, std=4.0).to(dev)
        y = torch.empty_like(x)
        for _ in range(args.iters):
            fa.softmax_online(x, out=y)
            fa.softmax_safe(x, out=y)
        torch.cuda.synchronize()
        print("ok")
        return
    q, k, v, do = (t.to(dev) for t in make_inputs(args.B, args.H, args.N, args.d, seed=99,
                                                   q_std=args.q_std, Hkv=args.Hkv or None))
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
