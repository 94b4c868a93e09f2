"""Cases run through both library flavours (release and the bounds-checked
FA_DEBUG build) by tests/test_gpu_debug_build.py: every kernel family on
valid inputs, ragged sizes included. Run as a script it writes the results
of the library selected by FA_DEBUG_LIBRARY to the file named on the
command line."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def run_cases():
    """Results of every case as {name: CPU tensor}; asserts no device error."""
    import exact_tiled_attention_24_gb300 as fa
    from exact_tiled_attention_24_gb300.workloads import make_inputs

    dev = torch.device("cuda")
    out = {}

    def check(name):
        torch.cuda.synchronize()
        status = fa.last_device_error()
        assert status == 0, f"{name}: device status {fa.FA_STATUS.get(status, status)}"

    # attention forward + backward: ragged N, both head dims, causal and not,
    # grouped-query heads
    for (B, H, Hkv, N, d) in ((1, 2, 2, 300, 64), (2, 4, 2, 257, 128), (1, 2, 1, 129, 128)):
        q, k, v, do = (t.to(dev) for t in make_inputs(B, H, N, d, seed=500 + N + d, Hkv=Hkv))
        for causal in (False, True):
            o, lse = fa.fwd(q, k, v, causal=causal)
            dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal)
            tag = f"attn_{B}_{H}_{Hkv}_{N}_{d}_{int(causal)}"
            check(tag)
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
                out[f"{tag}_{n}"] = t.cpu()
            # the dQ sweep that forms D itself, then dK/dV reading that D
            Dv = torch.empty((B, H, N), device=dev)
            dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            fa.bwd_dq_d(q, k, v, o, do, lse, Dv, dq2, causal=causal)
            fa.bwd_dkdv(q, k, v, do, lse, Dv, dk2, dv2, causal=causal)
            check(tag + "_dq_d")
            for n, t in (("D", Dv), ("dq", dq2), ("dk", dk2), ("dv", dv2)):
                out[f"{tag}_dq_d_{n}"] = t.cpu()
    # row softmax: vector (n % 4 == 0) and scalar paths
    g = torch.Generator().manual_seed(7)
    for rows, n in ((5, 1000), (3, 1001)):
        x = (torch.randn((rows, n), generator=g) * 4).to(dev)
        out[f"softmax_online_{rows}_{n}"] = fa.softmax_online(x).cpu()
        out[f"softmax_safe_{rows}_{n}"] = fa.softmax_safe(x).cpu()
        check(f"softmax_{rows}_{n}")
    # partial-attention merge and paged decode
    o_parts = torch.randn((3, 40, 128), generator=g).to(dev)
    lse_parts = (torch.randn((3, 40), generator=g) * 3).to(dev)
    mo, ml = fa.attn_merge(o_parts, lse_parts)
    check("merge")
    out["merge_o"], out["merge_lse"] = mo.cpu(), ml.cpu()
    # paged decode: TMA boxes (16-token blocks) and per-token gathering
    # (3: table entries loaded ahead; 24: looked up per tile)
    for bs in (16, 3, 24):
        B, H, Hkv, d = 3, 8, 2, 128
        lens = [37, 1, 160]
        nb = [(L + bs - 1) // bs for L in lens]
        total = sum(nb) + 2
        qd = torch.randn((B, H, d), generator=g).to(torch.bfloat16).to(dev)
        kc = torch.randn((total, Hkv, bs, d), generator=g).to(torch.bfloat16).to(dev)
        vc = torch.randn((total, Hkv, bs, d), generator=g).to(torch.bfloat16).to(dev)
        perm = torch.randperm(total, generator=g)
        table = torch.zeros((B, max(nb)), dtype=torch.int32)
        pos = 0
        for b in range(B):
            table[b, :nb[b]] = perm[pos:pos + nb[b]].to(torch.int32)
            pos += nb[b]
        od, ld = fa.decode_paged(qd, kc, vc, table.to(dev), torch.tensor(lens, dtype=torch.int32).to(dev),
                                 n_splits=3)
        check(f"decode_bs{bs}")
        out[f"decode_bs{bs}_o"], out[f"decode_bs{bs}_lse"] = od.cpu(), ld.cpu()
    return out


def main(path):
    import exact_tiled_attention_24_gb300 as fa
    assert fa.debug_checks() == (os.environ.get("FA_DEBUG_LIBRARY") == "1")
    torch.save(run_cases(), path)


if __name__ == "__main__":
    main(sys.argv[1])
