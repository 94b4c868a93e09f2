"""Grouped-query attention parity: CUDA kernels (through the C ABI) vs the
fp64 CPU oracle, with K/V heads shared by groups of consecutive query heads."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs, to_f64
from oracle import attention_bwd_gqa, attention_bwd_head, attention_fwd_gqa, attention_fwd_head
from gpu_helpers import assert_grad, assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def run(fa, q, k, v, do, causal, scale):
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", [
    (2, 8, 2, 300, 64, True),
    (2, 8, 2, 300, 64, False),
    (1, 8, 1, 257, 128, True),     # one K/V head for all (multi-query)
    (1, 6, 3, 129, 128, False),
    (1, 4, 4, 200, 64, True),      # groups of one: plain multi-head
    (1, 16, 4, 640, 128, True),
])
def test_gqa_fwd_bwd_small(fa, B, H, Hkv, N, d, causal):
    q, k, v, do = make_inputs(B, H, N, d, seed=H * 7 + Hkv + N + d, Hkv=Hkv)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run(fa, q, k, v, do, causal, scale)
    ro, rlse = attention_fwd_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    assert_o(o, ro)
    assert_lse(lse, rlse)
    rdq, rdk, rdv, _ = attention_bwd_gqa(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    assert_grad(dq, rdq, "dq")
    assert_grad(dk, rdk, "dk")
    assert_grad(dv, rdv, "dv")


def test_gqa_stages_match_fused_call(fa):
    """The stage entry points with grouped heads equal fa_bwd_gqa bitwise."""
    B, H, Hkv, N, d = 1, 8, 2, 390, 128
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, N, d, seed=77, Hkv=Hkv))
    o, lse = fa.fwd(q, k, v, causal=True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
    Dv = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.bwd_preprocess(o, do, Dv)
    fa.bwd_dkdv(q, k, v, do, lse, Dv, dk2, dv2, causal=True)
    fa.bwd_dq(q, k, v, do, lse, Dv, dq2, causal=True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_gqa_rejects_bad_head_counts(fa):
    q = torch.zeros((1, 6, 64, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 4, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fwd(q, k, k)


def test_gqa_llama_heads_sampled(fa):
    """32 query heads over 8 K/V heads at N = 2048, d = 128, causal: O and lse
    of sampled query heads, and dK, dV of one K/V head (the sum over its four
    query heads), against the oracle; dV summed over keys equals dO summed
    over the group (P rows sum to one)."""
    B, H, Hkv, N, d = 1, 32, 8, 2048, 128
    G = H // Hkv
    scale = d ** -0.5
    q, k, v, do = make_inputs(B, H, N, d, seed=4242, Hkv=Hkv)
    o, lse, dq, dk, dv = run(fa, q, k, v, do, True, scale)
    qf, kf, vf, dof = (to_f64(t) for t in (q, k, v, do))
    for h in (0, 5, 31):
        g = h // G
        ro, rlse = attention_fwd_head(qf[0, h], kf[0, g], vf[0, g], scale, True)
        assert_o(o[0, h], ro, f"o head {h}")
        assert_lse(lse[0, h], rlse)
    g = 3
    rdk = np.zeros((N, d))
    rdv = np.zeros((N, d))
    for h in range(g * G, (g + 1) * G):
        rdq, dkh, dvh, _ = attention_bwd_head(qf[0, h], kf[0, g], vf[0, g], dof[0, h], scale, True)
        rdk += dkh
        rdv += dvh
        assert_grad(dq[0, h], rdq, f"dq head {h}")
    assert_grad(dk[0, g], rdk, "dk")
    assert_grad(dv[0, g], rdv, "dv")
    dv_sum = to_f64(dv).sum(axis=2)
    do_sum = dof.reshape(B, Hkv, G, N, d).sum(axis=(2, 3))
    np.testing.assert_allclose(dv_sum, do_sum, rtol=0, atol=0.5)
