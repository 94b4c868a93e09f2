"""Backward parity: CUDA kernels (through the C ABI) vs the fp64 CPU oracle."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import WORKLOADS, make_inputs, to_f64, workload_inputs
from oracle import attention_bwd, attention_bwd_gqa, attention_bwd_head, attention_dq_rows_head, attention_fwd
from gpu_helpers import assert_grad, assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def run_bwd(fa, q, k, v, do, causal, scale):
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 300, 513])
def test_bwd_small_shapes(fa, N, d, causal):
    q, k, v, do = make_inputs(1, 2, N, d, seed=N * 3 + d + 11)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run_bwd(fa, q, k, v, do, causal, scale)
    rdq, rdk, rdv, _ = attention_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    assert_grad(dq, rdq, "dq")
    assert_grad(dk, rdk, "dk")
    assert_grad(dv, rdv, "dv")


def test_bwd_c2(fa):
    w = WORKLOADS["c2"]
    q, k, v, do = workload_inputs("c2")
    o, lse, dq, dk, dv = run_bwd(fa, q, k, v, do, True, w.scale)
    ro, rlse = attention_fwd(to_f64(q), to_f64(k), to_f64(v), w.scale, True)
    assert_o(o, ro)
    assert_lse(lse, rlse)
    rdq, rdk, rdv, _ = attention_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), w.scale, True)
    assert_grad(dq, rdq, "dq")
    assert_grad(dk, rdk, "dk")
    assert_grad(dv, rdv, "dv")


def test_bwd_stages_match_fused_call(fa):
    """The three stage entry points in sequence equal fa_bwd (bitwise: no
    stage uses atomics), and D equals rowsum(dO * O)."""
    B, H, N, d = 1, 2, 390, 128
    q, k, v, do = make_inputs(B, H, N, d, seed=21)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=True)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
    Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq2, dk2, dv2 = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
    fa.bwd_preprocess(o, dog, Dvec)
    fa.bwd_dkdv(qg, kg, vg, dog, lse, Dvec, dk2, dv2, causal=True)
    fa.bwd_dq(qg, kg, vg, dog, lse, Dvec, dq2, causal=True)
    torch.cuda.synchronize()
    ref_D = (dog.double() * o.double()).sum(-1)
    assert torch.allclose(Dvec.double(), ref_D, atol=1e-3, rtol=1e-3)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(dq, dq2)


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", [
    (1, 2, 2, 300, 128, True),
    (2, 3, 3, 129, 64, False),
    (1, 4, 2, 257, 128, True),   # grouped-query heads: D for every query head
])
def test_bwd_dq_d_then_dkdv_vs_oracle(fa, B, H, Hkv, N, d, causal):
    """The dQ sweep that forms D itself (no preprocess), then the dK/dV
    sweep reading that D: D against rowsum(dO ∘ O) of the GPU's own O, the
    gradients against the oracle."""
    q, k, v, do = make_inputs(B, H, N, d, seed=B * 31 + H + N + d, Hkv=Hkv)
    scale = d ** -0.5
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal, scale=scale)
    Dvec = torch.full((B, H, N), float("nan"), device=dev)
    dq, dk, dv = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
    fa.bwd_dq_d(qg, kg, vg, o, dog, lse, Dvec, dq, causal=causal, scale=scale)
    fa.bwd_dkdv(qg, kg, vg, dog, lse, Dvec, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    ref_D = (dog.double() * o.double()).sum(-1)
    assert torch.allclose(Dvec.double(), ref_D, atol=1e-4, rtol=1e-5)
    rdq, rdk, rdv, _ = attention_bwd_gqa(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    assert_grad(dq, rdq, "dq")
    assert_grad(dk, rdk, "dk")
    assert_grad(dv, rdv, "dv")


def test_bwd_fused_order_matches_its_stages(fa):
    """Where fa_bwd forms D inside the dQ sweep (one K/V head per query head,
    a dK/dV grid of at least 4 CTAs per SM), it equals bwd_dq_d then
    bwd_dkdv bit for bit; below the threshold it takes the D pass."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, N, d = 1, 4 * sms // 8 + 8, 1024, 64  # 8 key tiles per head
    assert fa.bwd_fuses_d(B, H, H, N, d) and not fa.bwd_fuses_d(1, 2, 2, N, d)
    assert not fa.bwd_fuses_d(B, H, H // 2, N, d)  # grouped-query heads
    q, k, v, do = make_inputs(B, H, N, d, seed=5)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=True)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
    Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq2, dk2, dv2 = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
    fa.bwd_dq_d(qg, kg, vg, o, dog, lse, Dvec, dq2, causal=True)
    fa.bwd_dkdv(qg, kg, vg, dog, lse, Dvec, dk2, dv2, causal=True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_bwd_deterministic(fa):
    """No atomics anywhere in the backward: repeated runs are bitwise equal."""
    q, k, v, do = make_inputs(2, 3, 700, 128, seed=8)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=True)
    r1 = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
    r2 = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_bwd_invariants(fa):
    """Σ_j dK_j = 0 and Σ_j dV_j = Σ_i dO_i per head (within bf16 rounding)."""
    B, H, N, d = 1, 2, 640, 64
    q, k, v, do = make_inputs(B, H, N, d, seed=31)
    _, _, dq, dk, dv = run_bwd(fa, q, k, v, do, True, 1.0 / d ** 0.5)
    assert dk.double().sum(2).abs().max().item() < 0.1
    assert (dv.double().sum(2) - do.to("cuda").double().sum(2)).abs().max().item() < 0.2


def test_bwd_c4_sampled(fa):
    """Full-size Llama-shaped workload in the benchmark's launch configuration:
    one head's dK/dV in full and sampled dQ rows of three heads."""
    w = WORKLOADS["c4"]
    q, k, v, do = workload_inputs("c4")
    o, lse, dq, dk, dv = run_bwd(fa, q, k, v, do, True, w.scale)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    b, h = 1, 7
    rdq, rdk, rdv, _ = attention_bwd_head(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]),
                                          to_f64(do[b, h]), w.scale, True)
    assert_grad(dk[b, h].cpu(), rdk, "dk")
    assert_grad(dv[b, h].cpu(), rdv, "dv")
    assert_grad(dq[b, h].cpu(), rdq, "dq")
    rows = np.array([0, 1, 127, 128, 4095, 4096, 8190, 8191])
    for b, h in [(0, 0), (1, 31)]:
        rq, _ = attention_dq_rows_head(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]),
                                       to_f64(do[b, h]), w.scale, True, rows)
        assert_grad(dq[b, h, rows].cpu(), rq, f"dq[{b},{h}]")


@pytest.mark.parametrize("d", [64, 128])
def test_many_heads_one_ragged_tile(fa, d):
    """2048 (batch, head) pairs of N = 70 (one ragged tile each), with K/V
    heads shared by pairs of query heads: head indexing over a large grid."""
    from oracle import attention_bwd_gqa, attention_fwd_gqa
    B, H, Hkv, N = 64, 32, 16, 70
    q, k, v, do = make_inputs(B, H, N, d, seed=2048 + d, Hkv=Hkv)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    scale = 1.0 / d ** 0.5
    for causal in (False, True):
        o, lse = fa.fwd(qg, kg, vg, causal=causal)
        dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal)
        torch.cuda.synchronize()
        assert fa.last_device_error() == 0
        ro, rlse = attention_fwd_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
        assert_o(o, ro)
        assert_lse(lse, rlse)
        rdq, rdk, rdv, _ = attention_bwd_gqa(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
        assert_grad(dq, rdq, "dq")
        assert_grad(dk, rdk, "dk")
        assert_grad(dv, rdv, "dv")
