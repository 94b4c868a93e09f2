"""Numerical corners of the attention path against the fp64 oracle: scales
other than 1/sqrt(d), and strongly peaked scores whose row maximum keeps
outgrowing the kernel's exponent reference (so the forward raises it, and
rescales O and the running sum, on tiles after the first)."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs, to_f64
from oracle import attention_bwd_gqa, attention_fwd_gqa
from gpu_helpers import assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def bf16_rounding_yardstick(q, k, v, do, scale, causal):
    """Gradients computed plainly in fp64 except for the roundings the path
    makes by design: the forward's output O is stored in bf16 and D is the row
    sum of dO∘O over that stored O; P and dS are rounded to bf16 before they
    enter the products (dV = Pᵀ dO, dK = scale·dSᵀ Q, dQ = scale·dS K). Its
    distance to the oracle is the error those roundings alone cause on these
    inputs."""
    qd, kd, vd, dd = (torch.from_numpy(to_f64(t)) for t in (q, k, v, do))
    H, Hkv = qd.shape[1], kd.shape[1]
    kd = kd.repeat_interleave(H // Hkv, dim=1)
    vd = vd.repeat_interleave(H // Hkv, dim=1)
    s = qd @ kd.transpose(-1, -2) * scale
    if causal:
        n = s.shape[-1]
        s = s.masked_fill(~torch.ones(n, n, dtype=torch.bool).tril(), float("-inf"))
    p = torch.softmax(s, dim=-1)
    pb = p.to(torch.bfloat16).to(torch.float64)
    dv = pb.transpose(-1, -2) @ dd
    dp = dd @ vd.transpose(-1, -2)
    ob = (p @ vd).to(torch.bfloat16).to(torch.float64)
    D = (dd * ob).sum(-1, keepdim=True)
    dsb = (p * (dp - D)).to(torch.bfloat16).to(torch.float64)
    dq = scale * dsb @ kd
    dk = scale * dsb.transpose(-1, -2) @ qd
    g = H // Hkv
    B, _, N, d = kd.shape
    dk = dk.view(B, Hkv, g, N, d).sum(2)
    dv = dv.view(B, Hkv, g, N, d).sum(2)
    return dq.numpy(), dk.numpy(), dv.numpy()


def check(fa, q, k, v, do, scale, causal):
    """o and lse within the fixed parity bounds. Gradients within those bounds
    too, or, where the gradients are large (peaked scores, big scales), within
    twice the error that the path's designed bf16 roundings alone cause (plus
    0.1% of the largest gradient): the fixed 5e-2 bound is set for the
    benchmark inputs, whose gradients are O(1)."""
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    ro, rlse = attention_fwd_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    assert_o(o, ro)
    assert_lse(lse, rlse)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    ref = attention_bwd_gqa(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)[:3]
    yard = bf16_rounding_yardstick(q, k, v, do, scale, causal)
    for name, got, r, y in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, yard):
        err = float(np.abs(to_f64(got) - r).max())
        if err <= 5e-2:
            continue
        bound = 2.0 * float(np.abs(y - r).max()) + 1e-3 * float(np.abs(r).max())
        assert err <= bound, f"{name}: max-abs {err} > {bound} (bf16-rounding yardstick)"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [0.02, 0.3])
def test_scales_other_than_inverse_sqrt_d(fa, d, scale):
    q, k, v, do = make_inputs(1, 4, 333, d, seed=int(scale * 1000) + d, Hkv=2)
    for causal in (False, True):
        check(fa, q, k, v, do, scale, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_peaked_scores_raise_the_reference_after_the_first_tile(fa, d, causal):
    # q ~ N(0, 8²): scaled scores have a standard deviation of 8 (11.5 in
    # log2 units), so the row maximum grows past the reference by more
    # than its 2^8 threshold on many tiles after the first.
    B, H, N = 1, 2, 1100
    q, k, v, do = make_inputs(B, H, N, d, seed=77 + d, q_std=8.0)
    scale = 1.0 / d ** 0.5
    qd, kd = to_f64(q), to_f64(k)
    s = np.einsum("bhid,bhjd->bhij", qd, kd) * scale * np.log2(np.e)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    tile_max = np.stack([s[..., t:t + 128].max(-1) for t in range(0, N, 128)], -1)
    running = np.maximum.accumulate(tile_max, axis=-1)
    # the scenario holds: on some row a later tile beats the first tile by > 8
    assert np.any(running[..., 1:] - tile_max[..., :1] > 8)
    check(fa, q, k, v, do, scale, causal)
