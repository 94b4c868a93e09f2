"""Numerical corners of the attention path against the fp64 oracle: scales
other than 1/sqrt(d), and strongly peaked scores whose row maximum keeps
outgrowing the kernel's exponent reference (so the forward raises it, and
rescales O and the running sum, on tiles after the first)."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs, to_f64
from oracle import attention_bwd_gqa, attention_fwd_gqa
from gpu_helpers import assert_grad_scaled, assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def check(fa, q, k, v, do, scale, causal):
    """o and lse within the fixed parity bounds; gradients against the oracle
    within the fixed bound or, where they are larger than unit scale (big
    scales, peaked scores), within 2^-6 of their largest entry."""
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
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad_scaled(got, r, name)


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
