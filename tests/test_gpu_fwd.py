"""Forward parity: CUDA kernels (through the C ABI) vs the fp64 CPU oracle on
the same seeded bf16 inputs."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import WORKLOADS, make_inputs, to_f64, workload_inputs
from oracle import attention_fwd, attention_fwd_head
from gpu_helpers import assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def run_full(fa, q, k, v, causal, scale):
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    ro, rlse = attention_fwd(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    assert_o(o, ro)
    assert_lse(lse, rlse)
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 255, 256, 300, 513])
def test_fwd_small_shapes(fa, N, d, causal):
    q, k, v = make_inputs(1, 2, N, d, seed=N * 7 + d, with_do=False)
    run_full(fa, q, k, v, causal, 1.0 / d ** 0.5)


def test_fwd_c1(fa):
    w = WORKLOADS["c1"]
    q, k, v = workload_inputs("c1")
    run_full(fa, q, k, v, False, w.scale)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_c3_ragged(fa, causal):
    w = WORKLOADS["c3"]
    q, k, v = workload_inputs("c3")
    run_full(fa, q, k, v, causal, w.scale)


def test_fwd_c2(fa):
    w = WORKLOADS["c2"]
    q, k, v, _ = workload_inputs("c2")
    run_full(fa, q, k, v, True, w.scale)


def sampled_rows(N, n_tiles=4):
    rows = set()
    for t in [0, 1, N // 256, N // 128 - 1]:
        base = t * 128
        rows.update(r for r in (base, base + 1, base + 63, base + 127) if r < N)
    rows.update([N - 1, N // 2])
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["c4", "c5"])
def test_fwd_full_size_sampled_rows(fa, name):
    """Full-size workloads in the benchmark's launch configuration; the
    oracle computes sampled rows of a few heads exactly."""
    w = WORKLOADS[name]
    q, k, v = workload_inputs(name, with_do=False)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = sampled_rows(w.N)
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (0, w.H // 2)]:
        ro, rlse = attention_fwd_head(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]), w.scale,
                                      True, rows=rows)
        assert_o(o[b, h, rows].cpu(), ro, what=f"o[{b},{h}]")
        assert_lse(lse[b, h, rows].cpu(), rlse)


def test_fwd_deterministic(fa):
    q, k, v = make_inputs(2, 3, 700, 128, seed=5, with_do=False)
    dev = torch.device("cuda")
    qg, kg, vg = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = fa.fwd(qg, kg, vg, causal=True)
    o2, l2 = fa.fwd(qg, kg, vg, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_canary_guard(fa, d):
    """Outputs sit at the start of larger buffers filled with a sentinel: the
    padding after o and lse must be untouched (ragged N, causal)."""
    B, H, N = 2, 3, 1028
    q, k, v = make_inputs(B, H, N, d, seed=77, with_do=False)
    dev = torch.device("cuda")
    pad = 4096
    obuf = torch.full((B * H * N * d + pad,), 7.0, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((B * H * N + pad,), -3.0, dtype=torch.float32, device=dev)
    o = obuf[: B * H * N * d].view(B, H, N, d)
    lse = lbuf[: B * H * N].view(B, H, N)
    fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(obuf[B * H * N * d:] == 7.0)
    assert torch.all(lbuf[B * H * N:] == -3.0)
    ro, rlse = attention_fwd(to_f64(q), to_f64(k), to_f64(v), 1.0 / d ** 0.5, True)
    assert_o(o, ro)
    assert_lse(lse, rlse)


def test_fwd_closed_form_zero_queries(fa):
    """Q = 0: O is the prefix mean of V and lse = ln(i+1) (causal)."""
    B, H, N, d = 1, 2, 300, 64
    _, k, v = make_inputs(B, H, N, d, seed=9, with_do=False)
    q = torch.zeros_like(k)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    vv = to_f64(v)
    prefix = np.cumsum(vv, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    assert_o(o, prefix)
    assert_lse(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), (B, H, N)))


def test_fwd_misaligned_pointer_rejected(fa):
    q, k, v = make_inputs(1, 1, 64, 64, seed=1, with_do=False)
    dev = torch.device("cuda")
    buf = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device=dev)
    qm = buf[1: 1 + 64 * 64].view(1, 1, 64, 64)
    with pytest.raises(fa.FAError) as e:
        fa.fwd(qm, k.to(dev), v.to(dev))
    assert e.value.status == 3


def test_fwd_long_context_sampled_rows(fa):
    """N = 131072 (four times the longest benchmark context) on two heads:
    TMA coordinates, tile counts and the causal bound at the largest N the
    tests reach; sampled rows against the oracle."""
    B, H, N, d = 1, 2, 131072, 128
    q, k, v = make_inputs(B, H, N, d, seed=1313, with_do=False)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    rows = np.array(sorted({0, 1, 127, 128, 65535, 65536, 100001, N - 129, N - 128, N - 2, N - 1}))
    for h in range(H):
        ro, rlse = attention_fwd_head(to_f64(q[0, h]), to_f64(k[0, h]), to_f64(v[0, h]), 1.0 / d ** 0.5,
                                      True, rows=rows)
        assert_o(o[0, h, rows].cpu(), ro, what=f"o[0,{h}]")
        assert_lse(lse[0, h, rows].cpu(), rlse)
