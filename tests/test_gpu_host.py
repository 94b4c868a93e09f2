"""Attention from host memory (fa_fwd_host, fa_fwd_bwd_host): the pipelined
copies and per-slice launches give the device calls' results bit for bit,
and those match the fp64 oracle."""
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs, to_f64
from oracle import attention_bwd_gqa, attention_fwd_gqa
from gpu_helpers import assert_grad, assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def host_bufs(q, k, with_bwd):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    pin = dict(pin_memory=True)
    h = {"o": torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16).pin_memory(),
         "lse": torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()}
    if with_bwd:
        for n, shp in (("dq", (B, H, N, d)), ("dk", (B, Hkv, N, d)), ("dv", (B, Hkv, N, d))):
            h[n] = torch.full(shp, float("nan"), dtype=torch.bfloat16, **pin)
    return h


def dev_bufs(q, k, with_bwd):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    dev = torch.device("cuda")
    e = lambda shp, dt=torch.bfloat16: torch.empty(shp, dtype=dt, device=dev)  # noqa: E731
    out = {"q": e((B, H, N, d)), "k": e((B, Hkv, N, d)), "v": e((B, Hkv, N, d)), "o": e((B, H, N, d)),
           "lse": e((B, H, N), torch.float32)}
    if with_bwd:
        out.update({"dO": e((B, H, N, d)), "dq": e((B, H, N, d)), "dk": e((B, Hkv, N, d)),
                    "dv": e((B, Hkv, N, d))})
    return out


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,chunks", [
    (2, 8, 2, 300, 64, True, 3),      # 4 K/V heads over 3 slices (uneven)
    (1, 6, 6, 257, 128, False, 0),    # library default, clamped to 6 pairs
    (3, 4, 1, 129, 128, True, 2),     # multi-query: one K/V head per request
    (1, 4, 4, 640, 64, True, 1),      # a single slice
    (2, 4, 2, 200, 128, False, 64),   # more slices asked than pairs exist
])
def test_fwd_bwd_host_matches_device_calls(fa, B, H, Hkv, N, d, causal, chunks):
    q, k, v, do = make_inputs(B, H, N, d, seed=500 + N + H + chunks, Hkv=Hkv)
    host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory(), "dO": do.pin_memory()}
    host.update(host_bufs(q, k, True))
    dev = dev_bufs(q, k, True)
    ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fwd_bwd_host(host, dev, ws, causal=causal, n_chunks=chunks)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0

    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal)
    torch.cuda.synchronize()
    for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(host[name], ref.cpu()), name
        assert torch.equal(dev[name], ref), name

    scale = 1.0 / d ** 0.5
    ro, rlse = attention_fwd_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    assert_o(host["o"], ro)
    assert_lse(host["lse"], rlse)
    rdq, rdk, rdv, _ = attention_bwd_gqa(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    assert_grad(host["dq"], rdq, "dq")
    assert_grad(host["dk"], rdk, "dk")
    assert_grad(host["dv"], rdv, "dv")


@pytest.mark.parametrize("chunks", [0, 5])
def test_fwd_host_matches_device_call(fa, chunks):
    B, H, Hkv, N, d = 2, 6, 3, 1028, 64
    q, k, v = make_inputs(B, H, N, d, seed=611 + chunks, Hkv=Hkv, with_do=False)
    host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory()}
    host.update(host_bufs(q, k, False))
    dev = dev_bufs(q, k, False)
    fa.fwd_host(host, dev, causal=True, n_chunks=chunks)
    torch.cuda.synchronize()
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert torch.equal(host["o"], o.cpu())
    assert torch.equal(host["lse"], lse.cpu())


def test_host_call_is_ordered_on_the_stream(fa):
    """Work queued on the stream after the call sees the copied-back results:
    a second call that reads the first call's host outputs as its inputs
    (after a synchronise) gives the device chain's result."""
    B, H, N, d = 1, 2, 384, 128
    q, k, v = make_inputs(B, H, N, d, seed=9, with_do=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory()}
        host.update(host_bufs(q, k, False))
        dev = dev_bufs(q, k, False)
        fa.fwd_host(host, dev, causal=False, n_chunks=2)
        # queued behind the call on the same stream: reads dev["o"] after it is final
        o2 = dev["o"].clone()
    s.synchronize()
    o, _ = fa.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o2, o)
    assert torch.equal(host["o"], o.cpu())


def test_fwd_bwd_host_with_pageable_memory(fa):
    """Host buffers that are not page-locked: the copies are staged by the
    driver (no overlap) but the results are the same."""
    B, H, Hkv, N, d = 1, 4, 2, 257, 64
    q, k, v, do = make_inputs(B, H, N, d, seed=808, Hkv=Hkv)
    host = {"q": q.clone(), "k": k.clone(), "v": v.clone(), "dO": do.clone()}
    for n, shp, dt in (("o", (B, H, N, d), torch.bfloat16), ("lse", (B, H, N), torch.float32),
                       ("dq", (B, H, N, d), torch.bfloat16), ("dk", (B, Hkv, N, d), torch.bfloat16),
                       ("dv", (B, Hkv, N, d), torch.bfloat16)):
        host[n] = torch.full(shp, float("nan"), dtype=dt)
    assert not host["q"].is_pinned() and not host["o"].is_pinned()
    dev = dev_bufs(q, k, True)
    ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fwd_bwd_host(host, dev, ws, causal=True, n_chunks=2)
    torch.cuda.synchronize()
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=True)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
    torch.cuda.synchronize()
    for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(host[name], ref.cpu()), name


def test_two_host_calls_in_flight_on_two_streams(fa):
    # double buffering: calls on two streams, each with its own inputs and
    # buffers, share the library's copy streams; each must give its own
    # device calls' bits (B=2 H=8 over 2 K/V heads, N=700, causal, d=128)
    B, H, Hkv, N, d = 2, 8, 2, 700, 128
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    calls = []
    for i, s in enumerate(streams):
        q, k, v, do = make_inputs(B, H, N, d, seed=900 + i, Hkv=Hkv)
        host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory(), "dO": do.pin_memory()}
        host.update(host_bufs(q, k, True))
        dev = dev_bufs(q, k, True)
        ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
        calls.append((q, k, v, do, host, dev, ws, s))
    torch.cuda.synchronize()
    for rnd in range(3):  # several rounds, so calls of one stream meet the other's in flight
        for q, k, v, do, host, dev, ws, s in calls:
            with torch.cuda.stream(s):
                fa.fwd_bwd_host(host, dev, ws, causal=True, n_chunks=3)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for q, k, v, do, host, dev, ws, s in calls:
        qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
        o, lse = fa.fwd(qg, kg, vg, causal=True)
        dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
        torch.cuda.synchronize()
        for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.equal(host[name], ref.cpu()), name


def _draw_host_cases(n, seed):
    import random
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        d = rng.choice((64, 128))
        Hkv = rng.randint(1, 4)
        G = rng.choice((1, 1, 2, 4))
        B = rng.randint(1, 3)
        N = rng.randint(1, 900)
        chunks = rng.choice((0, 1, 2, 3, 5, 64))
        cases.append((B, Hkv * G, Hkv, N, d, rng.random() < 0.5, chunks, 600 + i))
    return cases


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,chunks,seed", _draw_host_cases(12, seed=2028))
def test_random_host_pipeline_matches_device_calls(fa, B, H, Hkv, N, d, causal, chunks, seed):
    # seeded shapes and slice counts: the pipelined call gives the device calls'
    # bits (B*H <= 48 and N <= 900 keep every slice and the whole problem below
    # the dK/dV grid at which fa_bwd switches to forming D in the dQ sweep, so
    # all take one kernel order)
    q, k, v, do = make_inputs(B, H, N, d, seed=seed, Hkv=Hkv)
    host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory(), "dO": do.pin_memory()}
    host.update(host_bufs(q, k, True))
    dev = dev_bufs(q, k, True)
    ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fwd_bwd_host(host, dev, ws, causal=causal, n_chunks=chunks)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal)
    torch.cuda.synchronize()
    for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(host[name], ref.cpu()), name
