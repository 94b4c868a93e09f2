"""fa_bwd_noalloc: the backward for callers that cannot allocate device
memory (hosts whose device memory all belongs to their own fixed pool and
that give a plug-in no allocator, runtimes that forbid allocation after
start-up, code that cannot take cudaMalloc's implicit synchronisation).

It takes no workspace: its scratch is a fixed-size array inside the library.
These tests call it through the C ABI and compare it with fa_bwd, which
takes a caller-provided workspace, on two calls in a row (the second call
sees the array holding the first call's contents). This file is collected
last so that a failure here does not hide the other tests.
"""
import ctypes

import pytest
import torch

import exact_tiled_attention_24_gb300 as fa
from exact_tiled_attention_24_gb300 import build as fabuild
from exact_tiled_attention_24_gb300.workloads import make_inputs
from gpu_helpers import TOL_GRAD

SCRATCH_BYTES = 32 * 1024 * 1024  # FA_BWD_NOALLOC_SCRATCH_BYTES in include/fa.h


@pytest.fixture(scope="module")
def L():
    fabuild.build()
    return fa.lib()


def test_noalloc_rejects_problems_larger_than_its_scratch(L):
    """Checked on the host before any launch: B=64 H=64 N=4096 needs 64 MiB
    of scratch (one fp32 per query row), more than the 32 MiB array."""
    fake = ctypes.c_void_p(0x10000)
    assert fa.bwd_workspace_bytes(64, 64, 4096, 128) > SCRATCH_BYTES
    st = L.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                          64, 64, 4096, 128, 0.088, 1, ctypes.c_void_p(0))
    assert st == 6  # FA_ERR_WORKSPACE
    assert L.fa_bwd_noalloc(fake, fake, fake, fake, fake, ctypes.c_void_p(0), fake, fake, fake,
                            1, 1, 64, 64, 0.125, 0, ctypes.c_void_p(0)) == 1


def _call_noalloc(L, q, k, v, o, lse, do, causal):
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.fa_bwd_noalloc(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv),
                          B, H, N, d, 1.0 / d ** 0.5, int(causal),
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_two_calls_in_a_row(L):
    dev = torch.device("cuda")
    cases = [((2, 3, 700, 128), True, 41), ((1, 4, 1028, 64), False, 42)]
    for (B, H, N, d), causal, seed in cases:
        q, k, v, do = (t.to(dev) for t in make_inputs(B, H, N, d, seed=seed))
        o, lse = fa.fwd(q, k, v, causal=causal)
        ref = fa.bwd(q, k, v, o, lse, do, causal=causal)
        got = _call_noalloc(L, q, k, v, o, lse, do, causal)
        torch.cuda.synchronize()
        assert fa.last_device_error() == 0
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            err = (a.float() - b.float()).abs().max().item()
            assert err <= TOL_GRAD, f"{name} (N={N}, d={d}): max-abs {err}"
        # the backward uses no atomics: identical to the workspace path
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


@pytest.mark.gpu
def test_noalloc_call_captures_into_a_graph(L):
    # after an eager first call, a captured call (the scratch address looked up
    # inside the capture) replays to the same bits as fa_bwd
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in make_inputs(1, 4, 300, 128, seed=43))
    o, lse = fa.fwd(q, k, v, causal=True)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True)
    _call_noalloc(L, q, k, v, o, lse, do, True)
    torch.cuda.synchronize()
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st = L.fa_bwd_noalloc(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv),
                                  1, 4, 300, 128, 1.0 / 128 ** 0.5, 1,
                                  ctypes.c_void_p(s.cuda_stream))
    assert st == 0
    for t in (dq, dk, dv):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for a, b in zip((dq, dk, dv), ref):
        assert torch.equal(a, b)
