"""The library's calls are capturable into a CUDA graph: each entry point only
launches on the caller's stream (the host pipeline also records and waits on
events, which joins its copy streams to the capture), so a captured step
replays to the same bits as the eager calls."""
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


@pytest.mark.parametrize("d,Hkv", [(64, 4), (128, 2)])
def test_fwd_bwd_graph_replay_matches_eager(fa, d, Hkv):
    B, H, N = 2, 4, 777
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, N, d, seed=4242 + d, Hkv=Hkv))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dvec = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        fa.fwd(q, k, v, causal=True, out=o, lse=lse)
        fa.bwd_preprocess(o, do, dvec)
        fa.bwd_dkdv(q, k, v, do, lse, dvec, dk, dv, causal=True)
        fa.bwd_dq(q, k, v, do, lse, dvec, dq, causal=True)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture (module load, attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for name, got, want in zip(("o", "lse", "dq", "dk", "dv"), (o, lse, dq, dk, dv), ref):
        assert torch.equal(got, want), name


def test_host_pipeline_graph_replay_matches_eager(fa):
    B, H, Hkv, N, d = 2, 4, 2, 300, 128
    q, k, v, do = make_inputs(B, H, N, d, seed=99, Hkv=Hkv)
    host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory(), "dO": do.pin_memory()}
    for n, shp, dt in (("o", (B, H, N, d), torch.bfloat16), ("lse", (B, H, N), torch.float32),
                       ("dq", (B, H, N, d), torch.bfloat16), ("dk", (B, Hkv, N, d), torch.bfloat16),
                       ("dv", (B, Hkv, N, d), torch.bfloat16)):
        host[n] = torch.empty(shp, dtype=dt).pin_memory()
    dev = {n: torch.empty(host[n].shape, dtype=host[n].dtype, device="cuda") for n in host}
    ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.fwd_bwd_host(host, dev, ws, causal=True, n_chunks=3)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = {n: host[n].clone() for n in ("o", "lse", "dq", "dk", "dv")}
    for n in ref:
        host[n].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fwd_bwd_host(host, dev, ws, causal=True, n_chunks=3)
    g.replay()
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for n, want in ref.items():
        assert torch.equal(host[n], want), n


def test_fused_backward_graph_replay_matches_eager(fa):
    """fa.bwd forks the dQ sweep onto the library's side stream and joins it
    back; captured, it replays to the eager result."""
    B, H, Hkv, N, d = 1, 4, 2, 500, 128
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, N, d, seed=31, Hkv=Hkv))
    o, lse = fa.fwd(q, k, v, causal=True)
    ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    ref = fa.bwd(q, k, v, o, lse, do, causal=True, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    outs = {}
    with torch.cuda.stream(s):
        outs["warm"] = fa.bwd(q, k, v, o, lse, do, causal=True, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs["graph"] = fa.bwd(q, k, v, o, lse, do, causal=True, workspace=ws)
    for t in outs["graph"]:
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for name, got, want in zip(("dq", "dk", "dv"), outs["graph"], ref):
        assert torch.equal(got, want), name
