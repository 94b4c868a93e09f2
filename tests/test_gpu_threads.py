"""Entry points called from several host threads at once, each thread on its
own CUDA stream: every call builds its own descriptors, and the streams the
library keeps (copy and side streams) belong to the calling thread, so the
results equal those of one thread running the same calls alone."""
import threading

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


def work(fa, seed, stream, reps):
    B, H, Hkv, N, d = 1, 4, 2, 400 + seed % 7, 128 if seed % 2 else 64
    q, k, v, do = make_inputs(B, H, N, d, seed=seed, Hkv=Hkv)
    with torch.cuda.stream(stream):
        qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
        out = None
        for _ in range(reps):
            o, lse = fa.fwd(qg, kg, vg, causal=True)
            dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=True)
            host = {"q": q.pin_memory(), "k": k.pin_memory(), "v": v.pin_memory(), "dO": do.pin_memory(),
                    "o": torch.empty_like(q).pin_memory(),
                    "lse": torch.empty((B, H, N), dtype=torch.float32).pin_memory(),
                    "dq": torch.empty_like(q).pin_memory(), "dk": torch.empty_like(k).pin_memory(),
                    "dv": torch.empty_like(v).pin_memory()}
            dev = {n: torch.empty(t.shape, dtype=t.dtype, device="cuda") for n, t in host.items()}
            ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
            fa.fwd_bwd_host(host, dev, ws, causal=True, n_chunks=2)
            out = (o, lse, dq, dk, dv, host)
        stream.synchronize()
    o, lse, dq, dk, dv, host = out
    return [t.cpu() for t in (o, lse, dq, dk, dv)] + [host[n].clone() for n in ("o", "lse", "dq", "dk", "dv")]


def test_two_threads_match_one(fa):
    seeds = (11, 12)
    alone = [work(fa, s, torch.cuda.Stream(), 1) for s in seeds]
    results, errors = {}, []

    def run(s):
        try:
            results[s] = work(fa, s, torch.cuda.Stream(), 4)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(s,)) for s in seeds]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    for s, ref in zip(seeds, alone):
        for i, (a, b) in enumerate(zip(results[s], ref)):
            assert torch.equal(a, b), (s, i)
    # device results and the host pipeline's copies agree within each thread
    for s in seeds:
        r = results[s]
        for i in range(5):
            assert torch.equal(r[i], r[5 + i]), (s, i)
