"""The Python binding's argument checks, on CPU. The library is replaced by a
fake that records which entry points are called, and the binding's device
type is set to "meta" (tensors with shapes and dtypes but no storage)
standing in for CUDA. Every wrapper must pass the buffers that the GPU tests
and the benchmark pass, exactly as they shape them, on to the library. A
buffer the kernels would overrun, the wrong dtype, a non-contiguous view or a
tensor on the wrong device must raise ValueError before any library call.
With the real device type, host tensors are refused outright."""
import pytest
import torch

import exact_tiled_attention_24_gb300 as fa

BF, F32, I32 = torch.bfloat16, torch.float32, torch.int32
META = torch.device("meta")


class FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("fa_"):
            raise AttributeError(name)

        def entry(*args):
            self.calls.append(name)
            if name == "fa_bwd_workspace_bytes":
                B, H, N, d = args
                return B * H * N * 4
            if name == "fa_decode_workspace_bytes":
                B, H, d, S = args
                return S * B * H * (d + 1) * 4
            return 0
        return entry


@pytest.fixture
def fake(monkeypatch):
    L = FakeLib()
    monkeypatch.setattr(fa, "_DEVICE_TYPE", "meta")
    monkeypatch.setattr(fa, "lib", lambda: L)
    monkeypatch.setattr(fa, "_stream", lambda device: None)
    return L


def m(*shape, dtype=BF):
    return torch.empty(shape, dtype=dtype, device=META)


B, H, HKV, N, D = 2, 4, 2, 8, 64


def qkv():
    return m(B, H, N, D), m(B, HKV, N, D), m(B, HKV, N, D)


def launches(fake):
    """Library calls that queue device work (size queries excluded)."""
    return [c for c in fake.calls if not c.endswith("_workspace_bytes")]


def rejects(fake, fn, *args, **kw):
    before = len(launches(fake))
    with pytest.raises(ValueError):
        fn(*args, **kw)
    assert len(launches(fake)) == before, "the library was called despite a bad argument"


def test_attention_wrappers_accept_what_the_tests_pass(fake):
    q, k, v = qkv()
    o, lse = fa.fwd(q, k, v, causal=True)
    assert o.shape == q.shape and lse.shape == (B, H, N) and lse.dtype == F32
    # preallocated outputs, also as contiguous views of a padded buffer
    obuf, lbuf = m(B * H * N * D + 64), m(B * H * N + 16, dtype=F32)
    fa.fwd(q, k, v, out=obuf[:B * H * N * D].view(B, H, N, D), lse=lbuf[:B * H * N].view(B, H, N))
    do = m(B, H, N, D)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
    assert dk.shape == k.shape and dq.shape == q.shape
    ws = m(fa.bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8)
    fa.bwd(q, k, v, o, lse, do, workspace=ws)
    Dvec = m(B, H, N, dtype=F32)
    fa.bwd_preprocess(o, do, Dvec)
    fa.bwd_dkdv(q, k, v, do, lse, Dvec, torch.empty_like(k), torch.empty_like(v), causal=True)
    fa.bwd_dq(q, k, v, do, lse, Dvec, torch.empty_like(q), causal=True)
    assert fake.calls.count("fa_fwd_gqa") == 2 and fake.calls.count("fa_bwd_gqa") == 2
    for name in ("fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq"):
        assert name in fake.calls


def test_attention_wrappers_reject_bad_buffers(fake):
    q, k, v = qkv()
    o, lse, do = m(B, H, N, D), m(B, H, N, dtype=F32), m(B, H, N, D)
    rejects(fake, fa.fwd, q, k, v, out=m(B, H, N - 1, D))                 # too small
    rejects(fake, fa.fwd, q, k, v, out=m(B, H, N, D, dtype=torch.float16))
    rejects(fake, fa.fwd, q, k, v, out=m(B, H, D, N).transpose(2, 3))    # not contiguous
    rejects(fake, fa.fwd, q, k, v, out=torch.empty(B, H, N, D, dtype=BF))  # another device
    rejects(fake, fa.fwd, q, k, v, lse=m(B, H, N - 1, dtype=F32))
    rejects(fake, fa.fwd, q, k, v, lse=m(B, H, N))                       # bf16 lse
    rejects(fake, fa.bwd, q, k, v, o, m(B, H, N - 1, dtype=F32), do)
    rejects(fake, fa.bwd, q, k, v, o, lse, do, workspace=torch.empty(4096, dtype=torch.uint8))
    Dvec = m(B, H, N, dtype=F32)
    rejects(fake, fa.bwd_preprocess, o, do, m(B, H, N - 1, dtype=F32))
    rejects(fake, fa.bwd_preprocess, o, m(B, H, N, D // 2), Dvec)
    rejects(fake, fa.bwd_dkdv, q, k, v, do, lse, Dvec, torch.empty_like(q), torch.empty_like(v))  # H, not Hkv
    rejects(fake, fa.bwd_dkdv, q, k, v, do, lse, m(B, H, N), torch.empty_like(k), torch.empty_like(v))
    rejects(fake, fa.bwd_dq, q, k, v, do, lse, Dvec, torch.empty_like(k))
    rejects(fake, fa.bwd_dq, q, k, v, do, m(B, H, 1, dtype=F32), Dvec, torch.empty_like(q))


def test_softmax_and_merge(fake):
    x = m(8, 256, dtype=F32)
    y = fa.softmax_online(x)
    fa.softmax_safe(y, out=y)                     # in place
    fa.softmax_safe(x, out=m(8, 256, dtype=F32))
    rejects(fake, fa.softmax_online, x, out=m(8, 255, dtype=F32))
    rejects(fake, fa.softmax_online, x, out=m(8, 256))
    rejects(fake, fa.softmax_online, torch.empty(8, 256))
    S, rows = 3, 10
    o, lse = fa.attn_merge(m(S, rows, D, dtype=F32), m(S, rows, dtype=F32))
    assert o.shape == (rows, D) and o.dtype == BF and lse.shape == (rows,)
    rejects(fake, fa.attn_merge, m(S, rows, D, dtype=F32), torch.empty(S, rows))
    rejects(fake, fa.attn_merge, m(S, rows, D, dtype=F32), m(S, rows, dtype=F32), out=m(rows, D - 1))
    rejects(fake, fa.attn_merge, m(S, rows, D, dtype=F32), m(S, rows, dtype=F32), lse=m(rows + 1, dtype=F32))
    assert fake.calls.count("fa_attn_merge") == 1


def test_decode(fake):
    Bd, Hd, Hkvd, nb, bs, mb = 3, 8, 2, 12, 16, 5
    q, kc, vc = m(Bd, Hd, D), m(nb, Hkvd, bs, D), m(nb, Hkvd, bs, D)
    table, lens = m(Bd, mb, dtype=I32), m(Bd, dtype=I32)
    o, lse = fa.decode_paged(q, kc, vc, table, lens, n_splits=2)
    assert o.shape == (Bd, Hd, D) and lse.shape == (Bd, Hd)
    ws = m(fa.decode_workspace_bytes(Bd, Hd, D, 4), dtype=torch.uint8)
    fa.decode_paged(q, kc, vc, table, lens, n_splits=4, workspace=ws, out=torch.empty_like(q),
                    lse=m(Bd, Hd, dtype=F32))
    assert fake.calls.count("fa_decode_paged") == 2
    rejects(fake, fa.decode_paged, q, kc, vc, torch.zeros(Bd, mb, dtype=I32), lens)   # table on the host
    rejects(fake, fa.decode_paged, q, kc, vc, table, torch.zeros(Bd, dtype=I32))      # lens on the host
    rejects(fake, fa.decode_paged, q, kc, vc, table, m(Bd, 2, dtype=I32)[:, 0])      # lens not contiguous
    rejects(fake, fa.decode_paged, q, kc, vc, table, lens, workspace=torch.empty(1 << 16, dtype=torch.uint8))
    rejects(fake, fa.decode_paged, q, kc, vc, table, lens, out=m(Bd, Hd, D - 8))
    rejects(fake, fa.decode_paged, q, kc, vc, table, lens, lse=m(Bd, Hd + 1, dtype=F32))
    rejects(fake, fa.decode_paged, q, kc, m(nb, Hkvd, bs, D // 2), table, lens)


def host_dev(with_bwd):
    q, k, v = (torch.empty(t.shape, dtype=BF) for t in qkv())
    host = {"q": q, "k": k, "v": v, "o": torch.empty_like(q), "lse": torch.empty(B, H, N)}
    dev = {n: torch.empty_like(t, device=META) for n, t in host.items()}
    if with_bwd:
        for n, t in (("dO", q), ("dq", q), ("dk", k), ("dv", v)):
            host[n] = torch.empty_like(t)
            dev[n] = torch.empty_like(t, device=META)
    return host, dev


def test_host_pipeline_wrappers(fake):
    host, dev = host_dev(False)
    fa.fwd_host(host, dev, causal=True)
    host, dev = host_dev(True)
    ws = m(fa.bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8)
    fa.fwd_bwd_host(host, dev, ws, causal=True, n_chunks=3)
    fa.softmax_host(torch.empty(6, 32), torch.empty(6, 32), m(6, 32, dtype=F32), m(6, 32, dtype=F32))
    assert fake.calls == ["fa_fwd_host", "fa_bwd_workspace_bytes", "fa_fwd_bwd_host", "fa_softmax_host"]
    bad = dict(dev, o=torch.empty_like(host["o"]))                 # a device buffer on the host
    rejects(fake, fa.fwd_bwd_host, host, bad, ws)
    bad = dict(host, lse=m(B, H, N, dtype=F32))                    # a host buffer on the device
    rejects(fake, fa.fwd_bwd_host, bad, dev, ws)
    bad = dict(dev, dk=m(B, H, N, D))                              # H heads where Hkv are due
    rejects(fake, fa.fwd_bwd_host, host, bad, ws)
    rejects(fake, fa.fwd_bwd_host, host, dev, torch.empty(ws.shape, dtype=torch.uint8))
    rejects(fake, fa.softmax_host, torch.empty(6, 32), torch.empty(6, 32), torch.empty(6, 32),
            m(6, 32, dtype=F32))


def test_host_tensors_refused_with_the_real_device_type(monkeypatch):
    """No silent host path: CPU tensors raise before the library is touched."""
    def no_lib():
        raise AssertionError("library called")
    monkeypatch.setattr(fa, "lib", no_lib)
    q, k, v = (torch.empty(t.shape, dtype=BF) for t in qkv())
    with pytest.raises(ValueError):
        fa.fwd(q, k, v)
    with pytest.raises(ValueError):
        fa.softmax_online(torch.empty(4, 16))
    with pytest.raises(ValueError):
        fa.attn_merge(torch.empty(2, 3, D), torch.empty(2, 3))
    with pytest.raises(ValueError):
        fa.decode_paged(torch.empty(1, 2, D, dtype=BF), torch.empty(1, 1, 16, D, dtype=BF),
                        torch.empty(1, 1, 16, D, dtype=BF), torch.zeros(1, 1, dtype=I32),
                        torch.ones(1, dtype=I32))
