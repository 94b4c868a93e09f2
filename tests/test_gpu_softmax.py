"""Row softmax parity: the three-pass (safe) and two-pass (online) CUDA
kernels against the fp64 oracle's safe softmax, on the same seeded inputs."""
import numpy as np
import pytest
import torch

from oracle import softmax_safe

pytestmark = pytest.mark.gpu

# fp32 output with hardware 2^x: per-element relative error of a few ulp
# plus the rounding of an n-term fp32 sum in the denominator.
REL = 1e-4
ABS = 1e-7


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def draw(rows, n, seed, std=4.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((rows, n), generator=g, dtype=torch.float32) * std


def check(fa, x):
    ref = softmax_safe(x.to(torch.float64).numpy())
    xg = x.cuda()
    for fn in (fa.softmax_safe, fa.softmax_online):
        y = fn(xg)
        torch.cuda.synchronize()
        got = y.cpu().to(torch.float64).numpy()
        np.testing.assert_allclose(got, ref, rtol=REL, atol=ABS)
    return ref


@pytest.mark.parametrize("rows,n", [(1, 1), (3, 5), (7, 1000), (5, 1001), (64, 4096), (2, 262147),
                                    (4, 262144)])
def test_softmax_shapes(fa, rows, n):
    check(fa, draw(rows, n, seed=rows * 31 + n))


def test_softmax_extremes(fa):
    """Large magnitudes (no overflow: the maximum is subtracted first), -inf
    entries (weight 0), a one-hot row, a shifted copy (shift invariance)."""
    x = draw(6, 515, seed=5)
    x[0] *= 1e4
    x[1, ::3] = float("-inf")
    x[2] = -1e30
    x[2, 17] = 1e30
    x[3] = x[4] + 1000.0
    ref = check(fa, x)
    assert ref[2, 17] == 1.0
    y = fa.softmax_online(x.cuda()).cpu()
    assert torch.all(y[1, ::3] == 0)


def test_softmax_in_place_and_rows_sum_to_one(fa):
    x = draw(33, 20000, seed=9).cuda()
    ref = softmax_safe(x.cpu().to(torch.float64).numpy())
    for fn in (fa.softmax_safe, fa.softmax_online):
        y = x.clone()
        fn(y, out=y)
        torch.cuda.synchronize()
        np.testing.assert_allclose(y.cpu().double().numpy(), ref, rtol=REL, atol=ABS)
        np.testing.assert_allclose(y.double().sum(dim=1).cpu().numpy(), 1.0, atol=1e-5)


def test_softmax_misaligned_rows_use_the_scalar_path(fa):
    """A view starting one float into a buffer is 4-byte but not 16-byte
    aligned; the kernel takes 4-byte loads and the result is unchanged."""
    buf = draw(1, 8 * 256 + 1, seed=11).cuda().view(-1)
    x = buf[1:].view(8, 256)
    y = fa.softmax_safe(x.contiguous())  # aligned copy for the reference result
    for fn in (fa.softmax_online, fa.softmax_safe):
        out = torch.empty(8 * 256 + 1, device="cuda")[1:].view(8, 256)
        fn(x, out=out)
        torch.cuda.synchronize()
        np.testing.assert_allclose(out.cpu().numpy(), y.cpu().numpy(), rtol=REL, atol=ABS)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("online", [True, False])
def test_softmax_host_matches_device_call(fa, pinned, online):
    """Rows from host memory through the pipelined call give the device
    call's bits (n % 4 != 0 exercises the scalar path on every slice)."""
    for rows, n, chunks in ((300, 1000, 0), (7, 4099, 3), (1, 64, 5)):
        x = draw(rows, n, seed=rows + n, std=3.0)
        xh = x.pin_memory() if pinned else x.clone()
        yh = torch.full_like(x, float("nan"))
        if pinned:
            yh = yh.pin_memory()
        xd, yd = torch.empty_like(x, device="cuda"), torch.empty_like(x, device="cuda")
        fa.softmax_host(xh, yh, xd, yd, online=online, n_chunks=chunks)
        torch.cuda.synchronize()
        ref = (fa.softmax_online if online else fa.softmax_safe)(x.cuda())
        torch.cuda.synchronize()
        assert torch.equal(yh, ref.cpu())
        assert torch.equal(yd, ref)
