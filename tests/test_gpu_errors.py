"""The device error path: a bounded pipeline wait that runs out reports
FA_ERR_TIMEOUT through fa_last_device_error, the status is cleared by the
read, and the context stays usable for the next calls. No fault is raised:
the wait that runs out is on an mbarrier that nothing arrives on."""
import time

import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs, to_f64
from oracle import attention_fwd
from gpu_helpers import assert_lse, assert_o

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def test_wait_limit_reports_timeout_and_context_survives(fa):
    assert fa.last_device_error() == FA_OK
    t0 = time.monotonic()
    fa.selftest_wait_limit()
    assert fa.last_device_error() == FA_ERR_TIMEOUT
    waited = time.monotonic() - t0
    assert 1.5 < waited < 30.0, waited      # the limit is 2 s of device time
    assert fa.last_device_error() == FA_OK  # the read cleared it

    # the next calls run normally and give correct results
    q, k, v = make_inputs(1, 2, 300, 64, seed=4242, with_do=False)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == FA_OK
    ro, rlse = attention_fwd(to_f64(q), to_f64(k), to_f64(v), 64 ** -0.5, True)
    assert_o(o.cpu(), ro)
    assert_lse(lse.cpu(), rlse)


def test_wait_limit_on_a_side_stream(fa):
    """The error word is per device, not per stream: a time-out on one
    stream is seen by a check on another once both are ordered."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fa.selftest_wait_limit()
    torch.cuda.current_stream().wait_stream(s)
    assert fa.last_device_error() == FA_ERR_TIMEOUT
    assert fa.last_device_error() == FA_OK
