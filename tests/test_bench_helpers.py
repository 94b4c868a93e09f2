"""Host-side checks of bench.py's reporting helpers: which measured bf16 peak a
timed region is held against, the oracle-vs-GPU error figures of the CPU
baseline, and the CPU model probe (no GPU needed)."""
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"bf16_tflops": 1943.4, "bf16_tflops_sustained": 1698.1}


def test_short_uncapped_region_takes_the_burst_peak():
    peak, name = bench.pick_peak(PEAKS, 0.058, {"reasons": []})
    assert (peak, name) == (1943.4, "bf16_tflops")


def test_long_region_takes_the_sustained_peak():
    peak, name = bench.pick_peak(PEAKS, 1.5, {"reasons": []})
    assert (peak, name) == (1698.1, "bf16_tflops_sustained")


def test_power_cap_takes_the_sustained_peak_even_when_short():
    peak, name = bench.pick_peak(PEAKS, 0.3, {"reasons": ["sw_power_cap"]})
    assert name == "bf16_tflops_sustained"


def test_missing_peaks_fall_back():
    peak, name = bench.pick_peak({}, 0.1, {"reasons": []})
    assert name == "bf16_tflops" and peak == bench.FALLBACK_PEAKS["bf16_tflops"]


def test_oracle_errors_per_output_and_grouped_heads():
    B, H, N, d = 1, 4, 5, 8
    g = torch.Generator().manual_seed(0)
    gpu = {"o": torch.randn(B, H, N, d, generator=g), "lse": torch.randn(B, H, N, generator=g),
           "dq": torch.randn(B, H, N, d, generator=g),
           "dk": torch.randn(B, 2, N, d, generator=g), "dv": torch.randn(B, 2, N, d, generator=g)}
    first = {"o": gpu["o"][0, 1].double().numpy() + 0.25, "lse": gpu["lse"][0, 1].double().numpy(),
             "dq": gpu["dq"][0, 1].double().numpy(), "dk": np.zeros((N, d)), "dv": np.zeros((N, d))}
    # two query heads per K/V head: dk, dv on the GPU sum over the group, so
    # they are not compared with one head's oracle gradients
    out = bench.oracle_errors(first, gpu, 0, 1, G=2)
    assert set(out) == {"o", "lse", "dq"}
    assert math.isclose(out["o"]["max_abs"], 0.25, rel_tol=1e-6)
    assert math.isclose(out["o"]["mean_abs"], 0.25, rel_tol=1e-6)
    assert out["lse"]["max_abs"] == 0.0
    # one K/V head per query head: all five are compared (K/V head = query head)
    gpu1 = dict(gpu, dk=torch.zeros(B, H, N, d), dv=torch.zeros(B, H, N, d))
    out1 = bench.oracle_errors(first, gpu1, 0, 1, G=1)
    assert set(out1) == {"o", "lse", "dq", "dk", "dv"}
    assert out1["dk"]["max_abs"] == 0.0


def test_cpu_model_is_a_string_or_none():
    m = bench.cpu_model()
    assert m is None or (isinstance(m, str) and m)
