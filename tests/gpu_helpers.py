"""Shared helpers for the GPU parity tests (inputs from the workload module,
expected values from the fp64 oracle, tolerances from the parity contract)."""
import numpy as np
import torch

from exact_tiled_attention_24_gb300.workloads import to_f64

# Parity bar: O max-abs <= 2e-2 and mean-abs <= 2e-3 (bf16 I/O, fp32
# accumulation), lse <= 1e-3, dQ/dK/dV max-abs <= 5e-2.
TOL_O_MAX = 2e-2
TOL_O_MEAN = 2e-3
TOL_LSE = 1e-3
TOL_GRAD = 5e-2


def errs(got, ref):
    g = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    diff = np.abs(g - ref)
    return float(diff.max()), float(diff.mean())


def assert_o(got, ref, what="o"):
    mx, mean = errs(got, ref)
    assert mx <= TOL_O_MAX, f"{what}: max-abs {mx}"
    assert mean <= TOL_O_MEAN, f"{what}: mean-abs {mean}"


def assert_lse(got, ref):
    mx, _ = errs(got.to(torch.float64), ref)
    assert mx <= TOL_LSE, f"lse: max-abs {mx}"


def assert_grad(got, ref, what):
    mx, _ = errs(got, ref)
    assert mx <= TOL_GRAD, f"{what}: max-abs {mx}"
