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
# Gradients larger than unit scale (scores far from unit variance): the
# bf16 path's error grows with the gradients themselves. Every product
# operand is bf16 (8 significant bits, unit roundoff u = 2^-9), and each
# gradient's chain carries at most three roundings (the stored O inside D,
# P or dS, the operand), each of relative size u against the terms it
# rounds; with fp32 sums on top, 8u = 2^-6 of the largest reference entry
# bounds them. This equals the fixed bound at a largest entry of 3.2 and
# widens it only above; the five benchmark configurations are held to the
# fixed bound itself (their largest entries are 1.5 to 5.4).
TOL_GRAD_REL = 2.0 ** -6


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


def grad_bound(ref):
    """The gradient bound for one tensor: the fixed bound, or 2^-6 of the
    tensor's largest reference entry where that is larger."""
    return max(TOL_GRAD, TOL_GRAD_REL * float(np.abs(ref).max()))


def assert_grad_scaled(got, ref, what):
    mx, _ = errs(got, ref)
    bound = grad_bound(ref)
    assert mx <= bound, f"{what}: max-abs {mx} > {bound} (max |ref| {float(np.abs(ref).max())})"
