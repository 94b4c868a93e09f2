"""Pins for the oracle's attention forward and backward.

Each test ties the oracle to something other than itself: closed forms of
softmax attention, a library routine (torch fp64 softmax / autograd), central
finite differences, and invariants of the gradients. Sources for what is
computed: dcwnkz.com FlashAttention walk-through ("先简要回顾注意力机制"), the
causal mask of the "07-16 下午" notes (section 自回归语言模型推理) and the
recomputation idea of the CMU 10-423 L17–L18 notes (section FlashAttention 本身).
"""
import math

import numpy as np
import pytest
import torch

from oracle import (
    attention_bwd,
    attention_dq_rows_head,
    attention_flops,
    attention_fwd,
    attention_fwd_head,
    attention_pairs,
)


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# ------------------------------------------------------------------ forward

@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_constant_output(causal):
    B, H, N, d = 1, 2, 37, 8
    q, k = rnd((B, H, N, d), 1), rnd((B, H, N, d), 2)
    c = rnd((B, H, 1, d), 3)
    v = np.broadcast_to(c, (B, H, N, d)).copy()
    o, _ = attention_fwd(q, k, v, 0.35, causal)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-13)


def test_zero_queries_noncausal_mean_and_log_n():
    B, H, N, d = 2, 1, 29, 4
    q = np.zeros((B, H, N, d))
    k, v = rnd((B, H, N, d), 4), rnd((B, H, N, d), 5)
    o, lse = attention_fwd(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-14)


def test_zero_queries_causal_prefix_means_and_log_i():
    B, H, N, d = 1, 2, 23, 3
    q = np.zeros((B, H, N, d))
    k, v = rnd((B, H, N, d), 6), rnd((B, H, N, d), 7)
    o, lse = attention_fwd(q, k, v, 0.5, True)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), atol=1e-14)


def test_causal_first_row_sees_only_itself():
    B, H, N, d = 1, 1, 16, 5
    q, k, v = rnd((B, H, N, d), 8), rnd((B, H, N, d), 9), rnd((B, H, N, d), 10)
    scale = 0.7
    o, lse = attention_fwd(q, k, v, scale, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    assert lse[0, 0, 0] == pytest.approx(scale * q[0, 0, 0] @ k[0, 0, 0], abs=1e-14)


def test_causal_last_row_equals_noncausal_last_row():
    B, H, N, d = 1, 1, 20, 6
    q, k, v = rnd((B, H, N, d), 11), rnd((B, H, N, d), 12), rnd((B, H, N, d), 13)
    oc, lc = attention_fwd(q, k, v, 0.4, True)
    on, ln = attention_fwd(q, k, v, 0.4, False)
    np.testing.assert_allclose(oc[..., -1, :], on[..., -1, :], atol=1e-14)
    np.testing.assert_allclose(lc[..., -1], ln[..., -1], atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 4), (5, 3), (64, 16), (130, 8)])
def test_forward_matches_torch_fp64(causal, N, d):
    B, H = 2, 3
    q, k, v = rnd((B, H, N, d), 14, 2.0), rnd((B, H, N, d), 15), rnd((B, H, N, d), 16)
    scale = 1.0 / math.sqrt(d)
    o, lse = attention_fwd(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        mask = torch.ones(N, N, dtype=torch.bool).tril()
        s = s.masked_fill(~mask, float("-inf"))
    ref_o = torch.softmax(s, dim=-1) @ tv
    ref_lse = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-13)


def test_lse_bounds():
    B, H, N, d = 1, 2, 50, 8
    q, k, v = rnd((B, H, N, d), 17, 3.0), rnd((B, H, N, d), 18), rnd((B, H, N, d), 19)
    scale = 0.3
    _, lse = attention_fwd(q, k, v, scale, False)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    smax = s.max(axis=-1)
    assert np.all(lse >= smax - 1e-12)
    assert np.all(lse <= smax + math.log(N) + 1e-12)


def test_row_subset_equals_full(monkeypatch):
    import oracle.attention as oa
    N, d = 300, 8
    q, k, v = rnd((N, d), 20), rnd((N, d), 21), rnd((N, d), 22)
    o, lse = attention_fwd_head(q, k, v, 0.3, True)
    rows = np.array([0, 1, 127, 128, 250, 299])
    monkeypatch.setattr(oa, "ROW_CHUNK", 4)  # chunking must not change values
    o2, lse2 = attention_fwd_head(q, k, v, 0.3, True, rows=rows)
    np.testing.assert_allclose(o2, o[rows], atol=1e-14)
    np.testing.assert_allclose(lse2, lse[rows], atol=1e-14)


# ----------------------------------------------------------------- backward

def _loss_and_grads(q, k, v, do, scale, causal):
    o, _ = attention_fwd(q, k, v, scale, causal)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(causal):
    B, H, N, d = 1, 1, 7, 4
    q, k, v, do = (rnd((B, H, N, d), s) for s in (30, 31, 32, 33))
    scale = 0.6
    dq, dk, dv, _ = attention_bwd(q, k, v, do, scale, causal)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            fp = _loss_and_grads(q, k, v, do, scale, causal)
            x[idx] = old - eps
            fm = _loss_and_grads(q, k, v, do, scale, causal)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(9, 4), (70, 16)])
def test_backward_matches_torch_autograd_fp64(causal, N, d):
    B, H = 2, 2
    q, k, v, do = (rnd((B, H, N, d), s) for s in (40, 41, 42, 43))
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, D = attention_bwd(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)
    # D_i = sum_j P_ij dP_ij equals dO_i . O_i
    np.testing.assert_allclose(D, np.sum(do * o.detach().numpy(), axis=-1), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    B, H, N, d = 1, 2, 45, 8
    q, k, v, do = (rnd((B, H, N, d), s) for s in (50, 51, 52, 53))
    dq, dk, dv, _ = attention_bwd(q, k, v, do, 0.4, causal)
    # each row of dS sums to zero, so the key gradients sum to zero
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # each row of P sums to one, so the value gradients sum to the output grads
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


def test_dq_rows_equal_full_backward():
    N, d = 130, 8
    q, k, v, do = (rnd((N, d), s) for s in (60, 61, 62, 63))
    dq, _, _, D = attention_bwd(q[None, None], k[None, None], v[None, None], do[None, None], 0.3, True)
    rows = np.array([0, 5, 64, 129])
    dqr, Dr = attention_dq_rows_head(q, k, v, do, 0.3, True, rows)
    np.testing.assert_allclose(dqr, dq[0, 0, rows], atol=1e-14)
    np.testing.assert_allclose(Dr, D[0, 0, rows], atol=1e-14)


# -------------------------------------------------------------- FLOP count

@pytest.mark.parametrize("N", [1, 2, 7, 64])
def test_pairs_brute_force(N):
    vis = sum(1 for i in range(N) for j in range(N) if j <= i)
    assert attention_pairs(N, True) == vis
    assert attention_pairs(N, False) == N * N


def test_flops_two_mkn_per_product():
    # forward: QK^T is [N,d]x[d,N] and PV is [N,N]x[N,d]: 2 * 2*N*d*N
    B, H, N, d = 2, 3, 16, 8
    assert attention_flops(B, H, N, d, False, "fwd") == B * H * 2 * (2 * N * d * N)
    assert attention_flops(B, H, N, d, False, "bwd") == B * H * 5 * (2 * N * d * N)
