"""Pins for the oracle's grouped-query attention (K/V heads shared by groups
of consecutive query heads; "07-16 下午" notes, section 自回归语言模型推理,
Prefill、Decode 与推理调度, where kv_heads < query heads).

Each test ties the oracle to something other than its own formula: a closed
form that exposes the head mapping, central finite differences taken on the
shared K/V tensor itself, and torch autograd through an explicit
repeat_interleave of the K/V heads.
"""
import numpy as np
import pytest
import torch

from oracle import attention_bwd, attention_bwd_gqa, attention_fwd, attention_fwd_gqa, kv_head_of


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


@pytest.mark.parametrize("H,Hkv", [(8, 2), (6, 3), (4, 1)])
def test_head_mapping_closed_form(H, Hkv):
    """K/V head g holds one constant value row c_g, so every output row of a
    query head equals c of the K/V head it reads: h // (H / Hkv)."""
    B, N, d = 2, 19, 5
    q, k = rnd((B, H, N, d), 1), rnd((B, Hkv, N, d), 2)
    c = rnd((B, Hkv, 1, d), 3)
    v = np.broadcast_to(c, (B, Hkv, N, d)).copy()
    for causal in (False, True):
        o, _ = attention_fwd_gqa(q, k, v, 0.4, causal)
        for h in range(H):
            np.testing.assert_allclose(o[:, h], np.broadcast_to(c[:, h * Hkv // H], (B, N, d)),
                                       atol=1e-13)
    assert [kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]


def test_one_group_per_head_is_multi_head():
    B, H, N, d = 1, 3, 21, 4
    q, k, v, do = (rnd((B, H, N, d), s) for s in (4, 5, 6, 7))
    o1, l1 = attention_fwd_gqa(q, k, v, 0.5, True)
    o2, l2 = attention_fwd(q, k, v, 0.5, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    g1 = attention_bwd_gqa(q, k, v, do, 0.5, True)
    g2 = attention_bwd(q, k, v, do, 0.5, True)
    for a, b in zip(g1, g2):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_shared_kv_gradient_central_differences(causal):
    """Perturbing one entry of a shared K/V head moves every query head of its
    group; the numerical derivative of sum(o ∘ dO) must equal the summed dK,
    dV the oracle returns."""
    B, H, Hkv, N, d = 1, 4, 2, 6, 3
    q, do = rnd((B, H, N, d), 10), rnd((B, H, N, d), 11)
    k, v = rnd((B, Hkv, N, d), 12), rnd((B, Hkv, N, d), 13)
    scale = 0.7
    _, dk, dv, _ = attention_bwd_gqa(q, k, v, do, scale, causal)

    def loss():
        o, _ = attention_fwd_gqa(q, k, v, scale, causal)
        return float(np.sum(o * do))

    eps = 1e-6
    for x, g in ((k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            fp = loss()
            x[idx] = old - eps
            fm = loss()
            x[idx] = old
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=2e-8)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_matches_torch_autograd_through_repeat(causal):
    B, H, Hkv, N, d = 2, 6, 2, 33, 8
    q, do = rnd((B, H, N, d), 20), rnd((B, H, N, d), 21)
    k, v = rnd((B, Hkv, N, d), 22), rnd((B, Hkv, N, d), 23)
    scale = d ** -0.5
    o, lse = attention_fwd_gqa(q, k, v, scale, causal)
    dq, dk, dv, _ = attention_bwd_gqa(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    ke = torch.repeat_interleave(tk, H // Hkv, dim=1)
    ve = torch.repeat_interleave(tv, H // Hkv, dim=1)
    s = scale * tq @ ke.transpose(-1, -2)
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    ref = torch.softmax(s, dim=-1) @ ve
    ref.backward(torch.from_numpy(do))
    np.testing.assert_allclose(o, ref.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_gqa_gradient_invariants():
    """dS rows sum to zero, so dK summed over keys is zero; P rows sum to one,
    so dV summed over keys equals dO summed over the group's query heads."""
    B, H, Hkv, N, d = 1, 6, 3, 40, 4
    q, do = rnd((B, H, N, d), 30), rnd((B, H, N, d), 31)
    k, v = rnd((B, Hkv, N, d), 32), rnd((B, Hkv, N, d), 33)
    _, dk, dv, _ = attention_bwd_gqa(q, k, v, do, 0.4, True)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    G = H // Hkv
    do_group = do.reshape(B, Hkv, G, N, d).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), do_group, atol=1e-12)
