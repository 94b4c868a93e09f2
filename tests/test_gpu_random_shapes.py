"""Seeded sweeps of random problem shapes against the fp64 oracle, so that
combinations no hand-picked case names are exercised too:
- attention: batch, grouped-query ratio, ragged length, head size, mask and
  scale drawn together, through the forward, the full backward (whichever
  kernel order fa_bwd takes) and the dQ-sweep-with-D stage order;
- paged decode: batch, query heads per K/V head (up to 20, so beyond one
  CTA's 16), block size (TMA boxes and per-token gathering), context
  lengths (empty and single-token ones included), splits and head size.
Each sweep has a second, larger draw: attention lengths 700 to 4000, decode
contexts up to 20,000 tokens over up to 32 splits."""
import random

import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import make_inputs, to_f64
from oracle import attention_bwd_gqa, attention_fwd_gqa
from gpu_helpers import assert_grad_scaled, assert_lse, assert_o

pytestmark = pytest.mark.gpu


def draw_cases(n, seed, large=False):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        d = rng.choice((64, 128))
        Hkv = rng.randint(1, 3)
        G = rng.choice((1, 1, 2, 3, 4))
        B = rng.randint(1, 2 if large else 3)
        if large:  # several hundred tiles per head, tile-boundary lengths among them
            N = rng.choice((1023, 1024, 1025, 2047, 2049, 4000)) if i % 4 == 0 else rng.randint(700, 4000)
        else:
            N = rng.choice((1, 2, 63, 127, 128, 129)) if i % 4 == 0 else rng.randint(1, 700)
        causal = rng.random() < 0.5
        scale = rng.uniform(0.5, 1.5) / d ** 0.5
        cases.append((B, Hkv * G, Hkv, N, d, causal, round(scale, 5), 9000 + i))
    return cases


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,scale,seed",
                         draw_cases(64, seed=2026) + draw_cases(20, seed=4041, large=True))
def test_random_shape_vs_oracle(fa, B, H, Hkv, N, d, causal, scale, seed):
    q, k, v, do = make_inputs(B, H, N, d, seed=seed, Hkv=Hkv)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fwd(qg, kg, vg, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qg, kg, vg, o, lse, dog, causal=causal, scale=scale)
    # the other kernel order: the dQ sweep forming D, then dK/dV
    Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq2, dk2, dv2 = torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)
    fa.bwd_dq_d(qg, kg, vg, o, dog, lse, Dvec, dq2, causal=causal, scale=scale)
    fa.bwd_dkdv(qg, kg, vg, dog, lse, Dvec, dk2, dv2, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    qd, kd, vd, dod = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    ro, rlse = attention_fwd_gqa(qd, kd, vd, scale, causal)
    assert_o(o, ro)
    assert_lse(lse, rlse)
    rdq, rdk, rdv, _ = attention_bwd_gqa(qd, kd, vd, dod, scale, causal)
    for got, ref, what in ((dq, rdq, "dq"), (dk, rdk, "dk"), (dv, rdv, "dv"),
                           (dq2, rdq, "dq (dq_d order)"), (dk2, rdk, "dk (dq_d order)"),
                           (dv2, rdv, "dv (dq_d order)")):
        assert_grad_scaled(got, ref, what)
    # D as the dQ sweep formed it, against rowsum(dO ∘ O) of the same bf16 O in fp64
    ref_D = (dog.double() * o.double()).sum(-1)
    assert torch.allclose(Dvec.double(), ref_D, atol=1e-4, rtol=1e-5)


def draw_decode_cases(n, seed, large=False):
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        d = rng.choice((64, 128))
        Hkv = rng.randint(1, 4)
        G = rng.choice((1, 2, 4, 8, 16, 20))
        B = rng.randint(1, 4)
        bs = rng.choice((1, 2, 3, 8, 16, 24, 32, 64, 128, 200))  # TMA boxes and per-token gathering
        lens = []
        for _ in range(B):
            r = rng.random()
            if large:  # long contexts, many splits
                lens.append(0 if r < 0.05 else (1 if r < 0.1 else rng.randint(2, 20000)))
            else:
                lens.append(0 if r < 0.1 else (1 if r < 0.2 else rng.randint(2, 3000)))
        splits = rng.choice((1, 2, 5, 8, 16, 32)) if large else rng.randint(1, 6)
        cases.append((B, Hkv * G, Hkv, d, bs, tuple(lens), splits, 7000 + i))
    return cases


@pytest.mark.parametrize("B,H,Hkv,d,bs,lens,splits,seed",
                         draw_decode_cases(48, seed=2027) + draw_decode_cases(20, seed=4042, large=True))
def test_random_decode_vs_oracle(fa, B, H, Hkv, d, bs, lens, splits, seed):
    from oracle import decode_paged
    g = torch.Generator().manual_seed(seed)
    nb = [(L + bs - 1) // bs for L in lens]
    total = sum(nb) + 2
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    kc = torch.randn((total, Hkv, bs, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((total, Hkv, bs, d), generator=g).to(torch.bfloat16)
    perm = torch.randperm(total, generator=g)
    table = torch.zeros((B, max(max(nb), 1)), dtype=torch.int32)
    pos = 0
    for b in range(B):
        table[b, :nb[b]] = perm[pos:pos + nb[b]].to(torch.int32)
        pos += nb[b]
    seq = torch.tensor(lens, dtype=torch.int32)
    scale = d ** -0.5
    o, lse = fa.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), seq.cuda(), n_splits=splits, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    ro, rlse = decode_paged(to_f64(q), to_f64(kc), to_f64(vc), table.numpy(), seq.numpy(), scale)
    live = seq.numpy() > 0
    if live.any():
        assert_o(o[live], ro[live])
        assert_lse(lse[live], rlse[live])
    if not live.all():  # no cached token: o = 0, lse = -inf
        dead = ~torch.from_numpy(live)
        assert torch.all(o[dead].float() == 0) and torch.all(torch.isneginf(lse[dead]))
