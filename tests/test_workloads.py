"""The seeded input generators that feed both the CUDA path and the oracle:
the documented recipe (generator, draw order, scaling, bf16 rounding), the
workload table, and the invariants of the paged decode inputs. CPU only."""
import dataclasses

import torch

from exact_tiled_attention_24_gb300.workloads import (DECODE_WORKLOADS, ROW_WORKLOADS, WORKLOADS, DecodeWorkload,
                                                      make_decode, make_inputs, make_rows, workload_inputs)


def test_recipe_draw_order_and_scaling():
    """torch.Generator().manual_seed(seed); fp32 normal draws in the order
    q, k, v, dO, each times its standard deviation; then bf16."""
    B, H, Hkv, N, d, seed = 2, 4, 2, 9, 64, 1234
    q, k, v, do = make_inputs(B, H, N, d, seed, q_std=3.0, kv_std=0.5, do_std=2.0, Hkv=Hkv)
    g = torch.Generator().manual_seed(seed)
    rq = (torch.randn((B, H, N, d), generator=g) * 3.0).to(torch.bfloat16)
    rk = (torch.randn((B, Hkv, N, d), generator=g) * 0.5).to(torch.bfloat16)
    rv = (torch.randn((B, Hkv, N, d), generator=g) * 0.5).to(torch.bfloat16)
    rdo = (torch.randn((B, H, N, d), generator=g) * 2.0).to(torch.bfloat16)
    for got, want in ((q, rq), (k, rk), (v, rv), (do, rdo)):
        assert got.dtype == torch.bfloat16 and torch.equal(got, want)


def test_same_seed_same_bytes_other_seed_other_bytes():
    a = make_inputs(1, 2, 33, 128, seed=7)
    b = make_inputs(1, 2, 33, 128, seed=7)
    c = make_inputs(1, 2, 33, 128, seed=8)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[0], c[0])
    # forward-only draws are the first three of the full draw
    f = make_inputs(1, 2, 33, 128, seed=7, with_do=False)
    assert len(f) == 3 and all(torch.equal(x, y) for x, y in zip(f, a[:3]))


def test_workload_table():
    want = {"c1": (1, 1, 256, 64), "c2": (8, 12, 1024, 64), "c3": (4, 12, 1028, 64),
            "c4": (2, 32, 8192, 128), "c5": (1, 16, 32768, 128), "g4": (2, 32, 8192, 128)}
    for name, shape in want.items():
        w = WORKLOADS[name]
        assert w.shape == shape, name
        assert abs(w.scale - shape[3] ** -0.5) < 1e-12
    assert [WORKLOADS[n].seed for n in ("c1", "c2", "c3", "c4", "c5")] == [1001, 1002, 1003, 1004, 1005]
    assert WORKLOADS["c5"].q_std == 4.0
    assert WORKLOADS["g4"].kv_heads == 8 and WORKLOADS["c4"].kv_heads == 32
    assert "bwd" in WORKLOADS["c4"].directions and "bwd" not in WORKLOADS["c5"].directions
    q, k, v = workload_inputs("c1")
    assert q.shape == (1, 1, 256, 64) and k.shape == q.shape


def test_rows_generator():
    rw = ROW_WORKLOADS["s1"]
    assert rw.rows % 608 == 0 and rw.rows * rw.n * 4 > 129 * 2 ** 20  # whole waves; beyond L2
    x = make_rows(5, 11, seed=3, std=2.0)
    g = torch.Generator().manual_seed(3)
    assert torch.equal(x, torch.randn((5, 11), generator=g) * 2.0)


def test_decode_generator_invariants():
    d1 = DECODE_WORKLOADS["d1"]
    assert (d1.B, d1.H, d1.Hkv, d1.d, d1.block_size, d1.min_len, d1.max_len) == (32, 32, 8, 128, 16, 2048, 8192)
    # d2: the same step and draws with one-token blocks
    d2 = DECODE_WORKLOADS["d2"]
    assert dataclasses.replace(d2, name="d1", block_size=16) == d1
    # the same generator on a small workload of the same kind
    dw = DecodeWorkload("small", 6, 8, 2, 64, 16, 20, 300, 4, 3101)
    q, kc, vc, table, lens = make_decode(dw, torch.device("cpu"))
    assert q.shape == (dw.B, dw.H, dw.d) and q.dtype == torch.bfloat16
    assert kc.shape == vc.shape and kc.shape[1:] == (dw.Hkv, dw.block_size, dw.d)
    assert lens.dtype == torch.int32 and table.dtype == torch.int32
    assert int(lens.min()) >= dw.min_len and int(lens.max()) <= dw.max_len
    nb = (lens.long() + dw.block_size - 1) // dw.block_size
    assert table.shape == (dw.B, int(nb.max()))
    used = torch.cat([table[b, :nb[b]] for b in range(dw.B)])
    # every physical block belongs to exactly one request, and all are used
    assert used.numel() == kc.shape[0]
    assert torch.equal(torch.sort(used).values, torch.arange(kc.shape[0], dtype=torch.int32))
    # the placement is shuffled, not the identity
    assert not torch.equal(used, torch.arange(kc.shape[0], dtype=torch.int32))
    # same seed, same table
    _, _, _, table2, lens2 = make_decode(dw, torch.device("cpu"))
    assert torch.equal(table, table2) and torch.equal(lens, lens2)
