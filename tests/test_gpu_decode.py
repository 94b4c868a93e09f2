"""Paged-KV decode and partial-attention merge: CUDA kernels (through the C
ABI) against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_24_gb300.workloads import to_f64
from oracle import attention_merge, decode_paged
from gpu_helpers import assert_lse, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_tiled_attention_24_gb300 import build
    build.build()
    import exact_tiled_attention_24_gb300 as m
    return m


def paged_case(B, H, Hkv, d, bs, seq_lens, seed, spare_blocks=3):
    """Seeded bf16 q and a paged cache with a random physical placement of
    every request's blocks (unused slots hold other random values)."""
    g = torch.Generator().manual_seed(seed)
    nb = [(L + bs - 1) // bs for L in seq_lens]
    total = sum(nb) + spare_blocks
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    kc = torch.randn((total, Hkv, bs, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((total, Hkv, bs, d), generator=g).to(torch.bfloat16)
    perm = torch.randperm(total, generator=g)
    table = torch.zeros((B, max(max(nb), 1)), dtype=torch.int32)
    pos = 0
    for b in range(B):
        table[b, :nb[b]] = perm[pos:pos + nb[b]].to(torch.int32)
        pos += nb[b]
    return q, kc, vc, table, torch.tensor(seq_lens, dtype=torch.int32)


def run_case(fa, q, kc, vc, table, lens, n_splits, scale):
    o, lse = fa.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), lens.cuda(),
                             n_splits=n_splits, scale=scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    return o, lse


@pytest.mark.parametrize("B,H,Hkv,d,bs,seq_lens,n_splits", [
    (3, 4, 4, 64, 16, [1, 17, 100], 1),
    (3, 8, 2, 128, 16, [1, 64, 1000], 4),
    (2, 8, 1, 128, 32, [5000, 333], 8),
    (2, 4, 2, 64, 1, [50, 7], 2),           # one token per block
    (2, 32, 8, 128, 128, [4097, 256], 3),
    (1, 16, 1, 128, 16, [777], 5),           # 16 query heads on one K/V head
    (3, 4, 2, 128, 16, [0, 1, 129], 2),      # an empty context
    (3, 8, 2, 128, 16, [0, 300, 5], 1),      # one split (no merge): an empty context too
    (2, 8, 2, 64, 3, [0, 1000], 1),          # one split, gathered
    (1, 2, 1, 64, 48, [2000], 7),            # block size not a power of two
    (2, 32, 1, 128, 16, [300, 1500], 3),     # 32 query heads on one K/V head: two CTAs of 16
    (1, 24, 1, 64, 32, [777], 2),            # 24 = 16 + 8
    # blocks that are a multiple of 8 dividing 128 arrive as TMA boxes; 1, 48
    # above and the sizes below are gathered token by token
    (2, 8, 2, 128, 8, [100, 37], 2),         # eight-token blocks: 16 boxes per tile
    (2, 12, 3, 128, 64, [700, 129], 3),      # 64-token blocks
    (1, 40, 5, 128, 16, [1025], 4),          # 8 query heads per K/V head
    (2, 16, 2, 128, 3, [700, 131], 2),       # gathered, 8 query heads per K/V head
    (2, 32, 2, 64, 5, [900, 1], 3),          # gathered, 16 heads per K/V head (two K stages)
    (1, 16, 1, 128, 1, [3000], 1),           # one split over 3000 one-token blocks
    (1, 4, 1, 128, 200, [1000], 2),          # blocks larger than a tile
])
def test_decode_paged_vs_oracle(fa, B, H, Hkv, d, bs, seq_lens, n_splits):
    q, kc, vc, table, lens = paged_case(B, H, Hkv, d, bs, seq_lens, seed=B * 100 + H + bs + sum(seq_lens))
    scale = d ** -0.5
    o, lse = run_case(fa, q, kc, vc, table, lens, n_splits, scale)
    ro, rlse = decode_paged(to_f64(q), to_f64(kc), to_f64(vc), table.numpy(), lens.numpy(), scale)
    live = lens.numpy() > 0
    assert_o(o[live], ro[live])
    assert_lse(lse[live], rlse[live])
    if not live.all():  # no cached token: o = 0, lse = -inf
        assert torch.all(o[~torch.from_numpy(live)].float() == 0)
        assert torch.all(torch.isneginf(lse[~torch.from_numpy(live)]))


def test_decode_split_count_does_not_change_the_result(fa):
    q, kc, vc, table, lens = paged_case(4, 8, 2, 128, 16, [3000, 10, 640, 2049], seed=7)
    outs = [run_case(fa, q, kc, vc, table, lens, S, 0.1) for S in (1, 2, 7, 40)]
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max() <= 2e-2
        assert (lse - outs[0][1]).abs().max() <= 1e-4


@pytest.mark.parametrize("d,bs,L,bad", [
    (64, 16, 40, 1), (128, 16, 40, 1),  # TMA boxes
    (128, 3, 40, 1),                    # gathered, entries loaded before the CTA's setup
    (128, 1, 800, 300),                 # gathered, an entry loaded two tiles ahead (tile 2 of 4)
    (128, 24, 400, 11),                 # gathered, entries looked up per tile
])
def test_decode_bad_block_index_is_reported_not_read(fa, d, bs, L, bad):
    q, kc, vc, table, lens = paged_case(2, 4, 2, d, bs, [L, L], seed=9)
    table[1, bad] = kc.shape[0] + 5  # outside the cache
    fa.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), lens.cuda(), n_splits=2)
    assert fa.last_device_error() == 7  # FA_ERR_BAD_INDEX
    assert fa.last_device_error() == 0  # read and cleared
    # request 0 does not use the bad entry and is still right
    scale = d ** -0.5
    o, lse = run_case(fa, q[:1].contiguous(), kc, vc, table[:1].contiguous(), lens[:1].contiguous(), 2, scale)
    ro, rlse = decode_paged(to_f64(q[:1]), to_f64(kc), to_f64(vc), table[:1].numpy(), lens[:1].numpy(), scale)
    assert_o(o, ro)


@pytest.mark.parametrize("S,rows,d", [(1, 5, 64), (3, 300, 128), (17, 64, 128)])
def test_merge_vs_oracle(fa, S, rows, d):
    g = torch.Generator().manual_seed(S * 1000 + rows + d)
    o_parts = torch.randn((S, rows, d), generator=g)
    lse_parts = torch.randn((S, rows), generator=g) * 5
    lse_parts[0, ::4] = float("-inf")       # parts that saw no key
    if S > 1:
        lse_parts[:, 1] = float("-inf")      # a row with no key at all
    o, lse = fa.attn_merge(o_parts.cuda(), lse_parts.cuda())
    torch.cuda.synchronize()
    ro, rlse = attention_merge(o_parts.double().numpy(), lse_parts.double().numpy())
    assert_o(o, ro, "merged o")
    fin = np.isfinite(rlse)
    np.testing.assert_allclose(lse.cpu().numpy()[fin], rlse[fin], rtol=0, atol=1e-4)
    assert np.all(np.isneginf(lse.cpu().numpy()[~fin]))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_peaked_scores_raise_the_reference(fa, d):
    # q ~ N(0, 8²): scaled scores have a standard deviation of 8 (11.5 in log2
    # units), so a head's maximum keeps outgrowing its exponent reference by
    # more than 2^8 after the first tile, and the output columns are rescaled.
    q, kc, vc, table, lens = paged_case(2, 8, 2, d, 16, [1500, 700], seed=31 + d)
    q = (q.float() * 8).to(torch.bfloat16)
    scale = d ** -0.5
    qd, kd = to_f64(q), to_f64(kc)
    # the scenario holds: for some head, a key past the first 128 outscores the
    # first 128 keys' maximum by more than 8 in log2 units
    t = table[0].long()
    keys = np.swapaxes(kd[t], 0, 1).reshape(kd.shape[1], -1, d)[:, :int(lens[0])]  # [Hkv, L, d]
    G = q.shape[1] // kc.shape[1]
    s = np.einsum("hd,hkd->hk", qd[0], np.repeat(keys, G, axis=0)) * scale * np.log2(np.e)
    assert np.any(s[:, 128:].max(1) - s[:, :128].max(1) > 8)
    for n_splits in (1, 3):
        o, lse = run_case(fa, q, kc, vc, table, lens, n_splits, scale)
        ro, rlse = decode_paged(qd, kd, to_f64(vc), table.numpy(), lens.numpy(), scale)
        assert_o(o, ro)
        assert_lse(lse, rlse)


@pytest.mark.parametrize("name", ["d1", "d2"])
def test_decode_workload_full_size_sampled_requests(fa, name):
    # the decode workloads at full size, in the launch configuration the bench
    # times (8 context splits), against the oracle on sampled requests: each
    # one's blocks are gathered in table order into a small cache of its own
    from exact_tiled_attention_24_gb300.workloads import DECODE_WORKLOADS, make_decode
    w = DECODE_WORKLOADS[name]
    q, kc, vc, table, lens = make_decode(w, torch.device("cuda"))
    o, lse = fa.decode_paged(q, kc, vc, table, lens, n_splits=w.n_splits)
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
    scale = w.d ** -0.5
    for b in sorted({0, int(lens.argmax()), w.B - 1}):  # first, longest, last request
        L = int(lens[b])
        nb = (L + w.block_size - 1) // w.block_size
        blocks = table[b, :nb].long()
        kc_b, vc_b = kc[blocks].cpu(), vc[blocks].cpu()
        tab_b = np.arange(nb, dtype=np.int32)[None, :]
        ro, rlse = decode_paged(to_f64(q[b:b + 1]), to_f64(kc_b), to_f64(vc_b), tab_b,
                                np.array([L], dtype=np.int32), scale)
        assert_o(o[b:b + 1], ro)
        assert_lse(lse[b:b + 1], rlse)
