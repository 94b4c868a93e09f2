"""Pins for the oracle's partial-attention merge and paged-KV decode.

Merge ("07-16 下午" notes, section 长上下文与序列并行): the running max /
normaliser / weighted-sum recurrence over blocks.  Pinned to the six-score
walk-through's printed denominators (dcwnkz.com article, FlashAttention
section), to attention over the union of the blocks, and to its neutral
element.  Decode (CMU 10-423 notes, section 解碼端：PagedAttention; "07-16 下午"
notes, section Prefill、Decode 与推理调度): pinned to the row of the full causal
forward that the decode step reproduces, to a single-token closed form, and
to invariance under moving blocks in physical memory.
"""
import json
import os

import numpy as np
import pytest

from oracle import (attention_fwd, attention_fwd_head, attention_merge, decode_paged, gather_paged,
                    softmax_safe)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "six_score_example.json")


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def test_merge_reproduces_printed_denominators():
    """Each block of two scores, merged in order: the carried normaliser,
    expressed relative to the running max, is 1+0.0082, 1.3098, 1.4955."""
    six = json.load(open(GOLDEN))
    s = np.array(six["reconstruction"]["scores"], dtype=np.float64)
    pr = six["printed"]
    v = np.eye(6)
    o_parts, lse_parts = [], []
    for b in range(3):
        blk = s[2 * b:2 * b + 2]
        o_b, l_b = attention_fwd_head(np.ones((1, 1)), blk[:, None], v[2 * b:2 * b + 2], 1.0, False)
        o_parts.append(o_b)
        lse_parts.append(l_b)
    printed = [pr["denominator_after_block1"], pr["denominator_after_blocks_1_2"],
               pr["denominator_after_blocks_1_2_3"]]
    for k in range(1, 4):
        o, lse = attention_merge(o_parts[:k], lse_parts[:k])
        m = s[:2 * k].max()
        assert abs(np.exp(lse[0] - m) - printed[k - 1]) <= 2 * pr["printed_precision"]
        np.testing.assert_allclose(o[0][:2 * k], softmax_safe(s[:2 * k]), atol=1e-15)


@pytest.mark.parametrize("splits", [[0, 40, 97], [0, 1, 2, 97], [0, 97]])
def test_merge_of_key_blocks_equals_attention_over_union(splits):
    rows, n, d = 5, 97, 6
    q, k, v = rnd((rows, d), 1), rnd((n, d), 2, 2.0), rnd((n, d), 3)
    full_o, full_lse = attention_fwd_head(q, k, v, 0.4, False)
    parts = [attention_fwd_head(q, k[a:b], v[a:b], 0.4, False) for a, b in zip(splits, splits[1:])]
    o, lse = attention_merge([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, full_o, atol=1e-13)
    np.testing.assert_allclose(lse, full_lse, atol=1e-13)
    # the order of the parts does not matter
    o2, lse2 = attention_merge([p[0] for p in parts[::-1]], [p[1] for p in parts[::-1]])
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


def test_merge_empty_part_is_neutral():
    o1, l1 = rnd((4, 3), 5), rnd(4, 6)
    empty_o, empty_l = np.zeros((4, 3)), np.full(4, -np.inf)
    o, lse = attention_merge([empty_o, o1, empty_o], [empty_l, l1, empty_l])
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(lse, l1, atol=1e-15)
    o, lse = attention_merge([empty_o], [empty_l])
    assert np.all(o == 0) and np.all(lse == -np.inf)


def make_paged(B, Hkv, d, bs, seq_lens, seed, shuffle=True):
    """Draw each request's contiguous K/V [Hkv, L, d] from the seed, then
    scatter it into a paged cache under a random (or identity) block
    placement; returns the cache, the block table and the contiguous K/V."""
    rng = np.random.default_rng(seed)
    nb = [(L + bs - 1) // bs for L in seq_lens]
    total = sum(nb) + 3
    k_seq = [rnd((Hkv, L, d), seed + 100 + b) for b, L in enumerate(seq_lens)]
    v_seq = [rnd((Hkv, L, d), seed + 200 + b) for b, L in enumerate(seq_lens)]
    perm = rng.permutation(total) if shuffle else np.arange(total)
    kc, vc = rnd((total, Hkv, bs, d), seed + 1), rnd((total, Hkv, bs, d), seed + 2)
    table = np.zeros((B, max(nb)), dtype=np.int64)
    pos = 0
    for b, L in enumerate(seq_lens):
        table[b, :nb[b]] = perm[pos:pos + nb[b]]
        pos += nb[b]
        for t in range(L):
            kc[table[b, t // bs], :, t % bs] = k_seq[b][:, t]
            vc[table[b, t // bs], :, t % bs] = v_seq[b][:, t]
        np.testing.assert_array_equal(gather_paged(kc, table[b], L), k_seq[b])
    return kc, vc, table, k_seq, v_seq


def test_decode_equals_last_row_of_causal_forward():
    """Decoding token t with the cache of tokens 0..t gives row t of the causal
    forward over the whole sequence (no recomputation of the history)."""
    Hkv, H, d, bs, L = 2, 4, 8, 4, 23
    q_all = rnd((1, H, L, d), 10)
    kc, vc, table, k_seq, v_seq = make_paged(1, Hkv, d, bs, [L], seed=11)
    G = H // Hkv
    kq = np.stack([k_seq[0][h // G] for h in range(H)])[None]
    vq = np.stack([v_seq[0][h // G] for h in range(H)])[None]
    o_full, lse_full = attention_fwd(q_all, kq, vq, 0.3, True)
    o, lse = decode_paged(q_all[:, :, L - 1], kc, vc, table, [L], 0.3)
    np.testing.assert_allclose(o[0], o_full[0, :, L - 1], atol=1e-13)
    np.testing.assert_allclose(lse[0], lse_full[0, :, L - 1], atol=1e-13)


def test_decode_single_token_and_block_placement():
    Hkv, H, d, bs = 1, 3, 5, 4
    q = rnd((3, H, d), 20)
    seq_lens = [1, 9, 17]
    kc, vc, table, k_seq, v_seq = make_paged(3, Hkv, d, bs, seq_lens, seed=21)
    o, lse = decode_paged(q, kc, vc, table, seq_lens, 0.5)
    # one cached token: the output is its value row, lse its scaled score
    np.testing.assert_allclose(o[0], np.repeat(v_seq[0][0], H, axis=0), atol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * q[0] @ k_seq[0][0, 0], atol=1e-14)
    # the same requests with an identity placement give the same result
    kc2, vc2, table2, _, _ = make_paged(3, Hkv, d, bs, seq_lens, seed=21, shuffle=False)
    o2, lse2 = decode_paged(q, kc2, vc2, table2, seq_lens, 0.5)
    np.testing.assert_allclose(o2, o, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, atol=1e-14)
