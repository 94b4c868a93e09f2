"""Pins for the oracle's softmax pieces against what the pages print.

Sources: the dcwnkz.com GPU-tricks article (CS336 tricks), FlashAttention
section (six-score walk-through) and its softmax appendix; the CMU 10-423
L17–L18 notes, section 前置二：online softmax and the self-study exercise; the
"07-16 下午：分布式大模型训练与推理" notes, section 长上下文与序列并行.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import softmax_blocks_naive_sum, softmax_online_blocks, softmax_safe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "six_score_example.json")


@pytest.fixture(scope="module")
def six():
    with open(GOLDEN) as f:
        return json.load(f)


def test_six_score_printed_denominators(six):
    """Running denominators after blocks 1, 1-2 and 1-3 match the printed
    1+0.0082, 1.3098 and 1.4955 (printed to 4 decimals)."""
    pr = six["printed"]
    s = np.array(six["reconstruction"]["scores"], dtype=np.float64)
    _, trace = softmax_online_blocks(s, np.eye(6), pr["block_size"])
    tol = 2 * pr["printed_precision"]
    assert len(trace) == 3
    assert abs(trace[0]["l"] - pr["denominator_after_block1"]) <= tol
    assert abs(trace[1]["l"] - pr["denominator_after_blocks_1_2"]) <= tol
    assert abs(trace[2]["l"] - pr["denominator_after_blocks_1_2_3"]) <= tol
    # block 1's second term is e^(7.2-12) = e^-4.8, the printed 0.0082
    assert abs((trace[0]["l"] - 1.0) - 0.0082) <= tol


def test_six_score_max_moves_and_rescale(six):
    """The max stays 12 through block 2 and becomes 13 at block 3; the carried
    state is multiplied by 1 at block 2 and by e^(12-13) = e^-1 at block 3."""
    pr = six["printed"]
    s = np.array(six["reconstruction"]["scores"], dtype=np.float64)
    _, trace = softmax_online_blocks(s, np.eye(6), pr["block_size"])
    assert [t["m"] for t in trace] == [12.0, pr["max_after_blocks_1_2"], pr["max_after_block_3"]]
    assert trace[1]["alpha"] == 1.0
    assert trace[2]["alpha"] == pytest.approx(math.exp(-1.0), abs=1e-15)


def test_six_score_online_equals_one_shot(six):
    """Processing the six scores in blocks of 2 gives the one-shot softmax
    result: with V = I6 the output is the probability row itself; with a
    seeded V it is the weighted sum A."""
    s = np.array(six["reconstruction"]["scores"], dtype=np.float64)
    out_eye, _ = softmax_online_blocks(s, np.eye(6), 2)
    np.testing.assert_allclose(out_eye, softmax_safe(s), rtol=0, atol=1e-15)
    v = np.random.default_rng(7).standard_normal((6, 5))
    out_v, _ = softmax_online_blocks(s, v, 2)
    np.testing.assert_allclose(out_v, softmax_safe(s) @ v, rtol=0, atol=1e-14)


def test_naive_per_block_sum_differs(six):
    """Normalising each block separately and adding is not softmax: the global
    denominator depends on all blocks."""
    s = np.array(six["reconstruction"]["scores"], dtype=np.float64)
    wrong = softmax_blocks_naive_sum(s, np.eye(6), 2)
    assert np.max(np.abs(wrong - softmax_safe(s))) > 0.1
    assert abs(np.sum(wrong) - 3.0) < 1e-12  # three blocks, each summing to 1


def test_appendix_overflow_and_shift_invariance(six):
    """e^12 ≈ 162,755 exceeds the fp16 maximum 65,504; subtracting the max
    leaves softmax unchanged and keeps every exponential <= 1."""
    ap = six["appendix"]
    assert round(math.exp(12)) == ap["exp_12_printed"]
    assert float(np.finfo(np.float16).max) == ap["fp16_max"]
    assert math.exp(12) > ap["fp16_max"]
    x = np.array(ap["scores"], dtype=np.float64)
    direct = np.exp(x) / np.sum(np.exp(x))
    np.testing.assert_allclose(softmax_safe(x), direct, rtol=1e-12, atol=0)
    # in fp16 the direct form overflows, the max-subtracted form does not
    with np.errstate(over="ignore"):
        assert not np.all(np.isfinite(np.exp(x.astype(np.float16))))
    shifted = np.exp((x - x.max()).astype(np.float16))
    assert np.all(np.isfinite(shifted)) and shifted.max() == 1.0
    np.testing.assert_allclose(softmax_safe(x + 1000.0), softmax_safe(x), rtol=1e-11)


def test_long_vector_three_blocks_vs_scipy():
    """Self-study exercise of the CMU 10-423 notes: sweep a long vector in
    three blocks keeping only the running max and denominator, and compare
    with scipy.special.softmax."""
    scipy_special = pytest.importorskip("scipy.special")
    x = np.random.default_rng(11).standard_normal(3001) * 5.0
    n = x.shape[0]
    out, trace = softmax_online_blocks(x, np.eye(n), block=(n + 2) // 3)
    assert len(trace) == 3
    np.testing.assert_allclose(out, scipy_special.softmax(x), rtol=1e-12, atol=1e-18)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rows_sum_to_one(seed):
    x = np.random.default_rng(seed).standard_normal((17, 33)) * 10
    p = softmax_safe(x)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-14)
    assert np.all(p >= 0)


@pytest.mark.parametrize("block", [1, 3, 7, 64])
def test_online_equals_safe_random(block):
    rng = np.random.default_rng(block)
    s = rng.standard_normal(200) * 6
    v = rng.standard_normal((200, 9))
    out, trace = softmax_online_blocks(s, v, block)
    np.testing.assert_allclose(out, softmax_safe(s) @ v, rtol=1e-13, atol=1e-14)
    # the running max never decreases and ends at the global max
    ms = [t["m"] for t in trace]
    assert all(b >= a for a, b in zip(ms, ms[1:])) and ms[-1] == s.max()
