"""fp64 CPU oracle for exact attention, its backward, and (online) softmax.

TEST INFRASTRUCTURE ONLY. Only the tests, the package's ``smoke()`` check and
the benchmark's CPU-baseline / reference leg may import this module. The
library's CUDA path never calls it and shares no code with it.

What it computes, and where the pages state it:

* Attention (dcwnkz.com FlashAttention walk-through, CS336 tricks, "先简要回顾
  注意力机制"): scores are the q·k dot products, i.e. Q Kᵀ; softmax turns each
  row of scores into weights that sum to 1; the output is the weighted sum of
  the value vectors.  The 1/sqrt(d) factor is not printed on the pages; it is
  passed in explicitly as ``scale``.
* Safe softmax, three passes (same article, appendix on softmax; CMU 10-423
  L17–L18 notes, section 前置二：online softmax): subtract the row maximum before
  exponentiating, sum, then normalise.
* Causal mask ("07-16 下午：分布式大模型训练与推理", section 自回归语言模型推理):
  position i only sees positions j <= i (itself included).
* Online softmax over blocks (dcwnkz.com six-score worked example; "07-16 下午"
  notes, section 长上下文与序列并行): carry the running max m, the running
  denominator l and the running weighted sum u; when a block raises the max,
  multiply l and u by e^(m_old - m_new) before adding the block.
* Backward: the pages only say the attention matrix is never stored and the
  needed block is recomputed (CMU 10-423 L17–L18 notes, section FlashAttention
  本身, item 2).  The gradients below are those of o = softmax(scale·q Kᵀ) V,
  written out plainly: dV = Pᵀ dO, dP = dO Vᵀ, D_i = Σ_j P_ij dP_ij,
  dS = P ∘ (dP − D), dQ = scale·dS K, dK = scale·dSᵀ Q.

Every function works in float64 on numpy arrays. Rows are processed in chunks
so that one chunk of S stays bounded in memory; chunking over rows is exact
(rows of softmax are independent), no other blocking or reordering is done.
"""
from __future__ import annotations

import math

import numpy as np

ROW_CHUNK = 1024


# --------------------------------------------------------------------------
# softmax
# --------------------------------------------------------------------------

def softmax_safe(x: np.ndarray) -> np.ndarray:
    """Three-pass safe softmax along the last axis (max, sum of exps, divide)."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)          # pass 1: the max
    e = np.exp(x - m)
    l = np.sum(e, axis=-1, keepdims=True)          # pass 2: the denominator
    return e / l                                   # pass 3: normalise


def softmax_online_blocks(scores, values, block):
    """Block-by-block online softmax-weighted sum of one row of scores.

    Follows the six-score walk-through: each block's exponentials are taken
    relative to the running max; when a later block holds a larger max, the
    carried numerator u and denominator l are both multiplied by
    e^(m_old - m_new); normalisation happens once, at the end.

    Returns (output, trace), where trace holds one dict per block with the
    running max ``m``, the factor ``alpha`` applied to the carried state, and
    the running denominator ``l`` after the block.
    """
    s = np.asarray(scores, dtype=np.float64)
    vals = np.asarray(values, dtype=np.float64)
    n = s.shape[0]
    m = -math.inf
    l = 0.0
    u = np.zeros(vals.shape[1:], dtype=np.float64)
    trace = []
    for start in range(0, n, block):
        sb = s[start:start + block]
        vb = vals[start:start + block]
        m_new = max(m, float(np.max(sb)))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        e = np.exp(sb - m_new)
        l = alpha * l + float(np.sum(e))
        u = alpha * u + np.tensordot(e, vb, axes=(0, 0))
        trace.append({"m": m_new, "alpha": alpha if start else 1.0, "l": l})
        m = m_new
    return u / l, trace


def softmax_blocks_naive_sum(scores, values, block):
    """The WRONG way the long-context notes warn about: normalise each block
    on its own and add the blocks.  Kept only so a test can show it differs."""
    s = np.asarray(scores, dtype=np.float64)
    vals = np.asarray(values, dtype=np.float64)
    out = np.zeros(vals.shape[1:], dtype=np.float64)
    for start in range(0, s.shape[0], block):
        p = softmax_safe(s[start:start + block])
        out = out + np.tensordot(p, vals[start:start + block], axes=(0, 0))
    return out


# --------------------------------------------------------------------------
# attention forward
# --------------------------------------------------------------------------

def _scores(qb, k, scale, rows, causal):
    """scale·q_i·k_j for the query rows ``rows`` against all keys, with the
    causal mask (key j visible to query i iff j <= i) applied as -inf."""
    s = scale * (qb @ k.T)
    if causal:
        cols = np.arange(k.shape[0])
        s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
    return s


def attention_fwd_head(q, k, v, scale, causal, rows=None):
    """One head. q: [Nq_rows..] k, v: [N, d].  Returns (o, lse) for ``rows``
    (all rows when None).  lse_i = m_i + ln l_i in natural-log units."""
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    o = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.empty(rows.shape[0], dtype=np.float64)
    for c0 in range(0, rows.shape[0], ROW_CHUNK):
        r = rows[c0:c0 + ROW_CHUNK]
        s = _scores(q[r], k, scale, r, causal)
        m = np.max(s, axis=1, keepdims=True)              # pass 1
        e = np.exp(s - m)
        l = np.sum(e, axis=1, keepdims=True)              # pass 2
        p = e / l                                         # pass 3
        o[c0:c0 + r.shape[0]] = p @ v
        lse[c0:c0 + r.shape[0]] = (m + np.log(l))[:, 0]
    return o, lse


def attention_fwd(q, k, v, scale, causal):
    """q, k, v: [B, H, N, d] float64.  Returns o [B, H, N, d], lse [B, H, N]."""
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_fwd_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return o, lse


# --------------------------------------------------------------------------
# attention backward
# --------------------------------------------------------------------------

def attention_bwd_head(q, k, v, do, scale, causal):
    """Gradients of o = softmax(scale·q kᵀ) v for one head, with P rebuilt
    from its definition chunk by chunk (nothing from a forward is reused).
    Returns dq, dk, dv [N, d] and D [N] (D_i = Σ_j P_ij dP_ij)."""
    n = q.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.empty(n, dtype=np.float64)
    for c0 in range(0, n, ROW_CHUNK):
        r = np.arange(c0, min(n, c0 + ROW_CHUNK))
        s = _scores(q[r], k, scale, r, causal)
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / np.sum(e, axis=1, keepdims=True)
        dv += p.T @ do[r]
        dp = do[r] @ v.T
        Dr = np.sum(p * dp, axis=1)
        ds = p * (dp - Dr[:, None])
        dq[r] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r])
        D[r] = Dr
    return dq, dk, dv, D


def attention_bwd(q, k, v, do, scale, causal):
    """[B, H, N, d] float64 inputs.  Returns dq, dk, dv [B, H, N, d] and D [B, H, N]."""
    B, H, N, d = q.shape
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    D = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h], D[b, h] = attention_bwd_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv, D


def attention_dq_rows_head(q, k, v, do, scale, causal, rows):
    """dQ for selected query rows of one head.  Row i of dQ depends on row i
    of Q and dO only (through row i of P), so each sampled row is computed
    from the same definitions as ``attention_bwd_head``."""
    rows = np.asarray(rows)
    s = _scores(q[rows], k, scale, rows, causal)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    p = e / np.sum(e, axis=1, keepdims=True)
    dp = do[rows] @ v.T
    Dr = np.sum(p * dp, axis=1)
    ds = p * (dp - Dr[:, None])
    return scale * (ds @ k), Dr


# --------------------------------------------------------------------------
# grouped-query attention
# --------------------------------------------------------------------------
# "07-16 下午" notes, section 自回归语言模型推理 (Prefill、Decode 与推理调度):
# with grouped-query attention the number of K/V heads is smaller than the
# number of query heads.  The pages give no head mapping; the reading used
# here is the usual one: H / Hkv consecutive query heads share one K/V head,
# query head h reading K/V head h // (H / Hkv).  Attention per query head is
# then exactly the attention above, and since one K/V head feeds several
# query heads, its gradient is the sum of theirs.

def kv_head_of(h, H, Hkv):
    """K/V head read by query head h."""
    return h // (H // Hkv)


def attention_fwd_gqa(q, k, v, scale, causal):
    """q: [B, H, N, d]; k, v: [B, Hkv, N, d] float64 (Hkv divides H).
    Returns o [B, H, N, d], lse [B, H, N]."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            o[b, h], lse[b, h] = attention_fwd_head(q[b, h], k[b, g], v[b, g], scale, causal)
    return o, lse


def attention_bwd_gqa(q, k, v, do, scale, causal):
    """Gradients for grouped-query heads: dq [B, H, N, d], dk, dv
    [B, Hkv, N, d] (each the sum over the query heads sharing that K/V
    head) and D [B, H, N]."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            dq[b, h], dkh, dvh, D[b, h] = attention_bwd_head(q[b, h], k[b, g], v[b, g], do[b, h],
                                                             scale, causal)
            dk[b, g] += dkh
            dv[b, g] += dvh
    return dq, dk, dv, D


# --------------------------------------------------------------------------
# merging partial attention over disjoint key blocks
# --------------------------------------------------------------------------
# "07-16 下午" notes, section 长上下文与序列并行: partial softmax results of
# different K/V blocks cannot be normalised separately and added, because
# the global denominator depends on every block.  Carry the running maximum
# m, the normaliser l and the weighted sum u; when a block arrives, rescale
# the old l and u by e^(m_old - m_new) and add the block's.  A partial result
# over a block is stored as (o_s, lse_s) with o_s = u_s / l_s and
# lse_s = m_s + ln l_s, i.e. the block state (m, l, u) = (lse_s, 1, o_s).

def attention_merge(o_parts, lse_parts):
    """o_parts [S, rows, d], lse_parts [S, rows] (natural log; -inf for a
    part that saw no key) -> o [rows, d], lse [rows], processing the parts
    in order with the rescaling recurrence above."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    rows, d = o_parts.shape[1], o_parts.shape[2]
    m = np.full(rows, -np.inf)
    l = np.zeros(rows)
    u = np.zeros((rows, d))
    for o_s, lse_s in zip(o_parts, lse_parts):
        m_new = np.maximum(m, lse_s)
        live = np.isfinite(m_new)  # some part so far saw a key
        with np.errstate(invalid="ignore"):
            a_old = np.where(live, np.exp(np.where(live, m - m_new, 0.0)), 0.0)
            a_new = np.where(live, np.exp(np.where(live, lse_s - m_new, 0.0)), 0.0)
        l = l * a_old + a_new
        u = u * a_old[:, None] + o_s * a_new[:, None]
        m = m_new
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(l[:, None] > 0, u / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


# --------------------------------------------------------------------------
# decode against a paged KV cache
# --------------------------------------------------------------------------
# CMU 10-423 L17–L18 notes, section 解碼端：PagedAttention: the KV cache is cut
# into blocks of a fixed number of tokens stored non-contiguously, and a
# block table maps a sequence's logical blocks to physical ones.  "07-16
# 下午" notes, section Prefill、Decode 与推理调度: a decode step feeds one new
# token per request, whose query attends to the keys and values of every
# cached token of that request (the new token's own included).
# Layout read here (the pages fix none): k_cache, v_cache
# [num_blocks, Hkv, block_size, d]; token t of request b sits in physical
# block block_table[b, t // block_size], slot t % block_size.

def gather_paged(cache, block_table_row, seq_len):
    """Contiguous [Hkv, seq_len, d] copy of one request's cached keys or values."""
    bs = cache.shape[2]
    t = np.arange(seq_len)
    blocks = np.asarray(block_table_row)[t // bs]
    return cache[blocks, :, t % bs, :].transpose(1, 0, 2)


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale):
    """q [B, H, d] (one query row per request) -> o [B, H, d], lse [B, H].
    Query head h reads K/V head h // (H / Hkv)."""
    B, H, d = q.shape
    Hkv = k_cache.shape[1]
    o = np.zeros((B, H, d))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        K = gather_paged(k_cache, block_table[b], L)
        V = gather_paged(v_cache, block_table[b], L)
        for h in range(H):
            g = kv_head_of(h, H, Hkv)
            ob, lb = attention_fwd_head(q[b, h][None, :], K[g], V[g], scale, False)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


# --------------------------------------------------------------------------
# FLOP convention used when this oracle is timed
# --------------------------------------------------------------------------

def attention_pairs(N, causal):
    """Query-key pairs the method computes: N² or N(N+1)/2 with the causal mask."""
    return N * (N + 1) // 2 if causal else N * N


def attention_flops(B, H, N, d, causal, direction):
    """Algorithmic tensor FLOPs: 2mkn per [m,k]x[k,n] product ("07-16 下午"
    notes, section Transformer 层的算力估算).  Forward = 2 products (QKᵀ, PV),
    backward = 5 products (recomputed S, dV, dP, dK, dQ)."""
    per_pair = {"fwd": 4 * d, "bwd": 10 * d}[direction]
    return per_pair * B * H * attention_pairs(N, causal)
