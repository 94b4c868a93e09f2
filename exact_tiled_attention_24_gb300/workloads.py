"""Seeded synthetic workloads for exact tiled attention.

This module only draws inputs; it holds none of the attention arithmetic, so
both the CUDA path and the fp64 CPU oracle can be fed from it without sharing
any computation.

Shapes follow the ``[B, heads, S, head_dim]`` activation layout of the
"07-16 下午：分布式大模型训练与推理" notes (section 自回归语言模型推理, step 3 of
the tensor walk-through), written here as ``[B, H, N, d]``. The five workloads
are the GPT-2-small, ragged-tile, Llama and long-context shapes this library is
measured on; the ragged one uses the context length 1028 with 64-wide tiles
that the dcwnkz.com FlashAttention walk-through (CS336 tricks, "回到
FlashAttention") uses as its example of tiling along N.

Recipe: ``torch.Generator().manual_seed(seed)`` on the CPU, fp32 normal draws
in the order q, k, v, dO, each multiplied by its standard deviation, then
rounded to bf16 (round-to-nearest-even). Seeds are ``1000 + config index``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple  # the causal settings this workload is run with
    directions: tuple  # ("fwd",) or ("fwd", "bwd")
    q_std: float = 1.0
    kv_std: float = 1.0
    seed: int = 1000
    Hkv: int = 0  # K/V heads (grouped-query attention); 0 means H

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 256, 64, (False,), ("fwd",), seed=1001),
    "c2": Workload("c2", 8, 12, 1024, 64, (True,), ("fwd", "bwd"), seed=1002),
    "c3": Workload("c3", 4, 12, 1028, 64, (False, True), ("fwd",), seed=1003),
    "c4": Workload("c4", 2, 32, 8192, 128, (True,), ("fwd", "bwd"), seed=1004),
    "c5": Workload("c5", 1, 16, 32768, 128, (True,), ("fwd",), q_std=4.0, seed=1005),
    # grouped-query heads: 32 query heads over 8 K/V heads (Llama-3-8B's head
    # layout), otherwise the c4 shape
    "g4": Workload("g4", 2, 32, 8192, 128, (True,), ("fwd", "bwd"), seed=1006, Hkv=8),
}

WORKLOAD_TITLES = {
    "c1": "attention fwd B=1 H=1 N=256 d=64 non-causal",
    "c2": "GPT-2-small-shaped attention fwd+bwd B=8 H=12 N=1024 d=64 causal",
    "c3": "ragged-tile attention fwd B=4 H=12 N=1028 d=64 non-causal and causal",
    "c4": "Llama-shaped attention fwd+bwd B=2 H=32 N=8192 d=128 causal",
    "c5": "long-context attention fwd B=1 H=16 N=32768 d=128 causal, Q ~ N(0, 4^2)",
    "g4": "grouped-query attention fwd+bwd B=2 H=32 Hkv=8 N=8192 d=128 causal",
}


def make_inputs(B, H, N, d, seed, q_std=1.0, kv_std=1.0, do_std=1.0, with_do=True, Hkv=None):
    """Draw q, k, v (and dO) as bf16 CPU tensors: q and dO [B, H, N, d], k and
    v [B, Hkv, N, d] (Hkv = H unless given)."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, N, d)
    kv_shape = (B, H if Hkv is None else Hkv, N, d)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * q_std).to(torch.bfloat16)
    k = (torch.randn(kv_shape, generator=g, dtype=torch.float32) * kv_std).to(torch.bfloat16)
    v = (torch.randn(kv_shape, generator=g, dtype=torch.float32) * kv_std).to(torch.bfloat16)
    out = [q, k, v]
    if with_do:
        do = (torch.randn(shape, generator=g, dtype=torch.float32) * do_std).to(torch.bfloat16)
        out.append(do)
    return tuple(out)


def workload_inputs(name: str, with_do=None):
    w = WORKLOADS[name]
    if with_do is None:
        with_do = "bwd" in w.directions
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, q_std=w.q_std, kv_std=w.kv_std, with_do=with_do,
                       Hkv=w.kv_heads)


@dataclass(frozen=True)
class RowsWorkload:
    """Rows for the standalone softmax kernels: x [rows, n] fp32 ~ N(0, std²).
    rows is a multiple of 608 (152 SMs x 4 resident 512-thread CTAs), so the
    one-CTA-per-row grid fills whole waves."""
    name: str
    rows: int
    n: int
    std: float
    seed: int


ROW_WORKLOADS = {
    # 1 MB rows: 608 rows in flight hold ~600 MB, so a pass's re-read of its
    # row misses the 126 MB L2 and goes to DRAM
    "s1": RowsWorkload("s1", 1216, 262144, 4.0, 2001),
    # 128 KB rows: ~78 MB in flight, so the re-reads can hit L2
    "s2": RowsWorkload("s2", 9728, 32768, 4.0, 2002),
}


@dataclass(frozen=True)
class DecodeWorkload:
    """One decode step of B requests against a paged KV cache: context
    lengths drawn uniformly from [min_len, max_len], cache blocks of
    block_size tokens placed in a random order, q, K, V ~ N(0, 1) in bf16."""
    name: str
    B: int
    H: int
    Hkv: int
    d: int
    block_size: int
    min_len: int
    max_len: int
    n_splits: int
    seed: int


DECODE_WORKLOADS = {
    # 32 requests with 2k-8k cached tokens, Llama-3-8B heads (32 over 8):
    # about 670 MB of K and V read per step, more than L2
    "d1": DecodeWorkload("d1", 32, 32, 8, 128, 16, 2048, 8192, 8, 3001),
    # the same step with one token per cache block (page size 1): the
    # blocks do not tile into TMA boxes and are gathered token by token
    "d2": DecodeWorkload("d2", 32, 32, 8, 128, 1, 2048, 8192, 8, 3001),
}


def make_decode(w: DecodeWorkload, device):
    """Seeded decode inputs, drawn on `device` (the cache is state that lives
    there): q [B, H, d], k_cache, v_cache [num_blocks, Hkv, bs, d],
    block_table [B, max_blocks] int32, seq_lens [B] int32."""
    g = torch.Generator().manual_seed(w.seed)
    lens = torch.randint(w.min_len, w.max_len + 1, (w.B,), generator=g, dtype=torch.int64)
    nb = (lens + w.block_size - 1) // w.block_size
    total = int(nb.sum())
    perm = torch.randperm(total, generator=g)
    table = torch.zeros((w.B, int(nb.max())), dtype=torch.int32)
    pos = 0
    for b in range(w.B):
        table[b, :nb[b]] = perm[pos:pos + int(nb[b])].to(torch.int32)
        pos += int(nb[b])
    gd = torch.Generator(device=device).manual_seed(w.seed + 1)
    q = torch.randn((w.B, w.H, w.d), generator=gd, device=device).to(torch.bfloat16)
    kc = torch.randn((total, w.Hkv, w.block_size, w.d), generator=gd, device=device).to(torch.bfloat16)
    vc = torch.randn((total, w.Hkv, w.block_size, w.d), generator=gd, device=device).to(torch.bfloat16)
    return q, kc, vc, table.to(device), lens.to(torch.int32).to(device)


def make_rows(rows, n, seed, std=1.0):
    """Draw x [rows, n] fp32 on the CPU from the seeded generator."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn((rows, n), generator=g, dtype=torch.float32) * std


def to_f64(t: torch.Tensor):
    """bf16 tensor -> exact float64 numpy array (bf16 values are exact in fp64)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
