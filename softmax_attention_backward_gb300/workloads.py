"""Seeded synthetic inputs for the five attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the fp64 CPU oracle (through the tests) and the
CUDA path consume the very same tensors.

Recipe (one reading of the workload descriptions, fixed here once):
  * every tensor is drawn as float32 ``torch.randn`` from its own
    ``torch.Generator().manual_seed(seed)`` on the CPU and rounded to bf16;
    draw order is Q, K, V, dO (sparse: Q, KV, dO);
  * the variable-length lengths come from a second generator with the same seed:
    ``torch.randint(512, 8193, (4,))``;
  * the top-k index sets come from a third generator: token t takes every key of
    ``[0, t]`` when ``t < k``, else the first ``k`` entries of
    ``torch.randperm(t + 1)`` sorted ascending; rows are padded with -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16 = torch.bfloat16


def _randn(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(BF16)


# ----------------------------------------------------------------------------
# Dense BSHD and THD inputs
# ----------------------------------------------------------------------------
def dense_inputs(batch: int, seqlen: int, heads_q: int, heads_kv: int, head_dim: int,
                 seed: int):
    """Q [B,S,Hq,D], K/V [B,S,Hkv,D], dO [B,S,Hq,D], bf16, CPU."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (batch, seqlen, heads_q, head_dim))
    k = _randn(g, (batch, seqlen, heads_kv, head_dim))
    v = _randn(g, (batch, seqlen, heads_kv, head_dim))
    do = _randn(g, (batch, seqlen, heads_q, head_dim))
    return q, k, v, do


def varlen_lengths(seed: int = 3, num_seqs: int = 4, lo: int = 512, hi: int = 8192):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (num_seqs,), generator=g).tolist()


def cu_seqlens_from(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def thd_inputs(capacity: int, heads_q: int, heads_kv: int, head_dim: int, seed: int):
    """Packed THD buffers of static capacity: Q/dO [cap,Hq,D], K/V [cap,Hkv,D].

    Rows past the last sequence hold finite random values as well: the kernels
    must ignore them, which the parity tests check."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (capacity, heads_q, head_dim))
    k = _randn(g, (capacity, heads_kv, head_dim))
    v = _randn(g, (capacity, heads_kv, head_dim))
    do = _randn(g, (capacity, heads_q, head_dim))
    return q, k, v, do


# ----------------------------------------------------------------------------
# Top-k sparse (one shared KV head, 576 = 512 latent + 64 rope)
# ----------------------------------------------------------------------------
SPARSE_DQK = 576
SPARSE_DV = 512


def topk_indices(tokens: int, topk: int, seed: int, causal_window: bool = True) -> torch.Tensor:
    """int32 [T, topk]: token t selects min(topk, t+1) distinct keys of [0, t],
    sorted ascending, padded with -1."""
    g = torch.Generator().manual_seed(seed)
    idx = torch.full((tokens, topk), -1, dtype=torch.int32)
    for t in range(tokens):
        n = t + 1
        if n <= topk:
            idx[t, :n] = torch.arange(n, dtype=torch.int32)
        else:
            sel = torch.randperm(n, generator=g)[:topk].sort().values
            idx[t, :] = sel.to(torch.int32)
    return idx


def sparse_inputs(tokens: int, heads: int, topk: int, seed: int):
    """Q [T,H,576], KV [T,576], dO [T,H,512] bf16 and idx [T,topk] int32."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (tokens, heads, SPARSE_DQK))
    kv = _randn(g, (tokens, SPARSE_DQK))
    do = _randn(g, (tokens, heads, SPARSE_DV))
    idx = topk_indices(tokens, topk, seed)
    return q, kv, do, idx


# ----------------------------------------------------------------------------
# DSA lightning indexer (H index heads of dim 128, one key per token)
# ----------------------------------------------------------------------------
INDEXER_D = 128


def indexer_inputs(tokens: int, heads: int, seed: int, topk: int = 0):
    """q bf16 [T,H,128], k bf16 [T,128] N(0,1); w fp32 [T,H] N(0,1)/sqrt(H); and,
    with topk > 0, grad fp32 [T,topk] N(0,1) (a gradient for the selected
    logits)."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (tokens, heads, INDEXER_D))
    k = _randn(g, (tokens, INDEXER_D))
    w = torch.randn(tokens, heads, generator=g, dtype=torch.float32) / math.sqrt(heads)
    out = dict(q=q, k=k, w=w)
    if topk > 0:
        out["grad"] = torch.randn(tokens, topk, generator=g, dtype=torch.float32)
    return out


# The indexer workload: the sparse attention workload's token count and top-k
# (one causal sequence of 8192 tokens, 2048 keys per query) with 64 index heads.
INDEXER_WORKLOAD = dict(name="indexer_t8192_h64_d128_top2048", tokens=8192, heads=64, topk=2048,
                        seed=5)


# ----------------------------------------------------------------------------
# CSA compressor gated pooling (THD packs, one head)
# ----------------------------------------------------------------------------
def csa_inputs(lengths, head_dim: int, ratio: int, coff: int, seed: int, pad_tokens: int = 0,
               pad_rows: int = 0):
    """kv, score bf16 [T, coff*D] and dout bf16 [C_cap, D] N(0,1), ape fp32
    [ratio, coff*D] N(0,1); cu_seqlens and cu_seqlens_comp int32 (floor(len/ratio)
    rows per segment).  T = sum(lengths) + pad_tokens, C_cap = total rows +
    pad_rows; padding rows hold finite random values too."""
    g = torch.Generator().manual_seed(seed)
    T = sum(int(n) for n in lengths) + pad_tokens
    comp = [int(n) // ratio for n in lengths]
    C = sum(comp) + pad_rows
    kv = _randn(g, (T, coff * head_dim))
    score = _randn(g, (T, coff * head_dim))
    ape = torch.randn(ratio, coff * head_dim, generator=g, dtype=torch.float32)
    dout = _randn(g, (C, head_dim))
    return dict(kv=kv, score=score, ape=ape, dout=dout, cu_seqlens=cu_seqlens_from(lengths),
                cu_seqlens_comp=cu_seqlens_from(comp), comp_capacity=C)


# Compressor shapes of the page's benchmark table: THD packs of 8192-token
# sequences, ratio 4, coff 2, head_dim 128 or 512.
CSA_WORKLOADS = {
    "csa_1x8192_d128": dict(lengths=[8192], head_dim=128, ratio=4, coff=2, seed=41),
    "csa_3x8192_d128": dict(lengths=[8192] * 3, head_dim=128, ratio=4, coff=2, seed=42),
    "csa_1x8192_d512": dict(lengths=[8192], head_dim=512, ratio=4, coff=2, seed=43),
    "csa_3x8192_d512": dict(lengths=[8192] * 3, head_dim=512, ratio=4, coff=2, seed=44),
}


# ----------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    kind: str                 # "dense", "thd" or "sparse"
    batch: int = 1
    seqlen: int = 0
    heads_q: int = 0
    heads_kv: int = 0
    head_dim: int = 0
    causal: bool = False
    seed: int = 0
    lengths: list = field(default_factory=list)
    capacity: int = 0
    topk: int = 0

    @property
    def scale(self) -> float:
        d = SPARSE_DQK if self.kind == "sparse" else self.head_dim
        return 1.0 / math.sqrt(d)


WORKLOADS = {
    "mha_s128_d64": Workload("mha_s128_d64", "dense", batch=1, seqlen=128, heads_q=2,
                             heads_kv=2, head_dim=64, causal=False, seed=0),
    "mha_causal_b8_h32_s1024_d64": Workload("mha_causal_b8_h32_s1024_d64", "dense", batch=8,
                                            seqlen=1024, heads_q=32, heads_kv=32,
                                            head_dim=64, causal=True, seed=1),
    "gqa_causal_b4_h32x8_s4096_d128": Workload("gqa_causal_b4_h32x8_s4096_d128", "dense",
                                               batch=4, seqlen=4096, heads_q=32, heads_kv=8,
                                               head_dim=128, causal=True, seed=2),
    "thd_varlen_causal_h16_d128": Workload("thd_varlen_causal_h16_d128", "thd", heads_q=16,
                                           heads_kv=16, head_dim=128, causal=True, seed=3,
                                           capacity=32768),
    "sparse_topk2048_t8192_h64": Workload("sparse_topk2048_t8192_h64", "sparse", seqlen=8192,
                                          heads_q=64, heads_kv=1, head_dim=SPARSE_DQK,
                                          seed=4, topk=2048),
}


def get_workload(name: str) -> Workload:
    w = WORKLOADS[name]
    if w.kind == "thd" and not w.lengths:
        w.lengths = varlen_lengths(w.seed)
    return w


def make_inputs(w: Workload):
    """Returns a dict of CPU tensors for the workload."""
    if w.kind == "dense":
        q, k, v, do = dense_inputs(w.batch, w.seqlen, w.heads_q, w.heads_kv, w.head_dim, w.seed)
        return dict(q=q, k=k, v=v, do=do)
    if w.kind == "thd":
        q, k, v, do = thd_inputs(w.capacity, w.heads_q, w.heads_kv, w.head_dim, w.seed)
        return dict(q=q, k=k, v=v, do=do, cu_seqlens=cu_seqlens_from(w.lengths))
    if w.kind == "sparse":
        q, kv, do, idx = sparse_inputs(w.seqlen, w.heads_q, w.topk, w.seed)
        return dict(q=q, kv=kv, do=do, idx=idx)
    raise ValueError(w.kind)
