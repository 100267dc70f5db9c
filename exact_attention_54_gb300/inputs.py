"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws i.i.d. N(0,1) values
(float32 draws rounded to the 16-bit storage type) and sequence lengths from a
seeded CPU generator, and names the workloads the library is measured on. The
CUDA path and the oracle both receive exactly these tensors.

Workloads (shapes from the pages' own benchmark tables; none is a dataset):
  tiny        B=1  H=2  Sq=Sk=128  D=64  fp16, causal and non-causal
  small       B=8  H=16 Sq=Sk=256  D=64  fp16, non-causal   ("Flash Attention 101", Benchmark)
  llama_prefill B=1 H=32 Sq=Sk=4096 D=128 bf16, causal     ("FlashAttention-2 MMA", LLaMA-7B Prefill row)
  decode      B=16 H=8  Sq=1 Sk=8192 D=128 bf16, 32 KV partitions ("FlashAttention-2 MMA", Decode KV row, batched)
  varlen      16 sequences, lengths uniform on [64, 2048], H=16 D=128 bf16, causal
  paged_decode the decode workload with K/V in 16-key pages behind a permuted block table
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "dense", "decode" or "varlen"
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    dtype: torch.dtype
    causal: bool
    seed: int
    num_splits: int = 0
    num_seqs: int = 0
    len_lo: int = 0
    len_hi: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    "tiny": Workload("tiny_b1h2s128d64_fp16", "dense", 1, 2, 128, 128, 64, torch.float16, False, 1001),
    "tiny_causal": Workload("tiny_b1h2s128d64_fp16_causal", "dense", 1, 2, 128, 128, 64, torch.float16, True, 1001),
    "small": Workload("small_b8h16s256d64_fp16", "dense", 8, 16, 256, 256, 64, torch.float16, False, 1002),
    "llama_prefill": Workload("llama7b_prefill_b1h32s4096d128_bf16_causal", "dense", 1, 32, 4096, 4096, 128,
                              torch.bfloat16, True, 1003),
    "decode": Workload("decode_b16h8sk8192d128_bf16_split32", "decode", 16, 8, 1, 8192, 128, torch.bfloat16,
                       False, 1004, num_splits=32),
    "varlen": Workload("varlen_16seq_len64to2048_h16d128_bf16_causal", "varlen", 0, 16, 0, 0, 128,
                       torch.bfloat16, True, 1005, num_seqs=16, len_lo=64, len_hi=2048),
    # the pages' large-head row, "GPT-4 style" (1, 16, 2048, 2048, 256): its
    # printed TFLOPS match the non-causal FLOP count; fp16 (the page's T4 has
    # no bf16)
    "d256": Workload("gpt4style_b1h16s2048d256_fp16", "dense", 1, 16, 2048, 2048, 256, torch.float16, False, 1007),
    # the pages' Split-D rows, "Large Head" (1, 8, 1024, 1024, 512) and
    # "Massive Head" (1, 4, 512, 512, 1024), non-causal fp16 like the row above
    "large_head": Workload("large_head_b1h8s1024d512_fp16", "dense", 1, 8, 1024, 1024, 512, torch.float16, False,
                           1008),
    "massive_head": Workload("massive_head_b1h4s512d1024_fp16", "dense", 1, 4, 512, 512, 1024, torch.float16, False,
                             1009),
    "paged_decode": Workload("paged_decode_b16h8sk8192d128_bf16_block16_split32", "paged", 16, 8, 1, 8192, 128,
                             torch.bfloat16, False, 1006, num_splits=32, extra={"block_size": 16}),
}


def randn(shape, dtype: torch.dtype, gen: torch.Generator) -> torch.Tensor:
    """N(0,1) drawn in float32 from ``gen`` and rounded to ``dtype`` (CPU tensor)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def make_dense(B: int, H: int, Sq: int, Sk: int, D: int, dtype: torch.dtype, seed: int):
    """Q [B,H,Sq,D], K and V [B,H,Sk,D]; drawn in the order Q, K, V from one generator."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = randn((B, H, Sq, D), dtype, g)
    k = randn((B, H, Sk, D), dtype, g)
    v = randn((B, H, Sk, D), dtype, g)
    return q, k, v


def make_lengths(num_seqs: int, lo: int, hi: int, gen: torch.Generator) -> torch.Tensor:
    """Sequence lengths uniform on the integers [lo, hi] (int64 CPU tensor)."""
    return torch.randint(lo, hi + 1, (num_seqs,), generator=gen)


def cu_from_lengths(lengths) -> torch.Tensor:
    """Cumulative offsets [0, L0, L0+L1, ...] as int32 (length num_seqs + 1)."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def make_varlen(num_seqs: int, lo: int, hi: int, H: int, D: int, dtype: torch.dtype, seed: int,
                lengths=None):
    """Packed self-attention batch: lengths (drawn first unless given), cu_seqlens,
    then Q, K, V as [total_tokens, H, D]."""
    g = torch.Generator("cpu").manual_seed(seed)
    if lengths is None:
        lengths = make_lengths(num_seqs, lo, hi, g)
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    q = randn((T, H, D), dtype, g)
    k = randn((T, H, D), dtype, g)
    v = randn((T, H, D), dtype, g)
    return lengths, cu, q, k, v


def make_paged(B: int, H: int, D: int, block_size: int, seq_lens, dtype: torch.dtype, seed: int,
               spare_blocks: int = 3):
    """Paged KV cache: pages [num_blocks, H, block_size, D] filled with N(0,1)
    (spare pages included), each sequence's logical blocks mapped to pages by a
    seeded permutation. Table entries past a sequence's blocks hold an
    out-of-range page number (they must never be read).
    Returns q [B,H,1,D], k_cache, v_cache, block_table [B, max_blocks] int32,
    seq_lens [B] int32."""
    g = torch.Generator("cpu").manual_seed(seed)
    lens = [int(x) for x in seq_lens]
    per = [-(-L // block_size) for L in lens]
    max_blocks = max(max(per), 1)
    num_blocks = sum(per) + spare_blocks
    perm = torch.randperm(num_blocks, generator=g)
    q = randn((B, H, 1, D), dtype, g)
    k_cache = randn((num_blocks, H, block_size, D), dtype, g)
    v_cache = randn((num_blocks, H, block_size, D), dtype, g)
    table = torch.full((B, max_blocks), num_blocks + 1000, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(per):
        table[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    return q, k_cache, v_cache, table, torch.tensor(lens, dtype=torch.int32)


def make_workload(w: Workload):
    """Inputs for a named workload (CPU tensors)."""
    if w.kind == "dense":
        return make_dense(w.B, w.H, w.Sq, w.Sk, w.D, w.dtype, w.seed)
    if w.kind == "decode":
        return make_dense(w.B, w.H, 1, w.Sk, w.D, w.dtype, w.seed)
    if w.kind == "varlen":
        return make_varlen(w.num_seqs, w.len_lo, w.len_hi, w.H, w.D, w.dtype, w.seed)
    if w.kind == "paged":
        return make_paged(w.B, w.H, w.D, w.extra["block_size"], [w.Sk] * w.B, w.dtype, w.seed)
    raise ValueError(w.kind)

