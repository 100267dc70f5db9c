"""Algorithmic work counts used to turn a measured time into throughput.

FLOPs follow the convention of the pages' TFLOPS columns: two contractions of
2*Sq*Sk*D each per head, i.e. 4*B*H*Sq*Sk*D ("FlashAttention-2 MMA",
Performance Benchmarks: e.g. 135.38 ms for (1,32,4096,4096,128) printed as
2.03 TFLOPS). Causal work is counted at half of that. Decode traffic counts the
bytes that must cross HBM: every K and V element once, plus q in and O out.
"""
from __future__ import annotations


def attention_flops(B: int, H: int, Sq: int, Sk: int, D: int, causal: bool) -> float:
    f = 4.0 * B * H * Sq * Sk * D
    return f / 2.0 if causal else f


def varlen_flops(lengths_q, lengths_k, H: int, D: int, causal: bool) -> float:
    f = sum(4.0 * float(lq) * float(lk) * H * D for lq, lk in zip(lengths_q, lengths_k))
    return f / 2.0 if causal else f


def decode_bytes(B: int, H: int, Sk: int, D: int, elem_bytes: int = 2) -> float:
    """K and V read once, q read, O written (the split partials are excluded:
    they are implementation scratch, not algorithmic traffic)."""
    return float(B * H * (2 * Sk * D + 2 * D) * elem_bytes)


def prefill_bytes(B: int, H: int, Sq: int, Sk: int, D: int, elem_bytes: int = 2) -> float:
    """Compulsory HBM bytes of a dense forward: Q, K, V read once, O written, fp32 LSE written."""
    return float(B * H * ((2 * Sq + 2 * Sk) * D * elem_bytes + 4 * Sq))
