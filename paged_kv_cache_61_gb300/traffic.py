"""Algorithmic byte and FLOP counts for decode attention.

These are the denominators of the roofline numbers ``bench.py`` reports. The
convention follows the drill page "L2 讲解：paged decode attention 与 GQA",
section ①: the algorithmic bytes of one decode step are the K and V bytes of
the ctx tokens actually attended (2 * B * ctx * Hkv * D * dtype_bytes for a
uniform batch). The cache-size arithmetic follows "Attention Kernel Variants:
MQA, GQA, and MLA", section "KV-Cache Arithmetic on Real Models":
  MHA/GQA/MQA: bytes/token = 2 * layers * kv_heads * head_dim * dtype_bytes
  MLA:         bytes/token = layers * (kv_lora_rank + rope_dim) * dtype_bytes
"""
from __future__ import annotations

from typing import Iterable


def gqa_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """Whole-model cached bytes per token for an MHA/GQA/MQA model (K and V)."""
    return 2 * layers * kv_heads * head_dim * dtype_bytes


def mla_bytes_per_token(layers: int, kv_lora_rank: int, rope_dim: int, dtype_bytes: int) -> int:
    """Whole-model cached bytes per token for an MLA model (latent + rope key, stored once)."""
    return layers * (kv_lora_rank + rope_dim) * dtype_bytes


def gqa_kv_bytes(context_lens: Iterable[int], kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """K+V bytes one decode step reads for one layer (only the ctx tokens of each sequence)."""
    return sum(int(c) for c in context_lens) * 2 * kv_heads * head_dim * dtype_bytes


def mla_kv_bytes(context_lens: Iterable[int], record_dim: int, dtype_bytes: int) -> int:
    """Latent-record bytes one MLA decode step reads (K and V share the record)."""
    return sum(int(c) for c in context_lens) * record_dim * dtype_bytes


def decode_flops(context_lens: Iterable[int], q_heads: int, head_dim_qk: int, head_dim_v: int) -> int:
    """Multiply-add FLOPs of one decode step: 2 * Hq * (Dqk + Dv) per attended token."""
    return sum(int(c) for c in context_lens) * q_heads * 2 * (head_dim_qk + head_dim_v)


def io_bytes(batch: int, q_heads: int, head_dim_qk: int, head_dim_v: int, dtype_bytes: int,
             num_pages_read: int) -> int:
    """Bytes outside the cache: q, out, fp32 lse, the block-table entries read and context_lens."""
    return (batch * q_heads * head_dim_qk * dtype_bytes + batch * q_heads * head_dim_v * dtype_bytes
            + batch * q_heads * 4 + num_pages_read * 4 + batch * 4)
