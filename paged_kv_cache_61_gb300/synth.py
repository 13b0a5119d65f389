"""Seeded synthetic inputs for paged decode attention.

This module only draws numbers: context lengths, block tables and 16-bit
query / cache values. It contains none of the attention arithmetic, so both the
float64 oracle (test side) and the CUDA path (product side) can take their
inputs from here without sharing any of the method's code.

Recipe (every workload):
  * one ``numpy.random.SeedSequence(seed)`` spawns independent streams for the
    context lengths, the block tables, q, the K cache and the V cache (the MLA
    latent cache uses the K stream), so the q values do not depend on how large
    the cache is;
  * values are N(0, 1) drawn in float32 and rounded to nearest-even to the
    16-bit storage type (fp16 or bf16); the arrays hold the raw 16-bit
    patterns (``uint16``);
  * block tables are random permutations of the physical block pool; table
    entries past a sequence's last page are filled with ``UNUSED_ENTRY`` (an
    out-of-range id) unless the workload says otherwise;
  * fp8 caches (``kv_format="e4m3"``): the same N(0, 1) float32 draws, divided by
    one per-tensor scale amax|x| / 448 (448 = the largest E4M3 value) and cast
    to E4M3 by PyTorch's float8_e4m3fn conversion; the arrays hold the codes
    (``uint8``) and the case carries the scales. q stays 16-bit.

Workload names follow the five decode workloads this library is measured on:
``gqa_tiny``, ``gqa_b64_ctx1k``, ``gqa_b1_ctx32k`` (``_mqa`` for one KV head),
``gqa_varlen_b128`` and ``mla_b16_ctx64k_h16`` / ``_h128``; ``mla_r256_b16_ctx64k_h16`` /
``_h128`` are the same MLA shapes with the kv_lora_rank 256 record (256 latent + 64 rope).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

FP16 = "fp16"
BF16 = "bf16"
FP8_E4M3 = "e4m3"          # cache format: one E4M3 byte per value, one scale per tensor
E4M3_MAX = 448.0
UNUSED_ENTRY = -1          # block-table filler past the last page of a sequence
_CHUNK = 1 << 22           # values drawn per call; fixed so results never depend on the caller


def _round_to_16bit(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to nearest-even fp16/bf16; return the bit patterns."""
    if dtype == FP16:
        return x32.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        bits = x32.view(np.uint32)
        rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        return rounded.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def normal_16bit(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) float32 draws rounded to ``dtype``; returns uint16 bit patterns of ``shape``."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    for start in range(0, n, _CHUNK):
        stop = min(n, start + _CHUNK)
        out[start:stop] = _round_to_16bit(rng.standard_normal(stop - start, dtype=np.float32), dtype)
    return out.reshape(shape)


def normal_e4m3(rng: np.random.Generator, shape):
    """N(0,1) float32 draws stored as E4M3 codes with one per-tensor scale.

    Returns (codes uint8 of ``shape``, scale) with scale = amax|x| / 448, so the
    largest draw maps to the largest finite code. The cast is PyTorch's.
    """
    import torch
    n = int(np.prod(shape, dtype=np.int64))
    x = np.empty(n, dtype=np.float32)
    for start in range(0, n, _CHUNK):
        stop = min(n, start + _CHUNK)
        x[start:stop] = rng.standard_normal(stop - start, dtype=np.float32)
    amax = float(np.abs(x).max()) if n else 1.0
    scale = np.float32(amax / E4M3_MAX if amax > 0 else 1.0)
    codes = np.empty(n, dtype=np.uint8)
    for start in range(0, n, _CHUNK):
        stop = min(n, start + _CHUNK)
        y = np.clip(x[start:stop] / scale, -E4M3_MAX, E4M3_MAX)
        codes[start:stop] = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes.reshape(shape), float(scale)


def float32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of float32 values (PyTorch's float8_e4m3fn cast; for structured inputs)."""
    import torch
    x = np.ascontiguousarray(x, dtype=np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bits_to_float32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of 16-bit patterns to float32 (for building structured inputs)."""
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def float32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to 16-bit patterns (nearest-even)."""
    return _round_to_16bit(np.ascontiguousarray(x, dtype=np.float32), dtype)


@dataclasses.dataclass
class DecodeCase:
    """One decode-attention problem in host memory (16-bit values stored as uint16 bits;
    with ``kv_format == "e4m3"`` the caches hold uint8 E4M3 codes, dequantized as
    code * k_scale (K, or the MLA record) and code * v_scale (V); with seq_len_q = S > 1
    there are S query tokens per sequence and q is [B, S, Hq, Dqk]).

    GQA (``kind == "gqa"``):
      q            [B, Hq, D]
      k_cache      [num_blocks, page_size, Hkv, D]
      v_cache      [num_blocks, page_size, Hkv, D]
    MLA (``kind == "mla"``):
      q            [B, Hq, Dqk]   (Dv absorbed-content dims then 64 rope dims; Dqk 576 or 320)
      kv_cache     [num_blocks, page_size, Dqk]  (K = all Dqk dims, V = the first Dv = Dqk - 64)
    Both:
      block_tables [B, max_blocks_per_seq] int32
      context_lens [B] int32
    """
    name: str
    kind: str
    dtype: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    page_size: int
    num_blocks: int
    scale: float
    context_lens: np.ndarray
    block_tables: np.ndarray
    q: np.ndarray
    k_cache: Optional[np.ndarray] = None
    v_cache: Optional[np.ndarray] = None
    kv_cache: Optional[np.ndarray] = None
    kv_format: Optional[str] = None
    k_scale: float = 1.0
    v_scale: float = 1.0
    seq_len_q: int = 1        # query tokens per sequence; > 1: q is [B, S, Hq, Dqk]

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(5)]


def _tables_from_pool(pool: np.ndarray, pages: np.ndarray, max_blocks: int,
                      fill_unused: Optional[int]) -> np.ndarray:
    """Hand consecutive entries of ``pool`` to each sequence, in batch order."""
    tables = np.full((len(pages), max_blocks), UNUSED_ENTRY if fill_unused is None else fill_unused,
                     dtype=np.int32)
    pos = 0
    for b, n in enumerate(pages):
        tables[b, :n] = pool[pos:pos + n]
        pos += int(n)
    return tables


def make_gqa_case(*, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  dtype: str, page_size: int = 16, context_lens=None, ctx_low: int = 1,
                  ctx_high: int = 256, ctx_dist: str = "fixed", num_blocks: Optional[int] = None,
                  max_blocks_per_seq: Optional[int] = None, scale: Optional[float] = None,
                  seed: int = 0, name: str = "gqa", table_layout: str = "pool",
                  kv_format: Optional[str] = None, seq_len_q: int = 1,
                  with_caches: bool = True) -> DecodeCase:
    """Build a GQA/MQA/MHA decode problem.

    ctx_dist: "fixed" (``context_lens`` given), "uniform" (integers in
    [ctx_low, ctx_high] inclusive) or "loguniform" (floor(exp(U(ln lo, ln hi))),
    clamped to [lo, hi]).
    table_layout: "pool" hands each sequence consecutive entries of a shuffled
    pool of exactly sum(pages) blocks (unused entries = UNUSED_ENTRY);
    "permutation" reshapes one random permutation of ``num_blocks`` ids into
    the [B, max_blocks_per_seq] table (every entry is a valid, distinct id).
    with_caches=False leaves the caches out (None): lengths, tables and q are the same
    draws either way, since every array has its own random stream.
    """
    r_ctx, r_tab, r_q, r_k, r_v = _streams(seed)
    if ctx_dist == "fixed":
        ctx = np.asarray(context_lens, dtype=np.int64).reshape(batch)
    elif ctx_dist == "uniform":
        ctx = r_ctx.integers(ctx_low, ctx_high, size=batch, endpoint=True)
    elif ctx_dist == "loguniform":
        u = r_ctx.uniform(math.log(ctx_low), math.log(ctx_high), size=batch)
        ctx = np.clip(np.floor(np.exp(u)), ctx_low, ctx_high)
    else:
        raise ValueError(ctx_dist)
    if seq_len_q > 1:
        ctx = np.maximum(ctx, seq_len_q)                   # every query token sees itself
    ctx = ctx.astype(np.int32)
    pages = (ctx.astype(np.int64) + page_size - 1) // page_size
    if max_blocks_per_seq is None:
        max_blocks_per_seq = int(max(1, pages.max(initial=1)))
    if table_layout == "permutation":
        if num_blocks is None:
            num_blocks = batch * max_blocks_per_seq
        assert num_blocks >= batch * max_blocks_per_seq
        perm = r_tab.permutation(num_blocks).astype(np.int32)
        tables = perm[: batch * max_blocks_per_seq].reshape(batch, max_blocks_per_seq).copy()
    elif table_layout == "pool":
        if num_blocks is None:
            num_blocks = int(pages.sum())
        assert num_blocks >= int(pages.sum())
        pool = r_tab.permutation(num_blocks).astype(np.int32)
        tables = _tables_from_pool(pool, pages, max_blocks_per_seq, None)
    else:
        raise ValueError(table_layout)
    q_shape = (batch, num_q_heads, head_dim) if seq_len_q == 1 else \
        (batch, seq_len_q, num_q_heads, head_dim)
    q = normal_16bit(r_q, q_shape, dtype)
    cache_shape = (num_blocks, page_size, num_kv_heads, head_dim)
    k_scale = v_scale = 1.0
    if not with_caches:
        k = v = None
    elif kv_format is None:
        k = normal_16bit(r_k, cache_shape, dtype)
        v = normal_16bit(r_v, cache_shape, dtype)
    elif kv_format == FP8_E4M3:
        k, k_scale = normal_e4m3(r_k, cache_shape)
        v, v_scale = normal_e4m3(r_v, cache_shape)
    else:
        raise ValueError(kv_format)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return DecodeCase(name=name, kind="gqa", dtype=dtype, batch=batch, num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads, head_dim_qk=head_dim, head_dim_v=head_dim,
                      page_size=page_size, num_blocks=int(num_blocks), scale=float(scale),
                      context_lens=ctx, block_tables=tables, q=q, k_cache=k, v_cache=v,
                      kv_format=kv_format, k_scale=k_scale, v_scale=v_scale,
                      seq_len_q=seq_len_q)


def make_mla_case(*, batch: int, num_q_heads: int, dtype: str = BF16, page_size: int = 64,
                  context_lens=None, ctx_low: int = 1, ctx_high: int = 4096, ctx_dist: str = "fixed",
                  latent_dim: int = 512, rope_dim: int = 64, num_blocks: Optional[int] = None,
                  scale: Optional[float] = None, seed: int = 0, name: str = "mla",
                  kv_format: Optional[str] = None, seq_len_q: int = 1,
                  with_caches: bool = True) -> DecodeCase:
    """Build an absorbed-MLA decode problem: one shared (latent_dim + rope_dim)-wide KV head.
    with_caches=False leaves the cache out (None), as for make_gqa_case."""
    r_ctx, r_tab, r_q, r_k, _ = _streams(seed)
    if ctx_dist == "fixed":
        ctx = np.asarray(context_lens, dtype=np.int64).reshape(batch)
    elif ctx_dist == "uniform":
        ctx = r_ctx.integers(ctx_low, ctx_high, size=batch, endpoint=True)
    else:
        raise ValueError(ctx_dist)
    if seq_len_q > 1:
        ctx = np.maximum(ctx, seq_len_q)                   # every query token sees itself
    ctx = ctx.astype(np.int32)
    pages = (ctx.astype(np.int64) + page_size - 1) // page_size
    max_blocks = int(max(1, pages.max(initial=1)))
    if num_blocks is None:
        num_blocks = int(pages.sum())
    pool = r_tab.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_pool(pool, pages, max_blocks, None)
    width = latent_dim + rope_dim
    q_shape = (batch, num_q_heads, width) if seq_len_q == 1 else \
        (batch, seq_len_q, num_q_heads, width)
    q = normal_16bit(r_q, q_shape, dtype)
    kv_scale = 1.0
    if not with_caches:
        kv = None
    elif kv_format is None:
        kv = normal_16bit(r_k, (num_blocks, page_size, width), dtype)
    elif kv_format == FP8_E4M3:
        kv, kv_scale = normal_e4m3(r_k, (num_blocks, page_size, width))
    else:
        raise ValueError(kv_format)
    if scale is None:
        scale = 1.0 / math.sqrt(192.0)
    return DecodeCase(name=name, kind="mla", dtype=dtype, batch=batch, num_q_heads=num_q_heads,
                      num_kv_heads=1, head_dim_qk=width, head_dim_v=latent_dim,
                      page_size=page_size, num_blocks=int(num_blocks), scale=float(scale),
                      context_lens=ctx, block_tables=tables, q=q, kv_cache=kv,
                      kv_format=kv_format, k_scale=kv_scale, v_scale=kv_scale,
                      seq_len_q=seq_len_q)


# The five decode workloads (seed 0 everywhere).
def workload(name: str, seed: int = 0, with_caches: bool = True) -> DecodeCase:
    """The named workload. Suffixes: ``_fp8`` gives the same workload with E4M3 caches,
    ``_mtp2`` two query tokens per sequence (causal, bottom-right aligned).
    with_caches=False: the same lengths, tables and q, without the caches."""
    fmt, sq = None, 1
    base = name
    if base.endswith("_fp8"):
        fmt, base = FP8_E4M3, base[: -len("_fp8")]
    if base.endswith("_mtp2"):
        sq, base = 2, base[: -len("_mtp2")]
    case = _workload16(base, seed, fmt, sq, with_caches)
    case.name = name
    return case


def _workload16(name: str, seed: int, kv_format: Optional[str], seq_len_q: int,
                with_caches: bool = True) -> DecodeCase:
    kw = dict(seed=seed, name=name, kv_format=kv_format, seq_len_q=seq_len_q,
              with_caches=with_caches)
    if name == "gqa_tiny":
        # B=4, Hq=8, Hkv=2, D=64, fp16, PAGE=16, ctx ~ U{1..256}, tables = one permutation of 64 blocks.
        return make_gqa_case(batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype=FP16,
                             ctx_dist="uniform", ctx_low=1, ctx_high=256, num_blocks=64,
                             max_blocks_per_seq=16, table_layout="permutation",
                             scale=1.0 / 8.0, **kw)
    if name == "gqa_b64_ctx1k":
        return make_gqa_case(batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype=FP16,
                             context_lens=[1024] * 64, table_layout="permutation", **kw)
    if name in ("gqa_b1_ctx32k", "gqa_b1_ctx32k_mqa", "gqa_b1_ctx32k_mqa_h64"):
        # _mqa: one KV head; _mqa_h64: one KV head shared by 64 query heads
        hkv = 1 if "_mqa" in name else 8
        hq = 64 if name.endswith("_h64") else 32
        return make_gqa_case(batch=1, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, dtype=BF16,
                             context_lens=[32768], table_layout="permutation", **kw)
    if name == "gqa_varlen_b128":
        return make_gqa_case(batch=128, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype=BF16,
                             ctx_dist="loguniform", ctx_low=16, ctx_high=32768,
                             max_blocks_per_seq=2048, table_layout="pool", **kw)
    if name in ("mla_b16_ctx64k_h16", "mla_b16_ctx64k_h128",
                "mla_r256_b16_ctx64k_h16", "mla_r256_b16_ctx64k_h128"):
        hq = 16 if name.endswith("h16") else 128
        latent = 256 if "_r256_" in name else 512
        return make_mla_case(batch=16, num_q_heads=hq, dtype=BF16, context_lens=[65536] * 16,
                             latent_dim=latent, **kw)
    raise KeyError(name)


WORKLOADS = ("gqa_tiny", "gqa_b64_ctx1k", "gqa_b1_ctx32k", "gqa_b1_ctx32k_mqa",
             "gqa_b1_ctx32k_mqa_h64", "gqa_b1_ctx32k_mqa_h64_fp8",
             "gqa_varlen_b128", "mla_b16_ctx64k_h16", "mla_b16_ctx64k_h128",
             "mla_r256_b16_ctx64k_h16", "mla_r256_b16_ctx64k_h128",
             "gqa_b64_ctx1k_fp8", "gqa_b1_ctx32k_fp8", "gqa_b1_ctx32k_mqa_fp8",
             "gqa_varlen_b128_fp8", "gqa_b64_ctx1k_mtp2", "gqa_b1_ctx32k_mtp2",
             "gqa_b64_ctx1k_mtp2_fp8", "mla_b16_ctx64k_h16_mtp2", "mla_b16_ctx64k_h128_mtp2",
             "mla_r256_b16_ctx64k_h128_mtp2", "mla_b16_ctx64k_h16_fp8",
             "mla_r256_b16_ctx64k_h16_fp8")
