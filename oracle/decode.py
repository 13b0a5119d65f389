"""Float64 CPU oracle for single-token decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA path.

What it computes is the plain definition, written out without blocking,
fusion or reordering:

  for each sequence b, query head h, logical token j < ctx_b:
      phys  = block_tables[b, j // P]                 (paged addressing)
      slot  = j %  P
      K_j   = k_cache[phys, slot, h // G, :]           (contiguous grouping, G = Hq / Hkv)
      V_j   = v_cache[phys, slot, h // G, :]
      s_j   = scale * <q[b, h], K_j>
  m = max_j s_j;  Z = sum_j exp(s_j - m)
  out[b, h] = sum_j exp(s_j - m) V_j / Z,   lse[b, h] = m + ln Z   (natural log)

Sources (web pages this library follows):
  * "From MHA to MLA: KV Caches and Attention Kernels" (g-u-n.github.io),
    section 2 (head mapping h -> h // G), section 3 (grouped decode: masked
    rows, online softmax whose end result is the expression above, LSE),
    section 4 (Flash-Decoding: per-split normalized output O_s and L_s and the
    weighted combine), section 5 (paged addressing: logical page n // P,
    offset n - page * P, physical page from the block table), section 6
    (absorbed MLA: score = content dot + rope dot, value = latent only).
  * "L2 讲解：paged decode attention 与 GQA" (kzhou003.github.io gpu-kernel-drills),
    section ④ (page loop: num_pages = cdiv(ctx, PAGE), phys looked up per
    page, last page masked) and the pitfalls list (contiguous grouping).
  * FlashMLA-ETAP README, "Supported configurations" and "Usage": K and V share
    one 576-wide cache tensor, head_dim_v = 512, lse is float32 log-sum-exp.

Inputs are the 16-bit bit patterns produced by the shared input generator; the
oracle widens them exactly to float64 itself.

fp8 caches ("Attention Kernel Variants: MQA, GQA, and MLA" (vanos001.github.io),
the KV-cache arithmetic table's fp8 MLA row and pitfall 5: an fp8 cache stores
one byte per cached value and kernels dequantize its tiles before the attention
arithmetic). The pages fix no format details beyond "fp8", so the oracle reads
each byte as an E4M3 code (the OCP 8-bit floating-point format: 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN) and
multiplies it by one per-tensor scale: K_j = e4m3(code) * k_scale, V_j likewise
with v_scale (MLA: one kv_scale for the record).
"""
from __future__ import annotations

import numpy as np

FP16 = "fp16"
BF16 = "bf16"


# --------------------------------------------------------------------------------------
# exact widening of stored 16-bit values
# --------------------------------------------------------------------------------------
def widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> float64, exactly (fp16 via numpy's float16; bf16 = high half of a float32)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


FP8_E4M3 = "e4m3"


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """E4M3 byte codes -> float64, exactly, from the format's definition.

    sign s = bit 7, exponent field e = bits 6..3, mantissa field m = bits 2..0:
      e == 15 and m == 7 -> NaN (the format has no infinities)
      e == 0             -> (-1)^s * 2^(1 - 7) * (m / 8)      (subnormal, zero)
      otherwise          -> (-1)^s * 2^(e - 7) * (1 + m / 8)
    """
    codes = np.asarray(codes, dtype=np.uint8)
    sign = np.where((codes >> 7) & 1, -1.0, 1.0)
    e = ((codes >> 3) & 0xF).astype(np.int64)
    m = (codes & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, e - 7)
    subnormal = sign * np.ldexp(m / 8.0, 1 - 7)
    out = np.where(e == 0, subnormal, normal)
    return np.where((e == 15) & (m == 7), np.nan, out)


def dequantize(stored: np.ndarray, dtype: str, kv_format: str = None, scale: float = 1.0):
    """Cached values as float64: 16-bit patterns widened (kv_format None), or E4M3 codes
    decoded and multiplied by the per-tensor scale (kv_format "e4m3")."""
    if kv_format is None:
        return widen(stored, dtype)
    if kv_format == FP8_E4M3:
        return decode_e4m3(stored) * float(scale)
    raise ValueError(kv_format)


# --------------------------------------------------------------------------------------
# paged addressing ("From MHA to MLA", section 5; drill page, section ④)
# --------------------------------------------------------------------------------------
def num_pages(ctx: int, page_size: int) -> int:
    """cdiv(ctx, PAGE): how many block-table entries a sequence of ``ctx`` tokens uses."""
    return (int(ctx) + page_size - 1) // page_size


def token_locations(block_table_row: np.ndarray, ctx: int, page_size: int):
    """(physical block, slot) of logical tokens 0..ctx-1.

    Logical token n lives on logical page n // P at offset n - (n // P) * P; the
    block table maps the logical page to a physical block. Only the first
    cdiv(ctx, P) table entries are read.
    """
    phys = []
    slots = []
    for n in range(int(ctx)):
        logical_page = n // page_size
        offset = n - logical_page * page_size
        phys.append(int(block_table_row[logical_page]))
        slots.append(offset)
    return np.asarray(phys, dtype=np.int64), np.asarray(slots, dtype=np.int64)


def gather_tokens(cache: np.ndarray, block_table_row: np.ndarray, ctx: int, page_size: int):
    """Rows of ``cache[num_blocks, P, ...]`` for logical tokens 0..ctx-1, in token order."""
    phys, slots = token_locations(block_table_row, ctx, page_size)
    return cache[phys, slots]


# --------------------------------------------------------------------------------------
# attention over one gathered sequence ("From MHA to MLA", sections 2-3)
# --------------------------------------------------------------------------------------
def attend(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """softmax(scale * q K^T) V and its natural-log LSE, in float64.

    q_rows [n, Dqk], keys [L, Dqk], values [L, Dv] (L >= 1) -> out [n, Dv], lse [n].
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    s = float(scale) * (q_rows @ keys.T)          # [n, L] scaled logits
    m = s.max(axis=1)                              # row maximum
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)                              # softmax denominator
    out = (e @ values) / z[:, None]
    lse = m + np.log(z)
    return out, lse


# --------------------------------------------------------------------------------------
# GQA / MQA / MHA paged decode
# --------------------------------------------------------------------------------------
def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Contiguous grouping: query head h reads KV head h // G, G = Hq / Hkv."""
    if num_q_heads % num_kv_heads:
        raise ValueError("H_q must be divisible by H_kv")
    return h // (num_q_heads // num_kv_heads)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, page_size, dtype,
                 rows=None, kv_format=None, k_scale=1.0, v_scale=1.0):
    """Oracle for GQA/MQA/MHA decode over a paged cache.

    q [B, Hq, D] (16-bit bits), k_cache/v_cache [NB, P, Hkv, D] (bits; E4M3 codes when
    kv_format is "e4m3", dequantized with k_scale / v_scale),
    block_tables [B, max_blocks] int32, context_lens [B] int32 (>= 1).
    rows: optional list of (b, h) pairs to evaluate (others left NaN).
    Returns out [B, Hq, Dv] float64 and lse [B, Hq] float64.
    """
    B, Hq, _ = q.shape
    Hkv = k_cache.shape[2]
    Dv = v_cache.shape[3]
    out = np.full((B, Hq, Dv), np.nan)
    lse = np.full((B, Hq), np.nan)
    wanted = None if rows is None else {(int(b), int(h)) for b, h in rows}
    for b in range(B):
        ctx = int(context_lens[b])
        if ctx < 1:
            raise ValueError("context length must be >= 1")
        heads_by_kv = {}
        for h in range(Hq):
            if wanted is not None and (b, h) not in wanted:
                continue
            heads_by_kv.setdefault(kv_head_of(h, Hq, Hkv), []).append(h)
        for kvh, heads in heads_by_kv.items():
            keys = dequantize(gather_tokens(k_cache[:, :, kvh, :], block_tables[b], ctx, page_size),
                              dtype, kv_format, k_scale)
            vals = dequantize(gather_tokens(v_cache[:, :, kvh, :], block_tables[b], ctx, page_size),
                              dtype, kv_format, v_scale)
            o, l = attend(widen(q[b, heads, :], dtype), keys, vals, scale)
            out[b, heads] = o
            lse[b, heads] = l
    return out, lse


# --------------------------------------------------------------------------------------
# multi-token queries (speculative / MTP decoding): causal, bottom-right aligned
# ("From MHA to MLA", section 2 kernel, its CAUSAL branch: with M query rows and N keys,
# query row m sits at position N - M + m and sees keys n <= N - M + m; FlashMLA-ETAP
# "Supported configurations" (any seq_len_q, causal masking for multi-token queries) and
# "Usage" (q (B, s_q, Hq, D), o (B, s_q, Hq, Dv), lse (B, Hq, s_q))).
# --------------------------------------------------------------------------------------
def causal_prefix(ctx: int, seq_len_q: int, i: int) -> int:
    """Number of cached tokens query i (of seq_len_q) attends: it sits at position
    ctx - seq_len_q + i and sees tokens 0 .. ctx - seq_len_q + i."""
    pos = int(ctx) - int(seq_len_q) + int(i)
    if pos < 0:
        raise ValueError("context length must be >= seq_len_q")
    return pos + 1


def paged_decode_mtp(q, k_cache, v_cache, block_tables, context_lens, scale, page_size, dtype,
                     rows=None, kv_format=None, k_scale=1.0, v_scale=1.0):
    """GQA/MQA/MHA decode of seq_len_q query tokens per sequence, causal bottom-right.

    q [B, S, Hq, D] (16-bit bits); caches, tables, lengths and fp8 arguments as for
    paged_decode. rows: optional (b, i, h) triples to evaluate (others left NaN).
    Returns out [B, S, Hq, Dv] and lse [B, Hq, S], float64.
    """
    B, S, Hq, _ = q.shape
    Hkv = k_cache.shape[2]
    Dv = v_cache.shape[3]
    out = np.full((B, S, Hq, Dv), np.nan)
    lse = np.full((B, Hq, S), np.nan)
    wanted = None if rows is None else {(int(b), int(i), int(h)) for b, i, h in rows}
    for b in range(B):
        ctx = int(context_lens[b])
        if ctx < 1:
            raise ValueError("context length must be >= 1")
        for kvh in range(Hkv):
            heads = [h for h in range(Hq) if kv_head_of(h, Hq, Hkv) == kvh]
            todo = [(i, h) for i in range(S) for h in heads
                    if wanted is None or (b, i, h) in wanted]
            if not todo:
                continue
            keys = dequantize(gather_tokens(k_cache[:, :, kvh, :], block_tables[b], ctx, page_size),
                              dtype, kv_format, k_scale)
            vals = dequantize(gather_tokens(v_cache[:, :, kvh, :], block_tables[b], ctx, page_size),
                              dtype, kv_format, v_scale)
            for i in range(S):
                hs = [h for (ii, h) in todo if ii == i]
                if not hs:
                    continue
                n = causal_prefix(ctx, S, i)
                o, l = attend(widen(q[b, i, hs, :], dtype), keys[:n], vals[:n], scale)
                out[b, i, hs] = o
                lse[b, hs, i] = l
    return out, lse


# --------------------------------------------------------------------------------------
# absorbed MLA decode ("From MHA to MLA", section 6; FlashMLA-ETAP "Supported configurations")
# --------------------------------------------------------------------------------------
def mla_decode(q, kv_cache, block_tables, context_lens, scale, page_size, dtype,
               head_dim_v=512, rows=None, kv_format=None, kv_scale=1.0):
    """Oracle for absorbed-MLA decode: every query head attends to one shared latent record.

    q [B, Hq, Dqk] (content dims then rope dims), kv_cache [NB, P, Dqk] (bits; E4M3 codes
    when kv_format is "e4m3", dequantized with kv_scale).
    Score = scale * (content dot + rope dot) = scale * <q, kv[:Dqk]>; value = kv[:head_dim_v].
    """
    B, Hq, Dqk = q.shape
    out = np.full((B, Hq, head_dim_v), np.nan)
    lse = np.full((B, Hq), np.nan)
    wanted = None if rows is None else {(int(b), int(h)) for b, h in rows}
    for b in range(B):
        ctx = int(context_lens[b])
        if ctx < 1:
            raise ValueError("context length must be >= 1")
        heads = [h for h in range(Hq) if wanted is None or (b, h) in wanted]
        if not heads:
            continue
        record = dequantize(gather_tokens(kv_cache, block_tables[b], ctx, page_size), dtype,
                            kv_format, kv_scale)                                     # [L, Dqk]
        qb = widen(q[b, heads, :], dtype)
        content = float(scale) * (qb[:, :head_dim_v] @ record[:, :head_dim_v].T)
        rope = float(scale) * (qb[:, head_dim_v:] @ record[:, head_dim_v:Dqk].T)
        s = content + rope
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        z = e.sum(axis=1)
        out[b, heads] = (e @ record[:, :head_dim_v]) / z[:, None]
        lse[b, heads] = m + np.log(z)
    return out, lse


# --------------------------------------------------------------------------------------
# Flash-Decoding split and combine ("From MHA to MLA", section 4)
# --------------------------------------------------------------------------------------
def attend_interval(q_rows, keys, values, scale, begin, end):
    """Stage 1 of Flash-Decoding for one split: normalized O_s and L_s over tokens [begin, end)."""
    return attend(q_rows, keys[begin:end], values[begin:end], scale)


def combine_splits(partial_out: np.ndarray, partial_lse: np.ndarray):
    """Combine S locally normalized split results of one head.

    partial_out [S, Dv], partial_lse [S] -> out [Dv], lse.
    L = max_s L_s + ln sum_s exp(L_s - max);  out = sum_s exp(L_s - L) O_s.
    A split with L_s = -inf (no keys) carries zero weight and is skipped.
    """
    partial_out = np.asarray(partial_out, dtype=np.float64)
    partial_lse = np.asarray(partial_lse, dtype=np.float64)
    keep = np.isfinite(partial_lse)
    po, pl = partial_out[keep], partial_lse[keep]
    mx = pl.max()
    w = np.exp(pl - mx)
    denom = w.sum()
    out = (w[:, None] * po).sum(axis=0) / denom
    return out, mx + np.log(denom)


def mla_decode_mtp(q, kv_cache, block_tables, context_lens, scale, page_size, dtype,
                   head_dim_v=512, rows=None, kv_format=None, kv_scale=1.0):
    """Absorbed-MLA decode of seq_len_q query tokens per sequence, causal bottom-right.

    q [B, S, Hq, Dqk]; the rest as for mla_decode. rows: optional (b, i, h) triples.
    Returns out [B, S, Hq, head_dim_v] and lse [B, Hq, S], float64.
    """
    B, S, Hq, Dqk = q.shape
    out = np.full((B, S, Hq, head_dim_v), np.nan)
    lse = np.full((B, Hq, S), np.nan)
    wanted = None if rows is None else {(int(b), int(i), int(h)) for b, i, h in rows}
    for b in range(B):
        ctx = int(context_lens[b])
        if ctx < 1:
            raise ValueError("context length must be >= 1")
        record = None
        for i in range(S):
            hs = [h for h in range(Hq) if wanted is None or (b, i, h) in wanted]
            if not hs:
                continue
            if record is None:
                record = dequantize(gather_tokens(kv_cache, block_tables[b], ctx, page_size),
                                    dtype, kv_format, kv_scale)
            n = causal_prefix(ctx, S, i)
            o, l = attend(widen(q[b, i, hs, :], dtype), record[:n], record[:n, :head_dim_v],
                          scale)
            out[b, i, hs] = o
            lse[b, hs, i] = l
    return out, lse


# --------------------------------------------------------------------------------------
# appending the new tokens' keys and values ("From MHA to MLA", section 2: at decode step
# t the new key and value are appended to the cache, and every later step rereads them;
# section 5: logical token n lives in block block_tables[b][n // P], slot n - (n // P) * P)
# --------------------------------------------------------------------------------------
def encode_e4m3(x) -> np.ndarray:
    """float32 values -> E4M3 codes: round to nearest, ties to an even mantissa, finite
    values beyond the largest code clamp to +-448 (saturating), NaN -> 0x7F.

    Written from the format's definition: the candidates are the 127 non-negative finite
    codes 0x00..0x7E, whose values decode_e4m3 gives and which increase with the code.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    codes = np.arange(0x7F, dtype=np.uint8)
    values = decode_e4m3(codes)                      # 0, 2^-9, ..., 448, increasing
    mag = np.minimum(np.abs(np.nan_to_num(x, nan=0.0)), values[-1])
    hi = np.searchsorted(values, mag, side="left")   # first code with value >= mag
    hi = np.minimum(hi, len(values) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - values[lo]
    d_hi = values[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0) & (hi != lo))
    out = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    out = np.where(mag == values[hi], codes[hi], out).astype(np.uint8)
    sign = (np.signbit(x) & ~np.isnan(x)).astype(np.uint8) << 7
    out = out | sign
    return np.where(np.isnan(x), np.uint8(0x7F), out).astype(np.uint8)


def quantize_e4m3(x_bits, dtype, scale) -> np.ndarray:
    """16-bit values -> E4M3 codes of value / scale, the division done in float32 (as the
    append kernel does) and rounded once to E4M3."""
    x32 = widen(x_bits, dtype).astype(np.float32)
    return encode_e4m3(x32 / np.float32(scale))


def append_tokens(cache, new, block_tables, context_lens, page_size, seq_len_q=1):
    """A copy of ``cache`` [NB, P, ...] with the new tokens written in place.

    new [B, S, ...] holds the S new tokens of each sequence (already in the cache's storage
    type); token i of sequence b is logical token n = ctx_b - S + i (ctx_b counts the new
    tokens), stored at (block_tables[b][n // P], n % P).
    """
    out = np.array(cache, copy=True)
    B = len(context_lens)
    for b in range(B):
        ctx = int(context_lens[b])
        if ctx < seq_len_q:
            raise ValueError("context length must be >= seq_len_q")
        for i in range(seq_len_q):
            n = ctx - seq_len_q + i
            logical_page = n // page_size
            slot = n - logical_page * page_size
            phys = int(block_tables[b][logical_page])
            out[phys, slot] = new[b, i]
    return out
