"""Pins for the float64 oracle: values and invariants the pages and the mathematics fix.

Each test would fail on a plausible mistake in the oracle (wrong page index or
slot, interleaved instead of contiguous grouping, a dropped scale, log2 instead
of ln, a transposed operand, reading unused table entries or stale slots,
using the rope dims as value dims, a wrong combine weight).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_61_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAN16 = {synth.FP16: 0x7E00, synth.BF16: 0x7FC0}


def _small_case(dtype=synth.FP16, seed=3, batch=3, hq=8, hkv=2, d=64, ctx=(37, 1, 50)):
    return synth.make_gqa_case(batch=batch, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               dtype=dtype, context_lens=list(ctx), table_layout="permutation",
                               num_blocks=24, max_blocks_per_seq=5, seed=seed)


def _run(case, **kw):
    if case.kv_format is not None:
        kw = dict(kv_format=case.kv_format, k_scale=case.k_scale, v_scale=case.v_scale, **kw)
    return oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                               case.context_lens, case.scale, case.page_size, case.dtype, **kw)


# ---------------------------------------------------------------- paged addressing
def _read_worked_example():
    ranges, meta = [], {}
    with open(os.path.join(GOLDEN, "worked_example_ctx37.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line.startswith("range"):
                ranges.append(tuple(int(x) for x in line.split()[1:]))
            else:
                k, v = (s.strip() for s in line.split("="))
                meta[k] = [int(x) for x in v.split()]
    return meta, ranges


def test_worked_example_ctx37_mapping():
    meta, ranges = _read_worked_example()
    ctx, page = meta["ctx"][0], meta["page_size"][0]
    assert oracle.num_pages(ctx, page) == meta["num_pages"][0] == 3
    # entries after the third are garbage that would break the gather if it were read
    row = np.array(meta["table_prefix"] + [10 ** 9, -7, 2 ** 31 - 1], dtype=np.int64)
    phys, slots = oracle.token_locations(row, ctx, page)
    expect_phys, expect_slots = [], []
    for t0, t1, blk, s0, s1 in ranges:
        assert t1 - t0 == s1 - s0
        expect_phys += [blk] * (t1 - t0 + 1)
        expect_slots += list(range(s0, s1 + 1))
    assert phys.tolist() == expect_phys and slots.tolist() == expect_slots


def test_worked_example_gather_reads_only_three_entries():
    meta, _ = _read_worked_example()
    nb, page = 10, 16
    cache = np.arange(nb * page, dtype=np.int64).reshape(nb, page)  # label = block*16 + slot
    row = np.array(meta["table_prefix"] + [10 ** 9], dtype=np.int64)  # entry 3 is out of range
    got = oracle.gather_tokens(cache, row, 37, page)
    assert got.tolist() == ([9 * 16 + s for s in range(16)] + [3 * 16 + s for s in range(16)]
                            + [7 * 16 + s for s in range(5)])


def test_unused_entries_and_stale_slots_never_matter():
    case = _small_case()
    out0, lse0 = _run(case)
    poisoned = synth.DecodeCase(**{**case.__dict__})
    k, v, tab = case.k_cache.copy(), case.v_cache.copy(), case.block_tables.copy()
    used = set()
    for b, ctx in enumerate(case.context_lens):
        npg = oracle.num_pages(ctx, case.page_size)
        used.update(int(x) for x in tab[b, :npg])
        last = int(tab[b, npg - 1])
        fill = int(ctx) - (npg - 1) * case.page_size
        k[last, fill:] = NAN16[case.dtype]
        v[last, fill:] = NAN16[case.dtype]
        tab[b, npg:] = 10 ** 8          # would raise IndexError if read
    for blk in range(case.num_blocks):
        if blk not in used:
            k[blk] = NAN16[case.dtype]
            v[blk] = NAN16[case.dtype]
    poisoned.k_cache, poisoned.v_cache, poisoned.block_tables = k, v, tab
    out1, lse1 = _run(poisoned)
    assert np.isfinite(out1).all() and np.isfinite(lse1).all()
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


def test_block_permutation_invariance():
    case = _small_case(dtype=synth.BF16)
    out0, lse0 = _run(case)
    rng = np.random.default_rng(11)
    perm = rng.permutation(case.num_blocks)
    moved = synth.DecodeCase(**{**case.__dict__})
    moved.k_cache = np.empty_like(case.k_cache)
    moved.v_cache = np.empty_like(case.v_cache)
    moved.k_cache[perm] = case.k_cache
    moved.v_cache[perm] = case.v_cache
    moved.block_tables = perm[case.block_tables].astype(np.int32)
    out1, lse1 = _run(moved)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


# ---------------------------------------------------------------- softmax closed forms
def test_ctx1_gives_first_value_row():
    case = _small_case(ctx=(1, 1, 1))
    out, lse = _run(case)
    G = case.group
    for b in range(case.batch):
        blk = int(case.block_tables[b, 0])
        for h in range(case.num_q_heads):
            kvh = h // G
            v0 = oracle.widen(case.v_cache[blk, 0, kvh], case.dtype)
            k0 = oracle.widen(case.k_cache[blk, 0, kvh], case.dtype)
            qv = oracle.widen(case.q[b, h], case.dtype)
            np.testing.assert_array_equal(out[b, h], v0)
            assert lse[b, h] == pytest.approx(case.scale * math.fsum(qv * k0), abs=1e-12)


def test_equal_keys_give_mean_value_and_log_length():
    case = _small_case(ctx=(37, 16, 5))
    G = case.group
    k = case.k_cache.copy()
    k[:] = case.k_cache[0, 0]                     # every key row identical (per kv head)
    case.k_cache = k
    out, lse = _run(case)
    for b, ctx in enumerate(case.context_lens):
        for h in range(case.num_q_heads):
            kvh = h // G
            s = case.scale * math.fsum(oracle.widen(case.q[b, h], case.dtype)
                                       * oracle.widen(k[0, 0, kvh], case.dtype))
            assert lse[b, h] == pytest.approx(s + math.log(int(ctx)), abs=1e-12)
            rows = [oracle.widen(case.v_cache[case.block_tables[b, j // 16], j % 16, kvh], case.dtype)
                    for j in range(int(ctx))]
            np.testing.assert_allclose(out[b, h], np.mean(rows, axis=0), rtol=0, atol=1e-12)


def test_constant_values_give_that_value():
    case = _small_case()
    v = np.empty_like(case.v_cache)
    for kvh in range(case.num_kv_heads):
        v[:, :, kvh, :] = case.q[0, kvh]          # any fixed 16-bit row per kv head
    case.v_cache = v
    out, _ = _run(case)
    G = case.group
    for b in range(case.batch):
        for h in range(case.num_q_heads):
            np.testing.assert_allclose(out[b, h], oracle.widen(case.q[0, h // G], case.dtype),
                                       rtol=0, atol=1e-12)


def test_needle_selects_one_token():
    case = _small_case(ctx=(37, 20, 50))
    one = synth.float32_to_bits(np.float32(1.0), case.dtype)
    sixteen = synth.float32_to_bits(np.float32(16.0), case.dtype)
    case.q[:] = one
    for target in (0, 15, 16, 36):
        k = np.zeros_like(case.k_cache)
        b = 0
        blk = int(case.block_tables[b, target // 16])
        k[blk, target % 16] = sixteen
        case.k_cache = k
        out, lse = _run(case)
        for h in range(case.num_q_heads):
            v = oracle.widen(case.v_cache[blk, target % 16, h // case.group], case.dtype)
            np.testing.assert_allclose(out[b, h], v, rtol=0, atol=1e-30)
            assert lse[b, h] == pytest.approx(case.scale * 16 * case.head_dim_qk, abs=1e-9)


# ---------------------------------------------------------------- head grouping
def test_gqa_equals_mha_with_repeated_kv_heads():
    case = _small_case(hq=8, hkv=2)
    out_gqa, lse_gqa = _run(case)
    mha = synth.DecodeCase(**{**case.__dict__})
    mha.k_cache = np.repeat(case.k_cache, case.group, axis=2)
    mha.v_cache = np.repeat(case.v_cache, case.group, axis=2)
    mha.num_kv_heads = case.num_q_heads
    out_mha, lse_mha = _run(mha)
    # same arithmetic; only the BLAS blocking differs (4 rows per call vs 1)
    np.testing.assert_allclose(out_gqa, out_mha, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_gqa, lse_mha, rtol=0, atol=1e-13)
    # the interleaved convention (kv head = h % Hkv) is a different operator on this input
    inter = synth.DecodeCase(**{**case.__dict__})
    order = [h % case.num_kv_heads for h in range(case.num_q_heads)]
    inter.k_cache = case.k_cache[:, :, order, :]
    inter.v_cache = case.v_cache[:, :, order, :]
    inter.num_kv_heads = case.num_q_heads
    out_int, _ = _run(inter)
    assert np.abs(out_int - out_gqa).max() > 1e-3


def test_mqa_is_single_kv_head_special_case():
    case = _small_case(hq=8, hkv=1)
    out, lse = _run(case)
    for b, ctx in enumerate(case.context_lens):
        keys = oracle.widen(oracle.gather_tokens(case.k_cache[:, :, 0], case.block_tables[b], ctx, 16), case.dtype)
        vals = oracle.widen(oracle.gather_tokens(case.v_cache[:, :, 0], case.block_tables[b], ctx, 16), case.dtype)
        o, l = oracle.attend(oracle.widen(case.q[b], case.dtype), keys, vals, case.scale)
        np.testing.assert_allclose(out[b], o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], l, rtol=0, atol=1e-13)


def test_rejects_indivisible_heads_and_empty_context():
    with pytest.raises(ValueError):
        oracle.kv_head_of(0, 6, 4)
    case = _small_case(ctx=(5, 0, 3))
    with pytest.raises(ValueError):
        _run(case)


# ---------------------------------------------------------------- textbook cross-check
def _torch_reference(case):
    """softmax(scale q K^T) V and logsumexp with torch float64 on a gather built from torch ops."""
    P = case.page_size
    out = torch.empty(case.batch, case.num_q_heads, case.head_dim_v, dtype=torch.float64)
    lse = torch.empty(case.batch, case.num_q_heads, dtype=torch.float64)
    tdt = torch.float16 if case.dtype == synth.FP16 else torch.bfloat16
    q = torch.from_numpy(case.q.view(np.int16)).view(tdt).double()
    if case.kv_format == synth.FP8_E4M3:      # torch's own float8 decoding, then the scales
        k = torch.from_numpy(case.k_cache).view(torch.float8_e4m3fn).double() * case.k_scale
        v = torch.from_numpy(case.v_cache).view(torch.float8_e4m3fn).double() * case.v_scale
    else:
        k = torch.from_numpy(case.k_cache.view(np.int16)).view(tdt).double()
        v = torch.from_numpy(case.v_cache.view(np.int16)).view(tdt).double()
    kf = k.reshape(-1, case.num_kv_heads, case.head_dim_qk)
    vf = v.reshape(-1, case.num_kv_heads, case.head_dim_v)
    for b in range(case.batch):
        n = torch.arange(int(case.context_lens[b]))
        rowidx = torch.from_numpy(case.block_tables[b].astype(np.int64))[n // P] * P + n % P
        for h in range(case.num_q_heads):
            kvh = h * case.num_kv_heads // case.num_q_heads
            logits = case.scale * (kf[rowidx, kvh] @ q[b, h])
            out[b, h] = torch.softmax(logits, dim=0) @ vf[rowidx, kvh]
            lse[b, h] = torch.logsumexp(logits, dim=0)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
def test_matches_torch_float64_softmax(dtype):
    case = _small_case(dtype=dtype, ctx=(37, 1, 80), hq=8, hkv=2)
    out, lse = _run(case)
    ref_out, ref_lse = _torch_reference(case)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_tiny_workload_matches_torch_float64():
    case = synth.workload("gqa_tiny")
    out, lse = _run(case)
    ref_out, ref_lse = _torch_reference(case)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_row_subset_matches_full():
    case = _small_case()
    out, lse = _run(case)
    rows = [(0, 3), (2, 7), (1, 0)]
    o2, l2 = _run(case, rows=rows)
    for b, h in rows:
        np.testing.assert_allclose(o2[b, h], out[b, h], rtol=0, atol=1e-13)
        assert l2[b, h] == pytest.approx(lse[b, h], abs=1e-13)
    assert np.isnan(o2[0, 0]).all()


# ---------------------------------------------------------------- split-KV combine
def test_split_combine_equals_whole():
    rng = np.random.default_rng(5)
    L, D = 300, 32
    q = rng.standard_normal((4, D))
    keys = rng.standard_normal((L, D))
    vals = rng.standard_normal((L, D))
    whole_o, whole_l = oracle.attend(q, keys, vals, 0.3)
    for cuts in ([0, 150, 300], [0, 1, 2, 299, 300], [0, 17, 64, 200, 233, 300]):
        parts = [oracle.attend_interval(q, keys, vals, 0.3, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
        for r in range(q.shape[0]):
            po = np.stack([p[0][r] for p in parts])
            pl = np.array([p[1][r] for p in parts])
            o, l = oracle.combine_splits(po, pl)
            np.testing.assert_allclose(o, whole_o[r], rtol=0, atol=1e-12)
            assert l == pytest.approx(whole_l[r], abs=1e-12)


def test_combine_weights_by_split_mass_and_skips_empty():
    # two splits with LSE ln 1 and ln 3: weights 1/4 and 3/4; an empty split (-inf) is ignored
    po = np.array([[1.0, 0.0], [0.0, 1.0], [np.nan, np.nan]])
    pl = np.array([0.0, math.log(3.0), -math.inf])
    o, l = oracle.combine_splits(po, pl)
    np.testing.assert_allclose(o, [0.25, 0.75], rtol=0, atol=1e-15)
    assert l == pytest.approx(math.log(4.0), abs=1e-15)


# ---------------------------------------------------------------- MLA
def _small_mla(hq=16, ctx=(70, 1, 129), seed=4, latent=512):
    return synth.make_mla_case(batch=len(ctx), num_q_heads=hq, dtype=synth.BF16,
                               context_lens=list(ctx), latent_dim=latent, seed=seed)


def test_mla_equals_generic_with_one_kv_head(latent=512):
    case = _small_mla(latent=latent)
    out, lse = oracle.mla_decode(case.q, case.kv_cache, case.block_tables, case.context_lens,
                                 case.scale, case.page_size, case.dtype, head_dim_v=latent)
    k = case.kv_cache[:, :, None, :]
    v = case.kv_cache[:, :, None, :latent]
    out2, lse2 = oracle.paged_decode(case.q, k, v, case.block_tables, case.context_lens,
                                     case.scale, case.page_size, case.dtype)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_mla_rope_only_needle_returns_latent_of_target(latent=512):
    case = _small_mla(hq=4, ctx=(100,), latent=latent)
    kv = case.kv_cache.copy()
    q = case.q.copy()
    q[..., :latent] = 0                                   # no content score at all
    q[..., latent:] = synth.float32_to_bits(np.float32(1.0), case.dtype)
    kv[..., latent:] = 0
    target = 77
    blk = int(case.block_tables[0, target // 64])
    kv[blk, target % 64, latent:] = synth.float32_to_bits(np.float32(16.0), case.dtype)
    out, lse = oracle.mla_decode(q, kv, case.block_tables, case.context_lens, case.scale,
                                 case.page_size, case.dtype, head_dim_v=latent)
    want = oracle.widen(kv[blk, target % 64, :latent], case.dtype)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], want, rtol=0, atol=1e-30)
        assert lse[0, h] == pytest.approx(case.scale * 16 * 64, abs=1e-9)
    assert out.shape[-1] == latent


def test_rank256_record_pins():
    """The same two pins on the kv_lora_rank 256 record (256 latent + 64 rope)."""
    test_mla_equals_generic_with_one_kv_head(latent=256)
    test_mla_rope_only_needle_returns_latent_of_target(latent=256)


# ---------------------------------------------------------------- fp8 (E4M3) caches
def test_e4m3_closed_forms():
    """Values fixed by the E4M3 definition (bias 7, 3 mantissa bits, no infinities)."""
    want = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x30: 0.5, 0x7E: 448.0, 0x77: 240.0,
            0x08: 2.0 ** -6, 0x07: 7 * 2.0 ** -9, 0x01: 2.0 ** -9, 0x58: 16.0, 0xB8: -1.0,
            0xFE: -448.0, 0x81: -(2.0 ** -9)}
    got = oracle.decode_e4m3(np.array(list(want), dtype=np.uint8))
    np.testing.assert_array_equal(got, np.array(list(want.values())))
    assert math.copysign(1.0, oracle.decode_e4m3(np.array([0x80], np.uint8))[0]) == -1.0
    assert np.isnan(oracle.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_order_and_sign_symmetry():
    pos = oracle.decode_e4m3(np.arange(0x00, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                       # codes 0x00..0x7E increase strictly
    neg = oracle.decode_e4m3(np.arange(0x80, 0xFF, dtype=np.uint8))
    np.testing.assert_array_equal(neg, -pos)
    # adjacent normal values differ by 2^(e-7)/8: a spacing that doubles every 8 codes
    steps = np.diff(oracle.decode_e4m3(np.arange(0x08, 0x7F, dtype=np.uint8)))
    for i, st in enumerate(steps):
        assert st == 2.0 ** (((0x08 + i) >> 3) - 10)


def test_e4m3_matches_torch_float8_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])


def _fp8_case(seed=3, ctx=(37, 1, 50), hq=8, hkv=2, d=64, dtype=synth.BF16):
    return synth.make_gqa_case(batch=len(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               dtype=dtype, context_lens=list(ctx), table_layout="permutation",
                               num_blocks=24, max_blocks_per_seq=5, seed=seed,
                               kv_format=synth.FP8_E4M3)


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
def test_fp8_cache_matches_torch_float64_softmax(dtype):
    case = _fp8_case(dtype=dtype, ctx=(37, 1, 80))
    assert case.k_scale != 1.0 and case.v_scale != 1.0 and case.k_scale != case.v_scale
    out, lse = _run(case)
    ref_out, ref_lse = _torch_reference(case)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_fp8_scales_enter_as_score_and_value_factors():
    """k_scale multiplies every logit like the softmax scale does; v_scale multiplies the
    output and leaves the LSE alone."""
    case = _fp8_case(ctx=(37, 16, 50))
    out, lse = _run(case)
    kw = dict(kv_format=case.kv_format)
    args = (case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens)
    o2, l2 = oracle.paged_decode(*args, case.scale * 4.0, case.page_size, case.dtype,
                                 k_scale=case.k_scale / 4.0, v_scale=case.v_scale, **kw)
    np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)
    o3, l3 = oracle.paged_decode(*args, case.scale, case.page_size, case.dtype,
                                 k_scale=case.k_scale, v_scale=case.v_scale * 3.0, **kw)
    np.testing.assert_allclose(o3, 3.0 * out, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(l3, lse)


def test_fp8_needle_returns_scaled_value_code():
    case = _fp8_case(ctx=(37, 20, 50))
    case.q[:] = synth.float32_to_bits(np.float32(1.0), case.dtype)
    case.k_scale, case.v_scale = 1.0, 0.25
    for target in (0, 15, 16, 36):
        k = np.zeros_like(case.k_cache)
        blk = int(case.block_tables[0, target // 16])
        k[blk, target % 16] = 0x58                     # 16.0
        case.k_cache = k
        out, lse = _run(case)
        for h in range(case.num_q_heads):
            codes = case.v_cache[blk, target % 16, h // case.group]
            np.testing.assert_array_equal(out[0, h], 0.25 * oracle.decode_e4m3(codes))
            assert lse[0, h] == pytest.approx(case.scale * 16 * case.head_dim_qk, abs=1e-9)


def test_fp8_mla_equals_generic_with_one_kv_head():
    case = synth.make_mla_case(batch=2, num_q_heads=4, dtype=synth.BF16, context_lens=[70, 129],
                               seed=4, kv_format=synth.FP8_E4M3)
    out, lse = oracle.mla_decode(case.q, case.kv_cache, case.block_tables, case.context_lens,
                                 case.scale, case.page_size, case.dtype, kv_format=case.kv_format,
                                 kv_scale=case.k_scale)
    k = case.kv_cache[:, :, None, :]
    v = case.kv_cache[:, :, None, :512]
    out2, lse2 = oracle.paged_decode(case.q, k, v, case.block_tables, case.context_lens,
                                     case.scale, case.page_size, case.dtype,
                                     kv_format=case.kv_format, k_scale=case.k_scale,
                                     v_scale=case.k_scale)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- multi-token queries
def _mtp_case(s=2, ctx=(37, 2, 50), hq=8, hkv=2, d=64, dtype=synth.FP16, seed=6, fmt=None):
    return synth.make_gqa_case(batch=len(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               dtype=dtype, context_lens=list(ctx), table_layout="permutation",
                               num_blocks=24, max_blocks_per_seq=5, seed=seed, seq_len_q=s,
                               kv_format=fmt)


def _run_mtp(case, **kw):
    return oracle.paged_decode_mtp(case.q, case.k_cache, case.v_cache, case.block_tables,
                                   case.context_lens, case.scale, case.page_size, case.dtype,
                                   kv_format=case.kv_format, k_scale=case.k_scale,
                                   v_scale=case.v_scale, **kw)


def test_mtp_causal_prefix_is_bottom_right():
    # query i of S sits at position ctx - S + i: the last query sees the whole context
    assert [oracle.causal_prefix(10, 3, i) for i in range(3)] == [8, 9, 10]
    assert oracle.causal_prefix(2, 2, 0) == 1
    with pytest.raises(ValueError):
        oracle.causal_prefix(1, 2, 0)


def test_mtp_one_token_is_single_token_decode():
    case = _mtp_case(s=1)
    single = synth.DecodeCase(**{**case.__dict__})
    single.q = case.q
    out, lse = _run(single)
    case.q = case.q[:, None]
    out1, lse1 = _run_mtp(case)
    np.testing.assert_array_equal(out1[:, 0], out)
    np.testing.assert_array_equal(lse1[:, :, 0], lse)


def test_mtp_row_i_is_single_token_decode_over_its_prefix():
    case = _mtp_case(s=3, ctx=(37, 3, 50))
    out, lse = _run_mtp(case)
    for i in range(3):
        pre = synth.DecodeCase(**{**case.__dict__})
        pre.q = np.ascontiguousarray(case.q[:, i])
        pre.context_lens = (case.context_lens - 3 + 1 + i).astype(np.int32)
        o, l = _run(pre)
        np.testing.assert_allclose(out[:, i], o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, i], l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("fmt", [None, synth.FP8_E4M3])
def test_mtp_matches_torch_sdpa_lower_right_causal(fmt):
    from torch.nn.attention.bias import causal_lower_right
    case = _mtp_case(s=2, ctx=(37, 2, 80), fmt=fmt)
    out, lse = _run_mtp(case)
    P, S, G = case.page_size, case.seq_len_q, case.group
    tdt = torch.float16 if case.dtype == synth.FP16 else torch.bfloat16
    q = torch.from_numpy(case.q.view(np.int16)).view(tdt).double()
    if fmt == synth.FP8_E4M3:
        k = torch.from_numpy(case.k_cache).view(torch.float8_e4m3fn).double() * case.k_scale
        v = torch.from_numpy(case.v_cache).view(torch.float8_e4m3fn).double() * case.v_scale
    else:
        k = torch.from_numpy(case.k_cache.view(np.int16)).view(tdt).double()
        v = torch.from_numpy(case.v_cache.view(np.int16)).view(tdt).double()
    kf = k.reshape(-1, case.num_kv_heads, case.head_dim_qk)
    vf = v.reshape(-1, case.num_kv_heads, case.head_dim_v)
    for b in range(case.batch):
        n = int(case.context_lens[b])
        idx = torch.arange(n)
        rowidx = torch.from_numpy(case.block_tables[b].astype(np.int64))[idx // P] * P + idx % P
        kk = kf[rowidx].permute(1, 0, 2)[:, None]             # [Hkv, 1, n, D]
        vv = vf[rowidx].permute(1, 0, 2)[:, None]
        qq = q[b].permute(1, 0, 2).reshape(case.num_kv_heads, G, S, -1)   # [Hkv, G, S, D]
        bias = causal_lower_right(S, n)
        o = torch.nn.functional.scaled_dot_product_attention(
            qq, kk.expand(-1, G, -1, -1), vv.expand(-1, G, -1, -1), attn_mask=bias,
            scale=case.scale)
        logits = case.scale * (qq @ kk.expand(-1, G, -1, -1).transpose(-1, -2))
        logits = logits.masked_fill(~bias._materialize(), float("-inf"))
        l = torch.logsumexp(logits, dim=-1)                      # [Hkv, G, S]
        np.testing.assert_allclose(out[b], o.reshape(case.num_q_heads, S, -1).permute(1, 0, 2),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], l.reshape(case.num_q_heads, S), rtol=0, atol=1e-12)


def test_mtp_mla_equals_generic_with_one_kv_head():
    case = synth.make_mla_case(batch=2, num_q_heads=4, dtype=synth.BF16, context_lens=[70, 2],
                               seed=4, seq_len_q=2)
    out, lse = oracle.mla_decode_mtp(case.q, case.kv_cache, case.block_tables,
                                     case.context_lens, case.scale, case.page_size, case.dtype)
    k = case.kv_cache[:, :, None, :]
    v = case.kv_cache[:, :, None, :512]
    out2, lse2 = oracle.paged_decode_mtp(case.q, k, v, case.block_tables, case.context_lens,
                                         case.scale, case.page_size, case.dtype)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- appending new tokens
def test_e4m3_encode_closed_forms():
    x = np.array([1.0625, 1.1875, 1.0, -2.5, 500.0, -1e30, 448.0, 464.0, 2.0 ** -10,
                  1.5 * 2.0 ** -10, 0.0, -0.0, np.nan, np.inf], dtype=np.float32)
    want = [0x38,   # midpoint of 1.0 and 1.125: ties to the even mantissa (1.0)
            0x3A,   # midpoint of 1.125 and 1.25: the even one is 1.25
            0x38, 0xC2, 0x7E, 0xFE, 0x7E, 0x7E,   # +-448 saturate
            0x00,   # 2^-10: midpoint of 0 and the smallest subnormal, ties to 0
            0x01, 0x00, 0x80, 0x7F, 0x7E]
    np.testing.assert_array_equal(oracle.encode_e4m3(x), np.array(want, dtype=np.uint8))


def test_e4m3_encode_inverts_decode_on_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.encode_e4m3(oracle.decode_e4m3(codes)), codes)


def test_e4m3_encode_matches_torch_float8_cast_in_range():
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32) * 60.0
    x = np.clip(x, -448.0, 448.0)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.encode_e4m3(x), lib)


def test_e4m3_quantize_divides_once_in_float32():
    # An fp8 cache stores one byte per value ("Attention Kernel Variants", KV-cache table,
    # fp8 row; pitfall 5); the stored code is that of x / scale with the division done in
    # IEEE float32 and rounded once more to E4M3. Each pair below is worked out by hand.
    bf = lambda x: synth.float32_to_bits(np.array([x], np.float32), synth.BF16)
    f16 = lambda x: synth.float32_to_bits(np.array([x], np.float32), synth.FP16)
    cases = [
        # 3 / 0.25 = 12 exactly: exponent 3 (field 10), mantissa 1.5 (field 4) -> 0x54
        (bf(3.0), synth.BF16, 0.25, 0x54),
        # 5.46875 / 3.5 = 1.5625 exactly, the midpoint of 1.5 (0x3C) and 1.625 (0x3D): ties
        # go to the even mantissa, 0x3C. Multiplying by the float32 reciprocal of 3.5
        # instead gives 1.5625001..., above the midpoint, hence 0x3D.
        (bf(5.46875), synth.BF16, 3.5, 0x3C),
        # 1.77 as a float32 is 1.76999998...; 5.53125 / that = 3.12500003..., which float32
        # rounds to 3.125 (the excess is below half a float32 step at 3.125, 1.2e-7).
        # 3.125 is the midpoint of 3.0 (0x44, even) and 3.25 (0x45) -> 0x44; the exact
        # quotient, rounded once, would give 0x45.
        (bf(5.53125), synth.BF16, float(np.float32(1.77)), 0x44),
        # scale = float32 0x3EFA38E4 (0.48871529...): -6.59765625 / scale = -13.49999996...
        # exactly, -13.5 in float32: the midpoint of 13 (odd mantissa 5) and 14 (even,
        # 6) -> 14, sign set: 0xD6; the exact quotient rounds to -13, 0xD5.
        (f16(-6.59765625), synth.FP16, float(np.uint32(0x3EFA38E4).view(np.float32)), 0xD6),
    ]
    for bits, dtype, scale, want in cases:
        got = int(oracle.quantize_e4m3(bits, dtype, scale)[0])
        assert got == want, (bits, scale, hex(got), hex(want))


def test_e4m3_quantize_matches_torch_float32_division_and_cast():
    # library cross-check: torch's float32 division, then its float8_e4m3fn cast (in range)
    rng = np.random.default_rng(4)
    x = rng.standard_normal(50000).astype(np.float32) * 3
    bits = synth.float32_to_bits(x, synth.BF16)
    for scale in (np.float32(1.77), np.float32(0.0123), np.float32(3.5), np.float32(0.37)):
        xw = synth.bits_to_float32(bits, synth.BF16)
        q32 = torch.from_numpy(xw) / torch.tensor(scale, dtype=torch.float32)
        q32 = q32.clamp(-448.0, 448.0)
        lib = q32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(oracle.quantize_e4m3(bits, synth.BF16, float(scale)), lib)


@pytest.mark.parametrize("s", [1, 2])
def test_append_puts_new_tokens_where_the_gather_reads_them(s):
    case = synth.make_gqa_case(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                               dtype=synth.BF16, context_lens=[37, 16, 17],
                               table_layout="permutation", num_blocks=24, max_blocks_per_seq=5,
                               seed=8, seq_len_q=s)
    rng = np.random.default_rng(3)
    new = rng.integers(0, 2 ** 16, size=(3, s, 2, 64), dtype=np.uint16)
    out = oracle.append_tokens(case.k_cache, new, case.block_tables, case.context_lens, 16, s)
    changed = np.zeros(out.shape[:2], dtype=bool)
    for b, ctx in enumerate(case.context_lens):
        got = oracle.gather_tokens(out, case.block_tables[b], int(ctx), 16)
        np.testing.assert_array_equal(got[int(ctx) - s:], new[b])
        np.testing.assert_array_equal(got[:int(ctx) - s],
                                      oracle.gather_tokens(case.k_cache, case.block_tables[b],
                                                           int(ctx) - s, 16))
        phys, slots = oracle.token_locations(case.block_tables[b], int(ctx), 16)
        changed[phys[-s:], slots[-s:]] = True
    # nothing else in the pool changes
    np.testing.assert_array_equal(out[~changed], case.k_cache[~changed])
    # as in the drill's worked example, token 36 of a 37-token sequence is slot 4 of the
    # block in the third table entry
    phys, slots = oracle.token_locations(case.block_tables[0], 37, 16)
    assert (int(phys[-1]), int(slots[-1])) == (int(case.block_tables[0][2]), 4)
