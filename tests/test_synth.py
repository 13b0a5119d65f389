"""The shared input generator: determinism, rounding and block-table structure."""
import numpy as np

from paged_kv_cache_61_gb300 import synth


def test_same_seed_same_inputs():
    a = synth.workload("gqa_tiny")
    b = synth.workload("gqa_tiny")
    for name in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0], dtype=np.float32)
    bits = synth.float32_to_bits(x, synth.BF16)
    back = synth.bits_to_float32(bits, synth.BF16)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 is a tie -> even (1+2^-6 ... i.e. 1.015625)
    assert back.tolist() == [1.0, 1.0, 1.015625, 1.0, -2.5, 0.0]


def test_tiny_workload_shape_and_tables():
    c = synth.workload("gqa_tiny")
    assert c.q.shape == (4, 8, 64) and c.k_cache.shape == (64, 16, 2, 64)
    assert ((c.context_lens >= 1) & (c.context_lens <= 256)).all()
    assert sorted(c.block_tables.ravel().tolist()) == list(range(64))   # one permutation of 64 blocks
    assert abs(c.scale - 0.125) < 1e-15


def test_pool_tables_cover_each_block_once():
    c = synth.make_gqa_case(batch=9, num_q_heads=4, num_kv_heads=2, head_dim=64, dtype=synth.BF16,
                            ctx_dist="loguniform", ctx_low=16, ctx_high=2000, seed=1)
    pages = (c.context_lens + 15) // 16
    used = np.concatenate([c.block_tables[b, :n] for b, n in enumerate(pages)])
    assert sorted(used.tolist()) == list(range(c.num_blocks))
    for b, n in enumerate(pages):
        assert (c.block_tables[b, n:] == synth.UNUSED_ENTRY).all()
    assert ((c.context_lens >= 16) & (c.context_lens <= 2000)).all()


def test_e4m3_caches_are_seeded_and_use_the_full_code_range():
    a = synth.workload("gqa_tiny_fp8")
    b = synth.workload("gqa_tiny_fp8")
    assert a.kv_format == synth.FP8_E4M3 and a.k_cache.dtype == np.uint8
    np.testing.assert_array_equal(a.k_cache, b.k_cache)
    assert a.k_scale == b.k_scale and a.v_scale == b.v_scale
    # the largest draw maps to the largest finite code (0x7E / 0xFE); no NaN code appears
    for codes in (a.k_cache, a.v_cache):
        mags = codes & 0x7F
        assert mags.max() == 0x7E and not np.any(mags == 0x7F)
    # q, the tables and the context lengths are those of the 16-bit workload
    c = synth.workload("gqa_tiny")
    np.testing.assert_array_equal(a.q, c.q)
    np.testing.assert_array_equal(a.block_tables, c.block_tables)
