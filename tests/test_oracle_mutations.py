"""The oracle's pins catch plausible mistakes: each mutation planted in the oracle here
(on the CPU, for the duration of one test) must make at least one pin fail."""
import numpy as np
import pytest

import oracle
import oracle.decode as od
import test_oracle_pins as pins
from paged_kv_cache_61_gb300 import synth

PIN_CALLS = [
    pins.test_worked_example_ctx37_mapping,
    pins.test_worked_example_gather_reads_only_three_entries,
    pins.test_unused_entries_and_stale_slots_never_matter,
    pins.test_block_permutation_invariance,
    pins.test_ctx1_gives_first_value_row,
    pins.test_equal_keys_give_mean_value_and_log_length,
    pins.test_constant_values_give_that_value,
    pins.test_needle_selects_one_token,
    pins.test_gqa_equals_mha_with_repeated_kv_heads,
    lambda: pins.test_matches_torch_float64_softmax(synth.FP16),
    pins.test_tiny_workload_matches_torch_float64,
    pins.test_split_combine_equals_whole,
    pins.test_combine_weights_by_split_mass_and_skips_empty,
    pins.test_mla_equals_generic_with_one_kv_head,
    pins.test_mla_rope_only_needle_returns_latent_of_target,
    pins.test_e4m3_closed_forms,
    pins.test_e4m3_order_and_sign_symmetry,
    pins.test_e4m3_matches_torch_float8_for_every_code,
    lambda: pins.test_fp8_cache_matches_torch_float64_softmax(synth.BF16),
    pins.test_fp8_scales_enter_as_score_and_value_factors,
    pins.test_fp8_needle_returns_scaled_value_code,
    pins.test_fp8_mla_equals_generic_with_one_kv_head,
    pins.test_mtp_causal_prefix_is_bottom_right,
    pins.test_mtp_one_token_is_single_token_decode,
    pins.test_mtp_row_i_is_single_token_decode_over_its_prefix,
    lambda: pins.test_mtp_matches_torch_sdpa_lower_right_causal(None),
    pins.test_mtp_mla_equals_generic_with_one_kv_head,
    pins.test_e4m3_encode_closed_forms,
    pins.test_e4m3_encode_inverts_decode_on_every_finite_code,
    pins.test_e4m3_encode_matches_torch_float8_cast_in_range,
    lambda: pins.test_append_puts_new_tokens_where_the_gather_reads_them(2),
    pins.test_e4m3_quantize_divides_once_in_float32,
    pins.test_e4m3_quantize_matches_torch_float32_division_and_cast,
]


def _attend_log2(q_rows, keys, values, scale):
    s = float(scale) * (np.asarray(q_rows, float) @ np.asarray(keys, float).T)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)
    return (e @ np.asarray(values, float)) / z[:, None], m + np.log2(z)


def _attend_no_scale(q_rows, keys, values, scale):
    return od.__dict__["_orig_attend"](q_rows, keys, values, 1.0)


def _attend_keys_as_values(q_rows, keys, values, scale):
    return od.__dict__["_orig_attend"](q_rows, keys, keys[:, : np.asarray(values).shape[1]], scale)


def _token_locations_next_entry(row, ctx, page):
    phys, slots = od.__dict__["_orig_token_locations"](row, ctx, page)
    shifted = [int(row[j // page + 1]) if j // page + 1 < len(row) else int(row[j // page])
               for j in range(int(ctx))]
    return np.asarray(shifted, dtype=np.int64), slots


def _token_locations_bad_slot(row, ctx, page):
    phys, _ = od.__dict__["_orig_token_locations"](row, ctx, page)
    return phys, np.asarray([j % (page - 1) for j in range(int(ctx))], dtype=np.int64)


def _kv_head_interleaved(h, hq, hkv):
    return h % hkv


def _combine_plain_mean(po, pl):
    po, pl = np.asarray(po, float), np.asarray(pl, float)
    keep = np.isfinite(pl)
    return po[keep].mean(axis=0), pl[keep].max()


def _mla_drops_rope(q, kv, tables, ctx, scale, page, dtype, head_dim_v=512, rows=None, **kw):
    q2 = q.copy()
    q2[..., head_dim_v:] = 0
    return od.__dict__["_orig_mla"](q2, kv, tables, ctx, scale, page, dtype, head_dim_v, rows,
                                    **kw)


def _e4m3_bias8(codes):
    return od.__dict__["_orig_e4m3"](codes) / 2.0


def _e4m3_no_subnormals(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    out = od.__dict__["_orig_e4m3"](codes)
    e = (codes >> 3) & 0xF
    m = (codes & 7).astype(np.float64)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    return np.where((e == 0) & (m > 0), sign * np.ldexp(1.0 + m / 8.0, -7), out)


def _dequantize_no_scale(stored, dtype, kv_format=None, scale=1.0):
    return od.__dict__["_orig_dequantize"](stored, dtype, kv_format, 1.0)


def _paged_decode_swapped_scales(q, k, v, tables, ctx, scale, page, dtype, rows=None,
                                 kv_format=None, k_scale=1.0, v_scale=1.0):
    return od.__dict__["_orig_paged"](q, k, v, tables, ctx, scale, page, dtype, rows, kv_format,
                                      v_scale, k_scale)


def _causal_top_left(ctx, seq_len_q, i):
    return int(i) + 1


def _causal_ignored(ctx, seq_len_q, i):
    return int(ctx)


def _causal_off_by_one(ctx, seq_len_q, i):
    return max(1, int(ctx) - int(seq_len_q) + int(i))


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float32)
    base = od.__dict__["_orig_encode"](x)
    up = od.__dict__["_orig_encode"](x * np.float32(1.0 + 2.0 ** -20))   # nudge ties upward
    return np.where(np.abs(x) > 0, up, base).astype(np.uint8)


def _encode_truncates(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    codes = np.arange(0x7F, dtype=np.uint8)
    values = od.decode_e4m3(codes)
    mag = np.minimum(np.abs(np.nan_to_num(x)), values[-1])
    idx = np.searchsorted(values, mag, side="right") - 1
    return (codes[idx] | ((x < 0).astype(np.uint8) << 7)).astype(np.uint8)


def _quantize_divides_in_float64(x_bits, dtype, scale):
    # the exact float64 quotient rounded once to E4M3 (no float32 step in between)
    x = od.widen(x_bits, dtype) / float(scale)
    codes = np.arange(0x7F, dtype=np.uint8)
    values = od.decode_e4m3(codes)
    mag = np.minimum(np.abs(x), values[-1])
    hi = np.minimum(np.searchsorted(values, mag, side="left"), len(values) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = mag - values[lo], values[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    out = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    return (out | (np.signbit(x).astype(np.uint8) << 7)).astype(np.uint8)


def _quantize_times_reciprocal(x_bits, dtype, scale):
    x32 = od.widen(x_bits, dtype).astype(np.float32)
    return od.encode_e4m3(x32 * (np.float32(1.0) / np.float32(scale)))


def _append_one_slot_late(cache, new, tables, ctx, page, seq_len_q=1):
    return od.__dict__["_orig_append"](cache, new, tables, np.asarray(ctx) + 1, page, seq_len_q)


MUTATIONS = {
    "lse in log2": ("attend", _attend_log2),
    "scale dropped": ("attend", _attend_no_scale),
    "keys used as values": ("attend", _attend_keys_as_values),
    "next table entry read": ("token_locations", _token_locations_next_entry),
    "wrong slot within the page": ("token_locations", _token_locations_bad_slot),
    "interleaved head grouping": ("kv_head_of", _kv_head_interleaved),
    "splits averaged without weights": ("combine_splits", _combine_plain_mean),
    "MLA rope dims ignored": ("mla_decode", _mla_drops_rope),
    "E4M3 exponent bias 8": ("decode_e4m3", _e4m3_bias8),
    "E4M3 subnormals read as normals": ("decode_e4m3", _e4m3_no_subnormals),
    "fp8 scales ignored": ("dequantize", _dequantize_no_scale),
    "k_scale and v_scale swapped": ("paged_decode", _paged_decode_swapped_scales),
    "causal mask aligned top-left": ("causal_prefix", _causal_top_left),
    "causal mask ignored": ("causal_prefix", _causal_ignored),
    "causal limit excludes the query's own token": ("causal_prefix", _causal_off_by_one),
    "E4M3 encoding rounds ties away from zero": ("encode_e4m3", _encode_ties_away),
    "E4M3 encoding truncates": ("encode_e4m3", _encode_truncates),
    "append writes one slot late": ("append_tokens", _append_one_slot_late),
    "E4M3 quantization divides in float64": ("quantize_e4m3", _quantize_divides_in_float64),
    "E4M3 quantization multiplies by the reciprocal": ("quantize_e4m3",
                                                       _quantize_times_reciprocal),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_mutation_is_caught_by_a_pin(name, monkeypatch):
    func, repl = MUTATIONS[name]
    monkeypatch.setitem(od.__dict__, "_orig_attend", od.attend)
    monkeypatch.setitem(od.__dict__, "_orig_token_locations", od.token_locations)
    monkeypatch.setitem(od.__dict__, "_orig_mla", od.mla_decode)
    monkeypatch.setitem(od.__dict__, "_orig_e4m3", od.decode_e4m3)
    monkeypatch.setitem(od.__dict__, "_orig_dequantize", od.dequantize)
    monkeypatch.setitem(od.__dict__, "_orig_paged", od.paged_decode)
    monkeypatch.setitem(od.__dict__, "_orig_encode", od.encode_e4m3)
    monkeypatch.setitem(od.__dict__, "_orig_append", od.append_tokens)
    monkeypatch.setattr(od, func, repl)
    monkeypatch.setattr(oracle, func, repl)
    caught = []
    for call in PIN_CALLS:
        try:
            call()
        except (AssertionError, IndexError, ValueError):
            caught.append(getattr(call, "__name__", "lambda"))
    assert caught, f"no pin fails when the oracle has the mistake: {name}"
