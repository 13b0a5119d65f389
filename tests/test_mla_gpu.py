"""Absorbed-MLA paged decode on the GPU (tcgen05 kernel, through the C ABI) vs the float64 oracle.

Two record widths: kv_lora_rank 512 (576 = 512 latent + 64 rope, V = first 512) and
kv_lora_rank 256 (320 = 256 latent + 64 rope, V = first 256).

Tolerances: out max-abs <= 1e-2 (bf16) / 2e-3 (fp16), fp32 LSE within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE, TOL_OUT, DeviceCase, compare, device_bits
from paged_kv_cache_61_gb300 import pda, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pda.lib()


def _oracle(case, rows=None):
    return oracle.mla_decode(case.q, case.kv_cache, case.block_tables, case.context_lens,
                             case.scale, case.page_size, case.dtype, head_dim_v=case.head_dim_v,
                             rows=rows)


def _case(hq, ctx, dtype=synth.BF16, seed=5, latent=512):
    return synth.make_mla_case(batch=len(ctx), num_q_heads=hq, dtype=dtype, context_lens=ctx,
                               latent_dim=latent, seed=seed)


def _assert_close(case, dc, rows=None):
    out, lse = dc.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = _oracle(case, rows)
    eo, el = compare(case, out, lse, ref_out, ref_lse, rows)
    assert eo <= TOL_OUT[case.dtype], f"out max-abs error {eo}"
    assert el <= TOL_LSE, f"lse max-abs error {el}"
    assert pda.read_device_error(dc.ws) == 0
    return out, lse


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [16, 32, 64, 128])
@pytest.mark.parametrize("force", [0, 1, 3, 17])
def test_small_cases(hq, force, latent):
    case = _case(hq, [1, 63, 64, 65, 130, 700], latent=latent)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [16, 128])
@pytest.mark.parametrize("scale", [-0.07, 0.0])
def test_negative_and_zero_scale(hq, latent, scale):
    # the softmax takes any finite scale: negative (the row maximum of the scaled scores
    # is scale times the smallest raw score) and zero (uniform weights over the context)
    case = _case(hq, [1, 64, 65, 700], latent=latent)
    case.scale = scale
    for force in (0, 3):
        _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [16, 128])
def test_fp16(hq, latent):
    case = _case(hq, [200, 64, 1], dtype=synth.FP16, latent=latent)
    _assert_close(case, DeviceCase(case))


@pytest.mark.parametrize("hq", [128, 192, 256])
@pytest.mark.parametrize("force", [0, 2, 5])
def test_rank256_several_head_groups_ragged_batch(hq, force):
    # the 320-wide record: head groups of 128 on one CTA each (Hq = 128, 256: one or two
    # groups per sequence), 64-head groups otherwise (Hq = 192: three); ragged last pages,
    # a one-token sequence, split sequences
    case = _case(hq, [1, 65, 127, 128, 129, 1000, 3000], seed=11, latent=256)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("hq", [128, 256])
@pytest.mark.parametrize("force", [0, 2, 5])
def test_head_groups_of_128_ragged_batch(hq, force):
    # head groups of 128 run on CTA pairs: ragged last pages, a one-token sequence and
    # sequences split over several pairs (merged in-kernel and by the merge kernel)
    case = _case(hq, [1, 65, 127, 128, 129, 1000, 3000], seed=11)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [64, 128])
def test_score_jumps_force_rescales(hq, latent):
    # q's rope half is all ones and the rope keys of pages >= 3 and >= 10 get a constant
    # added, so the scores jump twice by ~8.7 in log2 units: the running maximum must be
    # raised and the accumulated output rescaled within one piece. After each jump many
    # tokens share the weight, so the check stays inside the bf16 tolerance.
    case = _case(hq, [2000, 900], latent=latent)
    case.q[..., latent:] = synth.float32_to_bits(np.float32(1.0), case.dtype)
    kv = synth.bits_to_float32(case.kv_cache, case.dtype)
    step = 6.0 * np.sqrt(192.0) / 64.0          # +6 on the natural-log score per jump
    for b, c in enumerate(case.context_lens):
        npg = (int(c) + 63) // 64
        for pg in range(npg):
            blk = int(case.block_tables[b, pg])
            kv[blk, :, latent:] += step * ((pg >= 3) + (pg >= 10))
    case.kv_cache = synth.float32_to_bits(kv, case.dtype)
    for force in (0, 1):
        _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [16, 128])
def test_rope_needle_is_bit_exact(hq, latent):
    ctx = 300
    case = _case(hq, [ctx] * 6, seed=9, latent=latent)
    one = synth.float32_to_bits(np.float32(1.0), case.dtype)
    sixteen = synth.float32_to_bits(np.float32(16.0), case.dtype)
    case.q[..., :latent] = 0
    case.q[..., latent:] = one
    case.kv_cache[..., latent:] = 0
    targets = [0, 63, 64, 150, 255, 299]
    for b, t in enumerate(targets):
        blk = int(case.block_tables[b, t // 64])
        case.kv_cache[blk, t % 64, latent:] = sixteen
    for force in (0, 1, 5):
        dc = DeviceCase(case, force_num_ctas=force)
        out, _ = dc.run()
        torch.cuda.synchronize()
        got = device_bits(out)
        for b, t in enumerate(targets):
            blk = int(case.block_tables[b, t // 64])
            for h in range(hq):
                assert np.array_equal(got[b, h], case.kv_cache[blk, t % 64, :latent]), (force, b, h)


@pytest.mark.parametrize("latent", [512, 256])
def test_ctx1_returns_latent_of_token0(latent):
    case = _case(128, [1, 1], latent=latent)
    dc = DeviceCase(case)
    out, _ = _assert_close(case, dc)
    got = device_bits(out)
    for b in range(2):
        blk = int(case.block_tables[b, 0])
        for h in range(128):
            assert np.array_equal(got[b, h], case.kv_cache[blk, 0, :latent])


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [32, 128])
def test_poisoned_stale_slots_and_table_entries(hq, latent):
    case = _case(hq, [70, 129, 5], latent=latent)
    out0, lse0 = DeviceCase(case).run()
    torch.cuda.synchronize()
    kv, tab = case.kv_cache.copy(), case.block_tables.copy()
    for b, c in enumerate(case.context_lens):
        npg = (int(c) + 63) // 64
        last, fill = int(tab[b, npg - 1]), int(c) - (npg - 1) * 64
        kv[last, fill:] = 0x7FC0
        tab[b, npg:] = -99
    bad = synth.DecodeCase(**{**case.__dict__})
    bad.kv_cache, bad.block_tables = kv, tab
    dc = DeviceCase(bad)
    out1, lse1 = dc.run()
    torch.cuda.synchronize()
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(lse0, lse1)
    assert pda.read_device_error(dc.ws) == 0


@pytest.mark.parametrize("name", ["mla_b16_ctx64k_h16", "mla_b16_ctx64k_h128",
                                  "mla_r256_b16_ctx64k_h16", "mla_r256_b16_ctx64k_h128"])
def test_full_size_workload_sampled_rows(name):
    case = synth.workload(name)
    hq = case.num_q_heads
    # every head of six sequences: the oracle's cost is the gather of each sequence
    rows = [(b, h) for b in (0, 3, 7, 8, 12, 15) for h in range(hq)]
    _assert_close(case, DeviceCase(case), rows=rows)


# ---------------------------------------------------------------- several query tokens
def _oracle_mtp(case, rows=None):
    return oracle.mla_decode_mtp(case.q, case.kv_cache, case.block_tables, case.context_lens,
                                 case.scale, case.page_size, case.dtype,
                                 head_dim_v=case.head_dim_v, rows=rows)


def _assert_close_mtp(case, dc, rows=None):
    out, lse = dc.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = _oracle_mtp(case, rows)
    eo, el = compare(case, out, lse, ref_out, ref_lse, rows)
    assert eo <= TOL_OUT[case.dtype], f"out max-abs error {eo}"
    assert el <= TOL_LSE, f"lse max-abs error {el}"
    assert pda.read_device_error(dc.ws) == 0


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq,s", [(16, 2), (32, 2), (16, 4), (8, 2), (64, 2), (128, 2), (64, 3),
                                  (128, 3)])
@pytest.mark.parametrize("force", [0, 1, 3, 17])
def test_mtp_small_cases(hq, s, force, latent):
    # q [B, S, Hq, Dqk]: query token i sees tokens [0, ctx - S + 1 + i). Up to 64 rows
    # (S * Hq) form one head group per sequence; more form groups of one token's heads
    # (64 per group, or 128 on the heads-on-M kernel for the 320 record)
    case = synth.make_mla_case(batch=4, num_q_heads=hq, dtype=synth.BF16,
                               context_lens=[64 + s - 1, 65, 130, 700], latent_dim=latent,
                               seed=5, seq_len_q=s)
    _assert_close_mtp(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("hq,latent", [(16, 512), (128, 512), (128, 256)])
@pytest.mark.parametrize("ctx", [65, 129])
def test_mtp_piece_where_a_row_sees_no_token(ctx, hq, latent):
    # ctx = 64k + 1, S = 2: the last page holds one token that query token 0 may not see;
    # one page per CTA makes that page a split piece with no token for those rows (with
    # Hq = 128, a whole head group's piece)
    case = synth.make_mla_case(batch=1, num_q_heads=hq, dtype=synth.BF16, context_lens=[ctx],
                               seed=2, seq_len_q=2, latent_dim=latent)
    # head groups per sequence: all 2 * Hq rows (<= 64), else groups of one token's 128
    # heads (the two-CTA kernel for the 576 record, heads-on-M for the 320 one)
    groups = 1 if 2 * hq <= 64 else 2 * hq // 128
    for force in ((ctx // 64 + 1) * groups, 0):
        _assert_close_mtp(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("name", ["mla_b16_ctx64k_h16_mtp2", "mla_b16_ctx64k_h128_mtp2",
                                  "mla_r256_b16_ctx64k_h128_mtp2"])
def test_mtp_full_size_workload_sampled_rows(name):
    case = synth.workload(name)
    hq = case.num_q_heads
    rows = [(b, i, h) for b in (0, 3, 7, 8, 12, 15) for i in range(2) for h in range(hq)]
    _assert_close_mtp(case, DeviceCase(case), rows=rows)
