"""GQA/MQA decode with more than 32 query rows per KV head, on the GPU vs the float64 oracle.

"优化 decode attention 与 GQA", section ③: the G query heads of a KV head share its pages;
the pages' MQA discussion (the variants page, "MQA") takes Hq/Hkv up to the full head
count. The kernel's column tiles hold 32 rows, so a KV head's S*G rows are cut into equal
row chunks; each chunk is a segment of its own that reads the KV head's pages. These
cases check every chunk's rows (including a last chunk with fewer rows), their causal
limits for S > 1, split pieces merged in the kernel and by the split-merge kernel, fp8
caches, and that no row beyond the real ones is written. Tolerances as everywhere.
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
    fn = oracle.paged_decode_mtp if case.seq_len_q > 1 else oracle.paged_decode
    return fn(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
              case.scale, case.page_size, case.dtype, rows=rows, kv_format=case.kv_format,
              k_scale=case.k_scale, v_scale=case.v_scale)


def _case(dtype, d, hq, hkv, ctx, s=1, seed=7, fmt=None):
    return synth.make_gqa_case(batch=len(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               dtype=dtype, context_lens=ctx, seed=seed, seq_len_q=s,
                               kv_format=fmt)


def _assert_close(case, dc, ref=None, rows=None):
    out, lse = dc.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = ref if ref is not None else _oracle(case, rows)
    eo, el = compare(case, out, lse, ref_out, ref_lse, rows)
    assert eo <= TOL_OUT[case.dtype], f"out max-abs error {eo}"
    assert el <= TOL_LSE, f"lse max-abs error {el}"
    assert pda.read_device_error(dc.ws) == 0
    return out, lse


CASES = [
    # dtype, D, Hq, Hkv, S, context lengths: rows per KV head S*G -> row chunks
    (synth.BF16, 128, 64, 1, 1, [700, 31, 1]),          # MQA, 64 rows: 2 chunks of 32
    (synth.FP16, 64, 96, 2, 1, [300, 17, 64]),          # G = 48: 2 chunks of 24
    (synth.BF16, 128, 128, 1, 1, [2000, 5]),            # MQA, 128 rows: 4 chunks of 32
    (synth.FP16, 128, 40, 1, 1, [129, 16, 2]),          # G = 40: 2 chunks of 20
    (synth.FP16, 128, 64, 2, 2, [300, 2, 48]),          # S = 2, G = 32: 2 chunks of 32
    (synth.FP16, 64, 22, 2, 3, [90, 3, 200]),           # S = 3, G = 11: 33 rows, 17 + 16
    (synth.BF16, 128, 64, 4, 4, [500, 33, 64]),         # S = 4, G = 16: 2 chunks of 32
]


@pytest.mark.parametrize("fmt", [None, synth.FP8_E4M3])
@pytest.mark.parametrize("dtype,d,hq,hkv,s,ctx", CASES)
@pytest.mark.parametrize("force", [0, 1, 3, 50])
def test_row_chunks(dtype, d, hq, hkv, s, ctx, force, fmt):
    case = _case(dtype, d, hq, hkv, ctx, s, fmt=fmt)
    dc = DeviceCase(case, force_num_ctas=force)
    rows = s * hq // hkv
    assert dc.plan.num_ctas >= 1 and rows > 32
    _assert_close(case, dc)


@pytest.mark.parametrize("hq,hkv,s", [(64, 1, 1), (128, 1, 1), (22, 2, 3)])
def test_long_sequence_goes_through_the_split_merge(hq, hkv, s):
    # one long sequence: every row chunk is cut into up to 32 pieces, more than the
    # in-kernel merge takes, so the split-merge kernel merges them
    case = _case(synth.BF16, 128, hq, hkv, [20000], s, seed=11)
    dc = DeviceCase(case)
    assert dc.plan.num_launches == 2 and dc.plan.num_splits(0) > 4
    _assert_close(case, dc)


def test_chunks_agree_with_single_segment_heads():
    # The first 32 heads of a 64-head MQA problem form its first row chunk, which is the
    # whole of a 32-head problem on the same caches, lengths and tables. With the same
    # piece boundaries (a share of 9 pages either way: 14 and 7 CTAs; or one page per
    # CTA) the two compute those rows with the same arithmetic: bit-identical outputs.
    big = _case(synth.BF16, 128, 64, 1, [900, 40, 3], seed=5)
    small = synth.DecodeCase(**{**big.__dict__})
    small.q = big.q[:, :32].copy()
    small.num_q_heads = 32
    pages = sum((int(c) + 15) // 16 for c in big.context_lens)
    for f_big, f_small in ((14, 7), (2 * pages, pages)):
        db, ds = DeviceCase(big, force_num_ctas=f_big), DeviceCase(small, force_num_ctas=f_small)
        assert db.plan.num_splits(0) == ds.plan.num_splits(0) > 1
        ob, lb = db.run()
        os_, ls = ds.run()
        torch.cuda.synchronize()
        assert np.array_equal(device_bits(ob)[:, :32], device_bits(os_))
        assert torch.equal(lb[:, :32], ls)


def test_needle_reaches_every_chunk_exactly():
    # q = 1 everywhere and one key of 16s per sequence (at token b): every row of every
    # chunk takes that token's value row exactly (the other tokens' weights, exp(-16 D
    # scale) = exp(-128), underflow to 0)
    ctx = 40
    case = _case(synth.FP16, 64, 72, 1, [ctx] * ctx, seed=3)     # 72 rows: 3 chunks of 24
    one = synth.float32_to_bits(np.float32(1.0), case.dtype)
    sixteen = synth.float32_to_bits(np.float32(16.0), case.dtype)
    case.q[:] = one
    case.k_cache[:] = 0
    for b in range(ctx):
        blk = int(case.block_tables[b, b // 16])
        case.k_cache[blk, b % 16] = sixteen
    for force in (0, 1, 13):
        out, _ = DeviceCase(case, force_num_ctas=force).run()
        torch.cuda.synchronize()
        got = device_bits(out)
        for b in range(ctx):
            blk = int(case.block_tables[b, b // 16])
            for h in range(case.num_q_heads):
                assert np.array_equal(got[b, h], case.v_cache[blk, b % 16, 0]), (force, b, h)


def test_short_last_chunk_writes_only_real_rows():
    # S = 3, G = 11: 33 rows per KV head in chunks of 17 and 16. The last chunk's 17th
    # row does not exist; nothing may be written past the real rows.
    case = _case(synth.BF16, 128, 11, 1, [77, 300], 3)
    dc = DeviceCase(case, force_num_ctas=5)
    B, S, H, D = case.batch, 3, case.num_q_heads, case.head_dim_v
    guard = 4096
    n_out, n_lse = B * S * H * D, B * H * S
    big = torch.zeros(guard + n_out + guard, dtype=torch.bfloat16, device="cuda")
    big.view(torch.int16).fill_(0x5A5A)
    big_lse = torch.full((guard + n_lse + guard,), 7.25, device="cuda")
    out = big[guard:guard + n_out].view(B, S, H, D)
    lse = big_lse[guard:guard + n_lse].view(B, H, S)
    dc.run(out=out, lse=lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = _oracle(case)
    eo, el = compare(case, out, lse, ref_out, ref_lse)
    assert eo <= TOL_OUT[case.dtype] and el <= TOL_LSE
    g = big.view(torch.int16)
    assert (g[:guard] == 0x5A5A).all() and (g[guard + n_out:] == 0x5A5A).all()
    assert (big_lse[:guard] == 7.25).all() and (big_lse[guard + n_lse:] == 7.25).all()


@pytest.mark.parametrize("name", ["gqa_b1_ctx32k_mqa_h64", "gqa_b1_ctx32k_mqa_h64_fp8"])
def test_full_size_mqa_64_heads_all_rows(name):
    # B=1, ctx 32K, 64 query heads on one KV head: two row chunks of 32, each cut into
    # split pieces, in the launch configuration the benchmark times
    case = synth.workload(name)
    _assert_close(case, DeviceCase(case))
