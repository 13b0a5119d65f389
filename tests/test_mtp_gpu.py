"""Multi-token (speculative / MTP) GQA decode on the GPU vs the float64 oracle.

S query tokens per sequence; token i sits at position ctx - S + i and attends to tokens
0 .. ctx - S + i (causal, bottom-right aligned). q and out are [B, S, Hq, D], lse is
[B, Hq, S]. Tolerances as for single-token decode.
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
    return oracle.paged_decode_mtp(case.q, case.k_cache, case.v_cache, case.block_tables,
                                   case.context_lens, case.scale, case.page_size, case.dtype,
                                   rows=rows, kv_format=case.kv_format, k_scale=case.k_scale,
                                   v_scale=case.v_scale)


def _assert_close(case, dc, rows=None):
    out, lse = dc.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = _oracle(case, rows)
    eo, el = compare(case, out, lse, ref_out, ref_lse, rows)
    assert eo <= TOL_OUT[case.dtype], f"out max-abs error {eo}"
    assert el <= TOL_LSE, f"lse max-abs error {el}"
    assert pda.read_device_error(dc.ws) == 0
    return out, lse


def _case(dtype, d, hq, hkv, ctx, s, seed=7, fmt=None):
    return synth.make_gqa_case(batch=len(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               dtype=dtype, context_lens=ctx, seed=seed, seq_len_q=s,
                               kv_format=fmt)


# Contexts of ctx = S (the first query token sees one token) are in the fp16 cases: with
# so few tokens an output can reach |out| >= 4, where bf16's own rounding step (2^-6)
# is already above the 1e-2 bf16 tolerance. bf16 cases give every query row >= 16 tokens.
SMALL = [
    # q dtype, D, Hq, Hkv, S, context lengths (ctx = S, page boundaries at ctx - S + i)
    (synth.FP16, 64, 8, 2, 2, [2, 16, 17, 18, 33, 100, 256]),
    (synth.BF16, 128, 32, 8, 2, [33, 500, 17, 64]),
    (synth.FP16, 128, 4, 4, 3, [300, 3, 48, 129]),           # MHA, S = 3
    (synth.BF16, 128, 16, 1, 2, [700, 31]),                   # MQA, 32 rows
    (synth.FP16, 64, 24, 8, 4, [90, 200, 4]),                 # G = 3, S = 4
    (synth.BF16, 128, 64, 8, 2, [2000, 17, 257, 18]),         # G = 8
]


@pytest.mark.parametrize("fmt", [None, synth.FP8_E4M3])
@pytest.mark.parametrize("dtype,d,hq,hkv,s,ctx", SMALL)
@pytest.mark.parametrize("force", [0, 1, 3, 50])
def test_small_cases(dtype, d, hq, hkv, s, ctx, force, fmt):
    case = _case(dtype, d, hq, hkv, ctx, s, fmt=fmt)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("fmt", [None, synth.FP8_E4M3])
@pytest.mark.parametrize("ctx", [17, 33, 49])
def test_piece_where_a_row_sees_no_token(ctx, fmt):
    # ctx = 16k + 1, S = 2: the last page holds one token, which query token 0 may not see.
    # With one page per CTA that page is a split piece in which row 0 has no token at all.
    case = _case(synth.BF16, 128, 4, 1, [ctx], 2, seed=2, fmt=fmt)
    for force in (ctx // 16 + 1, 2, 0):
        _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("fmt", [None, synth.FP8_E4M3])
def test_causal_boundary_needles_are_bit_exact(fmt):
    # ctx 45, S = 2: token 43 has K = 16 and token 44 has K = 32, all others 0, q = 1.
    # Query token 1 sees both and selects token 44; query token 0 may not see token 44
    # and selects token 43. The other weights underflow to 0, so out = V exactly.
    ctx, S = 45, 2
    case = _case(synth.FP16, 64, 8, 2, [ctx] * 3, S, seed=3, fmt=fmt)
    case.q[:] = synth.float32_to_bits(np.float32(1.0), case.dtype)
    case.k_cache[:] = 0
    for b in range(3):
        for t, val in ((43, 16.0), (44, 32.0)):
            blk = int(case.block_tables[b, t // 16])
            if fmt == synth.FP8_E4M3:
                case.k_cache[blk, t % 16] = synth.float32_to_e4m3(np.float32(val))
            else:
                case.k_cache[blk, t % 16] = synth.float32_to_bits(np.float32(val), case.dtype)
    if fmt == synth.FP8_E4M3:
        case.k_scale, case.v_scale = 1.0, 1.0
    for force in (0, 1, 5):
        dc = DeviceCase(case, force_num_ctas=force)
        out, _ = dc.run()
        torch.cuda.synchronize()
        got = device_bits(out)
        for b in range(3):
            for i, t in ((0, 43), (1, 44)):
                blk = int(case.block_tables[b, t // 16])
                for h in range(case.num_q_heads):
                    v = case.v_cache[blk, t % 16, h // case.group]
                    want = (oracle.decode_e4m3(v).astype(np.float32) if fmt == synth.FP8_E4M3
                            else synth.bits_to_float32(v, case.dtype))
                    # equal values (the weighted sum turns a -0 into +0)
                    assert np.array_equal(synth.bits_to_float32(got[b, i, h], case.dtype),
                                          want), (force, b, i, h)


@pytest.mark.parametrize("name", ["gqa_b64_ctx1k_mtp2", "gqa_b1_ctx32k_mtp2",
                                  "gqa_b64_ctx1k_mtp2_fp8"])
def test_full_size_workload_sampled_rows(name):
    case = synth.workload(name)
    hq = case.num_q_heads
    bs = sorted({0, case.batch // 2, case.batch - 1})
    rows = [(b, i, h) for b in bs for i in range(case.seq_len_q) for h in range(hq)]
    _assert_close(case, DeviceCase(case), rows=rows)
