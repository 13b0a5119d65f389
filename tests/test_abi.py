"""The C-ABI library: it loads, exports every declared symbol and validates on the host.

No compute call runs here: every call below returns before touching a GPU.
"""
import ctypes
import os
import re

import pytest

from paged_kv_cache_61_gb300 import build, pda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(pda.LIB_PATH):
        build.build()
    return pda.lib()


def _declared_functions():
    names = []
    for header in os.listdir(os.path.join(ROOT, "include")):
        if header.endswith(".h"):
            text = open(os.path.join(ROOT, "include", header)).read()
            names += re.findall(r"PDA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported():
    names = _declared_functions()
    assert len(names) >= 12
    handle = ctypes.CDLL(pda.LIB_PATH)
    for name in names:
        assert hasattr(handle, name), f"{name} declared in include/ but not exported"


def test_status_strings():
    assert pda.status_name(pda.PDA_OK) == "PDA_OK"
    assert pda.status_name(pda.PDA_ERR_WORKSPACE) == "PDA_ERR_WORKSPACE"


def _plan(**kw):
    args = dict(kind=pda.PDA_KIND_GQA, dtype=pda.PDA_FP16, batch=2, num_q_heads=8, num_kv_heads=2,
                head_dim_qk=64, head_dim_v=64, page_size=16, max_blocks_per_seq=4, num_blocks=8,
                context_lens=[5, 64], num_sms=152)
    args.update(kw)
    return pda.Plan(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=6, num_kv_heads=4), pda.PDA_ERR_INVALID_ARG),      # H_q % H_kv != 0
    (dict(context_lens=[0, 5]), pda.PDA_ERR_INVALID_ARG),                 # ctx < 1
    (dict(context_lens=[65, 5]), pda.PDA_ERR_INVALID_ARG),                # ctx > max_blocks * P
    (dict(dtype=7), pda.PDA_ERR_INVALID_ARG),
    (dict(kind=9), pda.PDA_ERR_INVALID_ARG),
    (dict(head_dim_qk=96, head_dim_v=96), pda.PDA_ERR_UNSUPPORTED),
    (dict(page_size=32, context_lens=[5, 5]), pda.PDA_ERR_UNSUPPORTED),
    (dict(num_q_heads=2050, num_kv_heads=2), pda.PDA_ERR_UNSUPPORTED),    # G = 1025
    (dict(batch=-1), pda.PDA_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_problems(kw, status):
    with pytest.raises(pda.PdaError) as e:
        _plan(**kw)
    assert e.value.status == status
    assert pda.lib().pda_last_error().decode() != ""


def test_plan_properties():
    p = _plan()
    assert p.num_ctas >= 1
    assert p.workspace_bytes >= 256 and p.workspace_bytes % 256 == 0
    assert p.num_splits(0) >= 1 and p.num_splits(5) == 0
    one = _plan(force_num_ctas=1)
    assert one.num_ctas == 1 and one.num_splits(0) == one.num_splits(1) == 1


def test_uniform_batch_split_counts():
    # 64 sequences x 8 KV heads x 64 pages over 7 forced CTAs: each range holds
    # ceil(32768/7) tiles, so no segment is cut by more than 2 ranges
    p = _plan(batch=64, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, head_dim_v=128,
              max_blocks_per_seq=64, num_blocks=4096, context_lens=[1024] * 64, force_num_ctas=7)
    assert p.num_ctas == 7
    assert max(p.num_splits(b) for b in range(64)) == 2
    # one long sequence is split across every CTA
    p = _plan(batch=1, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, head_dim_v=128,
              max_blocks_per_seq=2048, num_blocks=2048, context_lens=[32768])
    assert p.num_ctas > 100 and p.num_splits(0) > 10


def test_empty_batch_is_a_no_op():
    p = _plan(batch=0, context_lens=[])
    assert p.num_ctas == 0
    # all pointers NULL: nothing is enqueued, so this is safe without a GPU
    pda.paged_decode_attn(0, 0, 0, 0, 0, 0.125, 0, None, p, 0, stream=0)


@pytest.mark.parametrize("which", ["q", "k", "out", "ws", "misaligned_q", "scale", "kind"])
def test_decode_rejects_bad_arguments_before_launch(which):
    p = _plan()
    args = dict(q=4096, k=8192, v=8192, tables=64, ctx=128, scale=0.125, out=4096, lse=None,
                ws=1 << 20)
    if which == "q":
        args["q"] = 0
    elif which == "k":
        args["k"] = 0
    elif which == "out":
        args["out"] = 0
    elif which == "ws":
        args["ws"] = 0
    elif which == "misaligned_q":
        args["q"] = 4098
    elif which == "scale":
        args["scale"] = float("inf")
    with pytest.raises(pda.PdaError) as e:
        if which == "kind":
            pda.mla_decode(args["q"], args["k"], args["tables"], args["ctx"], args["scale"],
                           args["out"], None, p, args["ws"], stream=0)
        else:
            pda.paged_decode_attn(args["q"], args["k"], args["v"], args["tables"], args["ctx"],
                                  args["scale"], args["out"], args["lse"], p, args["ws"], stream=0)
    assert e.value.status in (pda.PDA_ERR_INVALID_ARG, pda.PDA_ERR_WORKSPACE)


def test_combine_rejects_bad_sizes():
    with pytest.raises(pda.PdaError):
        pda.combine_splits(0, 0, 4, 0, 128, 0, pda.PDA_FP16, None, stream=0)
    with pytest.raises(pda.PdaError):
        pda.combine_splits(0, 0, 4, 2, 130, 0, pda.PDA_FP16, None, stream=0)
    pda.combine_splits(0, 0, 0, 2, 128, 0, pda.PDA_FP16, None, stream=0)  # rows == 0: no-op


def test_fp8_plans_and_calls_must_agree():
    f8 = _plan(kv_format=pda.PDA_KV_FP8_E4M3)
    same = _plan()
    args = (4096, 8192, 8192)
    # a 16-bit call with an fp8 plan, and the other way round, are refused on the host
    with pytest.raises(pda.PdaError) as e:
        pda.paged_decode_attn(*args, 64, 128, 0.125, 4096, None, f8, 1 << 20, stream=0)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    with pytest.raises(pda.PdaError) as e:
        pda.paged_decode_attn_fp8(*args, 1.0, 1.0, 64, 128, 0.125, 4096, None, same, 1 << 20,
                                  stream=0)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    with pytest.raises(pda.PdaError) as e:
        pda.paged_decode_attn_no_alloc(*args, 64, 128, 0.125, 4096, None, f8, stream=0)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    for ks, vs in ((float("nan"), 1.0), (1.0, float("inf"))):
        with pytest.raises(pda.PdaError) as e:
            pda.paged_decode_attn_fp8(*args, ks, vs, 64, 128, 0.125, 4096, None, f8, 1 << 20,
                                      stream=0)
        assert e.value.status == pda.PDA_ERR_INVALID_ARG


def test_fp8_plan_validation():
    with pytest.raises(pda.PdaError) as e:
        _plan(kv_format=5)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    mla = dict(kind=pda.PDA_KIND_MLA, num_kv_heads=1, head_dim_qk=576, head_dim_v=512,
               page_size=64, max_blocks_per_seq=2, context_lens=[5, 64],
               kv_format=pda.PDA_KV_FP8_E4M3)
    # E4M3 record caches: groups of 16 or 32 query rows; larger head counts are refused
    for hq in (16, 32):
        assert _plan(num_q_heads=hq, **mla).num_ctas >= 1
    assert _plan(num_q_heads=16, seq_len_q=2, **mla).num_ctas >= 1
    for hq in (64, 128):
        with pytest.raises(pda.PdaError) as e:
            _plan(num_q_heads=hq, **mla)
        assert e.value.status == pda.PDA_ERR_UNSUPPORTED
    # the fp8 call needs an fp8 plan, the 16-bit call a 16-bit one, the scale is finite
    f8m = _plan(num_q_heads=16, **mla)
    m16 = _plan(num_q_heads=16, **{**mla, "kv_format": pda.PDA_KV_SAME_AS_Q})
    margs = (4096, 8192, 64, 128, 0.07, 4096, None)
    with pytest.raises(pda.PdaError) as e:
        pda.mla_decode(*margs, f8m, 1 << 20, stream=0)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    for plan, ks in ((m16, 1.0), (f8m, float("nan"))):
        with pytest.raises(pda.PdaError) as e:
            pda.mla_decode_fp8(4096, 8192, ks, 64, 128, 0.07, 4096, None, plan, 1 << 20,
                               stream=0)
        assert e.value.status == pda.PDA_ERR_INVALID_ARG
    # appends: the 16-bit record append refuses an fp8 plan (it would store codes with a
    # scale of 1), the fp8 one a 16-bit plan and a scale that is not finite or is zero
    with pytest.raises(pda.PdaError) as e:
        pda.mla_append(4096, 8192, 64, 128, f8m, 1 << 20, stream=0)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    for plan, ks in ((m16, 1.0), (f8m, float("inf")), (f8m, 0.0)):
        with pytest.raises(pda.PdaError) as e:
            pda.mla_append_fp8(4096, 8192, ks, 64, 128, plan, 1 << 20, stream=0)
        assert e.value.status == pda.PDA_ERR_INVALID_ARG
    f8 = _plan(batch=0, context_lens=[], kv_format=pda.PDA_KV_FP8_E4M3)
    pda.paged_decode_attn_fp8(0, 0, 0, 1.0, 1.0, 0, 0, 0.125, 0, None, f8, 0, stream=0)


def test_multi_token_plan_validation():
    # S = 2 query tokens: every context must hold at least S tokens
    with pytest.raises(pda.PdaError) as e:
        _plan(seq_len_q=2, context_lens=[1, 64])
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    # S * G query rows per KV head are limited to 1024
    with pytest.raises(pda.PdaError) as e:
        _plan(seq_len_q=3, num_q_heads=684, num_kv_heads=2)
    assert e.value.status == pda.PDA_ERR_UNSUPPORTED
    with pytest.raises(pda.PdaError) as e:
        _plan(seq_len_q=-1)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    mla = dict(kind=pda.PDA_KIND_MLA, num_kv_heads=1, head_dim_qk=576, head_dim_v=512,
               page_size=64, max_blocks_per_seq=2, context_lens=[5, 64], seq_len_q=2)
    # MLA: the S * Hq rows of a sequence form one group when there are at most 64, else
    # groups of one query token's heads, which needs Hq a multiple of 64
    with pytest.raises(pda.PdaError) as e:
        _plan(num_q_heads=48, **mla)
    assert e.value.status == pda.PDA_ERR_UNSUPPORTED
    p = _plan(num_q_heads=16, **mla)            # 32 rows: one head group per sequence
    assert p.num_ctas >= 1
    for hq, dqk in ((64, 576), (128, 576), (128, 320)):
        p = _plan(num_q_heads=hq, **{**mla, "head_dim_qk": dqk, "head_dim_v": dqk - 64,
                                     "force_num_ctas": 1})
        # accepted: 2 groups of 64 rows (Hq=64) or 2 of 128 (Hq=128: the two-CTA kernel for
        # the 576 record, heads-on-M for the 320 one) per sequence
        assert p.num_ctas == 1 and p.workspace_bytes > 0
    # one tile per CTA (force_num_ctas above the tile count) makes num_ctas the tile count,
    # pages x head groups per sequence: ctx 5 and 64 are one 64-token page each
    for hq, dqk, groups in ((16, 576, 1), (64, 576, 2), (128, 576, 2), (128, 320, 2),
                            (256, 320, 4), (256, 576, 4)):
        p = _plan(num_q_heads=hq, **{**mla, "head_dim_qk": dqk, "head_dim_v": dqk - 64,
                                     "force_num_ctas": 1000})
        assert p.num_ctas == 2 * groups, (hq, dqk)
    # S = 2 doubles the rows of a segment, and so each split piece's partial
    one, two = _plan(), _plan(seq_len_q=2)
    assert two.workspace_bytes > one.workspace_bytes


@pytest.mark.parametrize("hq,hkv,s,chunks", [
    (64, 1, 1, 2),      # MQA with 64 heads: chunks of 32 rows
    (96, 2, 1, 2),      # G = 48: chunks of 24
    (40, 1, 1, 2),      # G = 40: chunks of 20
    (22, 2, 3, 2),      # S * G = 33: chunks of 17 and 16
    (128, 1, 2, 8),     # 256 rows: chunks of 32
    (32, 1, 1, 1),      # 32 rows: one segment per KV head
    (12, 2, 5, 1),      # S * G = 30
])
def test_planner_cuts_many_rows_into_chunks(hq, hkv, s, chunks):
    # more than 32 query rows per KV head: the rows are cut into equal chunks, each a
    # segment that reads the KV head's pages. With one page per CTA the CTA count is the
    # tile count: pages x Hkv x chunks (ctx 5 and 64 are 1 + 4 pages of 16 tokens).
    p = _plan(num_q_heads=hq, num_kv_heads=hkv, seq_len_q=s, context_lens=[max(5, s), 64],
              force_num_ctas=1000)
    assert p.num_ctas == 5 * hkv * chunks
    rows = s * hq // hkv
    group = -(-rows // chunks)
    # workspace: two split slots of `group` rows (fp32 LSE + 64 fp32 dims) per CTA
    assert p.workspace_bytes >= p.num_ctas * 2 * group * 4 * 65


@pytest.mark.parametrize("hkv,ctas,splits", [(8, 256, 32), (2, 64, 32), (1, 32, 32)])
def test_planner_cuts_a_long_segment_into_equal_pieces(hkv, ctas, splits):
    # B=1, ctx 32K (2048 pages of 16 tokens), 152 SMs: pieces of 2048 / k pages, so every
    # CTA range lies inside one segment, and at most 32 pieces per segment. Hkv=8: the
    # natural share is 54 pages, and 64-page pieces are within a quarter above it. Hkv=2
    # and MQA: the share is raised to 64 pages (32 pieces per segment).
    p = _plan(batch=1, num_q_heads=32, num_kv_heads=hkv, head_dim_qk=128, head_dim_v=128,
              page_size=16, max_blocks_per_seq=2048, num_blocks=2048, context_lens=[32768],
              num_sms=152)
    assert p.num_ctas == ctas and p.num_splits(0) == splits
    # pieces beyond the in-kernel merge's four go to the split-merge kernel
    assert p.num_launches == 2


def test_planner_merges_few_pieces_in_kernel():
    # a uniform batch cut into whole segments needs one launch; a sequence cut into a few
    # pieces is merged by its last piece, in the same launch
    p = _plan(batch=64, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, head_dim_v=128,
              page_size=16, max_blocks_per_seq=64, num_blocks=4096, context_lens=[1024] * 64,
              num_sms=152)
    assert p.num_launches == 1
    p = _plan(batch=1, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, head_dim_v=128,
              page_size=16, max_blocks_per_seq=2048, num_blocks=2048, context_lens=[32768],
              num_sms=152, force_num_ctas=24)
    assert 2 <= p.num_splits(0) <= 4 and p.num_launches == 1


def test_planner_keeps_a_tiny_problem_in_one_launch():
    # at most one tile per SM (B=4, ctx up to 242, Hkv=2: 72 tiles): the share is raised
    # until no segment has more pieces than the decode kernel merges itself
    lens = [206, 242, 2, 81]
    p = _plan(batch=4, num_q_heads=8, num_kv_heads=2, head_dim_qk=64, head_dim_v=64,
              page_size=16, max_blocks_per_seq=16, num_blocks=64, context_lens=lens,
              num_sms=152)
    assert p.num_launches == 1 and max(p.num_splits(b) for b in range(4)) <= 4
    # a forced CTA count is kept as asked, merge launch included
    f = _plan(batch=4, num_q_heads=8, num_kv_heads=2, head_dim_qk=64, head_dim_v=64,
              page_size=16, max_blocks_per_seq=16, num_blocks=64, context_lens=lens,
              num_sms=152, force_num_ctas=36)
    assert f.num_ctas == 36 and f.num_launches == 2


def test_planner_gives_whole_segments_to_a_uniform_batch():
    # B=64, ctx 1024, Hkv=8: 512 segments of 64 pages, two whole segments per CTA
    p = _plan(batch=64, num_q_heads=32, num_kv_heads=8, head_dim_qk=128, head_dim_v=128,
              page_size=16, max_blocks_per_seq=64, num_blocks=4096, context_lens=[1024] * 64,
              num_sms=152)
    assert p.num_ctas == 256 and all(p.num_splits(b) == 1 for b in range(64))
