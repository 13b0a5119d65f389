"""GQA/MQA/MHA paged decode on the GPU (through the C ABI) against the float64 oracle.

Tolerances (from the problem statement): max-abs error of out <= 2e-3 (fp16)
or 1e-2 (bf16); fp32 LSE within 1e-3. Indexing work is checked bit-exactly:
needle sweeps (every token position, including the last slot of a partial
page), poisoned stale slots and unused blocks, guard regions around the
outputs and never-written padded head rows.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE, TOL_OUT, DeviceCase, compare, device_bits, to_device_16
from paged_kv_cache_61_gb300 import pda, synth

pytestmark = pytest.mark.gpu

NAN16 = {synth.FP16: 0x7E00, synth.BF16: 0x7FC0}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pda.lib()


def _oracle(case, rows=None):
    return oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                               case.context_lens, case.scale, case.page_size, case.dtype, rows=rows)


def _assert_close(case, dc, ref=None, rows=None):
    out, lse = dc.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = ref if ref is not None else _oracle(case, rows)
    eo, el = compare(case, out, lse, ref_out, ref_lse, rows)
    assert eo <= TOL_OUT[case.dtype], f"out max-abs error {eo}"
    assert el <= TOL_LSE, f"lse max-abs error {el}"
    assert pda.read_device_error(dc.ws) == 0
    return out, lse


def _case(dtype, d, hq, hkv, ctx, seed=7, layout="pool"):
    return synth.make_gqa_case(batch=len(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               dtype=dtype, context_lens=ctx, table_layout=layout, seed=seed)


def test_tiny_workload():
    case = synth.workload("gqa_tiny")
    _assert_close(case, DeviceCase(case))


SMALL = [
    # dtype, D, Hq, Hkv, context lengths (several tiles, ragged tails, ctx = 1)
    (synth.FP16, 64, 8, 2, [1, 15, 16, 17, 37, 100, 256]),
    (synth.BF16, 128, 32, 8, [33, 500, 1, 64]),
    (synth.FP16, 128, 4, 4, [300, 2, 48, 129]),             # MHA
    (synth.BF16, 128, 16, 1, [700, 31]),                     # G = 16
    (synth.BF16, 128, 32, 1, [1000, 17, 1]),                 # MQA, G = 32
    (synth.FP16, 64, 24, 8, [90, 200, 3]),                   # G = 3
    (synth.BF16, 128, 64, 8, [2000, 16, 257, 5]),            # G = 8
    (synth.FP16, 128, 20, 2, [333, 1024]),                   # G = 10
]


@pytest.mark.parametrize("dtype,d,hq,hkv,ctx", SMALL)
@pytest.mark.parametrize("force", [0, 1, 3, 50])
def test_small_cases(dtype, d, hq, hkv, ctx, force):
    case = _case(dtype, d, hq, hkv, ctx)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("scale", [-0.09, 0.0])
@pytest.mark.parametrize("hkv", [8, 1])
def test_negative_and_zero_scale(scale, hkv):
    # any finite scale: negative (the scores' order flips) or zero (uniform weights)
    case = _case(synth.FP16, 128, 32, hkv, [300, 17, 64, 1], seed=14)
    case.scale = scale
    for force in (0, 5):
        _assert_close(case, DeviceCase(case, force_num_ctas=force))


def test_split_count_invariance():
    case = _case(synth.BF16, 128, 32, 8, [4000, 70, 1500])
    ref = _oracle(case)
    dc = DeviceCase(case)
    outs = []
    for force in (1, 2, 7, 64, 0):
        dc.replan(force)
        out, _ = _assert_close(case, dc, ref=ref)
        outs.append(out.float().clone())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= TOL_OUT[case.dtype]


@pytest.mark.parametrize("dtype,d", [(synth.FP16, 64), (synth.BF16, 128), (synth.FP16, 128)])
def test_needle_sweep_is_bit_exact(dtype, d):
    # sequence b has ctx = 45 and its needle at token b: every position, both page
    # boundaries and the last slot of the partial third page are visited.
    ctx = 45
    case = _case(dtype, d, 8, 2, [ctx] * ctx, seed=3)
    one = synth.float32_to_bits(np.float32(1.0), dtype)
    sixteen = synth.float32_to_bits(np.float32(16.0), dtype)
    case.q[:] = one
    case.k_cache[:] = 0
    for b in range(ctx):
        blk = int(case.block_tables[b, b // 16])
        case.k_cache[blk, b % 16] = sixteen
    for force in (0, 1, 17):
        dc = DeviceCase(case, force_num_ctas=force)
        out, lse = dc.run()
        torch.cuda.synchronize()
        got = device_bits(out)
        G = case.group
        for b in range(ctx):
            blk = int(case.block_tables[b, b // 16])
            for h in range(case.num_q_heads):
                assert np.array_equal(got[b, h], case.v_cache[blk, b % 16, h // G]), (force, b, h)


def test_ctx1_returns_first_value_row_exactly():
    case = _case(synth.BF16, 128, 32, 8, [1, 1, 1])
    dc = DeviceCase(case)
    out, lse = _assert_close(case, dc)
    got = device_bits(out)
    for b in range(3):
        blk = int(case.block_tables[b, 0])
        for h in range(32):
            assert np.array_equal(got[b, h], case.v_cache[blk, 0, h // 4])


@pytest.mark.parametrize("hkv", [8, 1])   # one page per ring stage; two (32-row segments)
def test_poisoned_stale_slots_unused_blocks_and_table_entries(hkv):
    case = _case(synth.FP16, 128, 32, hkv, [37, 100, 5, 250, 17], layout="permutation")
    clean = DeviceCase(case)
    out0, lse0 = _assert_close(case, clean)
    out0 = device_bits(out0)
    lse0 = lse0.cpu().numpy()
    k, v, tab = case.k_cache.copy(), case.v_cache.copy(), case.block_tables.copy()
    used = set()
    for b, c in enumerate(case.context_lens):
        npg = (int(c) + 15) // 16
        used.update(int(x) for x in tab[b, :npg])
        last, fill = int(tab[b, npg - 1]), int(c) - (npg - 1) * 16
        k[last, fill:] = NAN16[case.dtype]
        v[last, fill:] = NAN16[case.dtype]
        tab[b, npg:] = -123456
    for blk in range(case.num_blocks):
        if blk not in used:
            k[blk] = NAN16[case.dtype]
            v[blk] = NAN16[case.dtype]
    poisoned = synth.DecodeCase(**{**case.__dict__})
    poisoned.k_cache, poisoned.v_cache, poisoned.block_tables = k, v, tab
    for force in (0, 1, 9):
        dc = DeviceCase(poisoned, force_num_ctas=force)
        out1, lse1 = dc.run()
        torch.cuda.synchronize()
        if force == 0:
            assert np.array_equal(device_bits(out1), out0)
            assert np.array_equal(lse1.cpu().numpy(), lse0)
        assert torch.isfinite(out1.float()).all() and torch.isfinite(lse1).all()
        assert pda.read_device_error(dc.ws) == 0


def test_guard_regions_and_padded_heads_untouched():
    # G = 4 heads fill half of an 8-column MMA tile: the 4 padded columns must never be
    # written (they would land in the guard after the last head).
    case = _case(synth.BF16, 128, 4, 1, [77, 300])
    dc = DeviceCase(case, force_num_ctas=5)
    guard = 4096
    n_out = case.batch * case.num_q_heads * case.head_dim_v
    big = torch.full((guard + n_out + guard,), 0.0, dtype=torch.bfloat16, device="cuda")
    big.view(torch.int16).fill_(0x5A5A)
    big_lse = torch.full((guard + case.batch * case.num_q_heads + guard,), 7.25, device="cuda")
    out = big[guard:guard + n_out].view(case.batch, case.num_q_heads, case.head_dim_v)
    lse = big_lse[guard:guard + case.batch * case.num_q_heads].view(case.batch, case.num_q_heads)
    dc.run(out=out, lse=lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = _oracle(case)
    eo, el = compare(case, out, lse, ref_out, ref_lse)
    assert eo <= TOL_OUT[case.dtype] and el <= TOL_LSE
    g = big.view(torch.int16)
    assert (g[:guard] == 0x5A5A).all() and (g[guard + n_out:] == 0x5A5A).all()
    assert (big_lse[:guard] == 7.25).all() and (big_lse[guard + case.batch * 4:] == 7.25).all()
    # workspace beyond the plan's size is never touched either
    ws = torch.full((dc.plan.workspace_bytes + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    pda.workspace_init(dc.plan, ws)
    pda.paged_decode_attn(dc.q, dc.k, dc.v, dc.tables, dc.ctx, case.scale, out, lse, dc.plan, ws)
    torch.cuda.synchronize()
    assert (ws[dc.plan.workspace_bytes:] == 0xA5).all()


def test_lse_may_be_null():
    case = _case(synth.FP16, 64, 8, 2, [40, 3])
    dc = DeviceCase(case)
    out, _ = dc.run(lse=None)
    torch.cuda.synchronize()
    ref_out, _ = _oracle(case)
    assert np.abs(out.float().cpu().numpy() - ref_out).max() <= TOL_OUT[case.dtype]


def test_block_permutation_invariance_bitwise():
    case = _case(synth.BF16, 128, 32, 8, [600, 45], layout="permutation")
    out0, lse0 = DeviceCase(case).run()
    rng = np.random.default_rng(2)
    perm = rng.permutation(case.num_blocks)
    moved = synth.DecodeCase(**{**case.__dict__})
    moved.k_cache = np.empty_like(case.k_cache)
    moved.v_cache = np.empty_like(case.v_cache)
    moved.k_cache[perm] = case.k_cache
    moved.v_cache[perm] = case.v_cache
    moved.block_tables = perm[case.block_tables].astype(np.int32)
    out1, lse1 = DeviceCase(moved).run()
    torch.cuda.synchronize()
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(lse0, lse1)


def test_out_of_range_block_id_is_flagged():
    case = _case(synth.FP16, 64, 8, 2, [40, 20])
    bad = synth.DecodeCase(**{**case.__dict__})
    bad.block_tables = case.block_tables.copy()
    bad.block_tables[0, 1] = case.num_blocks + 5      # inside num_pages: a caller error
    dc = DeviceCase(bad)
    dc.run()
    torch.cuda.synchronize()
    assert pda.read_device_error(dc.ws) & 1
    assert pda.read_device_error(dc.ws) == 0          # reading clears it


def test_repeated_calls_reuse_workspace():
    case = _case(synth.BF16, 128, 32, 8, [3000, 10])
    dc = DeviceCase(case)
    ref = _oracle(case)
    first = None
    for _ in range(3):
        out, _ = _assert_close(case, dc, ref=ref)
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))


def test_combine_entry_point_matches_oracle():
    rng = np.random.default_rng(9)
    rows, splits, dv = 37, 5, 128
    po = rng.standard_normal((rows, splits, dv)).astype(np.float32)
    pl = (rng.standard_normal((rows, splits)) * 3).astype(np.float32)
    pl[3, 1] = -np.inf                      # an empty split
    pl[4, :] = pl[4, 0]                     # equal masses
    out = torch.empty(rows, dv, dtype=torch.float16, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    pda.combine_splits(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), rows, splits, dv,
                       out, pda.PDA_FP16, lse)
    torch.cuda.synchronize()
    for r in range(rows):
        o, l = oracle.combine_splits(po[r].astype(np.float64), pl[r].astype(np.float64))
        assert np.abs(out[r].float().cpu().numpy() - o).max() <= TOL_OUT[synth.FP16]
        assert abs(lse[r].item() - l) <= TOL_LSE


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["gqa_b64_ctx1k", "gqa_b1_ctx32k", "gqa_b1_ctx32k_mqa"])
def test_full_size_workload_all_rows(name):
    case = synth.workload(name)
    _assert_close(case, DeviceCase(case))


def test_full_size_varlen_sampled_rows():
    case = synth.workload("gqa_varlen_b128")
    order = np.argsort(case.context_lens)
    seqs = list(order[:4]) + list(order[-4:]) + list(range(0, 128, 16))
    rows = [(int(b), int(h)) for b in seqs for h in range(case.num_q_heads)]
    _assert_close(case, DeviceCase(case), rows=rows)
