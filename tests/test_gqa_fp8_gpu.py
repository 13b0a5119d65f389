"""GQA/MQA/MHA paged decode over fp8 (E4M3) caches on the GPU vs the float64 oracle.

The oracle decodes every cached byte exactly and applies the per-tensor scales in
float64; the kernel converts the codes exactly to q's 16-bit type, folds k_scale into
the softmax scale and v_scale into the final normalisation. Tolerances are those of
the 16-bit caches: out max-abs <= 2e-3 (fp16 q) / 1e-2 (bf16 q), LSE within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE, TOL_OUT, DeviceCase, compare, device_bits
from paged_kv_cache_61_gb300 import pda, synth

pytestmark = pytest.mark.gpu

NAN_E4M3 = 0x7F


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pda.lib()


def _oracle(case, rows=None):
    return oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                               case.context_lens, case.scale, case.page_size, case.dtype,
                               rows=rows, kv_format=case.kv_format, k_scale=case.k_scale,
                               v_scale=case.v_scale)


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
                               dtype=dtype, context_lens=ctx, table_layout=layout, seed=seed,
                               kv_format=synth.FP8_E4M3)


SMALL = [
    # q dtype, D, Hq, Hkv, context lengths (several tiles, ragged tails, ctx = 1)
    (synth.FP16, 64, 8, 2, [1, 15, 16, 17, 37, 100, 256]),
    (synth.BF16, 128, 32, 8, [33, 500, 1, 64]),
    (synth.FP16, 128, 4, 4, [300, 2, 48, 129]),             # MHA
    (synth.BF16, 128, 32, 1, [1000, 17, 1]),                 # MQA, G = 32
    (synth.FP16, 64, 24, 8, [90, 200, 3]),                   # G = 3
    (synth.BF16, 64, 16, 2, [513, 40]),                      # D = 64, G = 8
    (synth.FP16, 128, 20, 2, [333, 1024]),                   # G = 10
]


@pytest.mark.parametrize("dtype,d,hq,hkv,ctx", SMALL)
@pytest.mark.parametrize("force", [0, 1, 3, 50])
def test_small_cases(dtype, d, hq, hkv, ctx, force):
    case = _case(dtype, d, hq, hkv, ctx)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("k_scale", [-0.02, 0.0])
def test_negative_and_zero_k_scale(k_scale):
    # k_scale folds into the softmax scale: a negative one flips the scores' order, zero
    # gives uniform weights
    case = _case(synth.BF16, 128, 16, 2, [300, 17, 64, 1], seed=13)
    case.k_scale = k_scale
    for force in (0, 5):
        _assert_close(case, DeviceCase(case, force_num_ctas=force))


def test_tiny_workload():
    case = synth.workload("gqa_tiny_fp8")
    _assert_close(case, DeviceCase(case))


def test_split_count_invariance():
    case = _case(synth.BF16, 128, 32, 8, [4000, 70, 1500])
    ref = _oracle(case)
    dc = DeviceCase(case)
    for force in (1, 2, 7, 64, 0):
        dc.replan(force)
        _assert_close(case, dc, ref=ref)


@pytest.mark.parametrize("dtype,d", [(synth.FP16, 64), (synth.BF16, 128), (synth.BF16, 64)])
def test_needle_sweep_is_bit_exact(dtype, d):
    # sequence b (ctx 45) has its needle at token b: K = 16 there and 0 elsewhere, q = 1,
    # so every other weight underflows to 0 and out = e4m3(V code) * v_scale exactly
    # (a power-of-two v_scale keeps the product exact in the 16-bit output type).
    ctx = 45
    case = _case(dtype, d, 8, 2, [ctx] * ctx, seed=3)
    case.q[:] = synth.float32_to_bits(np.float32(1.0), dtype)
    case.k_scale, case.v_scale = 1.0, 0.5
    case.k_cache[:] = 0
    for b in range(ctx):
        blk = int(case.block_tables[b, b // 16])
        case.k_cache[blk, b % 16] = 0x58                 # 16.0
    for force in (0, 1, 17):
        dc = DeviceCase(case, force_num_ctas=force)
        out, _ = dc.run()
        torch.cuda.synchronize()
        got = device_bits(out)
        G = case.group
        for b in range(ctx):
            blk = int(case.block_tables[b, b // 16])
            for h in range(case.num_q_heads):
                want = oracle.decode_e4m3(case.v_cache[blk, b % 16, h // G]) * 0.5
                assert np.array_equal(got[b, h], synth.float32_to_bits(want.astype(np.float32),
                                                                       dtype)), (force, b, h)


def test_every_code_reaches_the_output_exactly():
    # ctx = 1: out = e4m3(code) * v_scale. The V rows hold every finite code.
    case = _case(synth.BF16, 128, 8, 2, [1] * 2, seed=5)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    for b in range(2):
        blk = int(case.block_tables[b, 0])
        for kvh in range(2):
            case.v_cache[blk, 0, kvh] = np.resize(np.roll(finite, 128 * b + 64 * kvh), 128)
    case.v_scale = 2.0 ** -3
    out, _ = DeviceCase(case).run()
    torch.cuda.synchronize()
    got = device_bits(out)
    for b in range(2):
        blk = int(case.block_tables[b, 0])
        for h in range(8):
            want = (oracle.decode_e4m3(case.v_cache[blk, 0, h // 4]) * case.v_scale)
            # equal values (the sum that forms the output turns -0 into +0)
            assert np.array_equal(synth.bits_to_float32(got[b, h], synth.BF16),
                                  want.astype(np.float32)), (b, h)


def test_poisoned_stale_slots_unused_blocks_and_table_entries():
    case = _case(synth.FP16, 128, 32, 8, [37, 100, 5, 250], layout="permutation")
    out0, lse0 = _assert_close(case, DeviceCase(case))
    out0 = device_bits(out0)
    lse0 = lse0.cpu().numpy()
    k, v, tab = case.k_cache.copy(), case.v_cache.copy(), case.block_tables.copy()
    used = set()
    for b, c in enumerate(case.context_lens):
        npg = (int(c) + 15) // 16
        used.update(int(x) for x in tab[b, :npg])
        last, fill = int(tab[b, npg - 1]), int(c) - (npg - 1) * 16
        k[last, fill:] = NAN_E4M3
        v[last, fill:] = NAN_E4M3
        tab[b, npg:] = -123456
    for blk in range(case.num_blocks):
        if blk not in used:
            k[blk] = NAN_E4M3
            v[blk] = NAN_E4M3
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


@pytest.mark.parametrize("name", ["gqa_b64_ctx1k_fp8", "gqa_b1_ctx32k_fp8",
                                  "gqa_b1_ctx32k_mqa_fp8"])
def test_full_size_workload_sampled_rows(name):
    case = synth.workload(name)
    hq = case.num_q_heads
    bs = sorted({0, case.batch // 2, case.batch - 1})
    rows = [(b, h) for b in bs for h in range(hq)]
    _assert_close(case, DeviceCase(case), rows=rows)


@pytest.mark.parametrize("layout", ["v_below_k", "one_buffer", "same_buffer"])
def test_cache_placements(layout):
    # The fp8 path reads a page's K and V with one copy through a map spanning both caches
    # when it can: K below V, V below K (its tiles land in the other order), K and V as
    # halves of one [2, ...] buffer; with K and V the same buffer it uses separate maps.
    case = _case(synth.BF16, 128, 16, 2, [300, 17, 64], seed=12)
    if layout == "same_buffer":
        case.v_cache = case.k_cache.copy()
        case.v_scale = case.k_scale
    dc = DeviceCase(case)
    k = torch.from_numpy(case.k_cache).cuda()
    v = torch.from_numpy(case.v_cache).cuda()
    if layout == "v_below_k":
        both = torch.empty((2,) + k.shape, dtype=torch.uint8, device="cuda")
        both[0].copy_(v)
        both[1].copy_(k)
        dc.v, dc.k = both[0], both[1]
    elif layout == "one_buffer":
        both = torch.stack([k, v])
        dc.k, dc.v = both[0], both[1]
    else:
        dc.k = dc.v = k
    _assert_close(case, dc)
