"""Appending new tokens to the paged caches on the GPU, and a serving loop built on it.

Append is byte work: the caches after the call must equal the oracle's append bit for bit
(for fp8 caches, the E4M3 codes of value / scale computed in float32). The serving loop
grows tables with the block pool, appends each step's token(s) and decodes, checking
every step against the oracle on a host mirror of the cache.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE, TOL_OUT, DeviceCase, to_device_16
from paged_kv_cache_61_gb300 import pda, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pda.lib()


def _bits(t):
    return t.contiguous().cpu().numpy().view(np.uint8 if t.dtype == torch.uint8 else np.uint16)


def _new_values(rng, shape, dtype, spread=1.0):
    return synth.float32_to_bits((rng.standard_normal(shape) * spread).astype(np.float32), dtype)


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
@pytest.mark.parametrize("s", [1, 2])
def test_gqa_append_is_bit_exact(dtype, s):
    case = synth.make_gqa_case(batch=5, num_q_heads=8, num_kv_heads=2, head_dim=128,
                               dtype=dtype, context_lens=[1 + s, 16, 17, 300, 33], seed=4,
                               seq_len_q=s)
    dc = DeviceCase(case)
    rng = np.random.default_rng(1)
    kn = _new_values(rng, (5, s, 2, 128), dtype)
    vn = _new_values(rng, (5, s, 2, 128), dtype)
    pda.kv_append(to_device_16(kn, dtype), to_device_16(vn, dtype), dc.k, dc.v, dc.tables,
                  dc.ctx, dc.plan, dc.ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(dc.k.view(torch.int16)), oracle.append_tokens(
        case.k_cache, kn, case.block_tables, case.context_lens, 16, s))
    np.testing.assert_array_equal(_bits(dc.v.view(torch.int16)), oracle.append_tokens(
        case.v_cache, vn, case.block_tables, case.context_lens, 16, s))
    assert pda.read_device_error(dc.ws) == 0


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
def test_fp8_append_quantizes_like_the_oracle(dtype):
    case = synth.make_gqa_case(batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype=dtype,
                               context_lens=[2, 17, 64, 129], seed=6, seq_len_q=2,
                               kv_format=synth.FP8_E4M3)
    dc = DeviceCase(case)
    rng = np.random.default_rng(2)
    # K: some values exceed 448 * scale (they saturate); V: many land on E4M3 subnormals
    kn = _new_values(rng, (4, 2, 2, 64), dtype, spread=3.0)
    vn = _new_values(rng, (4, 2, 2, 64), dtype, spread=0.00005)
    ks, vs = 0.0107, 0.00093
    pda.kv_append_fp8(to_device_16(kn, dtype), to_device_16(vn, dtype), dc.k, dc.v, ks, vs,
                      dc.tables, dc.ctx, dc.plan, dc.ws)
    torch.cuda.synchronize()
    kq = oracle.quantize_e4m3(kn, dtype, ks)
    vq = oracle.quantize_e4m3(vn, dtype, vs)
    assert (kq & 0x7F == 0x7E).any()                    # saturated codes occur
    assert ((vq & 0x78) == 0).sum() > 16                # subnormal codes occur
    np.testing.assert_array_equal(_bits(dc.k), oracle.append_tokens(
        case.k_cache, kq, case.block_tables, case.context_lens, 16, 2))
    np.testing.assert_array_equal(_bits(dc.v), oracle.append_tokens(
        case.v_cache, vq, case.block_tables, case.context_lens, 16, 2))


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("s", [1, 2])
def test_mla_append_is_bit_exact(latent, s):
    case = synth.make_mla_case(batch=3, num_q_heads=16, dtype=synth.BF16,
                               context_lens=[64 + s, 65, 700], latent_dim=latent, seed=3,
                               seq_len_q=s)
    dc = DeviceCase(case)
    new = _new_values(np.random.default_rng(5), (3, s, latent + 64), synth.BF16)
    pda.mla_append(to_device_16(new, synth.BF16), dc.kv, dc.tables, dc.ctx, dc.plan, dc.ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(dc.kv.view(torch.int16)), oracle.append_tokens(
        case.kv_cache, new, case.block_tables, case.context_lens, 64, s))


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("s", [1, 2])
def test_mla_fp8_append_quantizes_like_the_oracle_and_decodes(latent, s):
    # E4M3 record cache (the variants page's fp8 latent): the appended records are the
    # oracle's codes of value / kv_scale, bit for bit, and the decode that follows reads them
    case = synth.make_mla_case(batch=3, num_q_heads=16, dtype=synth.BF16,
                               context_lens=[64 + s, 65, 700], latent_dim=latent, seed=3,
                               seq_len_q=s, kv_format=synth.FP8_E4M3)
    dc = DeviceCase(case)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, s, latent + 64)).astype(np.float32)
    # rope dims far above 448 * kv_scale (saturated codes) on a record whose latent is
    # clipped to |x| <= 2: its score may dominate, and an output near 4 would round in bf16
    # by more than the 1e-2 tolerance
    x[0, 0, :latent] = np.clip(x[0, 0, :latent], -2.0, 2.0)
    x[0, 0, latent:] *= 1000.0
    x[1, -1, :128] *= 1e-4                      # E4M3 subnormals and zeros
    new = synth.float32_to_bits(x, synth.BF16)
    pda.mla_append_fp8(to_device_16(new, synth.BF16), dc.kv, case.k_scale, dc.tables, dc.ctx,
                       dc.plan, dc.ws)
    torch.cuda.synchronize()
    codes = oracle.quantize_e4m3(new, synth.BF16, case.k_scale)
    assert (codes & 0x7F == 0x7E).any() and ((codes & 0x78) == 0).sum() > 16
    want = oracle.append_tokens(case.kv_cache, codes, case.block_tables, case.context_lens,
                                64, s)
    np.testing.assert_array_equal(_bits(dc.kv), want)
    assert pda.read_device_error(dc.ws) == 0
    out, lse = dc.run()
    torch.cuda.synchronize()
    fn = oracle.mla_decode_mtp if s > 1 else oracle.mla_decode
    ref_out, ref_lse = fn(case.q, want, case.block_tables, case.context_lens, case.scale, 64,
                          case.dtype, head_dim_v=latent, kv_format=synth.FP8_E4M3,
                          kv_scale=case.k_scale)
    assert np.abs(out.float().cpu().numpy() - ref_out).max() <= TOL_OUT[case.dtype]
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= TOL_LSE


def test_bad_table_entry_is_flagged_and_skipped():
    case = synth.make_gqa_case(batch=3, num_q_heads=4, num_kv_heads=1, head_dim=64,
                               dtype=synth.FP16, context_lens=[20, 33, 5], seed=7)
    bad = synth.DecodeCase(**{**case.__dict__})
    bad.block_tables = case.block_tables.copy()
    bad.block_tables[1, 2] = 10 ** 6                    # the page of sequence 1's new token
    dc = DeviceCase(bad)
    rng = np.random.default_rng(9)
    kn = _new_values(rng, (3, 1, 1, 64), synth.FP16)
    vn = _new_values(rng, (3, 1, 1, 64), synth.FP16)
    pda.kv_append(to_device_16(kn, synth.FP16), to_device_16(vn, synth.FP16), dc.k, dc.v,
                  dc.tables, dc.ctx, dc.plan, dc.ws)
    torch.cuda.synchronize()
    assert pda.read_device_error(dc.ws) & 1
    keep = [0, 2]                                       # the other sequences are written
    want = oracle.append_tokens(case.k_cache, kn[keep], case.block_tables[keep],
                                case.context_lens[keep], 16, 1)
    np.testing.assert_array_equal(_bits(dc.k.view(torch.int16)), want)


@pytest.mark.parametrize("s", [1, 2])
def test_serving_loop_pool_append_decode(s):
    """Sequences grow step by step through the block pool; each step appends the new
    token(s) and decodes, and one sequence finishes and is replaced (its blocks reused)."""
    rng = np.random.default_rng(11)
    dtype, P, hq, hkv, d, nb, mb = synth.FP16, 16, 8, 2, 64, 24, 8
    pool = pda.BlockPool(nb)
    k_host = _new_values(rng, (nb, P, hkv, d), dtype)        # stale contents everywhere
    v_host = _new_values(rng, (nb, P, hkv, d), dtype)
    k_dev, v_dev = to_device_16(k_host, dtype), to_device_16(v_host, dtype)
    lens = [0, 0, 0]
    tables = np.full((3, mb), -1, dtype=np.int32)
    start = [5, 16, 30]
    # prefill: the first tokens of each sequence go in through the append path too
    for b in range(3):
        pool.grow(tables[b], P, 0, start[b])
    for b in range(3):
        for n in range(start[b]):
            lens[b] = n + 1
            new_k = _new_values(rng, (1, 1, hkv, d), dtype)
            new_v = _new_values(rng, (1, 1, hkv, d), dtype)
            row = tables[b:b + 1]
            k_host = oracle.append_tokens(k_host, new_k, row, [lens[b]], P, 1)
            v_host = oracle.append_tokens(v_host, new_v, row, [lens[b]], P, 1)
    k_dev, v_dev = to_device_16(k_host, dtype), to_device_16(v_host, dtype)
    for step in range(24):
        if step == 12:                                        # sequence 1 finishes
            pool.release(tables[1], P, lens[1])
            lens[1] = 0
            pool.grow(tables[1], P, 0, s)                     # a new one starts
            lens[1] = s
        else:
            for b in range(3):
                pool.grow(tables[b], P, lens[b], lens[b] + s)
                lens[b] += s
        ctx = np.array(lens, dtype=np.int32)
        plan = pda.Plan(kind=pda.PDA_KIND_GQA, dtype=pda.PDA_FP16, batch=3, num_q_heads=hq,
                        num_kv_heads=hkv, head_dim_qk=d, head_dim_v=d, page_size=P,
                        max_blocks_per_seq=mb, num_blocks=nb, context_lens=ctx.tolist(),
                        seq_len_q=s)
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        pda.workspace_init(plan, ws)
        tab_d = torch.from_numpy(tables.copy()).cuda()
        ctx_d = torch.from_numpy(ctx).cuda()
        new_k = _new_values(rng, (3, s, hkv, d), dtype)
        new_v = _new_values(rng, (3, s, hkv, d), dtype)
        pda.kv_append(to_device_16(new_k, dtype), to_device_16(new_v, dtype), k_dev, v_dev,
                      tab_d, ctx_d, plan, ws)
        k_host = oracle.append_tokens(k_host, new_k, tables, ctx, P, s)
        v_host = oracle.append_tokens(v_host, new_v, tables, ctx, P, s)
        q = _new_values(rng, (3, hq, d) if s == 1 else (3, s, hq, d), dtype)
        out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
        lse = torch.empty((3, hq) if s == 1 else (3, hq, s), dtype=torch.float32, device="cuda")
        pda.paged_decode_attn(to_device_16(q, dtype), k_dev, v_dev, tab_d, ctx_d, 0.125, out,
                              lse, plan, ws)
        torch.cuda.synchronize()
        assert pda.read_device_error(ws) == 0
        if s == 1:
            ref_o, ref_l = oracle.paged_decode(q, k_host, v_host, tables, ctx, 0.125, P, dtype)
        else:
            ref_o, ref_l = oracle.paged_decode_mtp(q, k_host, v_host, tables, ctx, 0.125, P,
                                                   dtype)
        eo = float(np.abs(out.float().cpu().numpy() - ref_o).max())
        el = float(np.abs(lse.cpu().numpy() - ref_l).max())
        assert eo <= TOL_OUT[dtype] and el <= TOL_LSE, (step, eo, el)
    # the device cache equals the host mirror byte for byte
    np.testing.assert_array_equal(_bits(k_dev.view(torch.int16)), k_host)
    np.testing.assert_array_equal(_bits(v_dev.view(torch.int16)), v_host)
