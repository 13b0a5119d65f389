"""Absorbed-MLA decode over an E4M3 record cache, on the GPU through the C ABI.

"Attention Kernel Variants: MQA, GQA, and MLA", KV-cache arithmetic table: DeepSeek-V3's
MLA cache with an fp8 latent holds 34.3 KiB per token, half of bf16. Each cached byte is an
E4M3 code and record = e4m3(code) * kv_scale (one scale per tensor), for the scores (all
Dqk values) and the values (the first Dv). The kernel converts each page's codes to the
16-bit record in shared memory before the tensor-core MMAs; the oracle decodes the same
codes in float64.

Tolerances as for 16-bit caches: out max-abs <= 1e-2 (bf16) / 2e-3 (fp16), LSE 1e-3.
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


def _case(hq, ctx, dtype=synth.BF16, seed=5, latent=512, s=1):
    return synth.make_mla_case(batch=len(ctx), num_q_heads=hq, dtype=dtype, context_lens=ctx,
                               latent_dim=latent, seed=seed, kv_format=synth.FP8_E4M3,
                               seq_len_q=s)


def _oracle(case, rows=None):
    fn = oracle.mla_decode_mtp if case.seq_len_q > 1 else oracle.mla_decode
    return fn(case.q, case.kv_cache, case.block_tables, case.context_lens, case.scale,
              case.page_size, case.dtype, head_dim_v=case.head_dim_v, rows=rows,
              kv_format=case.kv_format, kv_scale=case.k_scale)


def _assert_close(case, dc, rows=None):
    out, lse = dc.run()
    torch.cuda.synchronize()
    eo, el = compare(case, out, lse, *_oracle(case, rows), rows)
    assert eo <= TOL_OUT[case.dtype], f"out max-abs error {eo}"
    assert el <= TOL_LSE, f"lse max-abs error {el}"
    assert pda.read_device_error(dc.ws) == 0
    return out, lse


@pytest.mark.parametrize("latent", [512, 256])
@pytest.mark.parametrize("hq", [16, 32])
@pytest.mark.parametrize("force", [0, 1, 3, 17])
def test_small_cases(hq, force, latent):
    case = _case(hq, [1, 63, 64, 65, 130, 700], latent=latent)
    _assert_close(case, DeviceCase(case, force_num_ctas=force))


@pytest.mark.parametrize("latent", [512, 256])
def test_fp16_and_negative_scale(latent):
    case = _case(16, [200, 64, 1], dtype=synth.FP16, latent=latent)
    _assert_close(case, DeviceCase(case))
    case.scale = -0.05
    _assert_close(case, DeviceCase(case, force_num_ctas=3))


@pytest.mark.parametrize("force", [0, 1, 5])
def test_two_query_tokens(force):
    # S = 2 with 16 heads: one group of 32 rows per sequence, causal bottom-right
    case = _case(16, [65, 130, 700, 2], s=2)
    out, lse = DeviceCase(case, force_num_ctas=force).run()
    torch.cuda.synchronize()
    ro, rl = _oracle(case)
    assert np.abs(out.float().cpu().numpy() - ro).max() <= TOL_OUT[case.dtype]
    assert np.abs(lse.cpu().numpy() - rl).max() <= TOL_LSE


@pytest.mark.parametrize("latent", [512, 256])
def test_rope_needle_is_bit_exact(latent):
    # q: content 0, rope 1; records: rope codes 0 except the target's (16.0), kv_scale 1:
    # every other weight underflows against the needle, so out is the target's latent,
    # decoded exactly, bit for bit
    ctx = 300
    case = _case(16, [ctx] * 6, seed=9, latent=latent)
    case.k_scale = case.v_scale = 1.0
    one = synth.float32_to_bits(np.float32(1.0), case.dtype)
    case.q[..., :latent] = 0
    case.q[..., latent:] = one
    case.kv_cache[..., latent:] = 0
    sixteen = synth.float32_to_e4m3(np.array([16.0], np.float32))[0]
    targets = [0, 63, 64, 150, 255, 299]
    for b, t in enumerate(targets):
        case.kv_cache[int(case.block_tables[b, t // 64]), t % 64, latent:] = sixteen
    for force in (0, 1, 5):
        out, _ = DeviceCase(case, force_num_ctas=force).run()
        torch.cuda.synchronize()
        got = device_bits(out)
        for b, t in enumerate(targets):
            codes = case.kv_cache[int(case.block_tables[b, t // 64]), t % 64, :latent]
            want = synth.float32_to_bits(oracle.decode_e4m3(codes).astype(np.float32), case.dtype)
            for h in range(16):
                assert np.array_equal(got[b, h], want), (force, b, h)


def test_nan_codes_in_stale_slots_and_unused_entries():
    case = _case(32, [70, 129, 5])
    out0, lse0 = DeviceCase(case).run()
    torch.cuda.synchronize()
    kv, tab = case.kv_cache.copy(), case.block_tables.copy()
    for b, c in enumerate(case.context_lens):
        npg = (int(c) + 63) // 64
        last, fill = int(tab[b, npg - 1]), int(c) - (npg - 1) * 64
        kv[last, fill:] = 0x7F                     # E4M3 NaN
        tab[b, npg:] = -99
    bad = synth.DecodeCase(**{**case.__dict__})
    bad.kv_cache, bad.block_tables = kv, tab
    dc = DeviceCase(bad)
    out1, lse1 = dc.run()
    torch.cuda.synchronize()
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(lse0, lse1)
    assert pda.read_device_error(dc.ws) == 0


@pytest.mark.parametrize("name", ["mla_b16_ctx64k_h16_fp8", "mla_r256_b16_ctx64k_h16_fp8"])
def test_full_size_workload_sampled_rows(name):
    case = synth.workload(name)
    rows = [(b, h) for b in (0, 3, 7, 8, 12, 15) for h in range(case.num_q_heads)]
    _assert_close(case, DeviceCase(case), rows=rows)
