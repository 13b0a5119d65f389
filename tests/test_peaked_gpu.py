"""Peaked scores on every decode kernel: one token carries 0.45-0.95 of each row's mass.

"From MHA to MLA", section 2: P is rounded to the value dtype before the PV product, so
with one dominant token the rounding of that weight reaches the output almost in full.
The cases (tests/peaked.py) plant a dominant token per segment behind decoys whose
scores sit a little lower, so kernels with a lazily raised running maximum weigh it by a
rounded non-power-of-two factor (relative error up to 2^-8 in bf16). Values are clipped
to |v| <= 2, so the output's own bf16 rounding is at most 2^-8 too. Dividing by the sum
of the unrounded weights would then leave up to w * 2^-8 * 2 ~ 7.4e-3 of error on top;
normalising by the sum of the rounded weights (the output a convex combination of value
rows) leaves at most w (1 - w) * 2^-8 * 4 ~ 3.9e-3, inside the 1e-2 tolerance.

Tolerances as everywhere: out max-abs <= 1e-2 (bf16) / 2e-3 (fp16), fp32 LSE within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import peaked
from gpu_util import TOL_LSE, TOL_OUT, DeviceCase, compare
from paged_kv_cache_61_gb300 import pda, synth

pytestmark = pytest.mark.gpu

WEIGHTS = [0.95, 0.8, 0.6]
CTX = [300, 2000, 5000]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pda.lib()


def _check(case, ref, forces):
    for force in forces:
        dc = DeviceCase(case, force_num_ctas=force)
        out, lse = dc.run()
        torch.cuda.synchronize()
        eo, el = compare(case, out, lse, *ref)
        assert eo <= TOL_OUT[case.dtype], f"force {force}: out max-abs error {eo}"
        assert el <= TOL_LSE, f"force {force}: lse max-abs error {el}"
        assert pda.read_device_error(dc.ws) == 0


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("dtype,hq,hkv", [(synth.FP16, 32, 8), (synth.BF16, 32, 8),
                                          (synth.BF16, 32, 1)])
def test_gqa_dominant_token(dtype, hq, hkv, seed):
    case = synth.make_gqa_case(batch=3, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                               dtype=dtype, context_lens=CTX, seed=30 + seed)
    placed = peaked.plant_gqa(case, WEIGHTS, seed=seed)
    w = peaked.dominant_weights_gqa(case, placed)
    assert 0.45 <= min(w.values()) and max(w.values()) <= 0.97
    ref = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, case.page_size, case.dtype)
    _check(case, ref, (0, 1, 5, 40))


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("hq,latent,dtype", [
    (16, 512, synth.BF16),     # 64-head kernel, one 16-head group
    (64, 512, synth.BF16),     # 64-head kernel
    (16, 512, synth.FP16),
    (128, 512, synth.BF16),    # two-CTA kernel (head groups of 128)
    (16, 256, synth.BF16),     # 64-head kernel, 320 record
    (128, 256, synth.BF16),    # heads-on-M kernel (320 record, head groups of 128)
])
def test_mla_dominant_token(hq, latent, dtype, seed):
    case = synth.make_mla_case(batch=3, num_q_heads=hq, dtype=dtype, context_lens=CTX,
                               latent_dim=latent, seed=30 + seed)
    placed = peaked.plant_mla(case, WEIGHTS, seed=seed)
    w = peaked.dominant_weights_mla(case, placed)
    assert 0.45 <= min(w.values()) and max(w.values()) <= 0.97
    ref = oracle.mla_decode(case.q, case.kv_cache, case.block_tables, case.context_lens,
                            case.scale, case.page_size, case.dtype, head_dim_v=case.head_dim_v)
    _check(case, ref, (0, 1, 5, 40))
