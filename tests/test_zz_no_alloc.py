"""paged_decode_attn_no_alloc gives the results of paged_decode_attn without a workspace.

Some callers cannot allocate device memory at the moment they decode: code that runs
inside another framework's memory pool, a plug-in that is handed only its input and
output buffers, or a serving host that forbids cudaMalloc after start-up. For them the
library keeps its scratch space (split pieces, merge counters, error word) in one
device array of its own. These tests call that entry point through the C ABI, twice
in a row, and compare it bit for bit with the workspace-taking entry point: both run
the same kernels on the same plan, and every merge adds its pieces in a fixed order.

This file is named to be collected last, so a run that stops at the first failure
has already run every other test.
"""
import pytest
import torch

from gpu_util import DeviceCase
from paged_kv_cache_61_gb300 import pda, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pda.lib()
    pda.no_alloc_read_device_error()      # start from a clear error word


def _no_alloc_call(dc, stream=None):
    c = dc.case
    out = torch.full_like(dc.out, float("nan"))
    lse = torch.full_like(dc.lse, float("nan"))
    pda.paged_decode_attn_no_alloc(dc.q, dc.k, dc.v, dc.tables, dc.ctx, c.scale, out, lse,
                                   dc.plan, stream)
    return out, lse


def _case(name):
    if name == "split_heavy":
        # one long and two short sequences: pieces merged in-kernel and by the merge kernel
        return synth.make_gqa_case(batch=3, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                   dtype=synth.BF16, context_lens=[4000, 70, 1500], seed=21)
    if name == "mqa":
        return synth.make_gqa_case(batch=1, num_q_heads=32, num_kv_heads=1, head_dim=128,
                                   dtype=synth.BF16, context_lens=[9000], seed=22)
    return synth.workload("gqa_tiny")


@pytest.mark.parametrize("case_name", ["split_heavy", "tiny_workload", "mqa"])
def test_no_alloc_matches_workspace_entry_point_twice(case_name):
    dc = DeviceCase(_case(case_name))
    ref_out, ref_lse = dc.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    assert dc.plan.workspace_bytes <= 16 << 20
    for _ in range(2):
        out, lse = _no_alloc_call(dc)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)
    assert pda.no_alloc_read_device_error() == 0


def test_no_alloc_on_a_side_stream():
    dc = DeviceCase(_case("split_heavy"))
    ref_out, ref_lse = dc.run()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        outs = [_no_alloc_call(dc, side) for _ in range(2)]
    side.synchronize()
    for out, lse in outs:
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)
    assert pda.no_alloc_read_device_error(side) == 0


def test_no_alloc_reports_a_block_id_outside_the_pool():
    case = synth.make_gqa_case(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=64,
                               dtype=synth.FP16, context_lens=[40, 20], seed=7)
    bad = synth.DecodeCase(**{**case.__dict__})
    bad.block_tables = case.block_tables.copy()
    bad.block_tables[0, 1] = case.num_blocks + 5      # inside num_pages: a caller error
    dc = DeviceCase(bad)
    _no_alloc_call(dc)
    torch.cuda.synchronize()
    assert pda.no_alloc_read_device_error() & 1
    assert pda.no_alloc_read_device_error() == 0      # reading clears it
    _no_alloc_call(DeviceCase(case))                  # a good call leaves it clear
    assert pda.no_alloc_read_device_error() == 0


def test_no_alloc_rejects_a_plan_larger_than_its_array():
    # MQA over 2048 CTAs needs 2048 x 2 x 32 x 128 fp32 pieces (64 MiB) of workspace
    case = synth.make_gqa_case(batch=1, num_q_heads=32, num_kv_heads=1, head_dim=128,
                               dtype=synth.BF16, context_lens=[32768], seed=23)
    dc = DeviceCase(case, force_num_ctas=2048)
    assert dc.plan.workspace_bytes > 16 << 20
    with pytest.raises(pda.PdaError) as e:
        _no_alloc_call(dc)
    assert e.value.status == pda.PDA_ERR_WORKSPACE
