"""Helpers for GPU tests: move a synthetic case to the device and run it through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_61_gb300 import pda, synth

TOL_OUT = {synth.FP16: 2e-3, synth.BF16: 1e-2}   # max-abs error of out vs the float64 oracle
TOL_LSE = 1e-3                                   # max-abs error of the fp32 LSE


def torch_dtype(dtype: str):
    return torch.float16 if dtype == synth.FP16 else torch.bfloat16


def to_device_16(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch_dtype(dtype))


def device_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_plan(case: synth.DecodeCase, force_num_ctas: int = 0) -> pda.Plan:
    return pda.Plan(kind=pda.PDA_KIND_GQA if case.kind == "gqa" else pda.PDA_KIND_MLA,
                    dtype=pda.PDA_FP16 if case.dtype == synth.FP16 else pda.PDA_BF16,
                    batch=case.batch, num_q_heads=case.num_q_heads,
                    num_kv_heads=case.num_kv_heads, head_dim_qk=case.head_dim_qk,
                    head_dim_v=case.head_dim_v, page_size=case.page_size,
                    max_blocks_per_seq=case.max_blocks_per_seq, num_blocks=case.num_blocks,
                    context_lens=case.context_lens.tolist(), force_num_ctas=force_num_ctas,
                    kv_format=(pda.PDA_KV_FP8_E4M3 if case.kv_format == synth.FP8_E4M3
                               else pda.PDA_KV_SAME_AS_Q),
                    seq_len_q=case.seq_len_q)


def to_device_cache(case: synth.DecodeCase, arr: np.ndarray) -> torch.Tensor:
    """A cache array on the device: E4M3 codes as uint8, 16-bit patterns as fp16/bf16."""
    if case.kv_format == synth.FP8_E4M3:
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint8)).cuda()
    return to_device_16(arr, case.dtype)


class DeviceCase:
    """A case's inputs resident on the GPU plus output buffers and a zeroed workspace."""

    def __init__(self, case: synth.DecodeCase, force_num_ctas: int = 0):
        self.case = case
        self.q = to_device_16(case.q, case.dtype)
        if case.kind == "gqa":
            self.k = to_device_cache(case, case.k_cache)
            self.v = to_device_cache(case, case.v_cache)
        else:
            self.kv = to_device_cache(case, case.kv_cache)
        self.tables = torch.from_numpy(case.block_tables).cuda()
        self.ctx = torch.from_numpy(case.context_lens).cuda()
        S = case.seq_len_q
        out_shape = (case.batch, case.num_q_heads, case.head_dim_v) if S == 1 else \
            (case.batch, S, case.num_q_heads, case.head_dim_v)
        lse_shape = (case.batch, case.num_q_heads) if S == 1 else (case.batch, case.num_q_heads, S)
        self.out = torch.full(out_shape, float("nan"), dtype=torch_dtype(case.dtype), device="cuda")
        self.lse = torch.full(lse_shape, float("nan"), dtype=torch.float32, device="cuda")
        self.replan(force_num_ctas)

    def replan(self, force_num_ctas: int = 0):
        self.plan = make_plan(self.case, force_num_ctas)
        self.ws = torch.zeros(max(256, self.plan.workspace_bytes), dtype=torch.uint8, device="cuda")
        pda.workspace_init(self.plan, self.ws)

    def run(self, out=None, lse="default"):
        c = self.case
        out = self.out if out is None else out
        lse = self.lse if isinstance(lse, str) else lse
        if c.kind == "gqa" and c.kv_format == synth.FP8_E4M3:
            pda.paged_decode_attn_fp8(self.q, self.k, self.v, c.k_scale, c.v_scale, self.tables,
                                      self.ctx, c.scale, out, lse, self.plan, self.ws)
        elif c.kind == "gqa":
            pda.paged_decode_attn(self.q, self.k, self.v, self.tables, self.ctx, c.scale, out, lse,
                                  self.plan, self.ws)
        elif c.kv_format == synth.FP8_E4M3:
            pda.mla_decode_fp8(self.q, self.kv, c.k_scale, self.tables, self.ctx, c.scale, out,
                               lse, self.plan, self.ws)
        else:
            pda.mla_decode(self.q, self.kv, self.tables, self.ctx, c.scale, out, lse, self.plan,
                           self.ws)
        return out, lse


def compare(case, out_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref_out, ref_lse, rows=None):
    """Max-abs errors of (out, lse) over all rows or the listed (b, h) / (b, i, h) rows."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.cpu().numpy().astype(np.float64)
    if rows is None:
        return float(np.abs(o - ref_out).max()), float(np.abs(l - ref_lse).max())
    if len(rows[0]) == 3:                  # (b, i, h): out [B, S, Hq, Dv], lse [B, Hq, S]
        bs, is_, hs = ([r[k] for r in rows] for k in range(3))
        return (float(np.abs(o[bs, is_, hs] - ref_out[bs, is_, hs]).max()),
                float(np.abs(l[bs, hs, is_] - ref_lse[bs, hs, is_]).max()))
    bs = [r[0] for r in rows]
    hs = [r[1] for r in rows]
    return (float(np.abs(o[bs, hs] - ref_out[bs, hs]).max()),
            float(np.abs(l[bs, hs] - ref_lse[bs, hs]).max()))
