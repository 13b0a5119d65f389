#!/usr/bin/env python
"""Benchmark of paged decode attention on GB300 (one JSON line on stdout, rank 0).

Default workload: GQA paged decode, B=64, ctx=1024, Hq=32, Hkv=8, D=128, fp16,
PAGE=16, randomly permuted block tables (the workload the drill page measures
at 1520 GB/s on an RTX 5090). A step is one decode call: one pass of the whole
hot path (block-table walk, TMA page stream, scores, online softmax, PV, split
merge) over the batch. ``value`` is the achieved algorithmic HBM bandwidth:
the K+V bytes of the attended tokens divided by the device time of a step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Multi-GPU (torchrun, one rank per GPU): every rank decodes its own batch of the
same shape (weak scaling, no data-path collective); time = max over ranks.
``--impl reference`` times the float64 CPU oracle on the host cores instead
(rank 0 only), each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
if "reference" in sys.argv:
    # the reference arm reports one core: keep numpy's BLAS on one thread
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

from paged_kv_cache_61_gb300 import synth, traffic  # noqa: E402

DEFAULT_WORKLOAD = "gqa_b64_ctx1k"
L2_BYTES = 129 * 2 ** 20
KERNEL_SOURCES = {"gqa": ["gqa_decode.cu", "ptx.cuh", "tile_walk.cuh"],
                  "mla": ["mla_decode.cu", "ptx.cuh", "ptx_ext.cuh", "tile_walk.cuh"],
                  "mla_pair": ["mla_pair.cu", "ptx.cuh", "ptx_ext.cuh", "ptx_cluster.cuh",
                               "tile_walk.cuh"],
                  "mla_rows": ["mla_rows.cu", "ptx.cuh", "ptx_ext.cuh", "ptx_cluster.cuh",
                               "tile_walk.cuh"]}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- helpers
def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(kind: str) -> str:
    """Hash of a kernel's sources without comments and layout: recorded DRAM traffic stays
    valid across comment edits and goes stale on any change of code."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "paged_kv_cache_61_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def kernel_kind(case) -> str:
    """Which decode kernel a case runs on. MLA with head counts a multiple of 128: the
    two-CTA kernel for the 576-wide record (one query token), the heads-on-M kernel for the
    320-wide one; every other MLA shape the 64-head kernel."""
    if case.kind == "gqa":
        return "gqa"
    if case.num_q_heads % 128 == 0:
        if case.head_dim_qk == 576 and case.seq_len_q <= 1:
            return "mla_pair"
        if case.head_dim_qk == 320:
            return "mla_rows"
    return "mla"


def recorded_traffic(workload: str, kind: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("kernel_hash") != kernel_hash(kind):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in a background process."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((t, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t_start - 0.06 <= r[0] <= self.t_stop + 0.06]
        use = inside or sorted(rows, key=lambda r: abs(r[0] - self.t_stop))[:3]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------- workload accounting
def accounting(case):
    """Algorithmic bytes and FLOPs of one step (K+V of the attended tokens; 2 FLOP per MAC)."""
    ctx = case.context_lens.tolist()
    elem = 1 if case.kv_format == synth.FP8_E4M3 else 2     # bytes per cached value
    if case.kind == "gqa":
        kv = traffic.gqa_kv_bytes(ctx, case.num_kv_heads, case.head_dim_qk, elem)
    else:
        kv = traffic.mla_kv_bytes(ctx, case.head_dim_qk, elem)
    S = case.seq_len_q
    if S == 1:
        flops = traffic.decode_flops(ctx, case.num_q_heads, case.head_dim_qk, case.head_dim_v)
    else:   # query token i attends the first c - S + 1 + i tokens (causal, bottom-right)
        seen = [c - S + 1 + i for c in ctx for i in range(S)]
        flops = traffic.decode_flops(seen, case.num_q_heads, case.head_dim_qk, case.head_dim_v)
    return kv, flops


def workload_config(case, rotation_copies):
    cfg = {"workload": case.name, "kind": case.kind, "batch": case.batch,
           "num_q_heads": case.num_q_heads, "num_kv_heads": case.num_kv_heads,
           "head_dim_qk": case.head_dim_qk, "head_dim_v": case.head_dim_v,
           "page_size": case.page_size, "dtype": case.dtype,
           "kv_cache": ("fp8 e4m3, per-tensor scales" if case.kv_format == synth.FP8_E4M3
                        else case.dtype),
           "seq_len_q": case.seq_len_q,
           "context_lens": ("all " + str(int(case.context_lens[0]))
                            if (case.context_lens == case.context_lens[0]).all()
                            else f"varlen sum {int(case.context_lens.sum())}"),
           "seed": 0}
    if rotation_copies:
        cfg["l2"] = (f"inputs larger than L2: steps rotate over {rotation_copies} copies of the "
                     f"cache ({rotation_copies} x {accounting(case)[0] / 1e6:.0f} MB)")
    return cfg


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(case, budget_s: float):
    """Run the oracle on whole sequences until ~budget_s; return (kv_bytes_done, seconds)."""
    import oracle
    done_bytes, t0 = 0, time.perf_counter()
    b = 0
    while True:
        rows = [(b, h) for h in range(case.num_q_heads)]
        rows3 = [(b, i, h) for i in range(case.seq_len_q) for h in range(case.num_q_heads)]
        elem = 1 if case.kv_format == synth.FP8_E4M3 else 2
        if case.kind == "gqa" and case.seq_len_q > 1:
            oracle.paged_decode_mtp(case.q, case.k_cache, case.v_cache, case.block_tables,
                                    case.context_lens, case.scale, case.page_size, case.dtype,
                                    rows=rows3, kv_format=case.kv_format, k_scale=case.k_scale,
                                    v_scale=case.v_scale)
            done_bytes += traffic.gqa_kv_bytes([case.context_lens[b]], case.num_kv_heads,
                                               case.head_dim_qk, elem)
        elif case.kind == "gqa":
            oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                case.context_lens, case.scale, case.page_size, case.dtype,
                                rows=rows, kv_format=case.kv_format, k_scale=case.k_scale,
                                v_scale=case.v_scale)
            done_bytes += traffic.gqa_kv_bytes([case.context_lens[b]], case.num_kv_heads,
                                               case.head_dim_qk, elem)
        else:
            oracle.mla_decode(case.q, case.kv_cache, case.block_tables, case.context_lens,
                              case.scale, case.page_size, case.dtype,
                              head_dim_v=case.head_dim_v, rows=rows, kv_format=case.kv_format,
                              kv_scale=case.k_scale)
            done_bytes += traffic.mla_kv_bytes([case.context_lens[b]], case.head_dim_qk, elem)
        b = (b + 1) % case.batch
        if time.perf_counter() - t0 >= budget_s:
            return done_bytes, time.perf_counter() - t0, b


def cpu_baseline(workload: str, budget_s: float = 10.0):
    """Time the oracle single-threaded in a fresh process (BLAS pinned to one thread)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; from paged_kv_cache_61_gb300 "
            "import synth; c = synth.workload(%r); b, s, n = bench.oracle_sample(c, %r); "
            "print(json.dumps([b, s, n]))") % (ROOT, workload, budget_s)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    if r.returncode != 0:
        return {"value": None, "error": r.stderr.strip().splitlines()[-1:]}
    done, secs, nseq = json.loads(r.stdout.strip().splitlines()[-1])
    case = synth.workload(workload)
    gbs = done / secs / 1e9
    if case.kind == "gqa":
        value, unit = gbs, "GB/s"
    else:                                   # MLA lines are in TFLOP/s: same FLOPs per KV byte
        kv, flops = accounting(case)
        value, unit = gbs * (flops / kv) / 1e3, "TFLOP/s"
    return {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
            "sample": f"float64 numpy oracle, one thread, {max(nseq, 1)} whole sequences "
                      f"(all heads) of {workload} in {secs:.1f} s"}


def run_reference(args, workload):
    """The reference arm: the oracle, as it stands, on the host cores."""
    case = synth.workload(workload)
    kv, flops = accounting(case)
    per_step_budget = max(0.02, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(case, per_step_budget)
    total_bytes, total_s = 0, 0.0
    for _ in range(args.steps):
        b, s, _n = oracle_sample(case, per_step_budget)
        total_bytes += b
        total_s += s
    gbs = total_bytes / total_s / 1e9
    value = gbs if case.kind == "gqa" else gbs * (flops / kv) / 1e3
    unit = "GB/s" if case.kind == "gqa" else "TFLOP/s"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kv / (gbs * 1e9) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, seed 0)",
            "config": workload_config(case, 0),
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                             "sample": f"each step: whole sequences of {workload} for "
                                       f"~{per_step_budget:.2f} s, one thread"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# decode steps that append each sequence's new token first (see run_gpu)
STEP_WORKLOADS = ("gqa_b64_ctx1k_step", "gqa_b64_ctx1k_fp8_step", "mla_b16_ctx64k_h16_step")

METRIC = "paged decode attn achieved HBM GB/s (% of GB300 peak), μs/step; MLA TFLOPS"


# ---------------------------------------------------------------- GPU arm
def reduce_step_time(ms_per_step: float, dist, device) -> float:
    """Max over ranks of the time per step (weak scaling: the slowest rank sets it)."""
    if dist is None:
        return ms_per_step
    import torch
    t = torch.tensor([ms_per_step], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Units (bytes or FLOPs) all ranks process per second, every rank doing one step."""
    return units_per_rank_step * world / (ms_per_step * 1e-3)


def _has_merge(plan, case):
    """Whether a decode call on this plan also launches the split-merge kernel."""
    return plan.num_ctas > 0 and max(plan.num_splits(b) for b in range(case.batch)) > max(
        4, -(-plan.num_ctas // 64))


def run_gpu(args, workload, rank, world, local_rank):
    import numpy as np
    import torch

    from paged_kv_cache_61_gb300 import pda

    torch.cuda.set_device(local_rank)
    # everything on one non-default stream (CUDA graphs cannot capture the legacy stream)
    torch.cuda.set_stream(torch.cuda.Stream())
    dist = None
    if world > 1:
        import torch.distributed as dist
    # "<workload>_step": each step first appends one new token per sequence (the last of
    # its context) through the append call, then decodes: a serving step's cache work
    with_append = workload.endswith("_step")
    case = synth.workload(workload[: -len("_step")] if with_append else workload, seed=rank)
    case.name = workload
    kv_bytes, flops = accounting(case)
    tdt = torch.float16 if case.dtype == synth.FP16 else torch.bfloat16

    def dev16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(tdt)

    fp8 = case.kv_format == synth.FP8_E4M3

    def dev_cache(arr):
        return torch.from_numpy(np.ascontiguousarray(arr)).cuda() if fp8 else dev16(arr)

    copies = max(1, min(64, math.ceil(4 * L2_BYTES / kv_bytes)))
    q = dev16(case.q)
    if case.kind == "gqa":
        k0, v0 = dev_cache(case.k_cache), dev_cache(case.v_cache)
        caches = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(copies - 1)]
    else:
        kv0 = dev_cache(case.kv_cache)
        caches = [(kv0, None)] + [(kv0.clone(), None) for _ in range(copies - 1)]
    tables = torch.from_numpy(case.block_tables).cuda()
    ctx = torch.from_numpy(case.context_lens).cuda()
    S = case.seq_len_q
    out_shape = (case.batch, case.num_q_heads, case.head_dim_v) if S == 1 else \
        (case.batch, S, case.num_q_heads, case.head_dim_v)
    lse_shape = (case.batch, case.num_q_heads) if S == 1 else (case.batch, case.num_q_heads, S)
    out = torch.empty(out_shape, dtype=tdt, device="cuda")
    lse = torch.empty(lse_shape, dtype=torch.float32, device="cuda")
    plan = pda.Plan(kind=pda.PDA_KIND_GQA if case.kind == "gqa" else pda.PDA_KIND_MLA,
                    dtype=pda.PDA_FP16 if case.dtype == synth.FP16 else pda.PDA_BF16,
                    batch=case.batch, num_q_heads=case.num_q_heads,
                    num_kv_heads=case.num_kv_heads, head_dim_qk=case.head_dim_qk,
                    head_dim_v=case.head_dim_v, page_size=case.page_size,
                    max_blocks_per_seq=case.max_blocks_per_seq, num_blocks=case.num_blocks,
                    context_lens=case.context_lens.tolist(),
                    kv_format=pda.PDA_KV_FP8_E4M3 if fp8 else pda.PDA_KV_SAME_AS_Q,
                    seq_len_q=S)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    pda.workspace_init(plan, ws, stream)

    new_shape = ((case.batch, S, case.num_kv_heads, case.head_dim_qk) if case.kind == "gqa"
                 else (case.batch, S, case.head_dim_qk))
    gen = torch.Generator(device="cuda").manual_seed(rank)
    k_new = torch.randn(new_shape, generator=gen, device="cuda").to(tdt)
    v_new = torch.randn(new_shape, generator=gen, device="cuda").to(tdt)

    def append(i, tables_, ctx_, kn=k_new, vn=v_new):
        kc, vc = caches[i % copies]
        if case.kind == "gqa" and fp8:
            pda.kv_append_fp8(kn, vn, kc, vc, case.k_scale, case.v_scale, tables_, ctx_, plan,
                              ws, stream)
        elif case.kind == "gqa":
            pda.kv_append(kn, vn, kc, vc, tables_, ctx_, plan, ws, stream)
        else:
            pda.mla_append(kn, kc, tables_, ctx_, plan, ws, stream)

    def step(i, q_=q, out_=out, lse_=lse, tables_=tables, ctx_=ctx, kn_=k_new, vn_=v_new):
        kc, vc = caches[i % copies]
        if with_append:
            append(i, tables_, ctx_, kn=kn_, vn=vn_)
        if case.kind == "gqa" and fp8:
            pda.paged_decode_attn_fp8(q_, kc, vc, case.k_scale, case.v_scale, tables_, ctx_,
                                      case.scale, out_, lse_, plan, ws, stream)
        elif case.kind == "gqa":
            pda.paged_decode_attn(q_, kc, vc, tables_, ctx_, case.scale, out_, lse_, plan, ws,
                                  stream)
        else:
            pda.mla_decode(q_, kc, tables_, ctx_, case.scale, out_, lse_, plan, ws, stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # Per-call device time of each decode call (events around every call), used for
    # the roofline of the decode kernels.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # The timed region: the K steps captured once in a CUDA graph and replayed
    # back to back (launch gaps of the host loop removed; every step still runs).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(args.steps):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    t_all0.record(stream)
    graph.replay()
    t_all1.record(stream)
    torch.cuda.synchronize()
    barrier()
    if sampler:
        sampler.mark_stop()
    total_ms = t_all0.elapsed_time(t_all1)
    ms_per_step = total_ms / args.steps
    ms_per_step = reduce_step_time(ms_per_step, dist, "cuda")
    clocks = sampler.stop() if sampler else None
    if rank != 0:
        return

    # ---- end to end through the C ABI: pinned host inputs in, outputs back, every step.
    # A step's inputs (q, block tables, context lengths, and the new tokens' K/V of the
    # _step workloads) travel as one pinned host buffer, one copy in; its outputs (out,
    # lse) are views of one device buffer, one copy out. The decode call reads and writes
    # those views, as a caller batching its transfers would.
    e2e_steps = min(args.steps, 500)
    ins = [q, tables, ctx] + ([k_new, v_new] if with_append else [])
    outs = [out, lse]

    def packed(tensors):
        offs, n = [], 0
        for t in tensors:                    # 16-byte aligned, end to end
            offs.append(n)
            n += -(-t.numel() * t.element_size() // 16) * 16
        return offs, n

    def view(buf, off, like):
        nbytes = like.numel() * like.element_size()
        return buf[off:off + nbytes].view(like.dtype).view(like.shape)

    in_offs, h2d = packed(ins)
    out_offs, d2h = packed(outs)
    in_h = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    in_d = torch.empty(h2d, dtype=torch.uint8, device="cuda")
    res_h = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    res_d = torch.empty(d2h, dtype=torch.uint8, device="cuda")
    for t, off in zip(ins, in_offs):
        view(in_h, off, t).copy_(t.cpu())
    d_in = [view(in_d, off, t) for t, off in zip(ins, in_offs)]
    out_v, lse_v = (view(res_d, off, t) for t, off in zip(outs, out_offs))
    kn_v, vn_v = (d_in[3], d_in[4]) if with_append else (k_new, v_new)

    def e2e_step(i):
        in_d.copy_(in_h, non_blocking=True)
        step(i, q_=d_in[0], out_=out_v, lse_=lse_v, tables_=d_in[1], ctx_=d_in[2], kn_=kn_v,
             vn_=vn_v)
        res_h.copy_(res_d, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    launches_per_step = 1 + (1 if _has_merge(plan, case) else 0) + (1 if with_append else 0)
    pk, pk_src = peaks()
    # The kernel time the roofline divides by: the timed region's time per step. A step
    # is one decode launch, plus one split-merge launch when the plan has heavily split
    # segments (then the figure covers both, which understates the decode kernel alone).
    mean_launch_ms = ms_per_step
    if case.kind == "gqa":
        value = whole_job_rate(kv_bytes, world, ms_per_step) / 1e9
        unit = "GB/s"
        achieved = kv_bytes / (mean_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": f"hbm_gbs of {pk_src}",
                "frac_of_8TBs_spec": achieved / 8000.0}
        e2e_value = kv_bytes / (e2e_ms * 1e-3) / 1e9
    else:
        value = whole_job_rate(flops, world, ms_per_step) / 1e12
        unit = "TFLOP/s"
        t_bytes = kv_bytes / (pk["hbm_gbs"] * 1e9)
        t_flops = flops / (pk["bf16_tflops"] * 1e12)
        achieved_gbs = kv_bytes / (mean_launch_ms * 1e-3) / 1e9
        achieved_tf = flops / (mean_launch_ms * 1e-3) / 1e12
        if t_bytes >= t_flops:
            roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved_gbs / pk["hbm_gbs"], "peak_source": f"hbm_gbs of {pk_src}"}
        else:
            roof = {"bound": "tensor", "achieved": achieved_tf, "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": achieved_tf / pk["bf16_tflops"],
                    "peak_source": f"bf16_tflops of {pk_src}"}
        roof["tflops"] = achieved_tf
        roof["frac_of_slower_roof"] = max(t_bytes, t_flops) / (mean_launch_ms * 1e-3)
        e2e_value = flops / (e2e_ms * 1e-3) / 1e12
    roof["traffic"] = recorded_traffic(workload, kernel_kind(case))
    roof["algorithmic_bytes_per_launch"] = kv_bytes
    roof["mean_launch_us"] = mean_launch_ms * 1e3
    roof["scope"] = (("append kernel + " if with_append else "") + "decode kernel" +
                     (" + split-merge kernel" if _has_merge(plan, case) else "") + " per step")
    roof["event_us_per_call"] = statistics.median(per_launch_ms) * 1e3
    roof["event_us_per_call_min"] = min(per_launch_ms) * 1e3

    cpu = None if args.no_cpu_baseline else cpu_baseline(workload)
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if case.dtype == synth.FP16 else "bf16",
            "data": "synthetic (seeded N(0,1) values, random block tables, seed = rank)",
            "config": workload_config(case, copies), "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "path": "one pinned host buffer (q, block_tables, context_lens"
                            + (", new K/V" if with_append else "") + ") -> device, C-ABI "
                            "decode into one device buffer (out, lse) -> pinned host, every "
                            "step, eager launches; caches resident in HBM"},
            "gpu_launches": args.steps * launches_per_step, "clocks": clocks,
            "timing": "value: K steps captured in one CUDA graph and replayed (device events); "
                      "roofline: device events around each call",
            "plan": {"num_ctas": plan.num_ctas, "max_splits": max(plan.num_splits(b)
                                                                  for b in range(case.batch))}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=synth.WORKLOADS + STEP_WORKLOADS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = env_int("RANK", 0)
    world = env_int("WORLD_SIZE", 1)
    local_rank = env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, args.workload)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gpu(args, args.workload, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
