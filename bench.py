#!/usr/bin/env python
"""Benchmark of paged decode attention on GB300 (one JSON line on stdout, rank 0).

Headline workload: GQA paged decode, B=64, ctx=1024, Hq=32, Hkv=8, D=128, fp16,
PAGE=16, randomly permuted block tables (the workload the drill page measures
at 1520 GB/s on an RTX 5090). A step is one decode call: one pass of the whole
hot path (block-table walk, TMA page stream, scores, online softmax, PV, split
merge) over the batch. ``value`` is the achieved algorithmic HBM bandwidth:
the K+V bytes of the attended tokens divided by the device time of a step.

The default run (one GPU) also measures the other decode workloads the library is
held to and reports each under ``per_config``: the tiny parity workload, B=1 at
ctx 32K (Hkv=8 and Hkv=1), the varlen batch of 128 and absorbed MLA at B=16, ctx
64K with 16 and 128 heads; each with its time per step, bandwidth, TFLOP/s, its
roofline fraction and the float64 oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Multi-GPU (torchrun, one rank per GPU): every rank decodes its own batch of the
same shape (weak scaling, no data-path collective); time = max over ranks.
``--impl reference`` times the float64 CPU oracle on the host cores instead
(rank 0 only), each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# The oracle runs one BLAS thread per process; the all-cores figures use one process
# per core. Set before numpy is imported.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

from paged_kv_cache_61_gb300 import synth, traffic  # noqa: E402

DEFAULT_WORKLOAD = "gqa_b64_ctx1k"
# the other decode workloads of the default run, with their role
PER_CONFIG = ("gqa_tiny", "gqa_b1_ctx32k", "gqa_b1_ctx32k_mqa", "gqa_varlen_b128",
              "mla_b16_ctx64k_h16", "mla_b16_ctx64k_h128", "gqa_b64_ctx1k_fp8",
              "mla_b16_ctx64k_h16_fp8")
L2_BYTES = 129 * 2 ** 20
KERNEL_SOURCES = {"gqa": ["gqa_decode.cu", "ptx.cuh", "tile_walk.cuh"],
                  "mla": ["mla_decode.cu", "ptx.cuh", "ptx_ext.cuh", "tile_walk.cuh"],
                  "mla_pair": ["mla_pair.cu", "ptx.cuh", "ptx_ext.cuh", "ptx_cluster.cuh",
                               "tile_walk.cuh"],
                  "mla_rows": ["mla_rows.cu", "ptx.cuh", "ptx_ext.cuh", "ptx_cluster.cuh",
                               "tile_walk.cuh"]}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "paged decode attn achieved HBM GB/s (% of GB300 peak), μs/step; MLA TFLOPS"
# decode steps that append each sequence's new token first (see time_config)
STEP_WORKLOADS = ("gqa_b64_ctx1k_step", "gqa_b64_ctx1k_fp8_step", "mla_b16_ctx64k_h16_step",
                  "mla_b16_ctx64k_h16_fp8_step")


# ---------------------------------------------------------------- helpers
def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


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
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in a background process;
    summary() gives the samples that fall inside one timed window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

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
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)

    def summary(self, t_start: float, t_stop: float):
        if self.proc is None:
            return None
        time.sleep(0.1)                  # let the sample after the window arrive
        rows = []
        for t, line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((t, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t_start - 0.06 <= r[0] <= t_stop + 0.06]
        use = inside or sorted(rows, key=lambda r: abs(r[0] - t_stop))[:3]
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


def workload_config(case):
    """The workload description; the same keys on the GPU and the reference arm."""
    return {"workload": case.name, "kind": case.kind, "batch": case.batch,
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


def rate_of(case, kv_bytes, flops, ms):
    """(value, unit) of the metric: GB/s for GQA, TFLOP/s for MLA."""
    if case.kind == "gqa":
        return kv_bytes / (ms * 1e-3) / 1e9, "GB/s"
    return flops / (ms * 1e-3) / 1e12, "TFLOP/s"


# ---------------------------------------------------------------- CPU oracle timing
def sample_case(workload: str, nseq: int):
    """A host case holding the first ``nseq`` sequences of a workload: the same per-sequence
    shape, lengths, dtypes and value distribution (seeded), with a cache pool just large
    enough for them. The oracle's cost per sequence does not depend on the pool's layout."""
    full = synth.workload(workload, with_caches=False)
    ctx = full.context_lens[:max(1, min(nseq, full.batch))].tolist()
    fmt, S = full.kv_format, full.seq_len_q
    if full.kind == "gqa":
        c = synth.make_gqa_case(batch=len(ctx), num_q_heads=full.num_q_heads,
                                num_kv_heads=full.num_kv_heads, head_dim=full.head_dim_qk,
                                dtype=full.dtype, page_size=full.page_size, context_lens=ctx,
                                scale=full.scale, kv_format=fmt, seq_len_q=S, name=workload)
    else:
        c = synth.make_mla_case(batch=len(ctx), num_q_heads=full.num_q_heads, dtype=full.dtype,
                                page_size=full.page_size, context_lens=ctx,
                                latent_dim=full.head_dim_v, scale=full.scale, kv_format=fmt,
                                seq_len_q=S, name=workload)
    return c


def oracle_one(case, b):
    """The oracle on every head of sequence b; returns the K+V (record) bytes it attended."""
    import oracle
    elem = 1 if case.kv_format == synth.FP8_E4M3 else 2
    S = case.seq_len_q
    rows = [(b, h) for h in range(case.num_q_heads)]
    rows3 = [(b, i, h) for i in range(S) for h in range(case.num_q_heads)]
    if case.kind == "gqa":
        fn = oracle.paged_decode_mtp if S > 1 else oracle.paged_decode
        fn(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, case.scale,
           case.page_size, case.dtype, rows=rows3 if S > 1 else rows, kv_format=case.kv_format,
           k_scale=case.k_scale, v_scale=case.v_scale)
        return traffic.gqa_kv_bytes([case.context_lens[b]], case.num_kv_heads, case.head_dim_qk,
                                    elem)
    fn = oracle.mla_decode_mtp if S > 1 else oracle.mla_decode
    fn(case.q, case.kv_cache, case.block_tables, case.context_lens, case.scale, case.page_size,
       case.dtype, head_dim_v=case.head_dim_v, rows=rows3 if S > 1 else rows,
       kv_format=case.kv_format, kv_scale=case.k_scale)
    return traffic.mla_kv_bytes([case.context_lens[b]], case.head_dim_qk, elem)


def oracle_sample(case, budget_s: float, start: int = 0):
    """Whole sequences (all heads) from sequence ``start`` on, round robin, until
    ~budget_s; returns (kv_bytes_done, seconds, sequences_done)."""
    done, n, t0 = 0, 0, time.perf_counter()
    b = start % case.batch
    while True:
        done += oracle_one(case, b)
        n += 1
        b = (b + 1) % case.batch
        if time.perf_counter() - t0 >= budget_s:
            return done, time.perf_counter() - t0, n


def _worker_sample(args):
    case, budget_s, start = args
    return oracle_sample(case, budget_s, start)


def oracle_rates(workload: str, budget_s: float, cores: int):
    """Oracle throughput on one core and on ``cores`` processes (one BLAS thread each).
    Runs in a process that never touches CUDA, so the pool may fork."""
    import multiprocessing as mp
    case = sample_case(workload, 4)
    b1, s1, n1 = oracle_sample(case, budget_s)
    ctx = mp.get_context("fork")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_worker_sample, [(case, budget_s, i) for i in range(cores)])
    wall = time.perf_counter() - t0
    bn = sum(r[0] for r in res)
    nn = sum(r[2] for r in res)
    return {"one_core": [b1, s1, n1], "all_cores": [bn, wall, nn], "cores": cores,
            "sample_batch": case.batch}


def cpu_baseline(workload: str, budget_s: float):
    """The oracle, as it stands, timed on the host cores in a fresh process: on all cores
    (one process per core) and on one core. ``value`` is the all-cores figure."""
    cores = host_cores()
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.oracle_rates(%r, %r, %d)))") % (ROOT, workload, budget_s,
                                                                    cores)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                           text=True, timeout=900)
    except subprocess.TimeoutExpired:
        return {"value": None, "error": "oracle timing timed out"}
    if r.returncode != 0:
        return {"value": None, "error": r.stderr.strip().splitlines()[-1:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    case = synth.workload(workload, with_caches=False)
    kv, flops = accounting(case)

    def rate(done, secs):
        v, _ = rate_of(case, done, done * flops / kv, secs * 1e3)
        return v
    (b1, s1, n1), (bn, sn, nn) = d["one_core"], d["all_cores"]
    unit = "GB/s" if case.kind == "gqa" else "TFLOP/s"
    return {"value": rate(bn, sn), "unit": unit, "cores": d["cores"], "kind": "oracle",
            "one_core": {"value": rate(b1, s1), "cores": 1},
            "sample": f"float64 numpy oracle on whole sequences (all heads) of {workload}'s "
                      f"shape, drawn as a {d['sample_batch']}-sequence case: {nn} sequences in "
                      f"{sn:.1f} s wall on {d['cores']} processes (one BLAS thread each), and "
                      f"{n1} in {s1:.1f} s on one"}


def run_reference(args, workload):
    """The reference arm: the oracle, as it stands, on all host cores."""
    import multiprocessing as mp
    case_full = synth.workload(workload, with_caches=False)
    kv, flops = accounting(case_full)
    cores = host_cores()
    case = sample_case(workload, 4)
    per_step_budget = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    ctx = mp.get_context("fork")               # this arm never touches CUDA
    total_bytes, total_s = 0, 0.0
    with ctx.Pool(cores) as pool:
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            res = pool.map(_worker_sample, [(case, per_step_budget, i + w) for w in range(cores)])
            if i >= args.warmup:
                total_s += time.perf_counter() - t0
                total_bytes += sum(r[0] for r in res)
    value, unit = rate_of(case_full, total_bytes, total_bytes * flops / kv, total_s * 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kv / (total_bytes / total_s) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) values, random block tables)",
            "config": workload_config(case_full),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": f"each step: whole sequences of {workload}'s shape for "
                                       f"~{per_step_budget:.2f} s on {cores} processes"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


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
    return plan.num_launches > 1


def rotation_copies(kv_bytes: int) -> int:
    """Copies of the caches that steps rotate over, so that a copy is read again only after
    at least 4x L2 of other cache bytes (inputs larger than L2 between timed steps)."""
    return max(1, min(4096, math.ceil(4 * L2_BYTES / max(1, kv_bytes)) + 1))


def device_caches(case, copies, seed, torch):
    """The workload's caches drawn on the device: N(0,1) in fp32 from torch's seeded
    generator, rounded to nearest-even to the cache type (E4M3 codes with one per-tensor
    scale amax / 448 for fp8), then cloned ``copies`` times."""
    gen = torch.Generator(device="cuda").manual_seed(1000 + seed)
    fp8 = case.kv_format == synth.FP8_E4M3
    tdt = torch.float16 if case.dtype == synth.FP16 else torch.bfloat16

    def draw(shape):
        x = torch.randn(shape, generator=gen, device="cuda", dtype=torch.float32)
        if not fp8:
            return x.to(tdt), 1.0
        sc = float(x.abs().max()) / synth.E4M3_MAX
        return (x / sc).to(torch.float8_e4m3fn).view(torch.uint8), sc

    if case.kind == "gqa":
        shape = (case.num_blocks, case.page_size, case.num_kv_heads, case.head_dim_qk)
        (k0, case.k_scale), (v0, case.v_scale) = draw(shape), draw(shape)
        return [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(copies - 1)]
    (kv0, case.k_scale) = draw((case.num_blocks, case.page_size, case.head_dim_qk))
    case.v_scale = case.k_scale
    return [(kv0, None)] + [(kv0.clone(), None) for _ in range(copies - 1)]


def time_config(args, workload, rank, world, dist, sampler, e2e=False, steps=None):
    """Time one workload's decode step on this GPU; returns the measurement record."""
    import numpy as np
    import torch

    from paged_kv_cache_61_gb300 import pda

    # "<workload>_step": each step first appends one new token per sequence (the last of
    # its context) through the append call, then decodes: a serving step's cache work
    with_append = workload.endswith("_step")
    case = synth.workload(workload[: -len("_step")] if with_append else workload, seed=rank,
                          with_caches=False)
    case.name = workload
    kv_bytes, flops = accounting(case)
    tdt = torch.float16 if case.dtype == synth.FP16 else torch.bfloat16
    fp8 = case.kv_format == synth.FP8_E4M3

    def dev16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(tdt)

    copies = rotation_copies(kv_bytes)
    # a graph of at least `copies` steps, so that its replays never reread a copy from L2
    K = steps or max(args.steps, copies)
    caches = device_caches(case, copies, rank, torch)
    q = dev16(case.q)
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
        elif fp8:
            pda.mla_append_fp8(kn, kc, case.k_scale, tables_, ctx_, plan, ws, stream)
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
        elif fp8:
            pda.mla_decode_fp8(q_, kc, case.k_scale, tables_, ctx_, case.scale, out_, lse_, plan,
                               ws, stream)
        else:
            pda.mla_decode(q_, kc, tables_, ctx_, case.scale, out_, lse_, plan, ws, stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # Device time of each decode call on its own (events around every eager call).
    n_ev = min(K, 200)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for i in range(n_ev):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    per_call_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # The timed region: K steps captured once in a CUDA graph, replayed R times back to
    # back (each replay bracketed by a barrier and a synchronize and timed by events on the
    # launching stream; launch gaps of the host loop removed, every step still runs).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    est_ms = statistics.median(per_call_ms) * K
    R = int(max(5, min(2000, math.ceil(300.0 / max(est_ms, 1e-3)))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(R)]
    t_win0 = time.time()
    for e0, e1 in ev:
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    t_win1 = time.time()
    replay_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms_per_step = reduce_step_time(statistics.median(replay_ms) / K, dist, "cuda")
    clocks = sampler.summary(t_win0, t_win1) if sampler else None
    isolated_us = isolated_step_us(step, K, stream, torch)
    launches_per_step = 1 + (1 if _has_merge(plan, case) else 0) + (1 if with_append else 0)

    pk, pk_src = peaks()
    if case.kind == "gqa":
        achieved = kv_bytes / (ms_per_step * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": f"hbm_gbs of {pk_src}",
                "frac_of_8TBs_spec": achieved / 8000.0}
    else:
        t_bytes = kv_bytes / (pk["hbm_gbs"] * 1e9)
        t_flops = flops / (pk["bf16_tflops"] * 1e12)
        achieved_gbs = kv_bytes / (ms_per_step * 1e-3) / 1e9
        achieved_tf = flops / (ms_per_step * 1e-3) / 1e12
        if t_bytes >= t_flops:
            roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved_gbs / pk["hbm_gbs"],
                    "peak_source": f"hbm_gbs of {pk_src}"}
        else:
            roof = {"bound": "tensor", "achieved": achieved_tf, "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": achieved_tf / pk["bf16_tflops"],
                    "peak_source": f"bf16_tflops of {pk_src}"}
        roof["tflops"] = achieved_tf
        roof["gbs"] = achieved_gbs
        roof["frac_of_slower_roof"] = max(t_bytes, t_flops) / (ms_per_step * 1e-3)
    roof["traffic"] = recorded_traffic(workload, kernel_kind(case))
    roof["algorithmic_bytes_per_launch"] = kv_bytes
    roof["mean_launch_us"] = ms_per_step * 1e3
    roof["scope"] = (("append kernel + " if with_append else "") + "decode kernel" +
                     (" + split-merge kernel" if _has_merge(plan, case) else "") + " per step")
    roof["event_us_per_call"] = statistics.median(per_call_ms) * 1e3
    roof["event_us_per_call_min"] = min(per_call_ms) * 1e3
    value, unit = rate_of(case, kv_bytes * world, flops * world, ms_per_step)
    rec = {"case": case, "value": value, "unit": unit, "ms_per_step": ms_per_step, "steps": K,
           "replays": R, "replay_us_per_step": {
               "median": statistics.median(replay_ms) / K * 1e3,
               "min": min(replay_ms) / K * 1e3, "max": max(replay_ms) / K * 1e3},
           "roofline": roof, "clocks": clocks, "launches_per_step": launches_per_step,
           "isolated_us_per_step": isolated_us,
           "copies": copies, "kv_bytes": kv_bytes, "flops": flops,
           "plan": {"num_ctas": plan.num_ctas,
                    "max_splits": max(plan.num_splits(b) for b in range(case.batch))}}
    if e2e and rank == 0:
        rec["e2e"] = time_e2e(args, case, step, stream, [q, tables, ctx] +
                              ([k_new, v_new] if with_append else []), out, lse, with_append,
                              kv_bytes, flops)
    del graph, caches
    return rec


def isolated_step_us(step, K, stream, torch):
    """Device time of one step on its own, outside the timed window (information only).

    In the timed graph a decode grid may start while the step before it drains: the
    library's decode and split-merge kernels allow programmatic dependent launch, so
    consecutive steps overlap, as consecutive calls do when nothing else runs between them.
    Here every step is preceded by a one-element kernel, after which a grid starts only
    once everything before it has completed; the same K of those kernels alone are timed
    as well and subtracted."""
    sep = torch.zeros(1, device="cuda")
    g_iso, g_sep = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_iso, stream=stream):
        for i in range(K):
            sep.add_(1.0)
            step(i)
    with torch.cuda.graph(g_sep, stream=stream):
        for i in range(K):
            sep.add_(1.0)
    t_iso, t_sep = [], []
    for _ in range(5):
        for g, acc in ((g_iso, t_iso), (g_sep, t_sep)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            acc.append(e0.elapsed_time(e1))
    del g_iso, g_sep
    return (statistics.median(t_iso) - statistics.median(t_sep)) / K * 1e3


def time_e2e(args, case, step, stream, ins, out, lse, with_append, kv_bytes, flops):
    """The same step end to end through the C ABI: pinned host inputs in, outputs back,
    every step. A step's inputs (q, block tables, context lengths, and the new tokens'
    K/V of the _step workloads) travel as one pinned host buffer, one copy in; its outputs
    (out, lse) are views of one device buffer, one copy out. The decode call reads and
    writes those views, as a caller batching its transfers would.

    The copies run on two copy streams beside the compute stream, with the device buffers
    doubled, as a serving loop would overlap them: step i's inputs go in while step i-1
    decodes, and step i-1's outputs come back while step i decodes. Events order each copy
    after what it depends on (a buffer is rewritten only once its previous contents have
    been read). Every step's copies lie inside the timed region, which ends when the last
    outputs are back in host memory."""
    import torch
    e2e_steps = min(max(args.steps, 20), 500)
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
    res_h = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    in_d = [torch.empty(h2d, dtype=torch.uint8, device="cuda") for _ in range(2)]
    res_d = [torch.empty(d2h, dtype=torch.uint8, device="cuda") for _ in range(2)]
    for t, off in zip(ins, in_offs):
        view(in_h, off, t).copy_(t.cpu())
    d_in = [[view(buf, off, t) for t, off in zip(ins, in_offs)] for buf in in_d]
    d_out = [[view(buf, off, t) for t, off in zip(outs, out_offs)] for buf in res_d]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    n_ev = e2e_steps + 8
    ev_in = [torch.cuda.Event() for _ in range(n_ev)]      # step's inputs on the device
    ev_dec = [torch.cuda.Event() for _ in range(n_ev)]     # step decoded (inputs read)
    ev_out = [torch.cuda.Event() for _ in range(n_ev)]     # step's outputs on the host

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(ev_dec[i - 2])           # step i-2 has read in_d[b]
            in_d[b].copy_(in_h, non_blocking=True)
            ev_in[i].record(h2d_s)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])              # step i-2's outputs were copied out
        ins_b, outs_b = d_in[b], d_out[b]
        extra = dict(kn_=ins_b[3], vn_=ins_b[4]) if with_append else {}
        step(i, q_=ins_b[0], out_=outs_b[0], lse_=outs_b[1], tables_=ins_b[1], ctx_=ins_b[2],
             **extra)
        ev_dec[i].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_dec[i])
            res_h.copy_(res_d[b], non_blocking=True)
            ev_out[i].record(d2h_s)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_out[e2e_steps - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / e2e_steps
    value, unit = rate_of(case, kv_bytes, flops, ms)
    return {"value": value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms,
            "path": "one pinned host buffer (q, block_tables, context_lens"
                    + (", new K/V" if with_append else "") + ") -> device, C-ABI decode into "
                    "one device buffer (out, lse) -> pinned host, every step, eager launches; "
                    "copies on two copy streams overlapping the decode of the neighbouring "
                    "steps (device buffers doubled); caches resident in HBM"}


def config_entry(rec, cpu):
    """The per_config record of one workload (no multi-rank fields)."""
    case = rec["case"]
    roof = rec["roofline"]
    e = {"config": workload_config(case), "us_per_step": rec["ms_per_step"] * 1e3,
         "value": rec["value"], "unit": rec["unit"],
         "gbs": rec["kv_bytes"] / (rec["ms_per_step"] * 1e-3) / 1e9,
         "tflops": rec["flops"] / (rec["ms_per_step"] * 1e-3) / 1e12,
         "steps_per_replay": rec["steps"], "replays": rec["replays"],
         "replay_us_per_step": rec["replay_us_per_step"],
         "isolated_us_per_step": rec["isolated_us_per_step"],
         "roofline": roof, "frac_of_slower_roof": roof.get("frac_of_slower_roof", roof["frac"]),
         "clocks": rec["clocks"], "plan": rec["plan"],
         "l2": f"steps rotate over {min(rec['copies'], rec['steps'])} copies of the caches "
               f"({rec['kv_bytes'] / 1e6:.2f} MB of K+V read per step)",
         "cpu_baseline": cpu}
    return e


def run_gpu(args, workload, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    # everything on one non-default stream (CUDA graphs cannot capture the legacy stream)
    torch.cuda.set_stream(torch.cuda.Stream())
    dist = None
    if world > 1:
        import torch.distributed as dist
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    try:
        head = time_config(args, workload, rank, world, dist, sampler, e2e=True,
                           steps=args.steps)
        torch.cuda.empty_cache()
        others = []
        if args.per_config and world == 1:
            for name in PER_CONFIG:
                if name == workload:
                    continue
                others.append(time_config(args, name, rank, world, dist, sampler))
                torch.cuda.empty_cache()
    finally:
        if sampler:
            sampler.stop()
    if rank != 0:
        return
    case = head["case"]
    cpu = None if args.no_cpu_baseline else cpu_baseline(workload, 10.0)
    per_config = {}
    for rec in others:
        c = None if args.no_cpu_baseline else cpu_baseline(rec["case"].name, 3.0)
        per_config[rec["case"].name] = config_entry(rec, c)
    line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "us_per_step": head["ms_per_step"] * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if case.dtype == synth.FP16 else "bf16",
            "data": "synthetic: seeded N(0,1) values (caches drawn on the device by torch's "
                    "seeded generator), random block tables, seed = rank",
            "config": workload_config(case),
            "l2": f"inputs larger than L2: steps rotate over {min(head['copies'], args.steps)} "
                  f"copies of the caches ({head['kv_bytes'] / 1e6:.0f} MB each)",
            "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": head["e2e"],
            "gpu_launches": args.steps * head["launches_per_step"], "clocks": head["clocks"],
            "replays": head["replays"], "replay_us_per_step": head["replay_us_per_step"],
            "isolated_us_per_step": head["isolated_us_per_step"],
            "timing": "value: K steps captured in one CUDA graph, replayed R times (device "
                      "events per replay, median); consecutive steps overlap through "
                      "programmatic dependent launch. isolated_us_per_step: each step after a "
                      "one-element kernel that lets no grid start early (that kernel's own "
                      "time subtracted), outside the timed window; roofline.event_us_per_call: "
                      "events around each eager call",
            "plan": head["plan"], "per_config": per_config}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=synth.WORKLOADS + STEP_WORKLOADS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="time only the headline workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    # the other workloads are reported with the default headline run only
    if args.workload is not None:
        args.per_config = False
    workload = args.workload or DEFAULT_WORKLOAD
    rank = env_int("RANK", 0)
    world = env_int("WORLD_SIZE", 1)
    local_rank = env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, workload)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gpu(args, workload, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
