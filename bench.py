"""Benchmark: split-KV decode attention + merge on GB300.

One step = one pass of the whole path over one batch: the fused persistent
engine (``splitkv_decode``: every split's partial state, then the LSE merge)
on a batch whose inputs are already resident in HBM.  The default workload
is the largest single-GPU configuration, the multi-million-token decode
(4 requests x 1,048,576 tokens, 64/8 heads, D=128, page 128, planner splits
in [16, 64]), whose 16 GiB of KV is far larger than L2, so no flush is
needed between steps.  The same line carries one sub-record per other
configuration (``configs``), each timed the same way (the 0.5 MB fp32 case
with an L2 flush between calls).

Printed JSON line (rank 0):
  value      KV-cache bytes read per second (GB/s, algorithmic bytes: each
             cached K and V row once) over the whole job
  e2e        the same metric through the public API with host buffers:
             per step H2D of the query block, lengths and page table, host
             planning + plan upload, the decode, D2H of output and LSE (the
             next step's plan is built while the GPU runs this one)
  roofline   the dominant kernel against the measured HBM copy bandwidth
             (tensor-bound kernels: the measured sustained bf16 rate)
  configs    per configuration: us/call p10/p50/p90, KV GB/s, decode
             tokens/s, the step against the configuration's roofline
             max(KV bytes / HBM, flops / tensor) and the dominant kernel's
             roofline
  cpu_baseline  the float64 CPU oracle on a bounded sample, host cores

``--impl reference`` times the float64 CPU oracle alone on the same
workload (the reference arm of this comparison; there is no GPU reference).
Multi-GPU: replicas only -- each rank runs its own copy of the workload, no
data-path collective; value = all ranks' bytes / max rank time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "million_token_decode"
# configurations measured as sub-records of the default line (the main line's
# workload is skipped); the last two are the extension rows (FP8 cache,
# speculative 16-token query blocks)
SUB_CONFIGS = ["tiny_fp32_gqa", "llama405b_gqa_decode", "deepseek_mla_decode", "mixed_chunked_prefill",
               "million_token_decode", "llama405b_fp8_decode", "spec_decode_q16", "deepseek_mla_fp8_decode"]
L2_FLUSH_BYTES = 256 << 20
METRIC = "KV-cache HBM GB/s (% of peak) and decode tokens/s, split-KV attn+merge"
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, 0, 1, 0


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# sources each kernel's committed ncu traffic figure depends on
KERNEL_SOURCES = {
    "gqa_engine_kernel": ["long_context_split_gb300/csrc/gqa_engine.cu", "long_context_split_gb300/csrc/internal.h"],
    "chunk_tc_kernel": ["long_context_split_gb300/csrc/chunk_kernel.cu", "long_context_split_gb300/csrc/tc_common.cuh",
                        "long_context_split_gb300/csrc/internal.h"],
    "mla_partial_kernel": ["long_context_split_gb300/csrc/mla_kernel.cu", "long_context_split_gb300/csrc/tc_common.cuh",
                           "long_context_split_gb300/csrc/internal.h"],
    "generic_partial_kernel": ["long_context_split_gb300/csrc/generic_kernel.cu", "long_context_split_gb300/csrc/internal.h"],
    "merge_states_kernel": ["long_context_split_gb300/csrc/merge_kernel.cu", "long_context_split_gb300/csrc/internal.h"],
    "pair_tc_kernel": ["long_context_split_gb300/csrc/pair_kernel.cu", "long_context_split_gb300/csrc/tc_common.cuh",
                       "long_context_split_gb300/csrc/internal.h"],
    "mla_latent_convert_kernel": ["long_context_split_gb300/csrc/mla_kernel.cu",
                                  "long_context_split_gb300/csrc/tc_common.cuh",
                                  "long_context_split_gb300/csrc/internal.h"],
    "chunk_value_convert_kernel": ["long_context_split_gb300/csrc/chunk_kernel.cu",
                                   "long_context_split_gb300/csrc/tc_common.cuh",
                                   "long_context_split_gb300/csrc/internal.h"],
}
PROFILE_PREFIX = {"gqa_engine_kernel": "gqa_engine", "chunk_tc_kernel": "chunk_tiles",
                  "mla_partial_kernel": "mla_partial", "generic_partial_kernel": "generic_partial",
                  "merge_states_kernel": "merge_states", "pair_tc_kernel": "pair_tiles",
                  "mla_latent_convert_kernel": "mla_latent", "chunk_value_convert_kernel": "chunk_value"}


def _traffic_for(kernel: str, workload: str, kernel_hash: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"{PROFILE_PREFIX[kernel]}_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_launch")


def _peak_bf16():
    """Sustained bf16 dense throughput (TFLOP/s) for kernels timed inside a long
    run of back-to-back steps; the recipe's fallback when the file is absent."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured sustained bf16"
    return 1700.0, "fallback sustained bf16"


def _roofline(spec, wl, plan, kernels):
    """Roofline of the kernel with the most device time in the timed region:
    algorithmic bytes (HBM-bound kernels) or flops (tensor-bound ones) per
    launch over its mean launch time from the launch profiler's events."""
    from long_context_split_gb300 import roofline
    name = max(kernels, key=lambda k: kernels[k][1])
    n, ms = kernels[name]
    per_launch_s = ms / n * 1e-3
    eb = 1 if spec.kv_fp8 else 2 if spec.dtype == "bf16" else 4
    route = plan.chunk_requests()      # 1 chunk tiles, 2 paired tiles, 0 engine
    chunk = route == 1
    sl, ql = np.asarray(wl.seq_lens), np.asarray(wl.q_lens)
    kh = _source_hash(KERNEL_SOURCES[name])
    if name == "chunk_tc_kernel" or name == "mla_partial_kernel":
        sel = chunk if name == "chunk_tc_kernel" else np.ones(len(sl), dtype=bool)
        flops = roofline.attention_flops(sl[sel], ql[sel], spec.num_q_heads, spec.head_dim_qk, spec.head_dim_v)
        peak, src = _peak_bf16()
        achieved = flops / per_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "algorithmic_per_launch": flops}
        if name == "mla_partial_kernel":
            hbm, hsrc = _peaks()
            kvb = roofline.kv_bytes(spec.kind, sl, spec.num_kv_heads, spec.head_dim_qk, spec.head_dim_v, eb)
            roof["hbm_frac"] = kvb / per_launch_s / 1e9 / hbm
    else:
        # HBM-bound kernels: the KV bytes of the requests they attend (the latent copy's pre-pass:
        # the E4M3 latent rows it reads and the bf16 pages it writes)
        sel = route == 2 if name == "pair_tc_kernel" else route == 0
        kvb = roofline.kv_bytes(spec.kind, sl[sel], spec.num_kv_heads, spec.head_dim_qk, spec.head_dim_v, eb)
        if name == "mla_latent_convert_kernel":
            kvb += int(sum(-(-int(L) // spec.page_size) for L in sl)) * spec.page_size * spec.head_dim_qk * 2
        peak, src = _peaks()
        achieved = kvb / per_launch_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "algorithmic_per_launch": kvb}
        src = f"{src} HBM copy"
    roof.update({"traffic": _traffic_for(name, spec.name, kh), "peak_source": src, "kernel": name,
                 "launches": n, "ms_per_launch": ms / n, "kernel_source_hash": kh})
    return roof


def _make_problem(wl, dev):
    import long_context_split_gb300 as skv
    t = wl.device_tensors(dev)
    s = wl.spec
    prob = skv.AttentionProblem(
        q=t["q"], k_cache=t["k"], v_cache=t["v"], page_table=t["page_table"], seq_lens=t["seq_lens"],
        qo_indptr=t["qo_indptr"], num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads,
        head_dim_qk=s.head_dim_qk, head_dim_v=s.head_dim_v, page_size=s.page_size, scale=s.scale,
        kind=s.kind, seq_lens_host=wl.seq_lens, qo_indptr_host=wl.qo_indptr,
        k_scale=s.k_scale if s.kv_fp8 else None, v_scale=s.v_scale if s.kv_fp8 else None)
    return prob, t


def _plan_params(spec):
    import long_context_split_gb300 as skv
    n = W.uniform_splits(spec)
    if n is not None:
        return skv.plan_params("uniform", uniform_splits=n)
    lo, hi = W.planner_split_range(spec)
    return skv.plan_params("critical_wave", min_splits=lo, max_splits=hi)


def _kv_bytes(wl):
    from long_context_split_gb300 import roofline
    s = wl.spec
    eb = 1 if s.kv_fp8 else 2 if s.dtype == "bf16" else 4
    return roofline.kv_bytes(s.kind, wl.seq_lens, s.num_kv_heads, s.head_dim_qk, s.head_dim_v, eb)


class OracleSampler:
    """Times the float64 oracle on whole query rows of a few (request, KV
    head) groups regenerated on the host (regeneration is not timed).  Each
    row is credited with its share of its group's KV bytes, so a pass over
    every row of the batch would be credited exactly the batch's KV bytes."""

    def __init__(self, wl, n_groups: int = 2, seed: int = 1234):
        import oracle
        self.oracle = oracle
        s = wl.spec
        self.threads = oracle.num_threads()
        rng = np.random.default_rng(seed)
        groups = [(b, h) for b in range(s.batch) for h in range(s.num_kv_heads)]
        pick = [groups[i] for i in rng.permutation(len(groups))[:n_groups]]
        eb = 1 if s.kv_fp8 else 2 if s.dtype == "bf16" else 4
        self.items = []
        for b, h in pick:
            sub = oracle.subproblem_for_group(wl, b, h)
            L = int(wl.seq_lens[b])
            row_bytes = L * (s.head_dim_qk + (s.head_dim_v if s.kind == "gqa" else 0)) * eb / sub.num_q_heads
            self.items.append((sub, sub.all_rows(), row_bytes))
        self.total_groups = len(groups)
        self.cursor = 0

    def run(self, budget_s: float):
        """Rows in chunks of one per host thread until budget_s is spent."""
        done_bytes, spent, rows = 0.0, 0.0, 0
        while True:
            sub, all_rows, row_bytes = self.items[self.cursor % len(self.items)]
            start = (self.cursor // len(self.items)) * self.threads % len(all_rows)
            chunk = all_rows[start:start + self.threads]
            self.cursor += 1
            t0 = time.perf_counter()
            sub.attention_rows(chunk)
            spent += time.perf_counter() - t0
            done_bytes += row_bytes * len(chunk)
            rows += len(chunk)
            if spent >= budget_s:
                return done_bytes / spent / 1e9, rows, spent


def run_reference(args):
    dist, rank, ws, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    spec = W.get_config(args.workload)
    wl = W.build_workload(spec)
    sampler = OracleSampler(wl)
    budget = max(0.05, min(args.ref_step_seconds, 120.0 / max(1, args.steps + args.warmup)))
    per_step = []
    for i in range(args.warmup + args.steps):
        gbs, rows, spent = sampler.run(budget)
        if i >= args.warmup:
            per_step.append((gbs, rows, spent))
    value = statistics.median([p[0] for p in per_step])
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median([p[2] for p in per_step]), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(spec, wl, None),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{per_step[0][1]} query rows per step from {len(sampler.items)} of "
                                   f"{sampler.total_groups} (request, KV head) groups, ~{budget:.2f} s of CPU "
                                   f"work per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(spec, wl, plan):
    return {
        "workload": spec.name, "kind": spec.kind, "batch": spec.batch,
        "seq_len": int(wl.seq_lens.max()) if spec.name != "mixed_chunked_prefill" else "mixed",
        "mean_seq_len": float(np.mean(wl.seq_lens)), "total_q": int(wl.total_q),
        "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
        "head_dim_qk": spec.head_dim_qk, "head_dim_v": spec.head_dim_v, "page_size": spec.page_size,
        "splits": spec.split,
        "l2": ("L2 flushed between calls (256 MB write)" if spec.name == "tiny_fp32_gqa"
               else "inputs larger than L2 (KV cache >> 129 MB); no flush"),
        "parallelism": "replicas",
        **({"kv_cache": f"fp8 e4m3, k_scale {spec.k_scale}, v_scale {spec.v_scale}"} if spec.kv_fp8 else {}),
    }


def _step_roofline(spec, wl, kvb):
    """The configuration's roofline time: max(KV bytes / HBM copy bandwidth,
    attention flops / sustained bf16 rate) -- the step can go no faster than its
    bytes or its products allow (mixed batches: both overlapped perfectly)."""
    from long_context_split_gb300 import roofline
    hbm, _ = _peaks()
    tf, _ = _peak_bf16()
    flops = roofline.attention_flops(wl.seq_lens, wl.q_lens, spec.num_q_heads, spec.head_dim_qk, spec.head_dim_v)
    t_hbm = kvb / (hbm * 1e9)
    t_tc = flops / (tf * 1e12)
    return {"time_ms": 1e3 * max(t_hbm, t_tc), "hbm_ms": 1e3 * t_hbm, "tensor_ms": 1e3 * t_tc,
            "bound": "hbm" if t_hbm >= t_tc else "tensor", "flops": flops, "kv_bytes": kvb}


def _time_steps(att, out, lse, stream, steps, flush=None):
    """Per-step CUDA-event times (ms) of ``steps`` decode calls and the launch
    profiler's per-kernel totals over them; ``flush`` (a device buffer larger than
    L2) is overwritten before every call, outside the timed events."""
    import long_context_split_gb300 as skv
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    skv.profile_begin()          # events around each of the library's launches, on its stream
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        starts[i].record(stream)
        att.decode(out, lse)
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    kernels = skv.profile_end()
    per = sorted(st.elapsed_time(e) for st, e in zip(starts, ends))
    total = sum(per) if flush is not None else t_start.elapsed_time(t_end)
    return per, total, kernels


def _tail_idle(prob, params, dev):
    """Tail idle of each stage of one traced launch (a separate plan with trace
    records; the timed plan records nothing): per stage, each SM's wait after its
    last task until the stage finishes, over total SM-time (LiquidCP Section 3)."""
    import long_context_split_gb300 as skv
    p = type(params).from_buffer_copy(params)
    p.trace = 1
    att = skv.SplitKVAttention(prob, p)
    if att.plan.trace_records == 0:
        return None
    out, lse = att.out_like()
    for _ in range(3):
        att.decode(out, lse)
    torch.cuda.synchronize()
    att.check_device_error()
    rec = skv.trace_read(att.plan, att.workspace)
    res = {}
    for stage, kinds in (("engine", (skv.TRACE_ATTENTION, skv.TRACE_REDUCTION)), ("chunk_tiles", (skv.TRACE_CHUNK,)),
                         ("pair_tiles", (skv.TRACE_PAIR,)), ("mla", (skv.TRACE_MLA_ITEM,))):
        if np.isin(rec["kind"], kinds).any():
            # the SMs the stage ran on (a stage may share the GPU with another kernel)
            st = skv.trace_tail_idle(rec, kinds=kinds, num_sms=0)
            res[stage] = {"tail_idle_frac": st["tail_idle_frac"], "span_us": (st["end_ns"] - st["begin_ns"]) / 1e3,
                          "records": st["records"], "sms": st["sms"]}
    del att, out, lse
    return res


def _pcts(per):
    return {"p10": per[len(per) // 10], "p50": per[len(per) // 2], "p90": per[(9 * len(per)) // 10]}


def _sub_record(name, dev, steps, warmup):
    """One configuration measured like the main line (kernel time only, inputs
    resident): us/call percentiles, KV GB/s, tokens/s, the step against the
    configuration's roofline and the dominant kernel's roofline."""
    import long_context_split_gb300 as skv
    spec = W.get_config(name)
    wl = W.build_workload(spec)
    prob, tens = _make_problem(wl, dev)
    params = _plan_params(spec)
    att = skv.SplitKVAttention(prob, params)
    out, lse = att.out_like()
    stream = torch.cuda.current_stream()
    att.decode(out, lse)
    torch.cuda.synchronize()
    att.check_device_error()
    for _ in range(max(3, warmup)):
        att.decode(out, lse)
    flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if name == "tiny_fp32_gqa" else None)
    per, total, kernels = _time_steps(att, out, lse, stream, steps, flush)
    att.check_device_error()
    kvb = _kv_bytes(wl)
    med = per[len(per) // 2]
    roof = _step_roofline(spec, wl, kvb)
    hbm, _ = _peaks()
    rec = {
        "workload": name, "steps": steps, "us_per_call": {k: 1e3 * v for k, v in _pcts(per).items()},
        "kv_gbs": kvb / (med * 1e-3) / 1e9, "pct_of_measured_hbm": 100.0 * kvb / (med * 1e-3) / 1e9 / hbm,
        "pct_of_8000_gbs": 100.0 * kvb / (med * 1e-3) / 1e9 / 8000.0,
        "decode_tokens_per_s": int(wl.total_q) / (med * 1e-3),
        "step_roofline": dict(roof, frac=roof["time_ms"] / med),
        "roofline": _roofline(spec, wl, att.plan, kernels),
        "kernels": {k: {"launches": n, "ms_per_launch": ms / n} for k, (n, ms) in kernels.items()},
        "gpu_launches": sum(n for n, _ in kernels.values()),
        "plan": _plan_summary(att.plan),
        "config": _config(spec, wl, att.plan),
        "tail_idle": _tail_idle(prob, params, dev),
    }
    del att, out, lse, tens, prob, flush
    torch.cuda.empty_cache()
    return rec


def _plan_summary(plan):
    sp = plan.splits()
    return {"splits_min": int(sp.min()), "splits_max": int(sp.max()), "splits_mean": float(sp.mean()),
            "tasks": int(plan.num_tasks), "chunk_tasks": int(plan.num_chunk_tasks),
            "pair_tasks": int(plan.num_pair_tasks), "kernel_path": int(plan.kernel_path)}


def run_ours(args):
    import long_context_split_gb300 as skv
    dist, rank, ws, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = W.get_config(args.workload)
    wl = W.build_workload(spec, batch=args.batch or None)
    subset = bool(args.select or args.batch or args.max_len)
    if args.select:
        # a subset of the requests, same lengths (small cases for profiling; not a bench line)
        pick = [int(x) for x in args.select.split(",")]
        full = W.build_workload(spec)
        spec = dataclasses.replace(spec, batch=len(pick))
        wl = W.build_workload(spec, seq_lens=full.seq_lens[pick], q_lens=full.q_lens[pick])
    elif args.batch:
        spec = dataclasses.replace(spec, batch=len(wl.seq_lens))
        wl.spec = spec
    if args.max_len:
        # histories cut to at most max_len tokens (small cases for profiling; not a bench line)
        wl = W.build_workload(spec, seq_lens=np.minimum(wl.seq_lens, args.max_len), q_lens=wl.q_lens)
    prob, tens = _make_problem(wl, dev)
    params = _plan_params(spec)
    if args.interleave:
        params.interleave = 1
    if args.partial_bf16:
        params.partial_dtype = skv.BF16
    att = skv.SplitKVAttention(prob, params)
    out, lse = att.out_like()
    stream = torch.cuda.current_stream()
    kv = _kv_bytes(wl)
    tokens = int(wl.total_q)

    # correctness guard on the timed configuration (one launch, checked below)
    att.decode(out, lse)
    torch.cuda.synchronize()
    att.check_device_error()

    for _ in range(max(3, args.warmup)):
        att.decode(out, lse)
    torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        _barrier(dist)
        per, total_ms, kernels = _time_steps(att, out, lse, stream, args.steps)
        _barrier(dist)
    att.check_device_error()
    total_ms = _max_over_ranks(dist, total_ms)
    med = per[len(per) // 2]
    ms_per_step = total_ms / args.steps
    value = ws * kv * args.steps / (total_ms * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers ----
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_q = torch.empty(tens["q"].shape, dtype=tens["q"].dtype).pin_memory()
    h_q.copy_(tens["q"].cpu())
    h_pt, h_sl, h_qo = pin(wl.page_table), pin(wl.seq_lens), pin(wl.qo_indptr)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = h_q.numel() * h_q.element_size() + h_pt.numel() * 4 + h_sl.numel() * 4 + h_qo.numel() * 4
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * 4
    e2e_steps = max(3, min(args.steps, args.e2e_steps))

    # A decode loop knows the next step's lengths before this step ends, so the next plan is
    # built on the host while the GPU runs this step; every step still plans, uploads its
    # plan, copies its inputs in and reads its result back.
    pending = {"plan": skv.splitkv_plan(prob, params)}

    def e2e_step():
        plan = pending["plan"]
        tens["q"].copy_(h_q, non_blocking=True)
        tens["page_table"].copy_(h_pt, non_blocking=True)
        tens["seq_lens"].copy_(h_sl, non_blocking=True)
        tens["qo_indptr"].copy_(h_qo, non_blocking=True)
        skv.splitkv_plan_upload(plan, att.workspace)
        skv.splitkv_decode(prob, plan, att.workspace, out, lse, att.error_word)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
        pending["plan"] = skv.splitkv_plan(prob, params)
        torch.cuda.current_stream().synchronize()
        return plan

    for _ in range(3):
        e2e_step()
    _barrier(dist)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = _max_over_ranks(dist, time.perf_counter() - t0)
    att.check_device_error()
    e2e_value = ws * kv * e2e_steps / e2e_s / 1e9

    roof = _roofline(spec, wl, att.plan, kernels)
    roof["per_step_ms"] = {"median": med, "p10": per[len(per) // 10], "p90": per[(9 * len(per)) // 10]}
    step_roof = _step_roofline(spec, wl, kv)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("bf16 q, fp8-e4m3 kv, f16 mma" if spec.kv_fp8 else "bf16") if spec.dtype == "bf16" else "f32", "data": "synthetic",
        "config": _config(spec, wl, att.plan),
        "plan": _plan_summary(att.plan),
        "decode_tokens_per_s": ws * tokens * args.steps / (total_ms * 1e-3),
        "us_per_call": 1e3 * med,
        "us_per_call_pcts": {k: 1e3 * v for k, v in _pcts(per).items()},
        "pct_of_8000_gbs": 100.0 * value / ws / 8000.0,
        "step_roofline": dict(step_roof, frac=step_roof["time_ms"] / med),
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "includes": "H2D q+lengths+page table, plan upload, decode, D2H out+lse; the next step's host plan overlaps the GPU"},
        "roofline": roof,
        "gpu_launches": sum(n for n, _ in kernels.values()),
        "kernels": {k: {"launches": n, "ms_per_launch": ms / n} for k, (n, ms) in kernels.items()},
        "clocks": clk.summary(),
    }
    if args.select or args.batch:
        line["config"]["subset"] = args.select or f"first {args.batch} requests"
    if args.max_len:
        line["config"]["subset"] = f"histories cut to {args.max_len} tokens"
    if args.interleave:
        line["config"]["split_layout"] = "round-robin pages (split r: pages r, r+n, ...)"
    if args.partial_bf16:
        line["config"]["partial_dtype"] = "bf16 partial outputs, float32 LSE"
    line["tail_idle"] = _tail_idle(prob, params, dev)
    line["partial_state_bytes"] = int(att.plan.num_states) * spec.head_dim_v * (2 if args.partial_bf16 else 4)
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        sampler = OracleSampler(wl)
        gbs, rows, spent = sampler.run(args.cpu_seconds)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": sampler.threads, "kind": "oracle",
                                "sample": f"{rows} query rows of {len(sampler.items)} of {sampler.total_groups} "
                                          f"(request, KV head) groups, {spent:.1f} s of CPU work"}
    if not (args.no_configs or subset or args.interleave or args.partial_bf16):
        # the other configurations, one sub-record each (after the main line's memory is freed)
        del att, out, lse, tens, prob, h_q, h_out, h_lse
        torch.cuda.empty_cache()
        sub_steps = max(5, min(args.steps, args.config_steps))
        line["configs"] = [_sub_record(n, dev, sub_steps, args.warmup) for n in SUB_CONFIGS if n != spec.name]
        line["gpu_launches_configs"] = sum(r["gpu_launches"] for r in line["configs"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.CONFIG_ORDER)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=5.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--select", default="",
                    help="comma-separated request indices to keep (small cases for profiling; not a bench line)")
    ap.add_argument("--interleave", action="store_true",
                    help="round-robin interleaved splits (Helix staggered KV placement; not a bench line "
                         "of the five configurations)")
    ap.add_argument("--batch", type=int, default=0,
                    help="keep only the first N requests (small cases for profiling; not a bench line)")
    ap.add_argument("--max-len", type=int, default=0,
                    help="cut every history to at most N tokens (small cases for profiling; not a bench line)")
    ap.add_argument("--partial-bf16", action="store_true",
                    help="store partial outputs as bf16 (LSE float32); not a bench line of the five configurations")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration sub-records")
    ap.add_argument("--config-steps", type=int, default=30,
                    help="timed calls per configuration sub-record (at most --steps)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
