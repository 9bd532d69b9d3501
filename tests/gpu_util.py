"""Shared helpers of the GPU parity tests: seeded workloads on both sides,
the oracle on the host, the CUDA path through the C ABI, and the tolerance
checks stated for this path (fp32 inputs: max |err| <= 1e-5; bf16 inputs:
|err| <= 2e-3 + 1e-2 |ref|; LSE: |err| <= 1e-3)."""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W

FP32_ATOL = 1e-5
BF16_ATOL, BF16_RTOL = 2e-3, 1e-2
LSE_ATOL = 1e-3


def spec_like(base: str, **over) -> W.WorkloadSpec:
    return dataclasses.replace(W.get_config(base), **over)


def device_problem(wl: W.Workload, dev="cuda"):
    t = wl.device_tensors(dev)
    s = wl.spec
    prob = skv.AttentionProblem(
        q=t["q"], k_cache=t["k"], v_cache=t["v"], page_table=t["page_table"], seq_lens=t["seq_lens"],
        qo_indptr=t["qo_indptr"], num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads,
        head_dim_qk=s.head_dim_qk, head_dim_v=s.head_dim_v, page_size=s.page_size, scale=s.scale,
        kind=s.kind, seq_lens_host=wl.seq_lens, qo_indptr_host=wl.qo_indptr,
        k_scale=s.k_scale if s.kv_fp8 else None, v_scale=s.v_scale if s.kv_fp8 else None)
    return prob, t


def plan_params_for(spec: W.WorkloadSpec, **over):
    n = W.uniform_splits(spec)
    if n is not None and "min_splits" not in over:
        kw = dict(uniform_splits=n)
        kw.update(over)
        return skv.plan_params("uniform", **kw)
    lo, hi = W.planner_split_range(spec) or (1, 64)
    kw = dict(min_splits=lo, max_splits=hi)
    kw.update(over)
    return skv.plan_params("critical_wave", **kw)


def check_output(out: np.ndarray, ref: np.ndarray, dtype: str, what: str = "out"):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (what, out.shape, ref.shape)
    assert np.isfinite(out).all(), f"{what}: non-finite values"
    err = np.abs(out - ref)
    if dtype == "f32":
        bad = err > FP32_ATOL
        lim = FP32_ATOL
    else:
        lim = BF16_ATOL + BF16_RTOL * np.abs(ref)
        bad = err > lim
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"max err {err.max():.3e}; first {idx.tolist()}")


def check_lse(lse: np.ndarray, ref: np.ndarray, what: str = "lse"):
    lse = np.asarray(lse, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert (np.isneginf(lse) == inf_ref).all(), f"{what}: -inf pattern differs"
    fin = ~inf_ref
    if fin.any():
        err = np.abs(lse[fin] - ref[fin]).max()
        assert err <= LSE_ATOL, f"{what}: max err {err:.3e}"


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_partials(prob_o: oracle.Problem, wl: W.Workload, plan: skv.Plan):
    """Oracle partial states laid out like the plan's o_part / lse_part: contiguous
    page-aligned ranges, or for an interleaved plan the round-robin shards of one page
    per block."""
    s = wl.spec
    n_spl = plan.splits()
    if plan.interleaved:
        rows, sets = [], []
        for b in range(wl.spec.batch):
            shards = oracle.interleaved_split_keys(int(wl.seq_lens[b]), s.page_size, int(n_spl[b]))
            for i in range(int(wl.q_lens[b])):
                for h in range(s.num_q_heads):
                    for keys in shards:
                        rows.append((b, i, h))
                        sets.append(keys)
        return prob_o.partial_keysets(np.array(rows, dtype=np.int32), sets)
    rows = []
    for b in range(wl.spec.batch):
        ranges = oracle.split_bounds(int(wl.seq_lens[b]), s.page_size, int(n_spl[b]))
        for i in range(int(wl.q_lens[b])):
            for h in range(s.num_q_heads):
                for (kb, ke) in ranges:
                    rows.append((b, i, h, kb, ke))
    return prob_o.partial_rows(np.array(rows, dtype=np.int32))
