"""bf16 partial states (splitkv_plan_params.partial_dtype = BF16): the
precision LiquidCP Section 7 reports vLLM and MegaDCP exchanging partial
attention states in (SGLang exchanges float32).  Every kernel that writes
partial states (GQA engine, chunk tiles, MLA tcgen05, CUDA-core path) and both
readers (the engine's reduction phase, merge_states_typed) are compared with
the float64 oracle on the same seeded inputs.

Tolerances:
  * each partial output o_r is one bf16 rounding of a float32 value, so it is
    held to the bf16 output bound (2e-3 + 1e-2 |ref|), LSE to 1e-3;
  * a merged output o = sum_r w_r o_r (w_r = exp(lse_r - lse)) carries each
    partial's rounding, at most 2^-8 |o_r| (bf16 keeps 8 significant bits),
    weighted by w_r: the bound is the path's output bound plus
    2^-8 sum_r w_r |o_r|, computed per element from the oracle's partials.
"""
import math

import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from tests.gpu_util import (BF16_ATOL, BF16_RTOL, FP32_ATOL, check_lse, check_output, device_problem,
                            oracle_partials, spec_like, to_np)

pytestmark = pytest.mark.gpu

BF16_U = 2.0 ** -8


def merged_bound(ref, dtype, plan, ro, rl):
    """Per-element tolerance of a merged output built from bf16 partial states."""
    indptr = plan.state_indptr()
    ro = np.abs(np.asarray(ro, dtype=np.float64))
    rl = np.asarray(rl, dtype=np.float64)
    rows = len(indptr) - 1
    extra = np.zeros((rows, ro.shape[1]))
    for x in range(rows):
        s0, s1 = indptr[x], indptr[x + 1]
        l = rl[s0:s1]
        fin = np.isfinite(l)
        if not fin.any():
            continue
        m = l[fin].max()
        lse = m + math.log(np.exp(l[fin] - m).sum())
        w = np.where(fin, np.exp(np.where(fin, l, 0.0) - lse), 0.0)
        extra[x] = BF16_U * (w[:, None] * ro[s0:s1]).sum(0)
    ref = np.asarray(ref, dtype=np.float64).reshape(rows, -1)
    base = FP32_ATOL if dtype == "f32" else BF16_ATOL + BF16_RTOL * np.abs(ref)
    return base + extra


def check_merged(out, ref, lim, what):
    out = np.asarray(out, dtype=np.float64).reshape(lim.shape)
    ref = np.asarray(ref, dtype=np.float64).reshape(lim.shape)
    assert np.isfinite(out).all(), f"{what}: non-finite values"
    bad = np.abs(out - ref) > lim
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; max err {np.abs(out - ref).max():.3e}"


CASES = {
    # (base config, overrides, seq_lens, q_lens, splits, expected kernel path)
    "gqa_engine_decode": ("llama405b_gqa_decode", dict(num_q_heads=32, num_kv_heads=2), [1, 63, 700, 4096, 2500],
                          None, 5, 1),
    "gqa_engine_wide_rows": ("spec_decode_q16", dict(num_q_heads=16, num_kv_heads=2), [5000, 40, 160], [3, 4, 2],
                             3, 1),
    "pair_tiles": ("spec_decode_q16", dict(num_q_heads=8, num_kv_heads=2), [5000, 40, 16], [16, 4, 16], 3, 1),
    "chunk_tiles": ("mixed_chunked_prefill", dict(num_q_heads=16, num_kv_heads=2), [600, 90, 2100], [100, 1, 70],
                    3, 1),
    "mla_tcgen05": ("deepseek_mla_decode", {}, [1, 200, 777, 3000], [1, 1, 2, 1], 4, 2),
    "mla_fp8_copy": ("deepseek_mla_fp8_decode", {}, [1, 200, 777, 3000], [1, 1, 2, 1], 4, 2),
    "cuda_core_fp32": ("tiny_fp32_gqa", {}, [37, 128, 300, 513], None, 4, 0),
    "cuda_core_mla": ("deepseek_mla_decode", dict(num_q_heads=16), [9, 200, 1000], None, 3, 0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bf16_partial_states(name):
    base, over, lens, q_lens, splits, path = CASES[name]
    spec = spec_like(base, batch=len(lens), split=f"uniform:{splits}", seed=71, **over)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, skv.plan_params("uniform", uniform_splits=splits, partial_dtype=skv.BF16))
    assert att.plan.partial_dtype == torch.bfloat16 and att.plan.kernel_path == path
    if name == "chunk_tiles":
        assert att.plan.num_chunk_tasks > 0
    if name == "pair_tiles":
        assert att.plan.num_pair_tasks > 0
    if name == "gqa_engine_wide_rows":
        assert att.plan.num_pair_tasks == 0 and att.plan.num_chunk_tasks == 0
    po = oracle.problem_from_workload(wl)
    ref_o, ref_l = po.attention_rows()
    ro, rl = oracle_partials(po, wl, att.plan)
    lim = merged_bound(ref_o, spec.dtype, att.plan, ro, rl)

    o_part, lse_part = att.partial()
    torch.cuda.synchronize()
    att.check_device_error()
    assert o_part.dtype == torch.bfloat16
    check_output(to_np(o_part)[:len(rl)], ro, "bf16", f"{name} bf16 partial o")
    check_lse(to_np(lse_part)[:len(rl)], rl, f"{name} partial lse")

    for run in (att.decode, att.two_stage):
        out, lse = run()
        torch.cuda.synchronize()
        att.check_device_error()
        check_merged(to_np(out), ref_o, lim, f"{name} {run.__name__} out")
        check_lse(to_np(lse).reshape(-1), ref_l, f"{name} {run.__name__} lse")


def test_bf16_partials_planner_mla_full_size_sampled():
    """The MLA configuration (the one with the most partial states) at full size with
    planner splits and bf16 partial states, on sampled requests."""
    spec = W.get_config("deepseek_mla_decode")
    wl = W.build_workload(spec)
    prob, _ = device_problem(wl)
    lo, hi = W.planner_split_range(spec)
    att = skv.SplitKVAttention(prob, skv.plan_params("critical_wave", min_splits=lo, max_splits=hi,
                                                     partial_dtype=skv.BF16))
    assert att.plan.kernel_path == 2
    out, lse = att.decode()
    torch.cuda.synchronize()
    att.check_device_error()
    out, lse = to_np(out), to_np(lse)
    n_spl = att.plan.splits()
    rng = np.random.default_rng(72)
    picks = sorted({int(np.argmax(wl.seq_lens)), int(np.argmax(n_spl))} | set(rng.choice(spec.batch, 6, replace=False)))
    for b in picks:
        sub = oracle.subproblem_for_group(wl, b, 0)
        ro_full, rl_full = sub.attention_rows()
        ranges = att.plan.split_ranges(b)
        rows5 = np.array([(0, 0, h, kb, ke) for h in range(spec.num_q_heads) for (kb, ke) in ranges], dtype=np.int32)
        po, pl = sub.partial_rows(rows5)
        n = len(ranges)
        extra = np.zeros_like(ro_full)
        for h in range(spec.num_q_heads):
            l = pl[h * n:(h + 1) * n]
            fin = np.isfinite(l)
            w = np.where(fin, np.exp(np.where(fin, l, 0.0) - rl_full[h]), 0.0)
            extra[h] = BF16_U * (w[:, None] * np.abs(po[h * n:(h + 1) * n])).sum(0)
        t0 = int(wl.qo_indptr[b])
        lim = BF16_ATOL + BF16_RTOL * np.abs(ro_full) + extra
        check_merged(out[t0], ro_full, lim, f"mla bf16 partials b={b}")
        check_lse(lse[t0], rl_full, f"mla bf16 partials lse b={b}")
