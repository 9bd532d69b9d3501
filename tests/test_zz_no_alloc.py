"""splitkv_decode_static: the decode entry point for callers that cannot
allocate device memory (its scratch is a fixed static array inside the
library).  Collected last on purpose, so that a failure here leaves every
other test already run.

Checked through the C ABI against the ordinary splitkv_decode (with its own
workspace) on the same inputs, within the output tolerance used by the parity
tests, on two calls in a row, for the kernel paths that use scratch: the
fused GQA engine, the MLA tcgen05 kernel with its separate merge (which reads
the partial-state index from the array), and the chunk tiles and the paired
tiles ahead of the engine.  One call per case is also checked against the float64 oracle, and
the path without a caller-supplied error word is exercised.  On the host: a
plan too large for the array, and arguments that fail their checks, are
refused before anything is enqueued.
"""
import dataclasses

import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from tests.gpu_util import check_lse, check_output, device_problem, to_np

CASES = {
    # GQA decode rows on the fused engine (path 1, uniform splits)
    "gqa_engine": (dict(base="llama405b_gqa_decode", batch=5, num_q_heads=32, num_kv_heads=4, seed=29),
                   [1, 64, 999, 4096, 2500], None, 4),
    # MLA tcgen05 partial kernel, then the merge kernel (path 2)
    "mla": (dict(base="deepseek_mla_decode", batch=3, seed=30), [200, 777, 3000], None, 3),
    # chunked-prefill rows on the chunk tiles, decode rows on the engine
    "chunk_tiles": (dict(base="mixed_chunked_prefill", batch=3, num_q_heads=16, num_kv_heads=2, seed=31),
                    [600, 90, 2000], [100, 1, 1], 2),
    # speculative blocks on the paired tiles, decode rows on the engine
    "pair_tiles": (dict(base="spec_decode_q16", batch=3, num_q_heads=16, num_kv_heads=2, seed=32),
                   [600, 90, 2000], [16, 1, 5], 2),
}


def _case(name):
    over, lens, q_lens, splits = CASES[name]
    over = dict(over)
    base = over.pop("base")
    spec = dataclasses.replace(W.get_config(base), split=f"uniform:{splits}", **over)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    return spec, wl, skv.plan_params("uniform", uniform_splits=splits)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_decode_matches_workspace_decode_twice(name):
    spec, wl, params = _case(name)
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, params)
    ref_out, ref_lse = att.decode()
    torch.cuda.synchronize()
    att.check_device_error()
    plan = skv.splitkv_plan(prob, params)
    assert plan.workspace_bytes <= (32 << 20)
    if name == "mla":
        assert plan.kernel_path == 2
    if name == "chunk_tiles":
        assert plan.num_chunk_tasks > 0
    if name == "pair_tiles":
        assert plan.num_pair_tasks > 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        skv.splitkv_decode_static(prob, plan, out, lse, err)
        torch.cuda.synchronize()
        st, raw = skv.read_device_error(err)
        assert st == skv.OK, (call, hex(raw))
        check_output(to_np(out), to_np(ref_out), spec.dtype, f"static call {call}")
        check_lse(to_np(lse), to_np(ref_lse), f"static lse call {call}")
        outs.append((to_np(out), to_np(lse)))
    # the first call against the float64 oracle
    ref_o, ref_l = oracle.problem_from_workload(wl).attention_rows()
    check_output(outs[0][0], ref_o.reshape(outs[0][0].shape), spec.dtype, "static vs oracle")
    check_lse(outs[0][1], ref_l.reshape(outs[0][1].shape), "static lse vs oracle")


@pytest.mark.gpu
def test_static_scratch_without_an_error_word():
    # device errors go to the array's own word, read through splitkv_read_static_device_error
    spec, wl, params = _case("gqa_engine")
    prob, _ = device_problem(wl)
    plan = skv.splitkv_plan(prob, params)
    out = torch.empty(wl.total_q, spec.num_q_heads, spec.head_dim_v, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(wl.total_q, spec.num_q_heads, dtype=torch.float32, device="cuda")
    skv.splitkv_decode_static(prob, plan, out, lse, None)
    st, raw = skv.read_static_device_error()
    assert st == skv.OK and raw == 0
    ref_o, ref_l = oracle.problem_from_workload(wl).attention_rows()
    check_output(to_np(out), ref_o.reshape(out.shape), "bf16", "static, no error word")
    check_lse(to_np(lse), ref_l.reshape(lse.shape), "static lse, no error word")
    # an out-of-range page id is recorded in the array's word and cleared on request
    wl.page_table[2, 1] = wl.num_pages + 5
    prob2, _ = device_problem(wl)
    plan2 = skv.splitkv_plan(prob2, params)
    skv.splitkv_decode_static(prob2, plan2, out, lse, None)
    st, raw = skv.read_static_device_error(clear=True)
    assert st == skv.ERR_DEVICE_CHECK, hex(raw)
    st, raw = skv.read_static_device_error()
    assert st == skv.OK and raw == 0


def _host_problem(spec, wl, num_q_heads=None):
    q = torch.zeros(1, dtype=torch.bfloat16)
    k = torch.zeros(wl.num_pages, 1, dtype=torch.bfloat16)
    return skv.AttentionProblem(
        q=q, k_cache=k, v_cache=k, page_table=torch.from_numpy(wl.page_table),
        seq_lens=torch.from_numpy(wl.seq_lens), qo_indptr=torch.from_numpy(wl.qo_indptr),
        num_q_heads=num_q_heads or spec.num_q_heads, num_kv_heads=spec.num_kv_heads, head_dim_qk=spec.head_dim_qk,
        head_dim_v=spec.head_dim_v, page_size=spec.page_size, scale=spec.scale), q


def test_static_scratch_rejects_plans_larger_than_the_array():
    # host-side check: needs no GPU
    spec = W.get_config("mixed_chunked_prefill")
    wl = W.build_workload(spec)
    prob, q = _host_problem(spec, wl)
    plan = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=8))
    assert plan.workspace_bytes > (32 << 20)
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_decode_static(prob, plan, q, None)
    assert e.value.status == skv.ERR_WORKSPACE
    assert "static array" in str(e.value)


def test_static_scratch_checks_arguments_before_touching_the_device():
    # a problem that does not match the plan is refused with INVALID_ARG by the host
    # checks, before the array's address is looked up or anything is queued (on a
    # machine without a GPU any device step would fail with a CUDA error instead)
    spec, wl, params = _case("gqa_engine")
    prob, q = _host_problem(spec, wl)
    plan = skv.splitkv_plan(prob, params)
    other, _ = _host_problem(spec, wl, num_q_heads=spec.num_q_heads * 2)
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_decode_static(other, plan, q, None)
    assert e.value.status == skv.ERR_INVALID_ARG and "differs from the plan" in str(e.value)
