"""splitkv_decode_static: the decode entry point for callers that cannot
allocate device memory (its scratch is a fixed static array inside the
library).  Collected last on purpose, so that a failure here leaves every
other test already run.

Checked through the C ABI against the ordinary splitkv_decode (with its own
workspace) on the same inputs, within the bf16 output tolerance used by the
parity tests, on two calls in a row; and a plan too large for the array is
refused on the host before anything is enqueued.
"""
import dataclasses

import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import workloads as W
from tests.gpu_util import check_lse, check_output, device_problem, to_np


def _small_case():
    spec = dataclasses.replace(W.get_config("llama405b_gqa_decode"), batch=5, num_q_heads=32, num_kv_heads=4,
                               split="uniform:4", seed=29)
    return W.build_workload(spec, seq_lens=[1, 64, 999, 4096, 2500])


@pytest.mark.gpu
def test_static_scratch_decode_matches_workspace_decode_twice():
    wl = _small_case()
    prob, _ = device_problem(wl)
    params = skv.plan_params("uniform", uniform_splits=4)
    att = skv.SplitKVAttention(prob, params)
    ref_out, ref_lse = att.decode()
    torch.cuda.synchronize()
    att.check_device_error()
    plan = skv.splitkv_plan(prob, params)
    assert plan.workspace_bytes <= (32 << 20)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        skv.splitkv_decode_static(prob, plan, out, lse, err)
        torch.cuda.synchronize()
        st, raw = skv.read_device_error(err)
        assert st == skv.OK, (call, hex(raw))
        check_output(to_np(out), to_np(ref_out), "bf16", f"static call {call}")
        check_lse(to_np(lse), to_np(ref_lse), f"static lse call {call}")


def test_static_scratch_rejects_plans_larger_than_the_array():
    # host-side check: needs no GPU
    spec = W.get_config("mixed_chunked_prefill")
    wl = W.build_workload(spec)
    q = torch.zeros(1, dtype=torch.bfloat16)
    k = torch.zeros(wl.num_pages, 1, dtype=torch.bfloat16)
    prob = skv.AttentionProblem(
        q=q, k_cache=k, v_cache=k, page_table=torch.from_numpy(wl.page_table),
        seq_lens=torch.from_numpy(wl.seq_lens), qo_indptr=torch.from_numpy(wl.qo_indptr),
        num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads, head_dim_qk=spec.head_dim_qk,
        head_dim_v=spec.head_dim_v, page_size=spec.page_size, scale=spec.scale)
    plan = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=8))
    assert plan.workspace_bytes > (32 << 20)
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_decode_static(prob, plan, q, None)
    assert e.value.status == skv.ERR_WORKSPACE
    assert "static array" in str(e.value)
