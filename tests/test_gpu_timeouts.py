"""Bounded waits expire into an error status, not a hang or a fault.

With the test hook on, each persistent kernel's task claimer withholds every
task: nothing ever signals the other roles, so their bounded waits run out
(about 2 s each), the launch records SPLITKV_ERR_TIMEOUT in its device error
word and returns.  The context stays usable: the next launch, hook off, is
checked against the oracle.
"""
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from tests.gpu_util import check_lse, check_output, device_problem, plan_params_for, spec_like, to_np

pytestmark = pytest.mark.gpu


def _case(name):
    if name == "gqa_engine":
        spec = spec_like("llama405b_gqa_decode", batch=3, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=71)
        return W.build_workload(spec, seq_lens=[300, 1000, 65])
    if name == "chunk_tiles":
        spec = spec_like("mixed_chunked_prefill", batch=2, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=72)
        return W.build_workload(spec, seq_lens=[600, 90], q_lens=[100, 1])
    if name == "pair_tiles":
        spec = spec_like("spec_decode_q16", batch=2, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=74)
        return W.build_workload(spec, seq_lens=[600, 90], q_lens=[8, 1])
    spec = spec_like("deepseek_mla_decode", batch=2, split="uniform:2", seed=73)
    return W.build_workload(spec, seq_lens=[700, 130])


@pytest.mark.parametrize("name", ["gqa_engine", "chunk_tiles", "pair_tiles", "mla"])
def test_withheld_tasks_time_out_and_context_survives(name):
    wl = _case(name)
    spec = wl.spec
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    if name == "chunk_tiles":
        assert att.plan.num_chunk_tasks > 0
    if name == "pair_tiles":
        assert att.plan.num_pair_tasks > 0
    expected_path = 2 if name == "mla" else 1
    assert att.plan.kernel_path == expected_path
    skv.read_device_error(att.error_word, clear=True)
    skv.debug_set_inject(1)
    try:
        att.decode()
        torch.cuda.synchronize()
    finally:
        skv.debug_set_inject(0)
    st, raw = skv.read_device_error(att.error_word, clear=True)
    assert st == skv.ERR_TIMEOUT, (st, hex(raw))

    # the context and the workspace are usable: a normal launch matches the oracle
    out, lse = att.decode()
    torch.cuda.synchronize()
    att.check_device_error()
    po = oracle.problem_from_workload(wl)
    ref_o, ref_l = po.attention_rows()
    check_output(to_np(out).reshape(ref_o.shape), ref_o, spec.dtype, f"{name} after timeout")
    check_lse(to_np(lse).reshape(-1), ref_l, f"{name} lse after timeout")

