"""Task trace on the GPU (splitkv_plan_params.trace = 1): every traced unit of
a launch has one well-formed record -- its id in place, its kind, a start no
later than its end, an SM id of this device -- all inside the launch's own
span; a reduction starts only after some attention task has ended; a second
launch rewrites every record; and tracing leaves the results unchanged."""
import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from tests.gpu_util import check_lse, check_output, device_problem, spec_like, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "gqa_engine": ("llama405b_gqa_decode", dict(num_q_heads=32, num_kv_heads=2), [3000, 1, 700, 4096], None, 5),
    "chunk_and_engine": ("mixed_chunked_prefill", dict(num_q_heads=16, num_kv_heads=2), [600, 90, 2100],
                         [100, 1, 1], 3),
    "pair_and_engine": ("spec_decode_q16", dict(num_q_heads=8, num_kv_heads=2), [3000, 40, 700, 5000],
                        [16, 1, 9, 16], 3),
    "mla": ("deepseek_mla_decode", {}, [200, 777, 3000, 64], None, 4),
}


@pytest.mark.parametrize("name", list(CASES))
def test_trace_records_one_well_formed_record_per_unit(name):
    base, over, lens, q_lens, splits = CASES[name]
    spec = spec_like(base, batch=len(lens), split=f"uniform:{splits}", seed=81, **over)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, skv.plan_params("uniform", uniform_splits=splits, trace=1))
    plan = att.plan
    n = plan.trace_records
    assert n > 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    out, lse = att.decode()
    e1.record()
    torch.cuda.synchronize()
    att.check_device_error()
    rec = skv.trace_read(plan, att.workspace)
    launch_ns = e0.elapsed_time(e1) * 1e6
    kinds = rec["kind"]
    if name == "mla":
        assert (kinds == skv.TRACE_MLA_ITEM).all() and n == 2 * plan.num_tasks
        assert (rec["id"] == np.arange(n)).all()
    else:
        # engine tasks, reduction items, chunk-tile tasks, paired-tile tasks
        n_chunk, n_pair = plan.num_chunk_tasks, plan.num_pair_tasks
        n_att = plan.num_tasks - n_chunk - n_pair
        assert (kinds[:n_att] == skv.TRACE_ATTENTION).all()
        assert (rec["id"][:n_att] == np.arange(n_att)).all()
        if n_pair:
            assert (kinds[n - n_pair:] == skv.TRACE_PAIR).all()
            assert (rec["id"][n - n_pair:] == np.arange(n_pair)).all()
        if n_chunk:
            assert (kinds[n - n_pair - n_chunk:n - n_pair] == skv.TRACE_CHUNK).all()
            assert (rec["id"][n - n_pair - n_chunk:n - n_pair] == np.arange(n_chunk)).all()
        red = kinds == skv.TRACE_REDUCTION
        assert red.sum() == n - n_att - n_chunk - n_pair > 0
        assert (rec["id"][red] == np.arange(red.sum())).all()
        # a reduction waits for its request's tasks: none starts before the first task ends
        work = np.isin(kinds, (skv.TRACE_ATTENTION, skv.TRACE_CHUNK, skv.TRACE_PAIR))
        assert rec["start_ns"][red].min() >= rec["end_ns"][work].min()
    assert (rec["start_ns"] > 0).all() and (rec["end_ns"] >= rec["start_ns"]).all()
    assert ((rec["sm"] >= 0) & (rec["sm"] < sms)).all() and (rec["cta"] >= 0).all()
    span = int(rec["end_ns"].max() - rec["start_ns"].min())
    assert span <= 1.5 * launch_ns + 50_000, (span, launch_ns)
    st = skv.trace_tail_idle(rec, kinds=tuple(set(int(k) for k in kinds)), num_sms=sms)
    assert 0.0 <= st["tail_idle_frac"] < 1.0
    # a second launch rewrites every record
    att.decode(out, lse)
    torch.cuda.synchronize()
    rec2 = skv.trace_read(plan, att.workspace)
    assert rec2["start_ns"].min() >= rec["end_ns"].max()
    # tracing leaves the results unchanged
    ref_o, ref_l = oracle.problem_from_workload(wl).attention_rows()
    check_output(to_np(out), ref_o.reshape(out.shape), spec.dtype, f"{name} traced out")
    check_lse(to_np(lse), ref_l.reshape(lse.shape), f"{name} traced lse")
