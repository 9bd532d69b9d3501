"""Task trace on the host: record counts of traced plans, argument checks,
and the tail-idle arithmetic (LiquidCP Section 3: an SM's wait after its last
task in a stage until the stage finishes, summed over SMs, divided by total
SM-time) on synthetic traces with hand-computed answers."""
import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import workloads as W
from tests.test_abi_cpu import _cpu_problem


def _recs(rows):
    r = np.zeros(len(rows), dtype=skv._lib.TRACE_DTYPE)
    for k, (start, end, sm, kind) in enumerate(rows):
        r[k] = (start, end, k, sm, kind, sm)
    return r


def test_tail_idle_two_sms_by_hand():
    # SM 0 busy 0..100 then 100..400; SM 1 busy 50..250: the stage spans 0..400,
    # SM 1 waits 150, SM 0 waits 0 -> 150 / (2 * 400)
    r = _recs([(0, 100, 0, 0), (100, 400, 0, 0), (50, 250, 1, 0)])
    st = skv.trace_tail_idle(r, kinds=(0,))
    assert st["records"] == 3 and st["sms"] == 2
    assert st["begin_ns"] == 0 and st["end_ns"] == 400
    assert st["tail_idle_sm_ns"] == 150
    assert st["tail_idle_frac"] == pytest.approx(150 / 800)


def test_tail_idle_counts_sms_without_records_and_selects_kinds():
    # four SMs requested, two appear: the other two wait for the whole stage
    r = _recs([(10, 110, 0, 0), (10, 60, 3, 0), (0, 1000, 1, 2)])
    st = skv.trace_tail_idle(r, kinds=(0,), num_sms=4)
    assert st["records"] == 2 and st["sms"] == 4
    assert st["tail_idle_sm_ns"] == 0 + 50 + 2 * 100
    assert st["tail_idle_frac"] == pytest.approx(250 / 400)
    # the other kind alone: one SM, no tail
    st2 = skv.trace_tail_idle(r, kinds=(2,))
    assert st2["records"] == 1 and st2["tail_idle_frac"] == 0.0


def test_tail_idle_matches_a_direct_computation_on_random_traces():
    rng = np.random.default_rng(5)
    for _ in range(20):
        n, sms = int(rng.integers(1, 300)), int(rng.integers(1, 20))
        start = rng.integers(0, 10_000, n)
        end = start + rng.integers(0, 5_000, n)
        sm = rng.integers(0, sms, n)
        r = _recs(list(zip(start, end, sm, np.zeros(n, dtype=int))))
        st = skv.trace_tail_idle(r, kinds=(0,), num_sms=sms)
        b, e = start.min(), end.max()
        want = sum(e - (end[sm == s].max() if (sm == s).any() else b) for s in range(sms))
        assert st["tail_idle_sm_ns"] == pytest.approx(float(want))
        assert st["tail_idle_frac"] == pytest.approx(want / (sms * (e - b)) if e > b else 0.0)


def test_tail_idle_rejects_bad_traces():
    with pytest.raises(skv.SplitKVError):
        skv.trace_tail_idle(_recs([(10, 5, 0, 0)]), kinds=(0,))          # ends before it starts
    with pytest.raises(skv.SplitKVError):
        skv.trace_tail_idle(_recs([(0, 5, 7, 0)]), kinds=(0,), num_sms=4)  # SM outside [0, 4)
    with pytest.raises(skv.SplitKVError):
        skv.trace_tail_idle(_recs([(0, 5, 0, 1)]), kinds=(0,))          # nothing selected


@pytest.mark.parametrize("name,expect", [
    ("llama405b_gqa_decode", "tasks+red"),
    ("mixed_chunked_prefill", "tasks+red"),
    ("deepseek_mla_decode", "2tasks"),
    ("tiny_fp32_gqa", "none"),
])
def test_traced_plan_record_counts(name, expect):
    spec = W.get_config(name)
    wl, prob = _cpu_problem(spec)
    n = W.uniform_splits(spec) or 4
    plain = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=n, num_ctas=152))
    traced = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=n, num_ctas=152, trace=1))
    assert plain.trace_records == 0
    if expect == "none":
        assert traced.trace_records == 0 and traced.workspace_bytes == plain.workspace_bytes
        return
    if expect == "2tasks":
        assert traced.trace_records == 2 * traced.num_tasks
    else:
        # engine tasks + chunk tasks + one reduction item per run of rows of every split request
        assert traced.trace_records > traced.num_tasks
    assert traced.workspace_bytes >= plain.workspace_bytes + 32 * traced.trace_records
    with pytest.raises(skv.SplitKVError):
        skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=n, trace=2))
    with pytest.raises(skv.SplitKVError):
        skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=n, reserved=1))
    with pytest.raises(skv.SplitKVError):
        skv.trace_read(plain, torch.zeros(plain.workspace_bytes, dtype=torch.uint8))
