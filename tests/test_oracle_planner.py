"""Pins for the oracle's critical-wave planner (LiquidCP Section 5.2, Eqs.
5-6, Figure 8, Appendix A.2).

Pins: the three plan scores printed in Figure 8 and the plan the search
selects there; closed forms of Eq. 5/6 for one task and for one full wave;
the rho floor; the adoption margin; determinism; the tie-break order.
"""
import json
import os

import pytest

from oracle import planner as P

HERE = os.path.dirname(os.path.abspath(__file__))
FIG8 = json.load(open(os.path.join(HERE, "golden", "liquidcp_fig8.json")))


def _fig8():
    g = FIG8["params"]
    p = P.ModelParams(num_ctas=g["num_ctas"], rho=g["rho"], delta_attn=g["delta_attn"],
                      delta_red=g["delta_red"], gamma=g["gamma"])
    seqs = [P.SeqSpec(tiles=t, vectors=g["vectors_per_reduction"]) for t in FIG8["histories_tiles"]]
    return p, seqs


@pytest.mark.parametrize("entry", FIG8["plans"], ids=lambda e: e["name"])
def test_figure8_scores(entry):
    p, seqs = _fig8()
    assert P.simulate(seqs, entry["splits"], p).score == pytest.approx(entry["score"], abs=1e-9)


def test_figure8_search_selects_critical_wave_plan():
    p, seqs = _fig8()
    plan = P.plan(seqs, p)
    assert plan.splits == FIG8["selected"]
    assert plan.score == pytest.approx(104.0)
    assert plan.base_score == pytest.approx(152.0)


def test_single_task_closed_form():
    # one task, K CTAs: it runs alone at tau = max(rho, 1/K), then one reduction
    for K, rho in [(4, 0.75), (8, 0.1), (132, 0.43)]:
        p = P.ModelParams(num_ctas=K, rho=rho, delta_attn=3.0, delta_red=2.0, gamma=0.5)
        r = P.simulate([P.SeqSpec(tiles=10, vectors=1)], [1], p)
        assert r.attn_end == pytest.approx(13.0 * max(rho, 1.0 / K))
        assert r.score == pytest.approx(13.0 * max(rho, 1.0 / K) + 2.0 + 0.5)


def test_full_wave_closed_form():
    # K equal tasks on K CTAs run at tau = 1: all finish at c_attn
    K = 6
    p = P.ModelParams(num_ctas=K, rho=0.3, delta_attn=2.0, delta_red=1.0, gamma=1.0, warps_per_cta=1)
    seqs = [P.SeqSpec(tiles=10 * K)]
    r = P.simulate(seqs, [K], p)
    assert r.attn_end == pytest.approx(12.0)
    assert r.score == pytest.approx(12.0 + 1.0 + 1.0 * K)
    # a second wave of one task runs alone at the rho floor
    r = P.simulate([P.SeqSpec(tiles=10 * (K + 1))], [K + 1], p)
    assert r.attn_end == pytest.approx(12.0 + 12.0 * 0.3)


def test_adoption_margin_keeps_nosplit():
    # a split plan that is better by less than 10% is not adopted
    p = P.ModelParams(num_ctas=2, rho=0.5, delta_attn=0.0, delta_red=0.0, gamma=0.0, warps_per_cta=1)
    seqs = [P.SeqSpec(tiles=10), P.SeqSpec(tiles=9)]
    plan = P.plan(seqs, p)
    assert plan.splits == [1, 1]


def test_limits_and_min_splits():
    p = P.ModelParams(num_ctas=4)
    seqs = [P.SeqSpec(tiles=3), P.SeqSpec(tiles=100)]
    plan = P.plan(seqs, p, min_splits=8, max_splits=16)
    assert plan.base_splits == [3, 8]
    assert all(lo <= s <= hi for lo, s, hi in zip(plan.base_splits, plan.splits, plan.limits))
    assert plan.limits[0] == 3


def test_lpt_order_only_for_split_decode_only():
    p = P.ModelParams(num_ctas=2, delta_attn=0)
    seqs = [P.SeqSpec(tiles=2), P.SeqSpec(tiles=9)]
    q = P.attention_queue(seqs, [1, 2], p)
    assert [w for w, _ in q] == [5, 4, 2]
    q = P.attention_queue(seqs, [1, 1], p)
    assert [w for w, _ in q] == [2, 9]
    mixed = [P.SeqSpec(tiles=2), P.SeqSpec(tiles=9, q_len=64)]
    q = P.attention_queue(mixed, [2, 1], p)
    assert [b for _, b in q] == [1, 0, 0]


def test_tie_break_prefers_earlier_attention_then_fewer_tasks():
    a = (10.0, 8.0, 5, 3)
    assert P._cmp_key(a, (10.0, 9.0, 1, 1)) < 0
    assert P._cmp_key(a, (10.0, 8.0, 6, 1)) < 0
    assert P._cmp_key(a, (10.0, 8.0, 5, 4)) < 0
    assert P._cmp_key(a, (10.0 + 1e-13, 8.0, 5, 3)) == 0


def test_run_length_rule():
    p = P.ModelParams(num_ctas=4, warps_per_cta=12)   # 48 warps -> need >= 38.4 tasks
    seqs = [P.SeqSpec(tiles=5, vectors=8 * 16) for _ in range(10)]   # 1280 vectors
    assert P.run_length(seqs, 8, p) == 32     # candidates 32, 16, 8, 1 -> 1280/32 = 40 tasks
    assert P.run_length(seqs[:1], 8, p) == 1


def test_deterministic():
    p = P.ModelParams(num_ctas=16, rho=0.43, delta_attn=8, delta_red=2.5, gamma=0.47)
    seqs = [P.SeqSpec(tiles=t, tasks_per_split=2, vectors=16) for t in (300, 17, 80, 2, 150, 64)]
    a = P.plan(seqs, p, q_heads=8)
    b = P.plan(seqs, p, q_heads=8)
    assert a == b
