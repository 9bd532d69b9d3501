"""The product planner's final selection over uniform candidates (a rule of
this library with no counterpart on the pages), on the host: splitkv_plan's
split counts equal the oracle restatement (oracle.planner.plan_with_uniform),
and that restatement is pinned by brute force -- its score is the minimum over
the pages' selection and every adoptable uniform plan."""
import random

import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle.planner as OP
import workloads as W


def _gqa_decode_problem(lens, hq=32, hkv=4, page=64):
    spec = W.get_config("llama405b_gqa_decode")
    import dataclasses
    spec = dataclasses.replace(spec, batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, page_size=page)
    wl = W.build_workload(spec, seq_lens=lens)
    q = torch.zeros(1, dtype=torch.bfloat16)
    k = torch.zeros(wl.num_pages, 1, dtype=torch.bfloat16)
    prob = skv.AttentionProblem(
        q=q, k_cache=k, v_cache=k, page_table=torch.from_numpy(wl.page_table), seq_lens=torch.from_numpy(wl.seq_lens),
        qo_indptr=torch.from_numpy(wl.qo_indptr), num_q_heads=hq, num_kv_heads=hkv, head_dim_qk=128,
        head_dim_v=128, page_size=page, scale=spec.scale)
    return spec, wl, prob


@pytest.mark.parametrize("seed", range(24))
def test_product_selection_matches_oracle_and_brute_force(seed):
    rng = random.Random(500 + seed)
    n = rng.randint(1, 10)
    lens = [rng.choice([rng.randint(64, 4096), rng.randint(4096, 131072)]) for _ in range(n)]
    hq, hkv = rng.choice([(32, 4), (64, 8), (16, 2)])
    spec, wl, prob = _gqa_decode_problem(lens, hq, hkv)
    K = rng.choice([16, 38, 76, 152])
    prm = dict(rho=rng.choice([0.43, 0.7, 1.0]), delta_attn=rng.choice([0.0, 4.0, 32.0]),
               delta_red=rng.choice([1.0, 2.5]), gamma=rng.choice([0.47, 2.0]))
    lo, hi = rng.choice([(1, 64), (1, 16), (4, 64)])
    plan = skv.splitkv_plan(prob, skv.plan_params("critical_wave", min_splits=lo, max_splits=hi, num_ctas=K,
                                                  warps_per_cta=7, **prm))
    seqs = [OP.SeqSpec(tiles=-(-L // 64), tasks_per_split=hkv, vectors=hq, q_len=1) for L in lens]
    op = OP.ModelParams(num_ctas=K, warps_per_cta=7, **prm)
    want = OP.plan_with_uniform(seqs, op, q_heads=hq, min_splits=lo, max_splits=hi)
    assert list(plan.splits()) == want.splits
    assert plan.scores()[1] == pytest.approx(want.score, rel=1e-12)
    # brute force: the selection is the lowest score among the pages' selection and the
    # adoptable uniform plans
    pages_sel = OP.plan(seqs, op, q_heads=hq, min_splits=lo, max_splits=hi)
    best = pages_sel.score
    lo_b = [max(1, min(lo, s.tiles)) for s in seqs]
    hi_b = [max(lo_b[b], min(hi, s.tiles)) for b, s in enumerate(seqs)]
    for u in range(2, 65):
        c = [min(hi_b[b], max(lo_b[b], u)) for b in range(n)]
        if u not in OP.UNIFORM_CANDIDATES:
            continue
        sc = OP.simulate(seqs, c, op, hq).score
        if sc <= 0.9 * pages_sel.base_score + OP.EPS:
            best = min(best, sc)
    assert want.score == pytest.approx(best, rel=1e-12)
    assert want.score <= pages_sel.score + 1e-12


def test_uniform_candidates_never_raise_the_pages_score():
    seqs = [OP.SeqSpec(tiles=t, tasks_per_split=8, vectors=128) for t in (2048, 64, 300, 1500)]
    op = OP.ModelParams(num_ctas=152, warps_per_cta=7, rho=1.0, delta_attn=0.0, delta_red=2.5, gamma=2.0)
    a = OP.plan(seqs, op, q_heads=128, min_splits=1, max_splits=64)
    b = OP.plan_with_uniform(seqs, op, q_heads=128, min_splits=1, max_splits=64)
    assert b.score <= a.score and np.all(np.array(b.splits) >= 1)
