"""Host-side checks of libsplitkv that need no GPU: the library loads and
exports every entry point of include/splitkv.h, the planner (host C++)
matches the oracle planner and LiquidCP Figure 8, plans have the documented
layout, and bad arguments are rejected before anything reaches a device.
"""
import dataclasses
import json
import os
import random
import re

import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from oracle import planner as OP

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "splitkv.h")
FIG8 = json.load(open(os.path.join(ROOT, "tests", "golden", "liquidcp_fig8.json")))


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keep = {n for n in names if n.startswith("splitkv_") or n.startswith("merge_states")}
    return sorted(keep)


def test_library_exports_every_declared_function():
    lib = skv.load()
    names = declared_functions()
    assert "splitkv_plan" in names and "splitkv_decode" in names and "merge_states" in names
    assert "splitkv_partial" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(skv._lib.SIGNATURES), "binding signatures must mirror the header"
    assert lib.splitkv_abi_version() == 1


def _cpu_problem(spec, wl=None, **over):
    wl = wl or W.build_workload(spec, **over)
    q = torch.zeros(1, dtype=torch.bfloat16 if spec.dtype == "bf16" else torch.float32)
    k = torch.zeros(wl.num_pages, 1, dtype=q.dtype)
    return wl, skv.AttentionProblem(
        q=q, k_cache=k, v_cache=k if spec.kind == "gqa" else None,
        page_table=torch.from_numpy(wl.page_table), seq_lens=torch.from_numpy(wl.seq_lens),
        qo_indptr=torch.from_numpy(wl.qo_indptr), num_q_heads=spec.num_q_heads,
        num_kv_heads=spec.num_kv_heads, head_dim_qk=spec.head_dim_qk, head_dim_v=spec.head_dim_v,
        page_size=spec.page_size, scale=spec.scale, kind=spec.kind)


def test_uniform_plan_layout_matches_oracle_split_bounds():
    spec = W.get_config("tiny_fp32_gqa")
    wl, prob = _cpu_problem(spec)
    plan = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4))
    assert plan.kernel_path == 0
    assert list(plan.splits()) == [4, 4, 4, 4]
    def keys(ranges):   # the key set of each split (empty ranges compare equal)
        return [tuple(range(int(a), int(e))) for a, e in ranges]

    for b in range(spec.batch):
        got = keys(plan.split_ranges(b))
        assert got == keys(oracle.split_bounds(int(wl.seq_lens[b]), spec.page_size, 4))
    ind = plan.state_indptr()
    assert ind[0] == 0 and ind[-1] == plan.num_states
    assert plan.num_states == spec.batch * spec.num_q_heads * 4
    assert (np.diff(ind) == 4).all()
    # the 37-token request has 3 pages: its 4th split is empty
    assert tuple(plan.split_ranges(0)[3]) == (37, 37)
    # 4 requests x 1 KV head x 1 row block x 4 splits
    assert plan.num_tasks == 16


def test_llama_plan_uses_engine_path_and_eight_splits():
    spec = W.get_config("llama405b_gqa_decode")
    wl, prob = _cpu_problem(spec)
    plan = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=8))
    assert plan.kernel_path == 1
    assert (plan.splits() == 8).all()
    assert plan.num_tasks == 32 * 8 * 8
    assert plan.num_states == 32 * 128 * 8


def test_figure8_through_the_c_abi():
    g = FIG8["params"]
    seqs = [(t, 1, g["vectors_per_reduction"], 1) for t in FIG8["histories_tiles"]]
    kw = dict(num_ctas=g["num_ctas"], rho=g["rho"], delta_attn=g["delta_attn"], delta_red=g["delta_red"],
              gamma=g["gamma"])
    for entry in FIG8["plans"]:
        score, _ = skv.model_simulate(seqs, entry["splits"], **kw)
        assert score == pytest.approx(entry["score"], abs=1e-9)
    splits, scores = skv.model_plan(seqs, **kw)
    assert list(splits) == FIG8["selected"]
    assert scores[0] == pytest.approx(152.0) and scores[1] == pytest.approx(104.0)


def _random_case(rng):
    n = rng.randint(1, 7)
    seqs = []
    for _ in range(n):
        q_len = rng.choice([1, 1, 1, 4, 16, 40])
        seqs.append((rng.randint(1, 300), rng.randint(1, 3), rng.randint(1, 40), q_len))
    p = dict(num_ctas=rng.choice([2, 4, 8, 16]), warps_per_cta=rng.choice([1, 4, 12]),
             q_heads=rng.choice([1, 8]), rho=rng.choice([0.25, 0.43, 0.75]),
             delta_attn=rng.choice([0.0, 4.0, 32.0]), delta_red=rng.choice([0.0, 2.5, 4.0]),
             gamma=rng.choice([0.0, 0.47, 1.0]))
    return seqs, p


def _oracle_seqs(seqs):
    return [OP.SeqSpec(tiles=t, tasks_per_split=k, vectors=v, q_len=q) for t, k, v, q in seqs]


def _oracle_params(p):
    return OP.ModelParams(num_ctas=p["num_ctas"], rho=p["rho"], delta_attn=p["delta_attn"],
                          delta_red=p["delta_red"], gamma=p["gamma"], warps_per_cta=p["warps_per_cta"])


@pytest.mark.parametrize("seed", range(40))
def test_planner_matches_oracle_planner(seed):
    rng = random.Random(seed)
    seqs, p = _random_case(rng)
    osq, op = _oracle_seqs(seqs), _oracle_params(p)
    lo, hi = rng.choice([(1, 64), (1, 8), (2, 16)])
    want = OP.plan(osq, op, q_heads=p["q_heads"], min_splits=lo, max_splits=hi)
    got, scores = skv.model_plan(seqs, min_splits=lo, max_splits=hi, **p)
    assert list(got) == want.splits
    assert scores[0] == pytest.approx(want.base_score, rel=1e-12)
    assert scores[1] == pytest.approx(want.score, rel=1e-12)
    assert scores[2] == pytest.approx(want.search_score, rel=1e-12)
    assert scores[3] == pytest.approx(want.ref_score, rel=1e-12)
    # and the simulator on a random plan
    sp = [rng.randint(1, min(8, s[0])) for s in seqs]
    sc, at = skv.model_simulate(seqs, sp, **p)
    r = OP.simulate(osq, sp, op, q_heads=p["q_heads"])
    assert sc == pytest.approx(r.score, rel=1e-12) and at == pytest.approx(r.attn_end, rel=1e-12)


@pytest.mark.parametrize("name", ["deepseek_mla_decode", "mixed_chunked_prefill", "million_token_decode"])
def test_planner_on_configurations_respects_bounds(name):
    spec = W.get_config(name)
    wl, prob = _cpu_problem(spec)
    lo, hi = W.planner_split_range(spec)
    plan = skv.splitkv_plan(prob, skv.plan_params("critical_wave", min_splits=lo, max_splits=hi, num_ctas=152))
    sp = plan.splits()
    pages = (wl.seq_lens + spec.page_size - 1) // spec.page_size
    assert ((sp >= np.minimum(lo, pages)) & (sp <= np.maximum(np.minimum(hi, pages), 1))).all()
    sc = plan.scores()
    assert sc[1] <= sc[0] + 1e-9
    ind = plan.state_indptr()
    assert ind[-1] == plan.num_states
    for b in range(spec.batch):
        rng_ = plan.split_ranges(b)
        assert rng_[0, 0] == 0 and rng_[-1, 1] == wl.seq_lens[b]


def test_invalid_arguments_are_rejected():
    spec = W.get_config("tiny_fp32_gqa")
    _, prob = _cpu_problem(spec, seq_lens=[3, 5], q_lens=[4, 1])     # q_len > seq_len
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(prob)
    assert e.value.status == skv.ERR_INVALID_ARG
    wl, prob = _cpu_problem(spec)
    prob._s.num_kv_heads = 3
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(prob)
    assert e.value.status == skv.ERR_INVALID_ARG
    wl, prob = _cpu_problem(spec)
    prob._s.head_dim_v = prob._s.head_dim_qk = 48
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(prob)
    assert e.value.status == skv.ERR_UNSUPPORTED
    wl, prob = _cpu_problem(spec)
    prob._s.max_pages_per_req = 2
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(prob)
    assert e.value.status == skv.ERR_INVALID_ARG
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(prob, skv.plan_params("critical_wave", min_splits=4, max_splits=2))


def test_merge_states_checks_before_launch():
    t = torch.zeros(4)
    with pytest.raises(skv.SplitKVError) as e:
        skv.merge_states(t.view(1, 4)[:, :3].contiguous(), t[:1], torch.zeros(2, dtype=torch.int32), t.view(1, 4)[:, :3])
    assert e.value.status == skv.ERR_UNSUPPORTED


def test_debug_inject_mode_is_validated():
    with pytest.raises(skv.SplitKVError):
        skv.debug_set_inject(2)
    skv.debug_set_inject(0)


@pytest.mark.parametrize("seed", range(4))
def test_planner_matches_oracle_planner_many_sequences(seed):
    """Batches large enough for the library's search to run on several host threads, with
    GQA-like reduction runs (many warps, one vector per item) and MLA-like ones."""
    rng = random.Random(1000 + seed)
    n = rng.randint(8, 10)
    mla = seed % 2 == 1
    seqs = [(rng.randint(8, 400), 1 if mla else 8, 128 if mla else 64, 1) for _ in range(n)]
    p = dict(num_ctas=76 if mla else 152, warps_per_cta=1 if mla else 7, q_heads=128 if mla else 64,
             rho=rng.choice([0.43, 1.0]), delta_attn=rng.choice([0.0, 4.0]), delta_red=rng.choice([1.0, 2.5]),
             gamma=rng.choice([0.0, 2.0]))
    osq, op = _oracle_seqs(seqs), _oracle_params(p)
    want = OP.plan(osq, op, q_heads=p["q_heads"], min_splits=1, max_splits=64)
    got, scores = skv.model_plan(seqs, min_splits=1, max_splits=64, **p)
    assert list(got) == want.splits
    assert scores[2] == pytest.approx(want.search_score, rel=1e-12)
    sp = [rng.randint(1, 12) for _ in seqs]
    sc, at = skv.model_simulate(seqs, sp, **p)
    r = OP.simulate(osq, sp, op, q_heads=p["q_heads"])
    assert sc == pytest.approx(r.score, rel=1e-12) and at == pytest.approx(r.attn_end, rel=1e-12)


def test_interleaved_plan_on_the_host():
    """Round-robin interleaved splits (Helix Section 2.3): validated, flagged, the same split
    counts and states as contiguous splits, no chunk tiles, and no key ranges to report."""
    spec = W.get_config("mixed_chunked_prefill")
    wl, prob = _cpu_problem(spec)
    with pytest.raises(skv.SplitKVError):
        skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4, interleave=2))
    with pytest.raises(skv.SplitKVError):
        skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4, partial_dtype=7))
    contiguous = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4, num_ctas=152))
    inter = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4, interleave=1, num_ctas=152))
    assert inter.interleaved and not contiguous.interleaved
    assert (inter.splits() == contiguous.splits()).all()
    assert inter.num_states == contiguous.num_states
    assert contiguous.num_chunk_tasks > 0 and inter.num_chunk_tasks == 0
    with pytest.raises(skv.SplitKVError):
        inter.split_ranges(0)
    # MLA: the tcgen05 kernel takes interleaved plans too (its items walk page-strided units)
    mla = W.get_config("deepseek_mla_decode")
    _, mprob = _cpu_problem(mla)
    assert skv.splitkv_plan(mprob, skv.plan_params("uniform", uniform_splits=2, num_ctas=76)).kernel_path == 2
    assert skv.splitkv_plan(mprob, skv.plan_params("uniform", uniform_splits=2, interleave=1,
                                                   num_ctas=76)).kernel_path == 2


def _fp8_problem(spec, k_scale=0.0625, v_scale=0.05, **over):
    wl = W.build_workload(spec, **over)
    q = torch.zeros(1, dtype=torch.bfloat16 if spec.dtype == "bf16" else torch.float32)
    k = torch.zeros(wl.num_pages, 1, dtype=torch.uint8)
    return wl, skv.AttentionProblem(
        q=q, k_cache=k, v_cache=k if spec.kind == "gqa" else None,
        page_table=torch.from_numpy(wl.page_table), seq_lens=torch.from_numpy(wl.seq_lens),
        qo_indptr=torch.from_numpy(wl.qo_indptr), num_q_heads=spec.num_q_heads,
        num_kv_heads=spec.num_kv_heads, head_dim_qk=spec.head_dim_qk, head_dim_v=spec.head_dim_v,
        page_size=spec.page_size, scale=spec.scale, kind=spec.kind, k_scale=k_scale, v_scale=v_scale)


def test_fp8_kv_problems_on_the_host():
    """FP8 (E4M3) KV caches: the GQA engine serves the shapes it takes (no chunk or paired
    tiles), the CUDA-core path the others (absorbed MLA included), unsupported shapes are
    refused, scales are validated, and a plan is tied to the cache type it was made for."""
    spec = W.get_config("llama405b_fp8_decode")
    _, prob = _fp8_problem(spec)
    plan = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=8))
    assert plan.kernel_path == 1 and plan.num_chunk_tasks == 0
    # chunk-sized rows go to the engine's wide blocks
    mixed = dataclasses.replace(W.get_config("mixed_chunked_prefill"), kv_fp8=True, k_scale=0.1, v_scale=0.1)
    _, mprob = _fp8_problem(mixed)
    assert skv.splitkv_plan(mprob, skv.plan_params("uniform", uniform_splits=2, num_ctas=152)).num_chunk_tasks == 0
    # shapes outside the engine's: the CUDA-core path (kernel path 0)
    for over in (dict(page_size=16), dict(head_dim_qk=64, head_dim_v=64)):
        other = dataclasses.replace(spec, **over)
        _, oprob = _fp8_problem(other)
        assert skv.splitkv_plan(oprob, skv.plan_params("uniform", uniform_splits=2)).kernel_path == 0
    # absorbed MLA of the tcgen05 kernel's shape: that kernel over a bf16 copy of the batch's
    # latent pages in the workspace (73,728 bytes per page), contiguous or interleaved splits;
    # other head counts: the CUDA-core path
    mla = W.get_config("deepseek_mla_fp8_decode")
    mwl, mlaprob = _fp8_problem(mla)
    p8 = skv.splitkv_plan(mlaprob, skv.plan_params("uniform", uniform_splits=2))
    assert p8.kernel_path == 2
    _, mbf = _cpu_problem(W.get_config("deepseek_mla_decode"), wl=mwl)
    pbf = skv.splitkv_plan(mbf, skv.plan_params("uniform", uniform_splits=2))
    pages = int(sum(-(-int(L) // 64) for L in mwl.seq_lens))
    assert p8.workspace_bytes - pbf.workspace_bytes >= pages * 64 * 576 * 2
    assert skv.splitkv_plan(mlaprob, skv.plan_params("uniform", uniform_splits=2, interleave=1)).kernel_path == 2
    _, m16 = _fp8_problem(dataclasses.replace(mla, num_q_heads=16))
    assert skv.splitkv_plan(m16, skv.plan_params("uniform", uniform_splits=2)).kernel_path == 0
    # unsupported: head dims off the 16-code row granule, value widths without a kernel
    for over in (dict(head_dim_qk=40, head_dim_v=40), dict(head_dim_qk=96, head_dim_v=96)):
        bad = dataclasses.replace(spec, **over)
        _, bprob = _fp8_problem(bad)
        with pytest.raises(skv.SplitKVError, match="FP8"):
            skv.splitkv_plan(bprob, skv.plan_params("uniform", uniform_splits=2))
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0)):
        _, sprob = _fp8_problem(spec, k_scale=ks, v_scale=vs)
        with pytest.raises(skv.SplitKVError, match="scale"):
            skv.splitkv_plan(sprob, skv.plan_params("uniform", uniform_splits=2))
    # a uint8 cache needs its scales, and other caches take none
    with pytest.raises(TypeError):
        skv.AttentionProblem(q=torch.zeros(1, dtype=torch.bfloat16), k_cache=torch.zeros(4, 1, dtype=torch.uint8),
                             v_cache=torch.zeros(4, 1, dtype=torch.uint8), page_table=torch.zeros(1, 1, dtype=torch.int32),
                             seq_lens=torch.ones(1, dtype=torch.int32), qo_indptr=torch.tensor([0, 1], dtype=torch.int32),
                             num_q_heads=8, num_kv_heads=1, head_dim_qk=128, head_dim_v=128, page_size=64, scale=0.1)


def test_bf16_partial_plan_on_the_host():
    """bf16 partial states (LiquidCP Section 7): the plan records the storage type and its
    workspace holds half the partial-output bytes; the float32 LSEs are unchanged."""
    import torch
    spec = W.get_config("deepseek_mla_decode")
    wl, prob = _cpu_problem(spec)
    f32 = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4, num_ctas=76))
    b16 = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=4, num_ctas=76, partial_dtype=skv.BF16))
    assert f32.partial_dtype == torch.float32 and b16.partial_dtype == torch.bfloat16
    assert f32.num_states == b16.num_states > 0
    saved = f32.workspace_bytes - b16.workspace_bytes
    # half of num_states x 512 float32 values, up to the 256-byte alignment of the regions
    assert abs(saved - f32.num_states * spec.head_dim_v * 2) <= 512


def test_chunk_tiles_beside_the_engine_only_when_chunk_requests_are_unsplit():
    """The mixed batch's planner plan keeps its chunk requests unsplit, so the chunk tiles
    and the engine share the SMs; with split chunk requests (their states are merged by
    the engine's reduction phase) or without chunk requests the two run one after the
    other.  The engine model's units are the engine's share of the SMs."""
    spec = W.get_config("mixed_chunked_prefill")
    wl, prob = _cpu_problem(spec)
    p = skv.splitkv_plan(prob, skv.plan_params("critical_wave", min_splits=1, max_splits=64))
    assert 0 < p.overlap_ctas < 152 and p.num_chunk_tasks > 0
    assert (p.splits()[p.chunk_requests() == 1] == 1).all()
    assert skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=2)).overlap_ctas == 0
    assert skv.splitkv_plan(prob, skv.plan_params("critical_wave", min_splits=2, max_splits=64)).overlap_ctas == 0
    llama = W.get_config("llama405b_gqa_decode")
    _, prob2 = _cpu_problem(llama)
    assert skv.splitkv_plan(prob2, skv.plan_params("uniform", uniform_splits=8)).overlap_ctas == 0


def test_paired_tiles_plan_on_the_host():
    """Requests with 33..128 query rows per KV head go to the paired-tile kernel (one block
    of all their rows per (KV head, split), two blocks per task, an empty block after an odd
    last one); more rows go to the chunk tiles, up to 32 stay on the engine; FP8 caches,
    interleaved splits and 16-token pages keep every row block on the engine."""
    spec = dataclasses.replace(W.get_config("mixed_chunked_prefill"), batch=6)   # g = 8
    q_lens = [1, 3, 4, 5, 16, 17]                     # 8, 24, 32, 40, 128, 136 rows per KV head
    wl, prob = _cpu_problem(spec, seq_lens=[900, 300, 2000, 70, 4096, 5000], q_lens=q_lens)
    plan = skv.splitkv_plan(prob, skv.plan_params("uniform", uniform_splits=3, num_ctas=152))
    assert plan.chunk_requests().tolist() == [0, 0, 0, 2, 2, 1]
    blocks = 2 * spec.num_kv_heads * 3
    assert plan.num_pair_tasks == -(-blocks // 2)
    assert plan.num_chunk_tasks == spec.num_kv_heads * 3 * 1
    engine_tasks = 3 * spec.num_kv_heads * 3           # one 64-row (or 16-row) block per KV head and split
    assert plan.num_tasks == engine_tasks + plan.num_chunk_tasks + plan.num_pair_tasks
    assert plan.overlap_ctas == 0
    # an odd number of blocks (one KV head, three splits): the last task holds one block
    one = dataclasses.replace(spec, batch=1, num_q_heads=8, num_kv_heads=1)
    _, p1 = _cpu_problem(one, seq_lens=[700], q_lens=[8])
    assert skv.splitkv_plan(p1, skv.plan_params("uniform", uniform_splits=3, num_ctas=152)).num_pair_tasks == 2
    # the speculative-decode batch: every request on the paired tiles, planner splits
    sd = W.get_config("spec_decode_q16")
    _, sprob = _cpu_problem(sd)
    lo, hi = W.planner_split_range(sd)
    sp = skv.splitkv_plan(sprob, skv.plan_params("critical_wave", min_splits=lo, max_splits=hi))
    assert (sp.chunk_requests() == 2).all() and sp.num_chunk_tasks == 0 and sp.num_pair_tasks > 0
    assert sp.num_tasks == sp.num_pair_tasks
    blocks = int(sp.splits().sum()) * sd.num_kv_heads
    assert sp.num_pair_tasks == -(-blocks // 2)
    # no paired tiles: interleaved splits, FP8 caches, 16-token pages
    assert skv.splitkv_plan(sprob, skv.plan_params("uniform", uniform_splits=2, interleave=1)).num_pair_tasks == 0
    fp8 = dataclasses.replace(sd, kv_fp8=True, k_scale=0.1, v_scale=0.1)
    _, fprob = _fp8_problem(fp8)
    assert skv.splitkv_plan(fprob, skv.plan_params("uniform", uniform_splits=2)).num_pair_tasks == 0
    p16 = dataclasses.replace(sd, page_size=16)
    _, qprob = _cpu_problem(p16)
    assert skv.splitkv_plan(qprob, skv.plan_params("uniform", uniform_splits=2)).num_pair_tasks == 0
