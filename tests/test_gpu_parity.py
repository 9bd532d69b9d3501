"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle
on the same seeded inputs, element by element.

Small cases span several pages and a ragged tail and run the oracle over
every output; the full-size configurations run in the launch configuration
the benchmark times and are checked on sampled (request, KV head) groups the
oracle recomputes one by one.
"""
import math

import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from tests.gpu_util import (check_lse, check_output, device_problem, oracle_partials, plan_params_for,
                            spec_like, to_np)

pytestmark = pytest.mark.gpu


def _run_all_paths(wl, params=None, check_partials=True):
    """Run decode (fused), partial + merge, and compare each with the oracle."""
    s = wl.spec
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, params or plan_params_for(s))
    po = oracle.problem_from_workload(wl)
    ref_o, ref_lse = po.attention_rows()
    ref_o = ref_o.reshape(wl.total_q, s.num_q_heads, s.head_dim_v)
    ref_lse = ref_lse.reshape(wl.total_q, s.num_q_heads)

    out, lse = att.decode()
    torch.cuda.synchronize()
    att.check_device_error()
    check_output(to_np(out), ref_o, s.dtype, "decode out")
    check_lse(to_np(lse), ref_lse, "decode lse")

    out2, lse2 = att.two_stage()
    torch.cuda.synchronize()
    att.check_device_error()
    check_output(to_np(out2), ref_o, s.dtype, "two-stage out")
    check_lse(to_np(lse2), ref_lse, "two-stage lse")

    if check_partials:
        o_part, lse_part = att.partial()
        torch.cuda.synchronize()
        ro, rl = oracle_partials(po, wl, att.plan)
        check_output(to_np(o_part)[:len(rl)], ro, s.dtype, "partial o")
        check_lse(to_np(lse_part)[:len(rl)], rl, "partial lse")
    return att, out, lse


def test_tiny_fp32_config():
    wl = W.build_workload(W.get_config("tiny_fp32_gqa"))
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 0


@pytest.mark.parametrize("lens,splits", [
    ([37, 128, 300, 513], 4),   # short splits: staged in shared memory
    ([2000, 45], 1),            # a 2000-key split: streamed from the cache
])
def test_cuda_core_decode_merges_on_every_call(lens, splits):
    """The CUDA-core path merges each request's splits in the request's last task (a
    per-request count that the merging task resets for the next call): repeated calls on
    one workspace, with the outputs poisoned before each, write every row again."""
    spec = spec_like("tiny_fp32_gqa", batch=len(lens), head_dim_qk=128, head_dim_v=128,
                     split=f"uniform:{splits}", seed=71 + splits)
    wl = W.build_workload(spec, seq_lens=lens)
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    assert att.plan.kernel_path == 0
    ref_o, ref_lse = oracle.problem_from_workload(wl).attention_rows()
    ref_o = ref_o.reshape(wl.total_q, spec.num_q_heads, spec.head_dim_v)
    ref_lse = ref_lse.reshape(wl.total_q, spec.num_q_heads)
    out, lse = att.out_like()
    for call in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        att.decode(out, lse)
        torch.cuda.synchronize()
        att.check_device_error()
        check_output(to_np(out), ref_o, spec.dtype, f"call {call} out")
        check_lse(to_np(lse), ref_lse, f"call {call} lse")


@pytest.mark.parametrize("case", [
    # (q heads, kv heads, page, q_lens, seq_lens, splits): every engine block of at most 8 rows
    (8, 2, 64, [2, 1, 2, 2], [700, 1300, 64 * 3 + 5, 2], 3),   # g = 4: two tokens per block, all-new request
    (4, 4, 128, [8, 3], [900, 1030], 2),                       # g = 1: eight tokens, eight causal limits
    (16, 2, 128, [1, 1, 1], [5000, 129, 64], 4),               # g = 8, page 128: one token per block
])
def test_gqa_engine_transposed_blocks(case):
    """Blocks of at most 8 rows run in the engine's transposed form (keys as the MMA rows);
    rows of different tokens in one block keep their own causal limits."""
    hq, hkv, page, q_lens, lens, splits = case
    spec = spec_like("llama405b_gqa_decode", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv,
                     page_size=page, split=f"uniform:{splits}", seed=140 + hq)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 1
    assert att.plan.num_chunk_tasks == 0 and att.plan.num_pair_tasks == 0
    assert max(ql * (hq // hkv) for ql in q_lens) <= 8


@pytest.mark.parametrize("lens,splits", [
    ([1, 63, 64, 65, 700, 2000], 3),
    ([4096, 130, 777], 8),
    ([64, 128, 192], 1),
    ([5, 17], 6),            # more splits than pages: empty splits
    ([20000, 3000, 1], 32),  # many splits per request: long reduction runs
])
@pytest.mark.parametrize("heads", [(32, 2), (16, 2), (8, 8)])
def test_gqa_engine_decode(lens, splits, heads):
    hq, hkv = heads
    spec = spec_like("llama405b_gqa_decode", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv,
                     split=f"uniform:{splits}", seed=100 + splits)
    wl = W.build_workload(spec, seq_lens=lens, extra_pages=3)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 1


@pytest.mark.parametrize("page,dim", [(16, 128), (128, 128), (64, 64), (16, 64), (128, 64)])
def test_gqa_engine_page_sizes_and_head_dims(page, dim):
    lens = [1, page - 1, page + 1, 5 * page + 3, 900]
    spec = spec_like("llama405b_gqa_decode", batch=len(lens), num_q_heads=16, num_kv_heads=2,
                     head_dim_qk=dim, head_dim_v=dim, page_size=page, scale=1 / math.sqrt(dim),
                     split="uniform:4", seed=7)
    wl = W.build_workload(spec, seq_lens=lens)
    _run_all_paths(wl)


@pytest.mark.parametrize("q_lens,lens", [
    ([5, 1, 37], [300, 64, 1000]),
    ([16, 16], [2048, 16]),         # speculative blocks; second request is all new tokens
    ([130], [130]),                 # full causal prefill
])
def test_gqa_engine_causal_chunks(q_lens, lens):
    spec = spec_like("mixed_chunked_prefill", batch=len(lens), num_q_heads=16, num_kv_heads=2,
                     split="uniform:3", seed=11)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    _run_all_paths(wl)


@pytest.mark.parametrize("case", [
    # (q heads, kv heads, head dim, page, q_lens, seq_lens, splits)
    (16, 2, 128, 64, [100, 1, 300], [1000, 500, 300], 2),     # ragged tiles, all-new request, decode row
    (64, 8, 128, 64, [2048], [2048 + 700], 1),                # one split: outputs written directly
    (32, 2, 128, 128, [40, 9], [5000, 777], 3),               # page 128, g = 16 (8 tokens per tile)
    (16, 2, 64, 64, [70, 3], [2100, 90], 2),                  # head dim 64
    (8, 8, 128, 64, [200, 65], [260, 1065], 4),               # g = 1: 128 tokens per tile (65 rows: paired tiles)
])
def test_gqa_chunk_tiles(case):
    hq, hkv, d, page, q_lens, lens, splits = case
    spec = spec_like("mixed_chunked_prefill", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim_qk=d,
                     head_dim_v=d, page_size=page, scale=1 / math.sqrt(d), split=f"uniform:{splits}", seed=61 + d)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 1
    g = hq // hkv
    expect = sum(hkv * -(-ql * g // 256) * splits for ql in q_lens if ql * g > 128)
    assert att.plan.num_chunk_tasks == expect


@pytest.mark.parametrize("case", [
    # (q heads, kv heads, head dim, page, q_lens, seq_lens, splits)
    (32, 8, 128, 64, [16, 16, 16, 16, 16], [5000, 40, 16, 900, 2100], 3),   # speculative blocks (64 rows)
    (16, 2, 128, 64, [5, 16, 9], [300, 2000, 77], 2),         # 40, 128 and 72 rows; ragged pages
    (16, 2, 64, 128, [7, 12], [1000, 140], 3),                # head dim 64, page 128
    (8, 8, 128, 128, [100, 33], [260, 1065], 1),              # g = 1, unsplit: outputs written directly
    (64, 8, 128, 64, [5], [5], 1),                            # all new tokens, shorter than a page
    (8, 1, 128, 64, [8], [700], 3),                           # odd block count: an empty last block
    (16, 2, 128, 64, [6, 1, 40], [3000, 800, 4100], 4),       # paired tiles, engine and chunk tiles
])
def test_gqa_paired_tiles(case):
    hq, hkv, d, page, q_lens, lens, splits = case
    spec = spec_like("spec_decode_q16", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim_qk=d,
                     head_dim_v=d, page_size=page, scale=1 / math.sqrt(d), split=f"uniform:{splits}", seed=91 + d)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 1
    g = hq // hkv
    blocks = sum(hkv * splits for ql in q_lens if 32 < ql * g <= 128)
    assert att.plan.num_pair_tasks == -(-blocks // 2) > 0
    assert ((att.plan.chunk_requests() == 2) == np.array([32 < ql * g <= 128 for ql in q_lens])).all()


def test_gqa_paired_tiles_planner():
    # planner splits on the paired tiles' own model (two blocks per SM)
    spec = spec_like("spec_decode_q16", batch=6, split="planner:1:64", seed=93)
    wl = W.build_workload(spec, seq_lens=[20000, 300, 7000, 16, 65000, 4100], q_lens=[16] * 6)
    att, _, _ = _run_all_paths(wl, plan_params_for(spec, num_ctas=0))
    assert att.plan.num_pair_tasks > 0 and att.plan.num_chunk_tasks == 0


def _rescale_events(q_rows, k_rows, c2, limits, unit=64):
    """Per row, how many units after the first raise its running maximum of
    c2 * q.k by more than 8 (log2 units): the chunk tiles' lazy-rescale rule.
    q_rows [R, D], k_rows [L, D] float64; row r sees keys 0 .. limits[r]."""
    s = (q_rows @ k_rows.T) * c2
    events = np.zeros(len(q_rows), dtype=np.int64)
    for r in range(len(q_rows)):
        m = None
        for k0 in range(0, limits[r] + 1, unit):
            mx = s[r, k0:min(k0 + unit, limits[r] + 1)].max()
            if m is None:
                m = mx
            elif mx > m + 8.0:
                events[r] += 1
                m = mx
    return events


@pytest.mark.parametrize("q0,route", [(100, 1), (9, 2)])
def test_tile_kernels_running_max_growth_rescales(q0, route):
    """Keys of later pages are scaled by exact powers of two (the same bits go to
    the oracle), so the running maximum of the first request's scores grows unit
    after unit by more than 2^8 and the tile kernel's lazy rescale of O and l fires
    (chunk tiles for 100 query tokens, paired tiles for 9); the host checks that it
    must, from the inputs, before the comparison."""
    spec = spec_like("mixed_chunked_prefill", batch=2, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=63)
    q_lens, lens = [q0, 1], [q0 + 12 * 64 + 5, 700]
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    P, D, g = spec.page_size, spec.head_dim_qk, spec.num_q_heads // spec.num_kv_heads
    k = wl.k_host().copy()                        # uint16 bf16 bits [pages, Hkv, P, D]
    n_pages = -(-lens[0] // P)
    for j in range(n_pages):
        page = int(wl.page_table[0, j])
        k[page] = k[page] + np.uint16((j // 2) << 7)     # x 2^(j // 2): exact (no zeros, no overflow)
    q, v = wl.q_host(), wl.v_host()
    # by construction: rows of the chunk request see their running max grow by > 2^8
    bf = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # noqa: E731
    c2 = spec.scale * 1.4426950408889634
    krows = bf(np.concatenate([k[int(wl.page_table[0, j]), 1] for j in range(n_pages)]))[:lens[0]]
    qrows = bf(q[0:q_lens[0], g:2 * g].reshape(-1, D))           # KV head 1: token-major rows
    limits = np.array([lens[0] - q_lens[0] + r // g for r in range(len(qrows))])
    # first split: pages 0..6 (keys 0..447) -- the tile kernels restart the running max per split
    ev = _rescale_events(qrows, krows, c2, np.minimum(limits, 7 * P - 1))
    assert (ev > 0).sum() > len(qrows) // 2, "inputs do not force the lazy rescale"
    po = oracle.Problem(kind="gqa", q=q, k=k, v=v, page_table=wl.page_table, seq_lens=wl.seq_lens,
                        qo_indptr=wl.qo_indptr, num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                        head_dim_qk=D, head_dim_v=D, page_size=P, scale=spec.scale)
    ref_o, ref_l = po.attention_rows()
    ref_o = ref_o.reshape(wl.total_q, spec.num_q_heads, D)
    ref_l = ref_l.reshape(wl.total_q, spec.num_q_heads)
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to("cuda")  # noqa: E731
    prob = skv.AttentionProblem(
        q=to_dev(q), k_cache=to_dev(k), v_cache=to_dev(v), page_table=torch.from_numpy(wl.page_table).to("cuda"),
        seq_lens=torch.from_numpy(wl.seq_lens).to("cuda"), qo_indptr=torch.from_numpy(wl.qo_indptr).to("cuda"),
        num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads, head_dim_qk=D, head_dim_v=D, page_size=P,
        scale=spec.scale, seq_lens_host=wl.seq_lens, qo_indptr_host=wl.qo_indptr)
    att = skv.SplitKVAttention(prob, skv.plan_params("uniform", uniform_splits=2))
    assert att.plan.chunk_requests()[0] == route
    for run in (att.decode, att.two_stage):
        out, lse = run()
        torch.cuda.synchronize()
        att.check_device_error()
        check_output(to_np(out), ref_o, "bf16", f"rescaled chunk {run.__name__} out")
        check_lse(to_np(lse), ref_l, f"rescaled chunk {run.__name__} lse")
    ro, rl = oracle_partials(po, wl, att.plan)
    o_part, lse_part = att.partial()
    torch.cuda.synchronize()
    check_output(to_np(o_part)[:len(rl)], ro, "bf16", "rescaled chunk partial o")
    check_lse(to_np(lse_part)[:len(rl)], rl, "rescaled chunk partial lse")


def test_mla_small_generic_path():
    spec = spec_like("deepseek_mla_decode", batch=3, num_q_heads=16, split="uniform:3", seed=13)
    wl = W.build_workload(spec, seq_lens=[1, 200, 777])
    att, _, _ = _run_all_paths(wl)


@pytest.mark.parametrize("lens,splits,q_lens", [
    ([1, 200, 777], 3, None),
    ([64, 4096, 130], 1, None),
    ([65, 3000], 5, None),
    ([5, 2000], 4, [2, 3]),          # several query tokens per request, causal
    ([10, 12], 3, None),             # more splits than pages: empty splits
    # 128-key units: last units of 1..32, 33..64, 65..96, 97..127 and 128 keys (one to four
    # value slots, one or two pages), single- and many-unit tasks
    ([32, 33, 96, 97, 127, 128, 129, 192, 255, 256, 257, 1000], 1, None),
])
def test_mla_tcgen05_path(lens, splits, q_lens):
    spec = spec_like("deepseek_mla_decode", batch=len(lens), split=f"uniform:{splits}", seed=31 + splits)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 2


def test_mla_tcgen05_many_items_per_cta():
    # 12 requests x 16 splits = 192 tasks = 384 work items: every CTA runs several in turn
    lens = [700 + 97 * j for j in range(12)]
    spec = spec_like("deepseek_mla_decode", batch=len(lens), split="uniform:16", seed=41)
    wl = W.build_workload(spec, seq_lens=lens)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 2 and att.plan.num_tasks == 192


def test_mla_tcgen05_running_max_growth_rescales():
    """Latent rows of later pages are scaled by exact powers of two, so scores
    and their running maximum grow page after page and the lazy rescale of
    the output accumulator fires (the same bits go to the oracle)."""
    spec = spec_like("deepseek_mla_decode", batch=2, split="uniform:1", seed=43)
    wl = W.build_workload(spec, seq_lens=[9 * 64 + 5, 3 * 64])
    k = wl.k_host().copy()                       # uint16 bf16 bits [pages, 64, 576]
    for b in range(2):
        n_pages = -(-int(wl.seq_lens[b]) // 64)
        for j in range(n_pages):
            page = int(wl.page_table[b, j])
            k[page] = k[page] + np.uint16((j // 2) << 7)   # x 2^(j // 2), exact for these values
    q = wl.q_host()
    po = oracle.Problem(kind="mla", q=q, k=k, v=None, page_table=wl.page_table, seq_lens=wl.seq_lens,
                        qo_indptr=wl.qo_indptr, num_q_heads=spec.num_q_heads, num_kv_heads=1,
                        head_dim_qk=spec.head_dim_qk, head_dim_v=spec.head_dim_v, page_size=64,
                        scale=spec.scale)
    ref_o, ref_l = po.attention_rows()
    dev = "cuda"
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    prob = skv.AttentionProblem(
        q=to_dev(q), k_cache=to_dev(k), v_cache=None, page_table=torch.from_numpy(wl.page_table).to(dev),
        seq_lens=torch.from_numpy(wl.seq_lens).to(dev), qo_indptr=torch.from_numpy(wl.qo_indptr).to(dev),
        num_q_heads=spec.num_q_heads, num_kv_heads=1, head_dim_qk=spec.head_dim_qk,
        head_dim_v=spec.head_dim_v, page_size=64, scale=spec.scale, kind="mla")
    att = skv.SplitKVAttention(prob, skv.plan_params("uniform", uniform_splits=1))
    assert att.plan.kernel_path == 2
    out, lse = att.decode()
    torch.cuda.synchronize()
    att.check_device_error()
    check_output(to_np(out).reshape(ref_o.shape), ref_o, "bf16", "rescaled mla out")
    check_lse(to_np(lse).reshape(-1), ref_l, "rescaled mla lse")


def test_planner_plan_runs():
    spec = spec_like("million_token_decode", batch=3, split="planner:1:16", seed=17)
    wl = W.build_workload(spec, seq_lens=[5000, 300, 20000])
    _run_all_paths(wl, plan_params_for(spec, num_ctas=0))


def test_decode_is_deterministic():
    spec = spec_like("llama405b_gqa_decode", batch=4, split="uniform:5", seed=19)
    wl = W.build_workload(spec, seq_lens=[3000, 1, 4096, 999])
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    o1, l1 = att.decode()
    o2, l2 = att.decode()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("fused", [True, False])
def test_out_of_range_page_is_reported_not_faulted(fused):
    spec = spec_like("llama405b_gqa_decode", batch=2, split="uniform:2", seed=23)
    wl = W.build_workload(spec, seq_lens=[200, 300])
    wl.page_table[1, 2] = wl.num_pages + 5       # caught by the kernels' range check
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    if fused:
        att.decode()
    else:
        att.partial()
    st, raw = skv.read_device_error(att.error_word, clear=True)
    assert st == skv.ERR_DEVICE_CHECK, (st, hex(raw))
    # the context is still usable
    wl2 = W.build_workload(spec, seq_lens=[200, 300])
    prob2, _ = device_problem(wl2)
    att2 = skv.SplitKVAttention(prob2, plan_params_for(spec))
    att2.decode()
    torch.cuda.synchronize()
    att2.check_device_error()


@pytest.mark.parametrize("case", ["mla_tcgen05", "chunk_tiles", "pair_tiles", "mla_fp8_copy"])
def test_out_of_range_page_is_reported_by_the_tcgen05_kernels(case):
    # the TMA producers check each page id before issuing its copies: the launch records
    # SPLITKV_ERR_DEVICE_CHECK and completes; a following launch on sound inputs matches the oracle
    if case == "mla_tcgen05":
        spec = spec_like("deepseek_mla_decode", batch=2, split="uniform:2", seed=25)
        lens, qls, bad = [200, 700], None, (1, 3)
    elif case == "mla_fp8_copy":
        spec = spec_like("deepseek_mla_fp8_decode", batch=2, split="uniform:2", seed=23)
        lens, qls, bad = [200, 700], None, (1, 3)
    elif case == "pair_tiles":
        spec = spec_like("spec_decode_q16", batch=2, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=24)
        lens, qls, bad = [600, 90], [8, 1], (0, 3)
    else:
        spec = spec_like("mixed_chunked_prefill", batch=2, num_q_heads=16, num_kv_heads=2, split="uniform:2",
                         seed=26)
        lens, qls, bad = [600, 90], [100, 1], (0, 3)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=qls)
    wl.page_table[bad] = wl.num_pages + 5
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    if case in ("mla_tcgen05", "mla_fp8_copy"):
        assert att.plan.kernel_path == 2
    elif case == "pair_tiles":
        assert att.plan.num_pair_tasks > 0
    else:
        assert att.plan.num_chunk_tasks > 0
    att.decode()
    st, raw = skv.read_device_error(att.error_word, clear=True)
    assert st == skv.ERR_DEVICE_CHECK, (st, hex(raw))
    wl2 = W.build_workload(spec, seq_lens=lens, q_lens=qls)
    _run_all_paths(wl2)


@pytest.mark.parametrize("q0,route", [(100, 1), (9, 2)])
def test_values_outside_the_f16_range_are_reported(q0, route):
    """The tile kernels multiply values in f16: a bf16 value of 2^17 in a slot the rows
    attend has no f16 form.  The launch records SPLITKV_ERR_DEVICE_CHECK at the value-range
    site and completes (chunk tiles for 100 query tokens, paired tiles for 9)."""
    spec = spec_like("mixed_chunked_prefill", batch=2, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=27)
    wl = W.build_workload(spec, seq_lens=[q0 + 300, 90], q_lens=[q0, 1])
    prob, t = device_problem(wl)
    t["v"][int(wl.page_table[0, 1]), 0, 5, 7] = 2.0 ** 17     # key 69 of request 0, KV head 0
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    assert att.plan.chunk_requests()[0] == route
    skv.read_device_error(att.error_word, clear=True)
    att.decode()
    st, raw = skv.read_device_error(att.error_word, clear=True)
    assert st == skv.ERR_DEVICE_CHECK and (raw >> 8) & 0xFF == 6, (st, hex(raw))


# ---------------------------------------------------------------- full size
def _sample_groups(wl: W.Workload, plan, n: int = 8, seed: int = 0):
    """At least ``n`` seeded (request, KV head) groups of a full-size batch: always
    the longest request, the request with the most splits and every chunked-prefill
    request (q_len > 16); then seeded requests not yet covered, then seeded groups.
    Each request enters with a seeded KV head."""
    s = wl.spec
    hkv = s.num_kv_heads if s.kind == "gqa" else 1
    rng = np.random.default_rng(1000 + seed)
    must = [int(np.argmax(wl.seq_lens)), int(np.argmax(plan.splits()))]
    must += [int(b) for b in np.flatnonzero(np.asarray(wl.q_lens) > 16)]
    order = must + [int(b) for b in rng.permutation(s.batch)]
    groups = []
    for b in order:
        if len(groups) >= max(n, len(set(must))):
            break
        if all(g[0] != b for g in groups):
            groups.append((b, int(rng.integers(hkv))))
    cand = [(b, h) for b in range(s.batch) for h in range(hkv)]
    for i in rng.permutation(len(cand)):
        if len(groups) >= n:
            break
        if cand[i] not in groups:
            groups.append(cand[i])
    return groups


def _group_heads(spec, hk):
    if spec.kind == "gqa":
        g = spec.num_q_heads // spec.num_kv_heads
        return slice(hk * g, (hk + 1) * g)
    return slice(0, spec.num_q_heads)


def _sampled_full_size(name, params=None, n_groups=8, two_stage=False, partial=False, seed=0):
    """The full-size configuration in the benchmark's launch configuration, checked on
    sampled (request, KV head) groups the oracle recomputes one by one: the fused
    decode always; with ``two_stage`` also splitkv_partial + merge_states, and with
    ``partial`` every split's partial state of the sampled groups."""
    spec = W.get_config(name)
    wl = W.build_workload(spec)
    prob, _ = device_problem(wl)
    att = skv.SplitKVAttention(prob, params or plan_params_for(spec))
    runs = {"decode": att.decode()}
    torch.cuda.synchronize()
    att.check_device_error()
    if two_stage:
        runs["two-stage"] = att.two_stage()
        torch.cuda.synchronize()
        att.check_device_error()
    outs = {k: (to_np(o), to_np(l)) for k, (o, l) in runs.items()}
    del runs
    o_part = lse_part = None
    if partial:
        op, lp = att.partial()
        torch.cuda.synchronize()
        att.check_device_error()
        o_part, lse_part = to_np(op), to_np(lp)
        del op, lp
        indptr = att.plan.state_indptr()
        n_spl = att.plan.splits()
    groups = _sample_groups(wl, att.plan, n_groups, seed)
    assert len(groups) >= n_groups
    for b, hk in groups:
        sub = oracle.subproblem_for_group(wl, b, hk)
        ql = int(wl.q_lens[b])
        hq_sub = sub.num_q_heads
        t0 = int(wl.qo_indptr[b])
        heads = _group_heads(spec, hk)
        rows = None
        if ql * hq_sub > 4096:
            # long chunked-prefill groups: a seeded sample of query tokens (all heads of each),
            # always the first and the last token
            rng = np.random.default_rng(7 + b)
            toks = np.unique(np.concatenate([[0, ql - 1], rng.choice(ql, size=min(ql, 96), replace=False)]))
            rows = np.array([(0, i, h) for i in toks for h in range(hq_sub)], dtype=np.int32)
        else:
            toks = np.arange(ql)
        ro, rl = sub.attention_rows(rows)
        ro = ro.reshape(len(toks), hq_sub, spec.head_dim_v)
        rl = rl.reshape(len(toks), hq_sub)
        for what, (out, lse) in outs.items():
            check_output(out[t0 + toks][:, heads], ro, spec.dtype, f"{name} {what} b={b} kv={hk}")
            check_lse(lse[t0 + toks][:, heads], rl, f"{name} {what} lse b={b} kv={hk}")
        if partial:
            n = int(n_spl[b])
            ranges = att.plan.split_ranges(b)
            h0 = heads.start
            rows5 = np.array([(0, i, h, kb, ke) for i in toks for h in range(hq_sub) for (kb, ke) in ranges],
                             dtype=np.int32)
            po, pl = sub.partial_rows(rows5)
            idx = np.array([indptr[(t0 + i) * spec.num_q_heads + h0 + h] + r
                            for i in toks for h in range(hq_sub) for r in range(n)])
            check_output(o_part[idx], po, spec.dtype, f"{name} partial o b={b} kv={hk}")
            check_lse(lse_part[idx], pl, f"{name} partial lse b={b} kv={hk}")
    return att, groups


def test_full_llama405b_decode_sampled():
    att, _ = _sampled_full_size("llama405b_gqa_decode", two_stage=True, partial=True)
    assert att.plan.kernel_path == 1 and (att.plan.splits() == 8).all()


def test_full_million_token_decode_sampled():
    att, groups = _sampled_full_size("million_token_decode", n_groups=8, two_stage=True)
    assert len({b for b, _ in groups}) == 4      # every request of the batch


def test_full_million_token_partial_states_sampled():
    # every split's partial state of three groups (up to 64 splits of 16k+ keys each)
    _sampled_full_size("million_token_decode", n_groups=3, partial=True, seed=1)


def test_full_mixed_batch_sampled():
    # decode requests plus both chunked-prefill requests (sampled query tokens of those)
    att, groups = _sampled_full_size("mixed_chunked_prefill", two_stage=True)
    assert {48, 49} <= {b for b, _ in groups}
    assert att.plan.num_chunk_tasks > 0


def test_full_mla_sampled():
    att, _ = _sampled_full_size("deepseek_mla_decode", two_stage=True, partial=True)
    assert att.plan.kernel_path == 2


def test_full_speculative_decode_sampled():
    # 16 query tokens per request (causal among the drafts), 64 rows per KV head
    att, _ = _sampled_full_size("spec_decode_q16", two_stage=True)
    assert att.plan.kernel_path == 1


@pytest.mark.parametrize("q_lens,lens,splits", [
    ([16, 16, 16], [5000, 40, 16], 3),    # drafts after a history, a short one, all new tokens (paired tiles)
    ([16, 4, 16], [777, 300, 2100], 5),
    ([5, 8, 1], [900, 2000, 40], 3),      # 20 and 32 rows per KV head: the engine's wide row blocks
])
def test_speculative_blocks_wide_rows(q_lens, lens, splits):
    spec = spec_like("spec_decode_q16", batch=len(lens), num_q_heads=8, num_kv_heads=2,
                     split=f"uniform:{splits}", seed=21)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    _run_all_paths(wl)


# ------------------------------------------------- FP8 (E4M3) KV cache
@pytest.mark.parametrize("case", [
    # (q heads, kv heads, page, seq_lens, q_lens, splits)
    (128, 8, 64, [1000, 37, 5, 640], [1, 1, 1, 1], 3),       # g = 16, ragged last pages
    (16, 2, 128, [3000, 130, 64, 1], [1, 1, 1, 1], 4),       # page 128, more splits than pages
    (8, 8, 64, [777, 300], [1, 1], 1),                       # g = 1, unsplit (fused output)
    (16, 2, 64, [900, 300, 2100], [5, 100, 16], 5),          # wide and causal row blocks
])
def test_fp8_kv_cache(case):
    hq, hkv, page, lens, q_lens, splits = case
    spec = spec_like("llama405b_fp8_decode", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, page_size=page,
                     split=f"uniform:{splits}", seed=61)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 1 and att.plan.num_chunk_tasks == 0


@pytest.mark.parametrize("case", [
    # (base configuration, overrides, seq_lens, q_lens, splits)
    ("deepseek_mla_decode", dict(num_q_heads=16), [9, 1000], [1, 2], 3),               # 16 heads, causal rows
    ("llama405b_fp8_decode", dict(num_q_heads=16, num_kv_heads=2, head_dim_qk=64, head_dim_v=64, scale=0.125),
     [300, 1000, 5], [1, 3, 1], 3),                                                    # head dim 64
    ("llama405b_fp8_decode", dict(num_q_heads=16, num_kv_heads=2, page_size=16), [70, 999], None, 2),   # page 16
])
def test_fp8_kv_cache_on_the_cuda_core_path(case):
    """E4M3 caches the engine does not take (absorbed MLA, other head dims and pages) run on the
    CUDA-core kernel in float32: for MLA the latent rows take k_scale as keys and as values."""
    base, over, lens, q_lens, splits = case
    spec = spec_like(base, batch=len(lens), kv_fp8=True, k_scale=0.0625, v_scale=0.05, split=f"uniform:{splits}",
                     seed=66, **over)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 0


@pytest.mark.parametrize("lens,q_lens,splits", [
    ([200, 777, 3000, 64], None, 4),
    ([1, 130, 2000], [1, 2, 1], 3),          # a one-key request, causal rows, more splits than some pages
    ([5000, 64, 300], None, 1),              # unsplit
])
def test_fp8_mla_latent_copy_on_tcgen05(lens, q_lens, splits):
    """Absorbed MLA over an E4M3 latent cache on the tcgen05 kernel: a pre-pass copies the
    batch's pages to bf16 (exact) and the kernel reads the copy; both roles of the latent
    rows take k_scale."""
    spec = spec_like("deepseek_mla_fp8_decode", batch=len(lens), split=f"uniform:{splits}", seed=67)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl)
    assert att.plan.kernel_path == 2


def test_full_mla_fp8_sampled():
    att, _ = _sampled_full_size("deepseek_mla_fp8_decode", two_stage=True)
    assert att.plan.kernel_path == 2


def test_fp8_kv_cache_planner_and_interleaved():
    spec = spec_like("llama405b_fp8_decode", batch=3, num_q_heads=16, num_kv_heads=2, seed=62)
    wl = W.build_workload(spec, seq_lens=[20000, 3000, 64])
    _run_all_paths(wl, skv.plan_params("critical_wave", min_splits=1, max_splits=16))
    _run_all_paths(wl, skv.plan_params("uniform", uniform_splits=6, interleave=1))


def test_full_llama405b_fp8_sampled():
    att, _ = _sampled_full_size("llama405b_fp8_decode", two_stage=True)
    assert att.plan.kernel_path == 1


# ------------------------------------------------- round-robin interleaved splits
@pytest.mark.parametrize("case", [
    # (base config, q heads, kv heads, head dim, page, seq_lens, q_lens, splits)
    ("llama405b_gqa_decode", 16, 1, 128, 16, [1000, 37, 5, 640], [1, 1, 1, 1], 3),   # Helix's 16-token blocks
    ("llama405b_gqa_decode", 32, 2, 128, 64, [3000, 130, 64, 1], [1, 1, 1, 1], 4),   # more splits than pages
    ("llama405b_gqa_decode", 8, 2, 64, 128, [2000, 300], [1, 1], 7),
    ("mixed_chunked_prefill", 16, 2, 128, 64, [900, 300, 2100], [5, 100, 1], 5),     # wide blocks, causal rows
    ("tiny_fp32_gqa", 8, 1, 64, 16, [37, 128, 300, 513], [1, 1, 1, 1], 4),           # CUDA-core path
])
def test_round_robin_interleaved_splits(case):
    base, hq, hkv, d, page, lens, q_lens, splits = case
    spec = spec_like(base, batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim_qk=d, head_dim_v=d,
                     page_size=page, scale=1.0 / np.sqrt(d), seed=31)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl, skv.plan_params("uniform", uniform_splits=splits, interleave=1))
    assert att.plan.interleaved and att.plan.num_chunk_tasks == 0


@pytest.mark.parametrize("base,lens,q_lens,splits", [
    ("deepseek_mla_decode", [700, 64, 1500], None, 3),
    ("deepseek_mla_decode", [130, 1, 5000], [1, 1, 2], 5),       # more splits than pages, causal rows
    ("deepseek_mla_decode", [4000, 900], None, 7),               # split units of two strided pages
    ("deepseek_mla_fp8_decode", [700, 2100, 65], None, 4),       # over the E4M3 latent's bf16 copy
])
def test_round_robin_interleaved_mla_on_tcgen05(base, lens, q_lens, splits):
    # the MLA kernel's items walk the pages r, r + n, r + 2n, ... of split r in 128-key units
    spec = spec_like(base, batch=len(lens), seed=32)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens, extra_pages=2)
    att, _, _ = _run_all_paths(wl, skv.plan_params("uniform", uniform_splits=splits, interleave=1))
    assert att.plan.interleaved and att.plan.kernel_path == 2


def test_full_mla_round_robin_sampled():
    att, _ = _sampled_full_size("deepseek_mla_decode", params=skv.plan_params("uniform", uniform_splits=6,
                                                                               interleave=1), two_stage=True)
    assert att.plan.interleaved and att.plan.kernel_path == 2


def test_full_llama405b_round_robin_sampled():
    att, _ = _sampled_full_size("llama405b_gqa_decode", params=skv.plan_params("uniform", uniform_splits=8,
                                                                                interleave=1), two_stage=True)
    assert att.plan.interleaved and att.plan.kernel_path == 1


# ------------------------------------------------- unused cache slots
def _poison_unused_slots(wl: W.Workload, t: dict):
    """NaN into every cache slot no request owns: the tail of each request's
    last page and the pages no request references.  The result is defined
    by the keys below seq_len only, so it must not change."""
    s = wl.spec
    P = s.page_size
    nan = 0x7F if s.kv_fp8 else float("nan")      # E4M3 S.1111.111 is NaN
    used = np.zeros(wl.num_pages, dtype=bool)
    for b in range(s.batch):
        n = -(-int(wl.seq_lens[b]) // P)
        used[wl.page_table[b, :n]] = True
        tail = int(wl.seq_lens[b]) % P
        if n > 0 and tail:
            last = int(wl.page_table[b, n - 1])
            for key in ("k", "v"):
                if t.get(key) is not None:
                    if s.kind == "gqa":
                        t[key][last, :, tail:] = nan
                    else:
                        t[key][last, tail:] = nan
    free = torch.from_numpy(np.flatnonzero(~used)).to(t["k"].device)
    for key in ("k", "v"):
        if t.get(key) is not None and free.numel():
            t[key][free] = nan


@pytest.mark.parametrize("case", ["fp32_generic", "gqa_engine_d128", "gqa_engine_d64_p16", "gqa_causal_chunks",
                                  "mla_tcgen05", "mla_generic", "gqa_engine_fp8", "mla_fp8_copy"])
def test_unused_cache_slots_do_not_reach_the_result(case):
    if case == "mla_fp8_copy":
        spec = spec_like("deepseek_mla_fp8_decode", batch=3, split="uniform:2", seed=58)
        wl = W.build_workload(spec, seq_lens=[3, 100, 650], q_lens=[1, 2, 1], extra_pages=2)
    elif case == "gqa_engine_fp8":
        spec = spec_like("llama405b_fp8_decode", batch=3, num_q_heads=16, num_kv_heads=2, split="uniform:3", seed=57)
        wl = W.build_workload(spec, seq_lens=[1, 70, 300], q_lens=[1, 3, 1], extra_pages=3)
    elif case == "fp32_generic":
        spec = spec_like("tiny_fp32_gqa", batch=3, split="uniform:3", seed=51)
        wl = W.build_workload(spec, seq_lens=[5, 70, 130], extra_pages=2)
    elif case == "gqa_engine_d128":
        spec = spec_like("llama405b_gqa_decode", batch=4, num_q_heads=16, num_kv_heads=2, split="uniform:3", seed=52)
        wl = W.build_workload(spec, seq_lens=[1, 65, 300, 1000], extra_pages=3)
    elif case == "gqa_engine_d64_p16":
        spec = spec_like("llama405b_gqa_decode", batch=3, num_q_heads=16, num_kv_heads=2, head_dim_qk=64,
                         head_dim_v=64, page_size=16, scale=1 / 8.0, split="uniform:2", seed=53)
        wl = W.build_workload(spec, seq_lens=[7, 33, 250], extra_pages=3)
    elif case == "gqa_causal_chunks":
        spec = spec_like("mixed_chunked_prefill", batch=3, num_q_heads=16, num_kv_heads=2, split="uniform:2", seed=54)
        wl = W.build_workload(spec, seq_lens=[300, 70, 130], q_lens=[5, 1, 100], extra_pages=2)
    elif case == "mla_tcgen05":
        spec = spec_like("deepseek_mla_decode", batch=3, split="uniform:2", seed=55)
        wl = W.build_workload(spec, seq_lens=[3, 100, 650], q_lens=[1, 2, 1], extra_pages=2)
    else:
        spec = spec_like("deepseek_mla_decode", batch=2, num_q_heads=16, split="uniform:2", seed=56)
        wl = W.build_workload(spec, seq_lens=[9, 200], extra_pages=2)
    prob, t = device_problem(wl)
    _poison_unused_slots(wl, t)
    att = skv.SplitKVAttention(prob, plan_params_for(spec))
    po = oracle.problem_from_workload(wl)
    ref_o, ref_lse = po.attention_rows()
    ref_o = ref_o.reshape(wl.total_q, spec.num_q_heads, spec.head_dim_v)
    ref_lse = ref_lse.reshape(wl.total_q, spec.num_q_heads)
    for run in (att.decode, att.two_stage):
        out, lse = run()
        torch.cuda.synchronize()
        att.check_device_error()
        check_output(to_np(out), ref_o, spec.dtype, f"{case} {run.__name__} out")
        check_lse(to_np(lse), ref_lse, f"{case} {run.__name__} lse")
