"""splitkv_decode inside a CUDA graph: after one ordinary call (which sets the
kernels up), a decode captured on a stream replays with the same results as the
float64 oracle, and a replay after new query values are copied into the same
buffers follows them.  Covers the fused engine (with its reduction phase), the
paired tiles ahead of it, and the chunk tiles beside it on the side stream,
whose fork and join become graph edges."""
import numpy as np
import pytest
import torch

import long_context_split_gb300 as skv
import oracle
import workloads as W
from tests.gpu_util import check_lse, check_output, device_problem, plan_params_for, spec_like, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "gqa_engine": ("llama405b_gqa_decode", dict(num_q_heads=32, num_kv_heads=4), [3000, 1, 700, 4096], None, 3),
    "pair_tiles": ("spec_decode_q16", dict(num_q_heads=16, num_kv_heads=2), [900, 40, 2000], [16, 1, 5], 2),
    # unsplit chunk request and decode rows: the chunk tiles run beside the engine
    "chunk_beside_engine": ("mixed_chunked_prefill", {}, [2000] * 48 + [512 + 384], [1] * 48 + [384], 1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_replays_from_a_cuda_graph(name):
    base, over, lens, q_lens, splits = CASES[name]
    spec = spec_like(base, batch=len(lens), split=f"uniform:{splits}", seed=87, **over)
    wl = W.build_workload(spec, seq_lens=lens, q_lens=q_lens)
    prob, t = device_problem(wl)
    if name == "chunk_beside_engine":
        att = skv.SplitKVAttention(prob, skv.plan_params("critical_wave", min_splits=1, max_splits=1))
        assert att.plan.overlap_ctas > 0
    else:
        att = skv.SplitKVAttention(prob, plan_params_for(spec))
    if name == "pair_tiles":
        assert att.plan.num_pair_tasks > 0
    out, lse = att.out_like()
    att.decode(out, lse)                       # first call outside the capture
    torch.cuda.synchronize()
    att.check_device_error()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            att.decode(out, lse)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    att.check_device_error()
    po = oracle.problem_from_workload(wl)
    ref_o, ref_l = po.attention_rows()
    check_output(to_np(out), ref_o.reshape(out.shape), spec.dtype, f"{name} graph replay out")
    check_lse(to_np(lse), ref_l.reshape(lse.shape), f"{name} graph replay lse")
    # new query values in the same buffer (the tokens in reverse order): the replay follows them
    t["q"].copy_(torch.flip(t["q"], dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    att.check_device_error()
    q2 = np.ascontiguousarray(np.flip(wl.q_host(), axis=0))
    ref2, _ = oracle.Problem(kind="gqa", q=q2, k=wl.k_host(), v=wl.v_host(), page_table=wl.page_table,
                             seq_lens=wl.seq_lens, qo_indptr=wl.qo_indptr, num_q_heads=spec.num_q_heads,
                             num_kv_heads=spec.num_kv_heads, head_dim_qk=spec.head_dim_qk,
                             head_dim_v=spec.head_dim_v, page_size=spec.page_size,
                             scale=spec.scale).attention_rows()
    check_output(to_np(out), ref2.reshape(out.shape), spec.dtype, f"{name} graph replay, new queries")
