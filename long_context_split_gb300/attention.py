"""Convenience wrapper: plan once, upload once, run many times."""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib


class SplitKVAttention:
    """Split-KV attention for one batch layout.

    Builds the plan (``splitkv_plan``), allocates and fills the workspace
    (``splitkv_plan_upload``) and then runs the fused path (``splitkv_decode``)
    or the two-stage path (``splitkv_partial`` + ``merge_states``).  The plan
    and workspace are reusable for every layer that shares the batch lengths.
    """

    def __init__(self, problem: _lib.AttentionProblem, params: Optional[_lib.PlanParams] = None,
                 stream=None):
        self.problem = problem
        self.plan = _lib.splitkv_plan(problem, params)
        dev = problem.q.device
        self.workspace = _lib.alloc_workspace(self.plan, dev)
        self.state_indptr = torch.from_numpy(self.plan.state_indptr()).to(dev)
        self.error_word = torch.zeros(1, dtype=torch.int32, device=dev)
        _lib.splitkv_plan_upload(self.plan, self.workspace, stream)

    def out_like(self):
        p = self.problem
        dt = torch.bfloat16 if p.dtype == _lib.BF16 else torch.float32
        out = torch.empty(p.total_q, p.num_q_heads, p.head_dim_v, dtype=dt, device=p.q.device)
        lse = torch.empty(p.total_q, p.num_q_heads, dtype=torch.float32, device=p.q.device)
        return out, lse

    def decode(self, out=None, lse=None, stream=None):
        if out is None:
            out, lse = self.out_like()
        _lib.splitkv_decode(self.problem, self.plan, self.workspace, out, lse, self.error_word, stream)
        return out, lse

    def partial(self, stream=None):
        dev = self.problem.q.device
        o_part = torch.empty(max(1, self.plan.num_states), self.problem.head_dim_v, dtype=self.plan.partial_dtype,
                             device=dev)
        lse_part = torch.empty(max(1, self.plan.num_states), dtype=torch.float32, device=dev)
        _lib.splitkv_partial(self.problem, self.plan, self.workspace, o_part, lse_part, self.error_word, stream)
        return o_part, lse_part

    def two_stage(self, out=None, lse=None, stream=None):
        o_part, lse_part = self.partial(stream)
        if out is None:
            out, lse = self.out_like()
        _lib.merge_states(o_part, lse_part, self.state_indptr, out.view(-1, self.problem.head_dim_v),
                          lse.view(-1) if lse is not None else None, stream)
        return out, lse

    def check_device_error(self, clear: bool = True):
        st, raw = _lib.read_device_error(self.error_word, None, clear)
        if st != _lib.OK:
            raise _lib.SplitKVError(st, f"device error word 0x{raw:x}")
