"""ctypes binding of libsplitkv (``include/splitkv.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libsplitkv.so``.  PyTorch supplies device memory and streams.
Loading fails loudly when the library has not been built; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsplitkv.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_DEVICE_CHECK = 6

GQA, MLA = 0, 1
F32, BF16 = 0, 1
PLAN_UNIFORM, PLAN_CRITICAL_WAVE = 0, 1


class SplitKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libsplitkv status {status}: {message}")
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32), ("scale", ctypes.c_float),
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("qo_indptr", ctypes.c_void_p), ("seq_lens_host", ctypes.c_void_p),
        ("qo_indptr_host", ctypes.c_void_p),
        ("kv_fp8", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
        ("reserved0", ctypes.c_int32),
    ]


class PlanParams(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32), ("uniform_splits", ctypes.c_int32),
        ("min_splits", ctypes.c_int32), ("max_splits", ctypes.c_int32),
        ("num_ctas", ctypes.c_int32), ("warps_per_cta", ctypes.c_int32),
        ("tile_tokens", ctypes.c_int32), ("decode_qlen_max", ctypes.c_int32),
        ("rho", ctypes.c_double), ("delta_attn", ctypes.c_double),
        ("delta_red", ctypes.c_double), ("gamma", ctypes.c_double),
        ("adopt_margin", ctypes.c_double),
        ("interleave", ctypes.c_int32), ("partial_dtype", ctypes.c_int32),
        ("trace", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


class TraceRecord(ctypes.Structure):
    _fields_ = [("start_ns", ctypes.c_uint64), ("end_ns", ctypes.c_uint64), ("id", ctypes.c_int32),
                ("sm", ctypes.c_int32), ("kind", ctypes.c_int32), ("cta", ctypes.c_int32)]


class TraceStats(ctypes.Structure):
    _fields_ = [("records", ctypes.c_int32), ("sms", ctypes.c_int32), ("begin_ns", ctypes.c_double),
                ("end_ns", ctypes.c_double), ("tail_idle_sm_ns", ctypes.c_double),
                ("tail_idle_frac", ctypes.c_double)]


TRACE_ATTENTION, TRACE_REDUCTION, TRACE_CHUNK, TRACE_MLA_ITEM, TRACE_PAIR = 0, 1, 2, 3, 4
TRACE_DTYPE = np.dtype([("start_ns", "<u8"), ("end_ns", "<u8"), ("id", "<i4"), ("sm", "<i4"), ("kind", "<i4"),
                        ("cta", "<i4")])


class SeqModel(ctypes.Structure):
    _fields_ = [("tiles", ctypes.c_int32), ("tasks_per_split", ctypes.c_int32),
                ("vectors", ctypes.c_int32), ("q_len", ctypes.c_int32)]


class ModelParams(ctypes.Structure):
    _fields_ = [
        ("num_ctas", ctypes.c_int32), ("warps_per_cta", ctypes.c_int32),
        ("q_heads", ctypes.c_int32), ("decode_qlen_max", ctypes.c_int32),
        ("rho", ctypes.c_double), ("delta_attn", ctypes.c_double),
        ("delta_red", ctypes.c_double), ("gamma", ctypes.c_double),
        ("adopt_margin", ctypes.c_double),
    ]


class KernelTime(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int32), ("pad", ctypes.c_int32), ("total_ms", ctypes.c_double)]


# splitkv_kernel ids, in order
KERNEL_NAMES = ["generic_partial_kernel", "gqa_engine_kernel", "mla_partial_kernel", "chunk_tc_kernel",
                "merge_states_kernel", "chunk_value_convert_kernel", "pair_tc_kernel", "mla_latent_convert_kernel"]

# name -> (restype, argtypes); this list mirrors include/splitkv.h
_vp, _i32, _i64, _dp = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = {
    "splitkv_plan_params_default": (None, [ctypes.POINTER(PlanParams)]),
    "splitkv_plan": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.POINTER(PlanParams),
                                    ctypes.POINTER(ctypes.c_void_p)]),
    "splitkv_plan_destroy": (None, [_vp]),
    "splitkv_plan_num_tasks": (_i32, [_vp]),
    "splitkv_plan_num_chunk_tasks": (_i32, [_vp]),
    "splitkv_plan_num_pair_tasks": (_i32, [_vp]),
    "splitkv_plan_chunk_requests": (ctypes.c_int, [_vp, _ip]),
    "splitkv_plan_num_states": (_i64, [_vp]),
    "splitkv_plan_num_rows": (_i32, [_vp]),
    "splitkv_plan_splits": (ctypes.c_int, [_vp, _ip]),
    "splitkv_plan_state_indptr": (ctypes.c_int, [_vp, _ip]),
    "splitkv_plan_split_ranges": (ctypes.c_int, [_vp, _i32, _ip]),
    "splitkv_plan_interleaved": (_i32, [_vp]),
    "splitkv_plan_partial_dtype": (_i32, [_vp]),
    "splitkv_plan_trace_records": (_i32, [_vp]),
    "splitkv_plan_overlap_ctas": (_i32, [_vp]),
    "splitkv_trace_read": (ctypes.c_int, [_vp, _vp, ctypes.c_size_t, _vp, _vp]),
    "splitkv_trace_tail_idle": (ctypes.c_int, [_vp, _i32, _i32, _i32, ctypes.POINTER(TraceStats)]),
    "splitkv_plan_scores": (ctypes.c_int, [_vp, _dp]),
    "splitkv_plan_kernel_path": (_i32, [_vp]),
    "splitkv_workspace_bytes": (ctypes.c_size_t, [_vp]),
    "splitkv_plan_upload": (ctypes.c_int, [_vp, _vp, ctypes.c_size_t, _vp]),
    "splitkv_partial": (ctypes.c_int, [ctypes.POINTER(Problem), _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]),
    "merge_states": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp]),
    "merge_states_typed": (ctypes.c_int, [_vp, _i32, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp]),
    "splitkv_decode": (ctypes.c_int, [ctypes.POINTER(Problem), _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]),
    "splitkv_decode_static": (ctypes.c_int, [ctypes.POINTER(Problem), _vp, _vp, _vp, _vp, _vp]),
    "splitkv_read_device_error": (ctypes.c_int, [_vp, _vp, _i32, _ip, _vp]),
    "splitkv_read_static_device_error": (ctypes.c_int, [_i32, _ip, _vp]),
    "splitkv_last_error_message": (ctypes.c_char_p, []),
    "splitkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "splitkv_abi_version": (_i32, []),
    "splitkv_model_simulate": (ctypes.c_int, [ctypes.POINTER(SeqModel), _i32, _ip,
                                              ctypes.POINTER(ModelParams), _dp, _dp]),
    "splitkv_model_plan": (ctypes.c_int, [ctypes.POINTER(SeqModel), _i32, ctypes.POINTER(ModelParams),
                                          _i32, _i32, _ip, _dp]),
    "splitkv_profile_begin": (ctypes.c_int, []),
    "splitkv_debug_set_inject": (ctypes.c_int, [_i32]),
    "splitkv_profile_end": (ctypes.c_int, [ctypes.POINTER(KernelTime)]),
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libsplitkv.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _check(status: int):
    if status != OK:
        msg = load().splitkv_last_error_message().decode(errors="replace")
        raise SplitKVError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        if not torch.cuda.is_available():
            return ctypes.c_void_p(0)   # argument checks still run; no launch can follow
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}


class AttentionProblem:
    """A batch of attention over a paged KV cache (``splitkv_problem``).

    Tensors are on the GPU: ``q`` [total_q, Hq, D_qk]; GQA ``k_cache``/``v_cache``
    [num_pages, Hkv, P, D]; MLA ``k_cache`` [num_pages, P, 576] with
    ``v_cache=None``; ``page_table`` int32 [B, max_pages]; ``seq_lens`` int32
    [B]; ``qo_indptr`` int32 [B+1].  Host copies of the lengths are taken once
    here (or passed in) for the planner.  K/V caches of dtype uint8 hold E4M3
    codes (an FP8 KV cache) whose values are code * ``k_scale`` / ``v_scale``.
    """

    def __init__(self, *, q: torch.Tensor, k_cache: torch.Tensor, v_cache: Optional[torch.Tensor],
                 page_table: torch.Tensor, seq_lens: torch.Tensor, qo_indptr: torch.Tensor,
                 num_q_heads: int, num_kv_heads: int, head_dim_qk: int, head_dim_v: int,
                 page_size: int, scale: float, kind: str = "gqa",
                 seq_lens_host: Optional[Sequence[int]] = None,
                 qo_indptr_host: Optional[Sequence[int]] = None,
                 k_scale: Optional[float] = None, v_scale: Optional[float] = None):
        self.q, self.k_cache, self.v_cache = q, k_cache, v_cache
        self.page_table, self.seq_lens, self.qo_indptr = page_table, seq_lens, qo_indptr
        for name, t in (("page_table", page_table), ("seq_lens", seq_lens), ("qo_indptr", qo_indptr)):
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous int32 tensor")
        for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
            if t is not None and not t.is_contiguous():
                raise TypeError(f"{name} must be contiguous")
        if q.dtype not in _DTYPES:
            raise TypeError(f"unsupported dtype {q.dtype}")
        self.kv_fp8 = k_cache.dtype == torch.uint8
        if self.kv_fp8 != (k_scale is not None and v_scale is not None):
            raise TypeError("uint8 (E4M3) K/V caches come with k_scale and v_scale, other caches without")
        self.k_scale = float(k_scale) if self.kv_fp8 else 1.0
        self.v_scale = float(v_scale) if self.kv_fp8 else 1.0
        self.seq_lens_host = np.ascontiguousarray(
            seq_lens.cpu().numpy() if seq_lens_host is None else seq_lens_host, dtype=np.int32)
        self.qo_indptr_host = np.ascontiguousarray(
            qo_indptr.cpu().numpy() if qo_indptr_host is None else qo_indptr_host, dtype=np.int32)
        self.kind = kind
        self.dtype = _DTYPES[q.dtype]
        self.num_q_heads, self.num_kv_heads = num_q_heads, num_kv_heads
        self.head_dim_qk, self.head_dim_v = head_dim_qk, head_dim_v
        self.page_size, self.scale = page_size, scale
        self.batch = int(seq_lens.shape[0])
        self._s = Problem(
            kind=GQA if kind == "gqa" else MLA, dtype=self.dtype, batch=self.batch,
            num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim_qk=head_dim_qk,
            head_dim_v=head_dim_v, page_size=page_size, num_pages=int(k_cache.shape[0]),
            max_pages_per_req=int(page_table.shape[1]), scale=float(scale),
            q=q.data_ptr(), k_cache=k_cache.data_ptr(),
            v_cache=(v_cache.data_ptr() if v_cache is not None else None),
            page_table=page_table.data_ptr(), seq_lens=seq_lens.data_ptr(),
            qo_indptr=qo_indptr.data_ptr(), seq_lens_host=self.seq_lens_host.ctypes.data,
            qo_indptr_host=self.qo_indptr_host.ctypes.data, kv_fp8=int(self.kv_fp8),
            k_scale=self.k_scale, v_scale=self.v_scale, reserved0=0)

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr_host[-1])

    @property
    def num_rows(self) -> int:
        return self.total_q * self.num_q_heads


def plan_params(mode: str = "critical_wave", **kw) -> PlanParams:
    p = PlanParams()
    load().splitkv_plan_params_default(ctypes.byref(p))
    p.mode = PLAN_UNIFORM if mode == "uniform" else PLAN_CRITICAL_WAVE
    for k, v in kw.items():
        if not hasattr(p, k):
            raise TypeError(f"unknown plan parameter {k}")
        setattr(p, k, v)
    return p


class Plan:
    """Owner of a ``splitkv_plan_t`` (host-side split plan and task list)."""

    def __init__(self, handle: ctypes.c_void_p, problem: AttentionProblem):
        self._h = handle
        self.batch = problem.batch
        lib = load()
        self.num_tasks = int(lib.splitkv_plan_num_tasks(handle))
        self.num_chunk_tasks = int(lib.splitkv_plan_num_chunk_tasks(handle))
        self.num_pair_tasks = int(lib.splitkv_plan_num_pair_tasks(handle))
        self.num_states = int(lib.splitkv_plan_num_states(handle))
        self.num_rows = int(lib.splitkv_plan_num_rows(handle))
        self.workspace_bytes = int(lib.splitkv_workspace_bytes(handle))
        self.kernel_path = int(lib.splitkv_plan_kernel_path(handle))
        self.trace_records = int(lib.splitkv_plan_trace_records(handle))
        self.overlap_ctas = int(lib.splitkv_plan_overlap_ctas(handle))

    @property
    def handle(self):
        return self._h

    def splits(self) -> np.ndarray:
        out = np.zeros(self.batch, dtype=np.int32)
        _check(load().splitkv_plan_splits(self._h, out.ctypes.data_as(_ip)))
        return out

    def state_indptr(self) -> np.ndarray:
        out = np.zeros(self.num_rows + 1, dtype=np.int32)
        _check(load().splitkv_plan_state_indptr(self._h, out.ctypes.data_as(_ip)))
        return out

    def split_ranges(self, b: int) -> np.ndarray:
        n = int(self.splits()[b])
        out = np.zeros(2 * n, dtype=np.int32)
        _check(load().splitkv_plan_split_ranges(self._h, b, out.ctypes.data_as(_ip)))
        return out.reshape(n, 2)

    @property
    def partial_dtype(self):
        """torch dtype of the plan's partial outputs (float32, or bfloat16)."""
        return torch.bfloat16 if load().splitkv_plan_partial_dtype(self._h) == BF16 else torch.float32

    @property
    def interleaved(self) -> bool:
        """True when split r of each request holds its pages r, r + n, r + 2n, ..."""
        return bool(load().splitkv_plan_interleaved(self._h))

    def chunk_requests(self) -> np.ndarray:
        """Per request: 1 when it runs on the chunk-tile kernel, 2 on the paired-tile
        kernel, else 0."""
        out = np.zeros(self.batch, dtype=np.int32)
        _check(load().splitkv_plan_chunk_requests(self._h, out.ctypes.data_as(_ip)))
        return out

    def scores(self) -> np.ndarray:
        out = np.zeros(4, dtype=np.float64)
        _check(load().splitkv_plan_scores(self._h, out.ctypes.data_as(_dp)))
        return out

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.splitkv_plan_destroy(h)
            self._h = None


def splitkv_plan(problem: AttentionProblem, params: Optional[PlanParams] = None) -> Plan:
    h = ctypes.c_void_p()
    _check(load().splitkv_plan(ctypes.byref(problem._s), ctypes.byref(params) if params is not None else None,
                               ctypes.byref(h)))
    return Plan(h, problem)


def alloc_workspace(plan: Plan, device=None) -> torch.Tensor:
    """A device byte buffer of the plan's workspace size (256-byte aligned by the allocator)."""
    t = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device=device or "cuda")
    if t.data_ptr() % 256:
        raise RuntimeError("workspace allocation is not 256-byte aligned")
    return t


def splitkv_plan_upload(plan: Plan, workspace: torch.Tensor, stream=None):
    _check(load().splitkv_plan_upload(plan.handle, _ptr(workspace), workspace.numel(), _stream_handle(stream)))


def splitkv_partial(problem: AttentionProblem, plan: Plan, workspace: torch.Tensor, o_part: torch.Tensor,
                    lse_part: torch.Tensor, dev_error_word: Optional[torch.Tensor] = None, stream=None):
    _check(load().splitkv_partial(ctypes.byref(problem._s), plan.handle, _ptr(workspace), workspace.numel(),
                                  _ptr(o_part), _ptr(lse_part), _ptr(dev_error_word), _stream_handle(stream)))


def merge_states(o_part: torch.Tensor, lse_part: torch.Tensor, state_indptr: torch.Tensor, out: torch.Tensor,
                 lse_out: Optional[torch.Tensor] = None, stream=None):
    """merge_states for float32 o_part; merge_states_typed for bfloat16 o_part."""
    rows = int(state_indptr.shape[0]) - 1
    dim = int(o_part.shape[-1])
    if o_part.dtype == torch.float32:
        _check(load().merge_states(_ptr(o_part), _ptr(lse_part), _ptr(state_indptr), rows, dim, _ptr(out),
                                   _DTYPES[out.dtype], _ptr(lse_out), _stream_handle(stream)))
    else:
        _check(load().merge_states_typed(_ptr(o_part), _DTYPES[o_part.dtype], _ptr(lse_part), _ptr(state_indptr),
                                         rows, dim, _ptr(out), _DTYPES[out.dtype], _ptr(lse_out),
                                         _stream_handle(stream)))


def splitkv_decode(problem: AttentionProblem, plan: Plan, workspace: torch.Tensor, out: torch.Tensor,
                   lse_out: Optional[torch.Tensor] = None, dev_error_word: Optional[torch.Tensor] = None,
                   stream=None):
    _check(load().splitkv_decode(ctypes.byref(problem._s), plan.handle, _ptr(workspace), workspace.numel(),
                                 _ptr(out), _ptr(lse_out), _ptr(dev_error_word), _stream_handle(stream)))


def splitkv_decode_static(problem: AttentionProblem, plan: Plan, out: torch.Tensor,
                          lse_out: Optional[torch.Tensor] = None, dev_error_word: Optional[torch.Tensor] = None,
                          stream=None):
    """splitkv_decode for callers that cannot allocate device memory: the
    scratch is the library's own static device array (see include/splitkv.h)."""
    _check(load().splitkv_decode_static(ctypes.byref(problem._s), plan.handle, _ptr(out), _ptr(lse_out),
                                        _ptr(dev_error_word), _stream_handle(stream)))


def read_device_error(dev_error_word: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      clear: bool = False, stream=None):
    """(status, raw word) of the device error word; synchronises the stream."""
    raw = ctypes.c_int32(0)
    st = load().splitkv_read_device_error(_ptr(dev_error_word), _ptr(workspace), 1 if clear else 0,
                                          ctypes.byref(raw), _stream_handle(stream))
    return st, raw.value


def read_static_device_error(clear: bool = False, stream=None):
    """(status, raw word) of the static array's error word (splitkv_decode_static
    calls made without an error word); synchronises the stream."""
    raw = ctypes.c_int32(0)
    st = load().splitkv_read_static_device_error(1 if clear else 0, ctypes.byref(raw), _stream_handle(stream))
    return st, raw.value


def trace_read(plan: Plan, workspace: torch.Tensor, stream=None) -> np.ndarray:
    """The plan's trace records from the workspace (structured numpy array with
    fields start_ns, end_ns, id, sm, kind, cta); synchronises the stream."""
    out = np.zeros(plan.trace_records, dtype=TRACE_DTYPE)
    _check(load().splitkv_trace_read(plan.handle, _ptr(workspace), workspace.numel(),
                                     ctypes.c_void_p(out.ctypes.data), _stream_handle(stream)))
    return out


def trace_tail_idle(records: np.ndarray, kinds=(TRACE_ATTENTION, TRACE_REDUCTION), num_sms: int = 0) -> dict:
    """Tail idle of the stage made of the records of the given kinds (LiquidCP
    Section 3: each SM's wait after its last task until the stage finishes,
    summed, over total SM-time)."""
    rec = np.ascontiguousarray(records, dtype=TRACE_DTYPE)
    mask = 0
    for k in kinds:
        mask |= 1 << int(k)
    st = TraceStats()
    _check(load().splitkv_trace_tail_idle(ctypes.c_void_p(rec.ctypes.data), len(rec), mask, num_sms,
                                          ctypes.byref(st)))
    return {f: getattr(st, f) for f, _ in TraceStats._fields_}


def _model_args(seqs, num_ctas, warps_per_cta, q_heads, rho, delta_attn, delta_red, gamma, adopt_margin,
                decode_qlen_max=16):
    arr = (SeqModel * len(seqs))()
    for i, s in enumerate(seqs):
        arr[i] = SeqModel(int(s[0]), int(s[1]), int(s[2]), int(s[3]))
    mp = ModelParams(num_ctas=num_ctas, warps_per_cta=warps_per_cta, q_heads=q_heads,
                     decode_qlen_max=decode_qlen_max, rho=rho, delta_attn=delta_attn, delta_red=delta_red,
                     gamma=gamma, adopt_margin=adopt_margin)
    return arr, mp


def model_simulate(seqs, splits, *, num_ctas, warps_per_cta=12, q_heads=1, rho=0.43, delta_attn=32.0,
                   delta_red=2.5, gamma=0.47, adopt_margin=0.10, decode_qlen_max=16):
    """(score, attention completion) of a split plan under the critical-wave
    model; ``seqs`` are (tiles, tasks_per_split, vectors, q_len) tuples."""
    arr, mp = _model_args(seqs, num_ctas, warps_per_cta, q_heads, rho, delta_attn, delta_red, gamma,
                          adopt_margin, decode_qlen_max)
    sp = np.ascontiguousarray(splits, dtype=np.int32)
    score, attn = ctypes.c_double(), ctypes.c_double()
    _check(load().splitkv_model_simulate(arr, len(seqs), sp.ctypes.data_as(_ip), ctypes.byref(mp),
                                         ctypes.byref(score), ctypes.byref(attn)))
    return score.value, attn.value


def model_plan(seqs, *, num_ctas, warps_per_cta=12, q_heads=1, rho=0.43, delta_attn=32.0, delta_red=2.5,
               gamma=0.47, adopt_margin=0.10, min_splits=1, max_splits=64, decode_qlen_max=16):
    """(splits, [base, chosen, search, reference] scores) from the planner."""
    arr, mp = _model_args(seqs, num_ctas, warps_per_cta, q_heads, rho, delta_attn, delta_red, gamma,
                          adopt_margin, decode_qlen_max)
    out = np.zeros(len(seqs), dtype=np.int32)
    sc = np.zeros(4, dtype=np.float64)
    _check(load().splitkv_model_plan(arr, len(seqs), ctypes.byref(mp), min_splits, max_splits,
                                     out.ctypes.data_as(_ip), sc.ctypes.data_as(_dp)))
    return out, sc


def profile_begin():
    """Start recording every kernel launch of the library (events on its stream)."""
    _check(load().splitkv_profile_begin())


def profile_end() -> dict:
    """Stop recording; {kernel name: (launches, total device ms)} for kernels that ran."""
    arr = (KernelTime * len(KERNEL_NAMES))()
    _check(load().splitkv_profile_end(arr))
    return {KERNEL_NAMES[k]: (int(arr[k].launches), float(arr[k].total_ms))
            for k in range(len(KERNEL_NAMES)) if arr[k].launches > 0}


def debug_set_inject(mode: int):
    """Test hook: 1 makes the persistent kernels withhold their tasks so their
    bounded waits expire (SPLITKV_ERR_TIMEOUT in the error word); 0 restores."""
    _check(load().splitkv_debug_set_inject(int(mode)))
