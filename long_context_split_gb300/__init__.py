"""GB300-native split-KV decode attention with an exact LSE merge.

The compute path is ``libsplitkv.so`` (hand-written sm_103a CUDA kernels
behind the C ABI of ``include/splitkv.h``); this package is its thin Python
binding.  Names follow the C ABI: ``splitkv_plan``, ``splitkv_partial``,
``merge_states``, ``splitkv_decode``.
"""
from ._lib import (  # noqa: F401
    BF16, ERR_CUDA, ERR_DEVICE_CHECK, ERR_INVALID_ARG, ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_WORKSPACE, F32,
    GQA, MLA, OK, PLAN_CRITICAL_WAVE, PLAN_UNIFORM, AttentionProblem, Plan, SplitKVError, alloc_workspace,
    KERNEL_NAMES, debug_set_inject, load, merge_states, model_plan, model_simulate, plan_params, profile_begin, profile_end,
    read_device_error, read_static_device_error, trace_read, trace_tail_idle, TRACE_ATTENTION,
    TRACE_REDUCTION, TRACE_CHUNK, TRACE_MLA_ITEM, TRACE_PAIR, splitkv_decode, splitkv_decode_static, splitkv_partial, splitkv_plan, splitkv_plan_upload,
)
from .attention import SplitKVAttention  # noqa: F401
from . import roofline  # noqa: F401


def build(verbose: bool = False) -> str:
    """Compile libsplitkv.so in-tree for sm_103a (see ``_build.py``)."""
    from . import _build
    return _build.build(verbose=verbose)
