// Optional per-task trace records (splitkv_plan_params.trace): when the launch
// has a trace array, a task's claimer stamps its start (%globaltimer), SM and
// CTA, and every role that finishes a part of it raises its end with an atomic
// max -- the per-SM task timelines from which LiquidCP Section 3 measures tail
// idle (an SM's wait after its last task until the stage finishes).
#pragma once

#include <cuda_runtime.h>

#include "splitkv.h"

namespace skv {
namespace {

__device__ __forceinline__ unsigned long long trace_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int trace_smid() {
    int r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void trace_start(splitkv_trace_record* base, int id, int kind) {
    if (!base) return;
    splitkv_trace_record* r = base + id;
    const unsigned long long t = trace_now();
    r->start_ns = t;
    // the end starts at the start (the workspace may hold anything); the roles that finish
    // the unit raise it afterwards -- their atomic maxima come later in the same CTA's
    // release/acquire chain
    atomicExch((unsigned long long*)&r->end_ns, t);
    r->id = id;
    r->sm = trace_smid();
    r->kind = kind;
    r->cta = (int)blockIdx.x;
}

__device__ __forceinline__ void trace_end(splitkv_trace_record* base, int id) {
    if (!base) return;
    atomicMax((unsigned long long*)&base[id].end_ns, trace_now());
}

}  // namespace
}  // namespace skv
