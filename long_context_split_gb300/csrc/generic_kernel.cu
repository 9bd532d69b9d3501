// CUDA-core partial attention in float32 arithmetic, for any supported shape
// and for float32 storage (the reference-precision path).
//
// Partial state of a query row over one split (Helix Parallelism,
// "Attention-Phase Configuration" step 2; LiquidCP Section 3): scores
// s_j = scale * q.k_j over the split's keys (cut by the row's causal limit),
// online softmax in base 2, output normalised over the split and the
// natural-log LSE.  An empty key set writes o = 0, lse = -inf.
//
// One CTA per task, one warp per query row.  Lanes score 32 keys at a time
// (each lane walks one key row), then accumulate p_j * v_j with the value
// columns spread over the lanes (coalesced row reads).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "splitkv.h"
#include "internal.h"
#include "partial_io.cuh"

namespace skv {
namespace {

constexpr int kRows = 16;   // warps per CTA = rows per task

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float load_elem(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

// dot(q_s[0:d), k[0:d)) with 16-byte loads of the key row
__device__ __forceinline__ float dot_row(const float* q_s, const float* k, int d) {
    float acc = 0.f;
    const float4* k4 = (const float4*)k;
    for (int c = 0; c < d / 4; ++c) {
        float4 v = k4[c];
        acc = fmaf(q_s[4 * c + 0], v.x, acc);
        acc = fmaf(q_s[4 * c + 1], v.y, acc);
        acc = fmaf(q_s[4 * c + 2], v.z, acc);
        acc = fmaf(q_s[4 * c + 3], v.w, acc);
    }
    return acc;
}

__device__ __forceinline__ float dot_row(const float* q_s, const __nv_bfloat16* k, int d) {
    float acc = 0.f;
    const uint4* k8 = (const uint4*)k;
    for (int c = 0; c < d / 8; ++c) {
        uint4 raw = k8[c];
        const __nv_bfloat162* h = (const __nv_bfloat162*)&raw;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 f = __bfloat1622float2(h[e]);
            acc = fmaf(q_s[8 * c + 2 * e], f.x, acc);
            acc = fmaf(q_s[8 * c + 2 * e + 1], f.y, acc);
        }
    }
    return acc;
}

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

template <typename T, int DVL>
__global__ void __launch_bounds__(kRows * 32)
generic_partial_kernel(KernelArgs a) {
    extern __shared__ float q_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TaskDesc t = a.tasks[blockIdx.x];
    const ReqDesc rq = a.reqs[t.b];
    const int row = t.row_begin + warp;
    if (row >= t.row_end) return;
    const int g = a.group;
    const int i = row / g;
    const int h = t.kv_head * g + row % g;
    const int tok = rq.q_start + i;
    const int limit = rq.seq_len - rq.q_len + i;            // last key this row may see
    const int kb = t.key_begin;
    const int ke = min(t.key_end, limit + 1);
    const int Dqk = a.head_dim_qk, Dv = a.head_dim_v, P = a.page_size;
    const T* q = (const T*)a.q + ((size_t)tok * a.num_q_heads + h) * Dqk;
    const T* kc = (const T*)a.k_cache;
    const T* vc = (const T*)a.v_cache;
    float* q_s = q_smem + warp * Dqk;
    for (int d = lane; d < Dqk; d += 32) q_s[d] = load_elem(q, d);
    __syncwarp();

    float m = -INFINITY, l = 0.f;
    float acc[DVL];
#pragma unroll
    for (int c = 0; c < DVL; ++c) acc[c] = 0.f;

    // The task's keys: those of pages kb / P + k * ps (ps = 1: the range kb .. ke - 1), walked
    // as a dense index v = k * P + offset; key j = (kb / P + (v / P) ps) P + v % P, kept when < ke.
    const int ps = max(1, t.page_stride);
    const int pb = kb / P;
    const int pe = (ke + P - 1) / P;
    const int nv = (ke > kb) ? ((pe - pb + ps - 1) / ps) * P : 0;
    for (int c0 = 0; c0 < nv; c0 += 32) {
        const int v = c0 + lane;
        const int j = (pb + (v / P) * ps) * P + v % P;
        float s = -INFINITY;
        size_t row_off = 0;   // element offset of key j's row
        if (v < nv && j < ke) {
            const int page = a.page_table[rq.page_row + j / P];
            if (page < 0 || page >= a.num_pages) {
                set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
            } else {
                const int off = j % P;
                row_off = a.mla ? ((size_t)page * P + off) * Dqk
                                : (((size_t)page * a.num_kv_heads + t.kv_head) * P + off) * Dqk;
                s = dot_row(q_s, kc + row_off, Dqk) * a.scale_log2;
            }
        }
        const float cmax = warp_max(s);
        const float m_new = fmaxf(m, cmax);
        const float base = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m - base);
        const float p = exp2f(s - base);
        l = l * alpha + warp_sum(p);
#pragma unroll
        for (int c = 0; c < DVL; ++c) acc[c] *= alpha;
        const int cnt = min(32, nv - c0);
        for (int jj = 0; jj < cnt; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const size_t vo = __shfl_sync(0xffffffffu, row_off, jj);
            if (pj != 0.f) {
#pragma unroll
                for (int c = 0; c < DVL; ++c) acc[c] = fmaf(pj, load_elem(vc, vo + lane + 32 * c), acc[c]);
            }
        }
        m = m_new;
    }
    const size_t state = (size_t)rq.state_base + ((size_t)i * a.num_q_heads + h) * rq.n_splits + t.split;
    const bool empty = (ke <= kb) || !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
#pragma unroll
    for (int c = 0; c < DVL; ++c) store_part1(a.o_part, a.part_bf16, state * Dv + lane + 32 * c, acc[c] * inv);
    if (lane == 0) a.lse_part[state] = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
}

template <typename T, int DVL>
cudaError_t launch_t(const KernelArgs& a, cudaStream_t s) {
    size_t smem = (size_t)kRows * a.head_dim_qk * sizeof(float);
    auto kern = generic_partial_kernel<T, DVL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    {
        ProfileScope ps(SPLITKV_KERNEL_GENERIC, s);
        kern<<<a.num_tasks, kRows * 32, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic_partial(const KernelArgs& a, int bf16, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    const int dvl = a.head_dim_v / 32;
    if (a.head_dim_v % 32) return cudaErrorNotSupported;
    if (bf16 ? (a.head_dim_qk % 8) : (a.head_dim_qk % 4)) return cudaErrorNotSupported;
    if (bf16) {
        if (dvl == 2) return launch_t<__nv_bfloat16, 2>(a, s);
        if (dvl == 4) return launch_t<__nv_bfloat16, 4>(a, s);
        if (dvl == 16) return launch_t<__nv_bfloat16, 16>(a, s);
    } else {
        if (dvl == 2) return launch_t<float, 2>(a, s);
        if (dvl == 4) return launch_t<float, 4>(a, s);
        if (dvl == 16) return launch_t<float, 16>(a, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace skv
