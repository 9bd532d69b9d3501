// CUDA-core partial attention in float32 arithmetic, for any supported shape,
// for float32 storage (the reference-precision path) and for E4M3 KV caches
// the other kernels do not take (absorbed MLA, other head dims and pages).
//
// Partial state of a query row over one split (Helix Parallelism,
// "Attention-Phase Configuration" step 2; LiquidCP Section 3): scores
// s_j = scale * q.k_j over the split's keys (cut by the row's causal limit),
// online softmax in base 2, output normalised over the split and the
// natural-log LSE.  An empty key set writes o = 0, lse = -inf.
//
// One CTA per task, one warp per query row.  Lanes score 32 keys at a time
// (each lane walks one key row), then accumulate p_j * v_j with the value
// columns spread over the lanes (coalesced row reads).  Splits whose key and
// value rows fit in shared memory are staged first (STAGED): the CTA reads the
// split's page ids once and copies every key's rows with cp.async in one
// round, so a short split costs a few memory round trips instead of several
// per 32 keys -- what bounds a small batch, whose caches are cold in L2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// E4M3 code (OCP FP8, no infinities) as a distinct storage type
struct e4m3_t {
    uint8_t c;
};

// two E4M3 codes in the low 16 bits -> f16 pair (low code in the low half); exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(d) : "r"(w));
    return d;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float load_elem(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ float load_elem(const e4m3_t* p, size_t i) {
    return f16x2_to_float2(e4m3x2_to_f16x2(p[i].c)).x;
}

// dot(q_s[0:d), k[0:d)) with 16-byte loads of the key row
__device__ __forceinline__ float dot_row(const float* q_s, const float* k, int d) {
    float acc = 0.f;
    const float4* k4 = (const float4*)k;
#pragma unroll 16
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
#pragma unroll 8
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

// the same over a row of E4M3 codes (16-byte loads: sixteen codes)
__device__ __forceinline__ float dot_row(const float* q_s, const e4m3_t* k, int d) {
    float acc = 0.f;
    const uint4* k16 = (const uint4*)k;
#pragma unroll 4
    for (int c = 0; c < d / 16; ++c) {
        const uint4 raw = k16[c];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 lo = f16x2_to_float2(e4m3x2_to_f16x2(w[e]));
            const float2 hi = f16x2_to_float2(e4m3x2_to_f16x2(w[e] >> 16));
            acc = fmaf(q_s[16 * c + 4 * e], lo.x, acc);
            acc = fmaf(q_s[16 * c + 4 * e + 1], lo.y, acc);
            acc = fmaf(q_s[16 * c + 4 * e + 2], hi.x, acc);
            acc = fmaf(q_s[16 * c + 4 * e + 3], hi.y, acc);
        }
    }
    return acc;
}

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Shared-memory layout of a staged split: the rows' queries (float), the split's page ids,
// then each key's K row and (GQA) V row, each padded by 16 bytes so that the lanes' row
// reads fall on distinct banks
struct StagedLayout {
    int kstride, vstride;      // bytes per staged key / value row
    size_t pages_off, k_off, v_off, bytes;
    __host__ __device__ StagedLayout(int dqk, int dv, int elem, int mla, int rows, int max_keys, int page) {
        kstride = dqk * elem + 16;
        vstride = mla ? 0 : dv * elem + 16;
        pages_off = (size_t)rows * dqk * 4;
        const int max_pages = (max_keys + page - 1) / page + 1;
        k_off = (pages_off + (size_t)max_pages * 4 + 15) & ~(size_t)15;
        v_off = k_off + (size_t)max_keys * kstride;
        bytes = v_off + (size_t)max_keys * vstride;
    }
};

// T: storage type of the query; TKV: of the caches (T, or E4M3 codes with bf16 queries;
// their key scale is folded into the score scale, the value scale into the normalisation)
// LSE-weighted merge of one request's partial states into its output rows (LiquidCP
// Eq. 1; Helix Parallelism, "Attention-Phase Configuration" step 3): lse = log sum_r
// exp(lse_r), o = sum_r exp(lse_r - lse) o_r, splits added in index order.  A warp per
// row (row v = token * Hq + head), lanes over groups of four columns; the states were
// written by other CTAs, so they are read from L2.
__device__ void merge_request(const KernelArgs& a, const ReqDesc& rq, int warp, int lane) {
    const int n = rq.n_splits, Dv = a.head_dim_v;
    for (int v = warp; v < rq.q_len * a.num_q_heads; v += kRows) {
        const size_t st0 = (size_t)rq.state_base + (size_t)v * n;
        const size_t orow = (size_t)rq.q_start * a.num_q_heads + v;
        float m = -INFINITY;
        for (int r = lane; r < n; r += 32) m = fmaxf(m, __ldcg(a.lse_part + st0 + r));
        m = warp_max(m);
        float den = 0.f;
        if (m != -INFINITY)
            for (int r = lane; r < n; r += 32) den += expf(__ldcg(a.lse_part + st0 + r) - m);
        den = warp_sum(den);
        const float inv = den > 0.f ? 1.f / den : 0.f;
        for (int c = 4 * lane; c < Dv; c += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m != -INFINITY) {
                for (int r = 0; r < n; ++r) {
                    const float w = expf(__ldcg(a.lse_part + st0 + r) - m) * inv;
                    const float4 o = load_part4(a.o_part, a.part_bf16, (st0 + r) * Dv + c);
                    acc.x = fmaf(w, o.x, acc.x);
                    acc.y = fmaf(w, o.y, acc.y);
                    acc.z = fmaf(w, o.z, acc.z);
                    acc.w = fmaf(w, o.w, acc.w);
                }
            }
            if (a.out_bf16) {
                __nv_bfloat162* op = (__nv_bfloat162*)((__nv_bfloat16*)a.out + orow * Dv + c);
                op[0] = __floats2bfloat162_rn(acc.x, acc.y);
                op[1] = __floats2bfloat162_rn(acc.z, acc.w);
            } else {
                *(float4*)((float*)a.out + orow * Dv + c) = acc;
            }
        }
        if (lane == 0 && a.lse_out) a.lse_out[orow] = (m == -INFINITY) ? -INFINITY : m + logf(den);
    }
}

// STAGED: every task's dense key slots number at most max_keys (the launch sized shared
// memory for them)
template <typename T, typename TKV, int DVL, bool STAGED>
__global__ void __launch_bounds__(kRows * 32, 1)
generic_partial_kernel(KernelArgs a, int max_keys) {
    extern __shared__ __align__(16) float q_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the request table (when small) is read together with the task descriptor: one round
    // trip instead of two dependent ones
    constexpr int kReqCache = 64;
    __shared__ ReqDesc req_s[kReqCache];
    const TaskDesc t = a.tasks[blockIdx.x];
    const bool cached = a.num_reqs <= kReqCache;
    if (cached && threadIdx.x < a.num_reqs) req_s[threadIdx.x] = a.reqs[threadIdx.x];
    __syncthreads();
    const ReqDesc rq = cached ? req_s[t.b] : a.reqs[t.b];
    const int row = t.row_begin + warp;
    const StagedLayout lay(a.head_dim_qk, a.head_dim_v, (int)sizeof(TKV), a.mla, kRows, max_keys, a.page_size);
    int* pg_s = (int*)((unsigned char*)q_smem + lay.pages_off);
    unsigned char* k_s = (unsigned char*)q_smem + lay.k_off;
    unsigned char* v_s = (unsigned char*)q_smem + lay.v_off;
    if constexpr (STAGED) {
        // the keys the task's last row may see, as dense slots of the task's pages
        const int P = a.page_size, Dqk = a.head_dim_qk;
        const int i_last = (t.row_end - 1) / a.group;
        const int ke_blk = min(t.key_end, rq.seq_len - rq.q_len + i_last + 1);
        const int ps = max(1, t.page_stride), pb = t.key_begin / P;
        const int npg = ke_blk > t.key_begin ? ((ke_blk + P - 1) / P - pb + ps - 1) / ps : 0;
        for (int k = threadIdx.x; k < npg; k += blockDim.x) pg_s[k] = a.page_table[rq.page_row + pb + k * ps];
        __syncthreads();
        // each key's K row (and V row) in 16-byte copies, all in flight together; V row r
        // starts at element r * Dqk of the V cache, as in the streaming form
        const int kc = Dqk * (int)sizeof(TKV) / 16, vc = a.mla ? 0 : a.head_dim_v * (int)sizeof(TKV) / 16;
        const int per_key = kc + vc;
        for (int idx = threadIdx.x; idx < npg * P * per_key; idx += blockDim.x) {
            const int v = idx / per_key, c = idx - v * per_key;
            const int j = (pb + (v / P) * ps) * P + v % P;
            const int page = pg_s[v / P];
            if (j >= ke_blk || page < 0 || page >= a.num_pages) continue;
            const size_t r = a.mla ? ((size_t)page * P + v % P) : (((size_t)page * a.num_kv_heads + t.kv_head) * P + v % P);
            if (c < kc)
                cp_async16(k_s + (size_t)v * lay.kstride + c * 16, (const unsigned char*)a.k_cache + (r * Dqk) * sizeof(TKV) + c * 16);
            else
                cp_async16(v_s + (size_t)v * lay.vstride + (c - kc) * 16,
                           (const unsigned char*)a.v_cache + (r * Dqk) * sizeof(TKV) + (c - kc) * 16);
        }
        // the warp's query row, while the copies are in flight
        if (row < t.row_end) {
            const int i = row / a.group, h = t.kv_head * a.group + row % a.group;
            const T* qp = (const T*)a.q + ((size_t)(rq.q_start + i) * a.num_q_heads + h) * Dqk;
            for (int d = lane; d < Dqk; d += 32) q_smem[warp * Dqk + d] = load_elem(qp, d);
        }
        cp_async_wait_all();
        __syncthreads();
    }
    if (row < t.row_end) {
        const int g = a.group;
        const int i = row / g;
        const int h = t.kv_head * g + row % g;
        const int tok = rq.q_start + i;
        const int limit = rq.seq_len - rq.q_len + i;            // last key this row may see
        const int kb = t.key_begin;
        const int ke = min(t.key_end, limit + 1);
        const int Dqk = a.head_dim_qk, Dv = a.head_dim_v, P = a.page_size;
        const T* q = (const T*)a.q + ((size_t)tok * a.num_q_heads + h) * Dqk;
        const TKV* kc = (const TKV*)a.k_cache;
        const TKV* vc = (const TKV*)a.v_cache;
        float* q_s = q_smem + warp * Dqk;
        if constexpr (!STAGED)
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
        // each lane's page id is read one chunk ahead, off the chunk's chain of dependent loads
        auto key_of = [&](int c0) { const int v = c0 + lane; return (pb + (v / P) * ps) * P + v % P; };
        auto has_key = [&](int c0) { return c0 + lane < nv && key_of(c0) < ke; };
        int next_page = 0;
        if constexpr (!STAGED) next_page = (nv > 0 && has_key(0)) ? a.page_table[rq.page_row + key_of(0) / P] : 0;
        for (int c0 = 0; c0 < nv; c0 += 32) {
            const int j = key_of(c0);
            int page = next_page;
            if constexpr (STAGED) {
                if (has_key(c0)) page = pg_s[(c0 + lane) / P];
            } else {
                if (c0 + 32 < nv && has_key(c0 + 32)) next_page = a.page_table[rq.page_row + key_of(c0 + 32) / P];
            }
            float s = -INFINITY;
            // element offset of key j's value row (STAGED: the dense slot's row in shared memory)
            size_t row_off = 0;
            if (has_key(c0)) {
                if (page < 0 || page >= a.num_pages) {
                    set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
                } else if constexpr (STAGED) {
                    const int v = c0 + lane;
                    row_off = (size_t)v * (a.mla ? lay.kstride : lay.vstride) / sizeof(TKV);
                    s = dot_row(q_s, (const TKV*)(k_s + (size_t)v * lay.kstride), Dqk) * a.scale_log2;
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
            // p_j v_j over the chunk's keys, U keys at a time so that their value loads are in
            // flight together; a key of weight 0 loads nothing (its slot may hold anything, and
            // 0 * NaN is not 0)
            const int cnt = min(32, nv - c0);
            constexpr int U = DVL <= 2 ? 16 : (DVL <= 4 ? 8 : 2);
            // value rows: the cache, or (STAGED) the staged rows (MLA: the key rows)
            const TKV* vbase = STAGED ? (const TKV*)(a.mla ? k_s : v_s) : vc;
            int jj = 0;
            for (; jj + U <= cnt; jj += U) {
                float pj[U], vv[U][DVL];
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    pj[k] = __shfl_sync(0xffffffffu, p, jj + k);
                    const size_t vo = __shfl_sync(0xffffffffu, row_off, jj + k);
#pragma unroll
                    for (int c = 0; c < DVL; ++c) vv[k][c] = pj[k] != 0.f ? load_elem(vbase, vo + lane + 32 * c) : 0.f;
                }
#pragma unroll
                for (int k = 0; k < U; ++k)
#pragma unroll
                    for (int c = 0; c < DVL; ++c) acc[c] = fmaf(pj[k], vv[k][c], acc[c]);
            }
            for (; jj < cnt; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
                const size_t vo = __shfl_sync(0xffffffffu, row_off, jj);
                if (pj != 0.f) {
#pragma unroll
                    for (int c = 0; c < DVL; ++c) acc[c] = fmaf(pj, load_elem(vbase, vo + lane + 32 * c), acc[c]);
                }
            }
            m = m_new;
        }
        const size_t state = (size_t)rq.state_base + ((size_t)i * a.num_q_heads + h) * rq.n_splits + t.split;
        const bool empty = (ke <= kb) || !(l > 0.f);
        const float inv = empty ? 0.f : a.v_scale / l;   // v_scale: 1 unless the values are E4M3 codes
#pragma unroll
        for (int c = 0; c < DVL; ++c) store_part1(a.o_part, a.part_bf16, state * Dv + lane + 32 * c, acc[c] * inv);
        if (lane == 0) a.lse_part[state] = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
    }
    // fused decode: the task counts in for its request once every row's state is written;
    // the request's last task merges its splits into the output (no CTA waits on another)
    if (a.fused) {
        __shared__ int last;
        __syncthreads();
        if (threadIdx.x == 0) {
            // the barrier orders every thread's state stores before this fence, whose
            // cumulativity carries them ahead of the count
            __threadfence();
            last = atomicAdd(&a.counters[t.b], 1) == rq.n_tasks - 1;
            if (last) __threadfence();
        }
        __syncthreads();
        if (last) merge_request(a, rq, warp, lane);
        if (last && threadIdx.x == 0) a.counters[t.b] = 0;   // for the next launch
    }
}

// shared memory a staged launch may take (one CTA of 512 threads per SM)
constexpr size_t kStagedSmemLimit = 160 * 1024;

template <typename T, typename TKV, int DVL>
cudaError_t launch_t(const KernelArgs& a, int max_keys, cudaStream_t s) {
    const StagedLayout lay(a.head_dim_qk, a.head_dim_v, (int)sizeof(TKV), a.mla, kRows, max_keys, a.page_size);
    const bool staged = max_keys > 0 && lay.bytes <= kStagedSmemLimit;
    const size_t smem = staged ? lay.bytes : (size_t)kRows * a.head_dim_qk * sizeof(float);
    auto kern = staged ? generic_partial_kernel<T, TKV, DVL, true> : generic_partial_kernel<T, TKV, DVL, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    {
        ProfileScope ps(SPLITKV_KERNEL_GENERIC, s);
        kern<<<a.num_tasks, kRows * 32, smem, s>>>(a, max_keys);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic_partial(const KernelArgs& a, int bf16, int max_keys, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    const int dvl = a.head_dim_v / 32;
    if (a.head_dim_v % 32) return cudaErrorNotSupported;
    if ((((uintptr_t)a.k_cache) & 15) || (((uintptr_t)a.v_cache) & 15)) max_keys = 0;   // no 16-byte copies
    if (a.kv_fp8) {
        if (!bf16 || a.head_dim_qk % 16) return cudaErrorNotSupported;
        if (dvl == 2) return launch_t<__nv_bfloat16, e4m3_t, 2>(a, max_keys, s);
        if (dvl == 4) return launch_t<__nv_bfloat16, e4m3_t, 4>(a, max_keys, s);
        if (dvl == 16) return launch_t<__nv_bfloat16, e4m3_t, 16>(a, max_keys, s);
        return cudaErrorNotSupported;
    }
    if (bf16 ? (a.head_dim_qk % 8) : (a.head_dim_qk % 4)) return cudaErrorNotSupported;
    if (bf16) {
        if (dvl == 2) return launch_t<__nv_bfloat16, __nv_bfloat16, 2>(a, max_keys, s);
        if (dvl == 4) return launch_t<__nv_bfloat16, __nv_bfloat16, 4>(a, max_keys, s);
        if (dvl == 16) return launch_t<__nv_bfloat16, __nv_bfloat16, 16>(a, max_keys, s);
    } else {
        if (dvl == 2) return launch_t<float, float, 2>(a, max_keys, s);
        if (dvl == 4) return launch_t<float, float, 4>(a, max_keys, s);
        if (dvl == 16) return launch_t<float, float, 16>(a, max_keys, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace skv
