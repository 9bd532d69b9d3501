// LSE-weighted merge of partial attention states (LiquidCP Eq. 1; Helix
// Parallelism, "Attention-Phase Configuration" step 3):
//   lse = log sum_r exp(lse_r),  o = sum_r exp(lse_r - lse) * o_r.
// One warp per output row; lanes split the row into float4 columns, so each
// partial row is read once with coalesced 16-byte loads.  Splits are added in
// index order, so the result does not depend on timing.  A merge is a chain of
// dependent reads (offsets, LSEs, rows), so the kernel keeps several split rows'
// loads in flight at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "splitkv.h"
#include "internal.h"
#include "partial_io.cuh"

namespace skv {
namespace {

constexpr int kWarpsPerBlock = 8;

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

// C4: float4 columns per lane (rows up to 128 C4 floats).  Splits are read G rows at a
// time with all their loads in flight together, and the first G rows are requested
// with the LSEs, before the weights that need them are known.
template <int C4>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
merge_states_kernel(const void* __restrict__ o_part, int part_bf16, const float* __restrict__ lse_part,
                    const int32_t* __restrict__ indptr, int rows, int dim, void* __restrict__ out,
                    int out_bf16, float* __restrict__ lse_out) {
    constexpr int G = C4 == 1 ? 8 : (C4 == 2 ? 4 : 2);
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int s0 = indptr[row];
    const int n = indptr[row + 1] - s0;
    const int d4 = dim >> 2;
    // rows r0 .. r0 + G - 1 (those that exist) into v
    auto load_group = [&](int r0, float4 (&v)[G][C4]) {
#pragma unroll
        for (int k = 0; k < G; ++k)
#pragma unroll
            for (int u = 0; u < C4; ++u) {
                const int c = lane + 32 * u;
                v[k][u] = (r0 + k < n && c < d4) ? load_part4(o_part, part_bf16, (size_t)(s0 + r0 + k) * dim + 4 * c)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
    };
    float4 v[G][C4];
    load_group(0, v);
    float m = -INFINITY;
    for (int r = lane; r < n; r += 32) m = fmaxf(m, lse_part[s0 + r]);
    m = warp_max(m);
    if (m == -INFINITY) {
        for (int c = lane; c < d4; c += 32) {
            if (out_bf16) {
                __nv_bfloat162 z = __floats2bfloat162_rn(0.f, 0.f);
                __nv_bfloat162* o = (__nv_bfloat162*)out + ((size_t)row * dim + 4 * c) / 2;
                o[0] = z;
                o[1] = z;
            } else {
                ((float4*)out)[(size_t)row * d4 + c] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (lse_out && lane == 0) lse_out[row] = -INFINITY;
        return;
    }
    float denom = 0.f;
    for (int r = lane; r < n; r += 32) denom += expf(lse_part[s0 + r] - m);
    denom = warp_sum(denom);
    const float inv = 1.f / denom;
    float4 acc[C4];
#pragma unroll
    for (int u = 0; u < C4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    // splits in index order, G at a time; lane j of a 32-split window holds split j's weight
    float w = 0.f;
    for (int r0 = 0; r0 < n; r0 += G) {
        if (r0 % 32 == 0) w = (r0 + lane < n) ? expf(lse_part[s0 + r0 + lane] - m) * inv : 0.f;
        if (r0 > 0) load_group(r0, v);
#pragma unroll
        for (int k = 0; k < G; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, (r0 + k) & 31);
            if (r0 + k < n) {
#pragma unroll
                for (int u = 0; u < C4; ++u) {
                    acc[u].x = fmaf(wk, v[k][u].x, acc[u].x);
                    acc[u].y = fmaf(wk, v[k][u].y, acc[u].y);
                    acc[u].z = fmaf(wk, v[k][u].z, acc[u].z);
                    acc[u].w = fmaf(wk, v[k][u].w, acc[u].w);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < C4; ++u) {
        const int c = lane + 32 * u;
        if (c >= d4) continue;
        if (out_bf16) {
            __nv_bfloat162* o = (__nv_bfloat162*)out + ((size_t)row * dim + 4 * c) / 2;
            o[0] = __floats2bfloat162_rn(acc[u].x, acc[u].y);
            o[1] = __floats2bfloat162_rn(acc[u].z, acc[u].w);
        } else {
            ((float4*)out)[(size_t)row * d4 + c] = acc[u];
        }
    }
    if (lse_out && lane == 0) lse_out[row] = m + logf(denom);
}

}  // namespace

cudaError_t launch_merge(const void* o_part, int part_bf16, const float* lse_part, const int32_t* indptr,
                         int32_t rows, int32_t dim, void* out, int out_bf16, float* lse_out, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    dim3 grid((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
    const int c4 = (dim / 4 + 31) / 32;   // float4 columns per lane
    {
        ProfileScope ps(SPLITKV_KERNEL_MERGE, s);
        if (c4 <= 1)
            merge_states_kernel<1><<<grid, kWarpsPerBlock * 32, 0, s>>>(o_part, part_bf16, lse_part, indptr, rows,
                                                                      dim, out, out_bf16, lse_out);
        else if (c4 <= 2)
            merge_states_kernel<2><<<grid, kWarpsPerBlock * 32, 0, s>>>(o_part, part_bf16, lse_part, indptr, rows,
                                                                      dim, out, out_bf16, lse_out);
        else if (c4 <= 4)
            merge_states_kernel<4><<<grid, kWarpsPerBlock * 32, 0, s>>>(o_part, part_bf16, lse_part, indptr, rows,
                                                                      dim, out, out_bf16, lse_out);
        else if (c4 <= 8)
            merge_states_kernel<8><<<grid, kWarpsPerBlock * 32, 0, s>>>(o_part, part_bf16, lse_part, indptr, rows,
                                                                      dim, out, out_bf16, lse_out);
        else
            return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace skv
