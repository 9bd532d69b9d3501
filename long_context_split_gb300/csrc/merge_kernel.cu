// LSE-weighted merge of partial attention states (LiquidCP Eq. 1; Helix
// Parallelism, "Attention-Phase Configuration" step 3):
//   lse = log sum_r exp(lse_r),  o = sum_r exp(lse_r - lse) * o_r.
// One warp per output row; lanes split the row into float4 columns, so each
// partial row is read once with coalesced 16-byte loads.  Splits are added in
// index order, so the result does not depend on timing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "splitkv.h"
#include "internal.h"
#include "partial_io.cuh"

namespace skv {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxC4PerLane = 8;   // rows up to 8 * 32 * 4 = 1024 floats

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

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
merge_states_kernel(const void* __restrict__ o_part, int part_bf16, const float* __restrict__ lse_part,
                    const int32_t* __restrict__ indptr, int rows, int dim, void* __restrict__ out,
                    int out_bf16, float* __restrict__ lse_out) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int s0 = indptr[row];
    const int n = indptr[row + 1] - s0;
    float m = -INFINITY;
    for (int r = lane; r < n; r += 32) m = fmaxf(m, lse_part[s0 + r]);
    m = warp_max(m);
    const int d4 = dim >> 2;
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
    // columns in float4 units: lane handles c = lane + 32 u; every lane runs every
    // shuffle, lanes past the row's width only skip the loads
    float4 acc[kMaxC4PerLane];
#pragma unroll
    for (int u = 0; u < kMaxC4PerLane; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r0 = 0; r0 < n; r0 += 32) {
        // lane j holds the weight of split r0 + j
        float w = 0.f;
        if (r0 + lane < n) w = expf(lse_part[s0 + r0 + lane] - m) * inv;
        const int cnt = min(32, n - r0);
        int j = 0;
        // two splits at a time: both rows' loads in flight before their multiply-adds
        for (; j + 2 <= cnt; j += 2) {
            const float w0 = __shfl_sync(0xffffffffu, w, j), w1 = __shfl_sync(0xffffffffu, w, j + 1);
            const size_t src0 = (size_t)(s0 + r0 + j) * dim, src1 = src0 + dim;
            float4 v0[kMaxC4PerLane], v1[kMaxC4PerLane];
#pragma unroll
            for (int u = 0; u < kMaxC4PerLane; ++u) {
                const int c = lane + 32 * u;
                if (c < d4) {
                    v0[u] = load_part4(o_part, part_bf16, src0 + 4 * c);
                    v1[u] = load_part4(o_part, part_bf16, src1 + 4 * c);
                }
            }
#pragma unroll
            for (int u = 0; u < kMaxC4PerLane; ++u) {
                const int c = lane + 32 * u;
                if (c < d4) {
                    acc[u].x = fmaf(w1, v1[u].x, fmaf(w0, v0[u].x, acc[u].x));
                    acc[u].y = fmaf(w1, v1[u].y, fmaf(w0, v0[u].y, acc[u].y));
                    acc[u].z = fmaf(w1, v1[u].z, fmaf(w0, v0[u].z, acc[u].z));
                    acc[u].w = fmaf(w1, v1[u].w, fmaf(w0, v0[u].w, acc[u].w));
                }
            }
        }
        for (; j < cnt; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
            const size_t src = (size_t)(s0 + r0 + j) * dim;
#pragma unroll
            for (int u = 0; u < kMaxC4PerLane; ++u) {
                const int c = lane + 32 * u;
                if (c < d4) {
                    const float4 v = load_part4(o_part, part_bf16, src + 4 * c);
                    acc[u].x = fmaf(wj, v.x, acc[u].x);
                    acc[u].y = fmaf(wj, v.y, acc[u].y);
                    acc[u].z = fmaf(wj, v.z, acc[u].z);
                    acc[u].w = fmaf(wj, v.w, acc[u].w);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kMaxC4PerLane; ++u) {
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
    {
        ProfileScope ps(SPLITKV_KERNEL_MERGE, s);
        merge_states_kernel<<<grid, kWarpsPerBlock * 32, 0, s>>>(o_part, part_bf16, lse_part, indptr, rows, dim,
                                                               out, out_bf16, lse_out);
    }
    return cudaGetLastError();
}

}  // namespace skv
