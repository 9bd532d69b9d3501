// Loads and stores of partial attention states (the per-split normalised
// outputs o_r).  They are kept in float32, or -- when the plan asks for it --
// in bf16, rounded to nearest even once: the partial-state precision that
// LiquidCP Section 7 reports vLLM and MegaDCP exchanging between ranks (SGLang
// exchanges float32).  The LSE of every partial state stays float32 either way.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace skv {
namespace {

__device__ __forceinline__ uint32_t bf16x2_bits(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 bf16x2_floats(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// elements elem .. elem + 3 of a partial-state array (elem a multiple of 4), L2 only
__device__ __forceinline__ void store_part4(void* base, int bf16, size_t elem, float4 v) {
    if (bf16)
        __stcg((uint2*)((__nv_bfloat16*)base + elem), make_uint2(bf16x2_bits(v.x, v.y), bf16x2_bits(v.z, v.w)));
    else
        __stcg((float4*)((float*)base + elem), v);
}

__device__ __forceinline__ float4 load_part4(const void* base, int bf16, size_t elem) {
    if (bf16) {
        const uint2 w = __ldcg((const uint2*)((const __nv_bfloat16*)base + elem));
        const float2 a = bf16x2_floats(w.x), b = bf16x2_floats(w.y);
        return make_float4(a.x, a.y, b.x, b.y);
    }
    return __ldcg((const float4*)((const float*)base + elem));
}

__device__ __forceinline__ void store_part1(void* base, int bf16, size_t elem, float v) {
    if (bf16)
        ((__nv_bfloat16*)base)[elem] = __float2bfloat16_rn(v);
    else
        ((float*)base)[elem] = v;
}

}  // namespace
}  // namespace skv
