// Helpers shared by the tcgen05 kernels (absorbed-MLA and chunk tiles):
// mbarrier waits with a time limit, TMA bulk-tensor loads, shared-memory
// matrix descriptors, the kind::f16 instruction descriptor, tcgen05 MMA,
// commit, tensor-memory loads and stores, and the bf16 high/residual split.
// Each including translation unit gets its own copies (anonymous namespace).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace skv {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// Phase test of a barrier that only this CTA's threads, tcgen05.commit and TMA arrive on
// (CTA-scope acquire)
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait; false when it gave up (time limit, or the CTA is aborting)
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, bool watch) {
    const unsigned long long t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (watch && *abort_flag) return false;
            if (gtimer() - t0 > kWaitLimitNs) return false;
        }
    }
}

// Bounded wait; the completed-phase case (a ~14-cycle test) stays inline.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, bool watch) {
    if (mbar_try(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, watch);
}

// Warp-uniform bounded wait: when every lane's first test finds the phase complete the
// warp goes on at once; otherwise lane 0 waits, the verdict is broadcast, and every
// lane then tests the (completed) phase once for its own acquire ordering.  Keeps the
// warp converged for the warp-collective tcgen05 instructions that follow.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int lane) {
    // fast path, convergent: every lane tests the phase once (its own acquire).  Measured: the
    // chunk tiles 7 % and the MLA kernel 8 % faster than with lane 0 alone polling first.
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    int ok = 1;
    if (lane == 0) ok = wait_bar(bar, parity, abort_flag, true) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try(bar, parity);
    return ok != 0;
}

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // tcgen05 descriptor version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: bf16 x bf16 -> f32, M x N, B MN-major when b_mn
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// kind::f16 instruction descriptor: f16 x f16 -> f32, M x N, B MN-major when b_mn
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn) {
    return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// the same with the A operand (K-major, 16-bit elements packed two per 32-bit
// column, lower k in the low half) read from tensor memory at column address a_tmem
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
            d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// The same two with the accumulate flag a compile-time constant (no predicate set from a
// register: the issuing thread stays on straight-line code)
template <int ACC>
__device__ __forceinline__ void mma_f16c(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "n"(ACC));
}
template <int ACC>
__device__ __forceinline__ void mma_f16_tsc(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
            d),
        "r"(a_tmem), "l"(b), "r"(idesc), "n"(ACC));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// commit when `cond` holds, as a predicated instruction rather than a branch
__device__ __forceinline__ void mma_commit_if(uint32_t bar, uint32_t cond) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
        "r"(cond)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define SKV_LD32(taddr, r)                                                                                          \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"   \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                         \
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),  \
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),          \
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),        \
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),        \
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                                                            \
                 : "r"(taddr))

#define SKV_ST32(taddr, r)                                                                                          \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),               \
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),  \
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),      \
                 "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),     \
                 "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                 \
                 : "memory")

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x with the special-function unit's approximate exp2 (PTX ex2.approx.ftz.f32):
// one instruction; results below the smallest normal flush to zero, ex2(-inf) = 0
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (x, y) -> bf16 pair hi = (x, y) truncated to bf16 (a byte permute: no conversion
// instruction) and residual pair lo = round((x, y) - hi), exact differences in fp32:
// hi + lo is within 2^-15 of each probability
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
    const uint32_t xb = __float_as_uint(x), yb = __float_as_uint(y);
    hi = __byte_perm(xb, yb, 0x7632);
    __nv_bfloat162 l = __floats2bfloat162_rn(x - __uint_as_float(xb & 0xFFFF0000u), y - __uint_as_float(yb & 0xFFFF0000u));
    lo = *reinterpret_cast<uint32_t*>(&l);
}

#define SKV_ST8(taddr, r)                                                                                         \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]), \
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])                       \
                 : "memory")

// P = 2^(s * c2 - base) for 64 keys of one row, masked keys (key0 + j > limit) 0,
// written to the row's P columns in tensor memory as bf16 pairs: columns 0..31
// the high parts, 32..63 the residuals (key 2k in the low half of column k).
// Returns the row's sum of P.
template <bool MASK>
__device__ __forceinline__ float write_p(const uint32_t (&sr)[64], float c2, float base, int key0, int limit,
                                         uint32_t pcol) {
    float part[4];                          // one running sum per 16 keys: four independent chains
#pragma unroll
    for (int h = 0; h < 4; ++h) {           // 16 keys -> 8 columns of each part
        uint32_t hi[8], lo[8];
        part[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 16 * h + 2 * e;
            float x0 = ex2_ftz(fmaf(__uint_as_float(sr[j]), c2, -base));
            float x1 = ex2_ftz(fmaf(__uint_as_float(sr[j + 1]), c2, -base));
            if (MASK) {
                if (key0 + j > limit) x0 = 0.f;
                if (key0 + j + 1 > limit) x1 = 0.f;
            }
            part[h] += x0 + x1;
            split_bf16(x0, x1, hi[e], lo[e]);
        }
        SKV_ST8(pcol + 8 * h, hi);          // high parts: columns 8h .. 8h + 7
        SKV_ST8(pcol + 32 + 8 * h, lo);     // residuals: columns 32 + 8h ..
    }
    return (part[0] + part[1]) + (part[2] + part[3]);
}

// P = 2^(s * c2 - base) for 64 keys of one row, masked keys (key0 + j > limit) 0,
// written over the row's S columns in tensor memory as f16 pairs (key 2k in the low
// half of column k: 32 columns).  Returns the row's sum of P (float32, before rounding).
template <bool MASK>
__device__ __forceinline__ float write_p16(const uint32_t (&sr)[64], float c2, float base, int key0, int limit,
                                           uint32_t pcol) {
    float part[4];                          // one running sum per 16 keys: four independent chains
#pragma unroll
    for (int h = 0; h < 4; ++h) {           // 16 keys -> 8 columns
        uint32_t pk[8];
        part[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = 16 * h + 2 * e;
            float x0 = ex2_ftz(fmaf(__uint_as_float(sr[j]), c2, -base));
            float x1 = ex2_ftz(fmaf(__uint_as_float(sr[j + 1]), c2, -base));
            if (MASK) {
                if (key0 + j > limit) x0 = 0.f;
                if (key0 + j + 1 > limit) x1 = 0.f;
            }
            part[h] += x0 + x1;
            __half2 p2 = __floats2half2_rn(x0, x1);
            pk[e] = *reinterpret_cast<uint32_t*>(&p2);
        }
        SKV_ST8(pcol + 8 * h, pk);
    }
    return (part[0] + part[1]) + (part[2] + part[3]);
}

// bf16 pair -> f16 pair, each rounded to nearest (exact for magnitudes in [2^-14, 65504])
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return *reinterpret_cast<uint32_t*>(&h);
}

// row max of 64 scores (keys j < valid when MASK), four independent chains
template <bool MASK>
__device__ __forceinline__ float row_max64(const uint32_t (&sr)[64], int valid) {
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 64; ++j)
        if (!MASK || j < valid) m4[j & 3] = fmaxf(m4[j & 3], __uint_as_float(sr[j]));
    return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// cuTensorMapEncodeTiled from the driver, looked up once (null if unavailable)
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace
}  // namespace skv
