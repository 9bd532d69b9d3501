// Persistent split-KV engine for bf16 GQA attention on sm_103a.
//
// What it computes (Helix Parallelism, "Attention-Phase Configuration" steps
// 2-3; LiquidCP Section 3 Eq. 1): for every task -- query rows of one
// (request, KV head) over one split of the history -- the split's partial
// state (output normalised over the split, natural-log LSE); in fused mode
// also the LSE-weighted merge of each split request's states into the final
// output, in the same launch.
//
// How (LiquidCP Section 6: a persistent GPU-resident engine dispatching
// host-prepared task descriptors):
//  * one CTA per SM with four roles: a scheduler warp, a producer warp,
//    NWC consumer warps and a finaliser warp;
//  * the scheduler claims tasks from a device queue (atomic head, plan
//    order) and prepares the next one -- descriptors, page range, first page
//    ids -- while the current one still streams: the producer asks for it a
//    few pages before the current task's end, so the claim and its dependent
//    loads stay off the copy stream;
//  * the producer streams each (page, KV head) K and V block into a ring of
//    NSTAGE shared-memory stages (as many as fit) with TMA bulk-tensor copies
//    (128-byte swizzle), completion on an mbarrier per stage;
//  * consumer warps split each page's keys (decode row blocks) or its rows
//    (chunked-prefill row blocks); each keeps a 16-row online softmax state
//    (base-2 exponent, scale folded in), computes S = Q K^T and O += P V with
//    bf16 m16n8k16 tensor-core MMA (fp32 accumulate), reading K and V from
//    the swizzled stages with ldmatrix; P enters the MMA as a bf16 high part
//    plus a bf16 residual, so rows that see few keys keep float-like weight
//    precision;
//  * at a task's last page each consumer warp drops its state into the
//    combine buffer and goes on with the next task; the finaliser combines
//    the warps' states and writes the partial state (or, for an unsplit
//    request in fused mode, the output);
//  * fused mode: the finaliser counts each finished task in for its request;
//    when the task queue is empty every warp takes reduction items (row
//    ranges of split requests, plan order), waits until the request's tasks
//    are all counted, and merges its rows' splits.
// FP8 KV caches (8-bit E4M3 codes, one scale per tensor): the stages hold the
// codes (half the bytes); consumer warps convert fragments to f16 in registers
// (exact: every E4M3 value is an f16 normal) and run f16 MMAs with the query
// and P in f16.  Key fragments come from ldmatrix over code pairs: one 8x8
// matrix of 16-bit pairs covers 16 dimensions of 8 keys, and the MMA's
// reduction index is permuted the same way in the query fragment (dims
// 4t..4t+3 of each 16-dim chunk feed k-slots 2t, 2t+1, 2t+8, 2t+9), which
// leaves every dot product unchanged.  Value fragments come from transposed
// ldmatrix plus a byte permute, which yields keys (2t, 2t+1) for dimension
// 2g and for 2g+1: each 16-dim chunk feeds an even-dim and an odd-dim output
// tile, put back in order when a warp hands its output over.  P enters the
// f16 product whole (11 significant bits; the bf16 path needs a residual).  The key scale is
// folded into the score scale, the value scale into the final normalisation.
// Every wait is bounded (globaltimer); on expiry the kernel records an error
// word, stops, waits for its own copies in flight and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "splitkv.h"
#include "internal.h"
#include "partial_io.cuh"
#include "trace.cuh"

namespace skv {
namespace {

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after kWaitLimitNs or
// when another warp raised the abort flag.  Returns false on give-up.
__device__ __noinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               bool watch_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (watch_abort && *abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate
__device__ __forceinline__ void mma_f16h(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x with the special-function unit's approximate exp2 (PTX ex2.approx.ftz.f32): one
// instruction instead of the accurate exp2f's range handling (measured: the E4M3 engine 7 %
// faster; its consumer warps are latency-bound); results below 2^-126 flush to 0, which the
// softmax's sums and products do not distinguish from it
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two E4M3 codes (low byte first) -> f16 pair (low half first); exact.  _lo converts the
// word's low two bytes, _hi its high two (one cvt.rn.f16x2.e4m3x2 on a half of the word)
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t w) {
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(d) : "r"(w));
    return d;
}
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t w) {
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(d) : "r"(w));
    return d;
}

// bytes (b0, b1, b2, b3) -> (b0, b2, b1, b3)
__device__ __forceinline__ uint32_t interleave_bytes(uint32_t r) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(d) : "r"(r));
    return d;
}

__device__ __forceinline__ uint32_t pack_f16(float x, float y) {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
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

// bf16 pair of keys (k, k + 1) in the low / high half: zero each half whose key is >= end
__device__ __forceinline__ uint32_t keep_keys(uint32_t pair, int k, int end) {
    const uint32_t lo = (k < end) ? 0x0000ffffu : 0u;
    const uint32_t hi = (k + 1 < end) ? 0xffff0000u : 0u;
    return pair & (lo | hi);
}

// 8x8 matrix of 16-bit elements spread over the warp in the MMA fragment layout (thread t
// holds row t / 4, columns 2 (t % 4) and + 1) -> its transpose in the same layout
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

// ---------------------------------------------------------------------------
// configuration
// ---------------------------------------------------------------------------
constexpr size_t kSmemLimit = 232448;                    // 227 KB per CTA on sm_103

template <int D_, int P_, int S_, bool F8_ = false, bool T8_ = false>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int P = P_;
    static constexpr int S = S_;                         // pages per stage
    static constexpr bool F8 = F8_;                      // E4M3 K/V codes
    static constexpr bool T8 = T8_;                      // every task holds at most 8 rows: transposed products
    static constexpr int EB = F8 ? 1 : 2;                // bytes per cached element
    static constexpr int T = P * S;                      // keys per stage
    static constexpr int NWC = (P == 16) ? 1 : 4;        // consumer warps
    static constexpr int KPW = T / NWC;                  // keys per consumer warp per stage
    static constexpr int NT = KPW / 8;                   // score n-tiles per warp
    static constexpr int KSTEP_PV = KPW / 16;            // PV k-steps per warp
    static constexpr int TILE_BYTES = P * D * EB;        // one (page, KV head) K or V block
    static constexpr int PAGE_BYTES = 2 * TILE_BYTES;    // K + V of one page
    static constexpr int STAGE_BYTES = S * PAGE_BYTES;   // pages in order, each K then V
    static constexpr int BOXES = D * EB / 128;           // 128-byte-wide TMA boxes per row
    static constexpr int DT = D / 8;                     // output n-tiles
    static constexpr int KT = D / 16;                    // QK k-steps
    static constexpr size_t COMB_BYTES = (size_t)NWC * 16 * D * 4;
    // as many stages as shared memory holds (each also needs a header and two barriers)
    static constexpr int NSTAGE_FIT = (int)((kSmemLimit - 1024 - COMB_BYTES - 1024) / (STAGE_BYTES + 112));
    static constexpr int NSTAGE = NSTAGE_FIT < 16 ? NSTAGE_FIT : 16;
    static constexpr size_t STAGES_BYTES = (size_t)NSTAGE * STAGE_BYTES;
    // roles: warp 0 producer, 1..NWC consumers, NWC+1 scheduler, NWC+2 finaliser
    static constexpr int W_SCHED = NWC + 1;
    static constexpr int W_FIN = NWC + 2;
    static constexpr int THREADS = (NWC + 3) * 32;
    // the scheduler is asked for the next task this many pages before the current one's end
    static constexpr int AHEAD = (4 * 32768 / PAGE_BYTES) > 2 ? (4 * 32768 / PAGE_BYTES) : 2;
    static_assert(KPW % 16 == 0 && NT * 8 == KPW && KSTEP_PV * 16 == KPW, "keys per warp must be a multiple of 16");
    static_assert(S == 1 || P % KPW == 0, "a warp's keys lie in one page of the stage");
    static_assert(32 % S == 0, "stages do not straddle the producer's 32-page id chunks");
    static_assert(!F8 || (D == 128 && KPW % 32 == 0), "E4M3 path: one 128-byte row per key, 32-key groups per warp");
    static_assert(!(T8 && F8), "transposed products: bf16 caches");
    static_assert(NSTAGE >= 2, "stage ring");
};

// Stage header written by the producer before it arrives on the stage's full barrier.
enum : int { F_FIRST = 1, F_LAST = 2, F_EMPTY = 4, F_END = 8, F_MASK = 16 };
struct StageHdr {
    TaskDesc t;
    ReqDesc r;
    int page;     // index within the request of the stage's first page (the next: + t.page_stride)
    int flags;
    int npages;   // pages loaded into the stage (1..S)
    int task;     // queue index of the task (trace records)
    int pad[4];
};
static_assert(sizeof(StageHdr) == 96, "StageHdr");

// The next task, prepared by the scheduler warp: descriptors, page range and the
// physical ids of its first 32 pages.
struct TaskSlot {
    TaskDesc t;
    ReqDesc r;
    int task, pb, pe, mask_from;
    int pad[4];
    int ids[32];
};

template <class C>
struct SmemExtra {
    StageHdr hdr[C::NSTAGE];
    unsigned long long full[C::NSTAGE];
    unsigned long long empty[C::NSTAGE];
    unsigned long long sched_req, sched_ready;   // producer -> scheduler, scheduler -> producer
    unsigned long long comb_full, comb_empty;    // consumers -> finaliser, finaliser -> consumers
    TaskSlot slot;
    TaskDesc fin_t;                              // the task whose states the combine buffer holds
    ReqDesc fin_r;
    int fin_task;                                // its queue index
    float comb_m[C::NWC][16];
    float comb_l[C::NWC][16];
    int fin_end;
    int exit_last;
    int abort_flag;
};

template <class C>
constexpr size_t smem_bytes() {
    return 1024 + C::STAGES_BYTES + C::COMB_BYTES + sizeof(SmemExtra<C>);
}

// byte offset of (key, dim) in a 128B-swizzled tile made of BOXES boxes of P x 64
template <class C>
__device__ __forceinline__ uint32_t tile_off(int key, int dim) {
    return (uint32_t)((dim >> 6) * (C::P * 128) + key * 128 + ((((dim & 63) >> 3) ^ (key & 7)) << 4) +
                      (dim & 7) * 2);
}

// float index of (row, col) in one warp's 16 x D slot of the combine buffer: 32-byte
// column groups are rotated by row so a warp's fragment stores hit distinct banks
template <class C>
__device__ __forceinline__ int comb_idx(int row, int col) {
    return row * C::D + (col ^ ((row & 3) << 3));
}

// One warp, KPW keys of one staged page (keys kw0 .. kw0 + KPW - 1 of the tile,
// key index key_page + kw0 + j in the request) against its 16 query rows:
// S = Q K^T on mma.sync, online softmax in base 2 over the warp's running
// (m, l) of rows qr and qr + 8, and O += P V with P = P_hi + P_lo (two bf16
// terms carry about 16 significant bits of each weight).  MASK: the page holds
// keys a row may not see (key >= key_end, or past the row's causal limit).
template <class C, bool MASK>
__device__ __forceinline__ void attend_keys(uint32_t kbase, int kw0, int key_page, int key_end, int lim0, int lim1,
                                            float scale_log2, const uint32_t (&qa)[C::KT][4], float (&o)[C::DT][4],
                                            float& m0, float& m1, float& l0, float& l1, int lane) {
    const uint32_t vbase = kbase + C::TILE_BYTES;
    const int qc = (lane & 3) * 2;
    float s[C::NT][4];
#pragma unroll
    for (int n = 0; n < C::NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < C::KT; ++kk) {
#pragma unroll
        for (int n = 0; n < C::NT; n += 2) {
            const int mi = lane >> 3;
            const int key = kw0 + n * 8 + ((mi >> 1) << 3) + (lane & 7);
            const int dim = kk * 16 + ((mi & 1) << 3);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + tile_off<C>(key, dim), b0, b1, b2, b3);
            mma_bf16(s[n], qa[kk], b0, b1);
            mma_bf16(s[n + 1], qa[kk], b2, b3);
        }
    }
    const int key0 = key_page + kw0;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v0 = s[n][e] * scale_log2;
            float v1 = s[n][2 + e] * scale_log2;
            if (MASK) {
                const int kidx = key0 + n * 8 + qc + e;
                if (kidx > lim0 || kidx >= key_end) v0 = -INFINITY;
                if (kidx > lim1 || kidx >= key_end) v1 = -INFINITY;
            }
            s[n][e] = v0;
            s[n][2 + e] = v1;
            mx0 = fmaxf(mx0, v0);
            mx1 = fmaxf(mx1, v1);
        }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float b0s = (mn0 == -INFINITY) ? 0.f : mn0;
    const float b1s = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = exp2f(m0 - b0s), al1 = exp2f(m1 - b1s);
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
        s[n][0] = ex2_approx(s[n][0] - b0s);
        s[n][1] = ex2_approx(s[n][1] - b0s);
        s[n][2] = ex2_approx(s[n][2] - b1s);
        s[n][3] = ex2_approx(s[n][3] - b1s);
        ps0 += s[n][0] + s[n][1];
        ps1 += s[n][2] + s[n][3];
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int n = 0; n < C::DT; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
    }
#pragma unroll
    for (int j = 0; j < C::KSTEP_PV; ++j) {
        uint32_t ph[4], pl[4];
        split_bf16(s[2 * j][0], s[2 * j][1], ph[0], pl[0]);
        split_bf16(s[2 * j][2], s[2 * j][3], ph[1], pl[1]);
        split_bf16(s[2 * j + 1][0], s[2 * j + 1][1], ph[2], pl[2]);
        split_bf16(s[2 * j + 1][2], s[2 * j + 1][3], ph[3], pl[3]);
#pragma unroll
        for (int nd = 0; nd < C::DT; nd += 2) {
            const int mi = lane >> 3;
            const int key = kw0 + j * 16 + ((mi & 1) << 3) + (lane & 7);
            const int dim = (nd + (mi >> 1)) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vbase + tile_off<C>(key, dim), b0, b1, b2, b3);
            if (MASK) {
                // Slots past the task's last key (the unused tail of a request's
                // last page) may hold anything: their weight is 0, but 0 * NaN is
                // not, so their V values go to 0.
                const int ka = key0 + j * 16 + 2 * (lane & 3);
                b0 = keep_keys(b0, ka, key_end);
                b2 = keep_keys(b2, ka, key_end);
                b1 = keep_keys(b1, ka + 8, key_end);
                b3 = keep_keys(b3, ka + 8, key_end);
            }
            mma_bf16(o[nd], ph, b0, b1);
            mma_bf16(o[nd + 1], ph, b2, b3);
            mma_bf16(o[nd], pl, b0, b1);
            mma_bf16(o[nd + 1], pl, b2, b3);
        }
    }
}

// The same for row blocks of at most 8 rows (decode with g <= 8 query heads per KV head),
// computed transposed so that no MMA row is padding: S^T = K Q^T with keys as the MMA's
// 16 rows and the 8 query rows as its columns (A = K from the stage by ldmatrix, B = Q^T
// from registers), and O^T += V^T P^T (A = V^T by transposed ldmatrix, B = P^T, formed
// from the score fragments by an in-register 8x8 transpose).  Half the MMAs of the
// 16-row form per key, half its exponentials and output registers.  Thread t keeps the
// softmax state of rows 2 (t % 4) and + 1 (limits limA, limB; state mA/lA, mB/lB, each
// l a partial sum over this thread's keys) and o[md] = O^T rows (output dims) 16 md +
// t / 4 and + 8 of those two query rows.
template <class C, bool MASK>
__device__ __forceinline__ void attend_keys_t(uint32_t kbase, int kw0, int key_page, int key_end, int limA,
                                              int limB, float scale_log2, const uint32_t (&qa)[C::KT][4],
                                              float (&o)[C::DT][4], float& mA, float& mB, float& lA, float& lB,
                                              int lane) {
    constexpr int MT = C::KPW / 16;   // 16-key tiles of the warp's keys
    constexpr int OT = C::D / 16;     // 16-dim output tiles
    const uint32_t vbase = kbase + C::TILE_BYTES;
    const int kr = lane >> 2;         // fragment key row (and + 8)
    const int mi = lane >> 3;         // ldmatrix: the 8x8 matrix this lane addresses
    float s[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < C::KT; ++kk) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            // matrices: keys +0 / +8 (mi & 1) x dims +0 / +8 (mi >> 1) -> a0a1, a2a3, a4a5, a6a7
            const int key = kw0 + mt * 16 + ((mi & 1) << 3) + (lane & 7);
            const int dim = kk * 16 + ((mi >> 1) << 3);
            uint32_t ka[4];
            ldsm_x4(kbase + tile_off<C>(key, dim), ka[0], ka[1], ka[2], ka[3]);
            mma_bf16(s[mt], ka, qa[kk][0], qa[kk][1]);
        }
    }
    // s[mt][2e + c]: key mt * 16 + kr + 8 e, query row 2 (lane % 4) + c
    const int key0 = key_page + kw0;
    float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float vA = s[mt][2 * e] * scale_log2;
            float vB = s[mt][2 * e + 1] * scale_log2;
            if (MASK) {
                const int kidx = key0 + mt * 16 + kr + 8 * e;
                if (kidx > limA || kidx >= key_end) vA = -INFINITY;
                if (kidx > limB || kidx >= key_end) vB = -INFINITY;
            }
            s[mt][2 * e] = vA;
            s[mt][2 * e + 1] = vB;
            mxA = fmaxf(mxA, vA);
            mxB = fmaxf(mxB, vB);
        }
    }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, x));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, x));
    }
    const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
    const float bA = (mnA == -INFINITY) ? 0.f : mnA;
    const float bB = (mnB == -INFINITY) ? 0.f : mnB;
    const float alA = exp2f(mA - bA), alB = exp2f(mB - bB);
    float psA = 0.f, psB = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        s[mt][0] = ex2_approx(s[mt][0] - bA);
        s[mt][1] = ex2_approx(s[mt][1] - bB);
        s[mt][2] = ex2_approx(s[mt][2] - bA);
        s[mt][3] = ex2_approx(s[mt][3] - bB);
        psA += s[mt][0] + s[mt][2];
        psB += s[mt][1] + s[mt][3];
    }
    lA = lA * alA + psA;
    lB = lB * alB + psB;
    mA = mnA;
    mB = mnB;
#pragma unroll
    for (int md = 0; md < OT; ++md) {
        o[md][0] *= alA;
        o[md][1] *= alB;
        o[md][2] *= alA;
        o[md][3] *= alB;
    }
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        // P^T of keys 16 j .. 16 j + 15 as the B operand: the score fragment holds rows
        // (keys) kr, kr + 8 x columns (query rows) 2 (lane % 4), + 1; transposed, keys
        // 2 (lane % 4), + 1 (+ 8) x query row lane / 4 -- the B fragment's layout
        uint32_t h0, l0, h1, l1;
        split_bf16(s[j][0], s[j][1], h0, l0);
        split_bf16(s[j][2], s[j][3], h1, l1);
        const uint32_t bh0 = movmatrix_t(h0), bh1 = movmatrix_t(h1);
        const uint32_t bl0 = movmatrix_t(l0), bl1 = movmatrix_t(l1);
#pragma unroll
        for (int md = 0; md < OT; ++md) {
            // V^T tile (dims 16 md.., keys 16 j..): matrices keys +0 / +8 (mi >> 1) x dims
            // +0 / +8 (mi & 1), transposed on load
            const int key = kw0 + j * 16 + ((mi >> 1) << 3) + (lane & 7);
            const int dim = md * 16 + ((mi & 1) << 3);
            uint32_t va[4];
            ldsm_x4_t(vbase + tile_off<C>(key, dim), va[0], va[1], va[2], va[3]);
            if (MASK) {
                // value slots past the task's last key may hold anything (0 * NaN is not 0)
                const int ka = key0 + j * 16 + 2 * (lane & 3);
                va[0] = keep_keys(va[0], ka, key_end);
                va[1] = keep_keys(va[1], ka, key_end);
                va[2] = keep_keys(va[2], ka + 8, key_end);
                va[3] = keep_keys(va[3], ka + 8, key_end);
            }
            mma_bf16(o[md], va, bh0, bh1);
            mma_bf16(o[md], va, bl0, bl1);
        }
    }
}

// The same over E4M3 K/V tiles (P rows x 128 bytes, 128-byte swizzle: 16-byte
// chunk c of row r sits at c ^ (r & 7)) with f16 MMAs; see the file comment for
// the permuted reduction index (keys) and output tiles (values).  qa holds the
// query in f16 in the matching order; output tile 2c (2c + 1) holds the even
// (odd) dims of chunk c: its column j is dim 16c + 2j (+ 1).
template <class C, bool MASK>
__device__ __forceinline__ void attend_keys_f8(uint32_t kbase, int kw0, int key_page, int key_end, int lim0, int lim1,
                                               float scale_log2, const uint32_t (&qa)[C::KT][4], float (&o)[C::DT][4],
                                               float& m0, float& m1, float& l0, float& l1, int lane) {
    const uint32_t vbase = kbase + C::TILE_BYTES;
    const int qc = (lane & 3) * 2;
    float s[C::NT][4];
#pragma unroll
    for (int n = 0; n < C::NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    {
        // per 32-key group g, one x4 load per 16-dim chunk: matrix n = keys kw0 + 32g + 8n .. + 7
        // (this lane's row address); the groups' products are independent chains
#pragma unroll
        for (int kk = 0; kk < C::KT; ++kk) {
#pragma unroll
            for (int g = 0; g < C::KPW / 32; ++g) {
                const int key = kw0 + 32 * g + 8 * (lane >> 3) + (lane & 7);
                uint32_t r[4];
                ldsm_x4(kbase + key * 128 + ((kk ^ (key & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int n = 0; n < 4; ++n)
                    mma_f16h(s[4 * g + n], qa[kk], e4m3x2_lo_to_f16x2(r[n]), e4m3x2_hi_to_f16x2(r[n]));
            }
        }
    }
    const int key0 = key_page + kw0;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v0 = s[n][e] * scale_log2;
            float v1 = s[n][2 + e] * scale_log2;
            if (MASK) {
                const int kidx = key0 + n * 8 + qc + e;
                if (kidx > lim0 || kidx >= key_end) v0 = -INFINITY;
                if (kidx > lim1 || kidx >= key_end) v1 = -INFINITY;
            }
            s[n][e] = v0;
            s[n][2 + e] = v1;
            mx0 = fmaxf(mx0, v0);
            mx1 = fmaxf(mx1, v1);
        }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float b0s = (mn0 == -INFINITY) ? 0.f : mn0;
    const float b1s = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = exp2f(m0 - b0s), al1 = exp2f(m1 - b1s);
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
        s[n][0] = ex2_approx(s[n][0] - b0s);
        s[n][1] = ex2_approx(s[n][1] - b0s);
        s[n][2] = ex2_approx(s[n][2] - b1s);
        s[n][3] = ex2_approx(s[n][3] - b1s);
        ps0 += s[n][0] + s[n][1];
        ps1 += s[n][2] + s[n][3];
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int n = 0; n < C::DT; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
    }
#pragma unroll
    for (int j = 0; j < C::KSTEP_PV; ++j) {
        // P in f16 (11 significant bits: each weight within 2^-12 of its float value, so no
        // residual product is needed)
        uint32_t ph[4];
        ph[0] = pack_f16(s[2 * j][0], s[2 * j][1]);
        ph[1] = pack_f16(s[2 * j][2], s[2 * j][3]);
        ph[2] = pack_f16(s[2 * j + 1][0], s[2 * j + 1][1]);
        ph[3] = pack_f16(s[2 * j + 1][2], s[2 * j + 1][3]);
        // x4 transposed load per 32 dims: matrices (keys 0-7 | 8-15 of the step) x (chunk 2G | 2G + 1)
        const int mi = lane >> 3;
        const int key = kw0 + j * 16 + ((mi & 1) << 3) + (lane & 7);
        const int ka = key0 + j * 16 + 2 * (lane & 3);
#pragma unroll
        for (int G = 0; G < C::D / 32; ++G) {
            const int chunk = 2 * G + (mi >> 1);
            uint32_t r[4];
            ldsm_x4_t(vbase + key * 128 + ((chunk ^ (key & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                // r[2c]: keys 2t, 2t+1 x dims 2g, 2g+1 of chunk 2G + c; r[2c + 1]: keys 2t+8, 2t+9
                const uint32_t pa = interleave_bytes(r[2 * c]);
                const uint32_t pb = interleave_bytes(r[2 * c + 1]);
                uint32_t e0 = e4m3x2_lo_to_f16x2(pa), e1 = e4m3x2_lo_to_f16x2(pb);
                uint32_t d0 = e4m3x2_hi_to_f16x2(pa), d1 = e4m3x2_hi_to_f16x2(pb);
                if (MASK) {
                    // value slots past the task's last key may hold anything (0 * NaN is not 0)
                    e0 = keep_keys(e0, ka, key_end);
                    d0 = keep_keys(d0, ka, key_end);
                    e1 = keep_keys(e1, ka + 8, key_end);
                    d1 = keep_keys(d1, ka + 8, key_end);
                }
                const int te = 2 * (2 * G + c);
                mma_f16h(o[te], ph, e0, e1);
                mma_f16h(o[te + 1], ph, d0, d1);
            }
        }
    }
}

// Wait (bounded) for a phase: when every lane's first test finds it complete the warp
// goes on at once; otherwise lane 0 waits, broadcasts the outcome, and every lane
// gets acquire ordering with one more test of the completed phase (it cannot move on
// before this warp's next arrive).  On give-up the first warp to notice records
// `site` and raises the CTA's abort flag.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          int32_t site, int lane) {
    // fast path, convergent and inline: every lane tests the phase once (its own acquire)
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int okw = 1;
    if (lane == 0) {
        okw = mbar_wait_bounded(bar, parity, abort_flag, true) ? 1 : 0;
        if (!okw && !*abort_flag) {
            set_error(err, ERR_TIMEOUT | site);
            *abort_flag = 1;
        }
    }
    if (!__shfl_sync(0xffffffffu, okw, 0)) return false;
    (void)mbar_try_wait(bar, parity);
    return true;
}

// ---------------------------------------------------------------------------
// reduction phase of the fused engine (LiquidCP Section 5.2: history reductions
// run in plan order on warps released by attention, each once every attention
// task of its sequence has finished; the merge itself is LiquidCP Eq. 1)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *ctr >= target; gives up after kWaitLimitNs or on the abort flag.
__device__ __noinline__ bool wait_count(const int32_t* ctr, int target, volatile int* abort_flag) {
    if (ld_acquire(ctr) >= target) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(200);
        if (ld_acquire(ctr) >= target) return true;
        if ((it & 15) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) return false;
        }
    }
}

// One warp: claim items until none is left; each item merges rows
// [row_begin, row_end) of one request: o = sum_r exp(lse_r - M) o_r / den,
// lse = M + log(den), M = max_r lse_r, den = sum_r exp(lse_r - M).
template <class C>
__device__ void reduce_items(const KernelArgs& a, volatile int* abort_flag, int lane) {
    const int Hq = a.num_q_heads;
    const int c = lane * 4;   // this lane's four output columns
    while (true) {
        int item = 0;
        if (lane == 0) item = atomicAdd(&a.ctrl->red_head, 1);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= a.num_red) return;
        const RedItem it = a.red_items[item];
        const ReqDesc r = a.reqs[it.b];
        int ok = 1;
        if (lane == 0) {
            ok = wait_count(a.counters + it.b, r.n_tasks, abort_flag) ? 1 : 0;
            if (!ok && !*abort_flag) {
                set_error(a.err, ERR_TIMEOUT | SITE_REDUCE_WAIT);
                *abort_flag = 1;
            }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        // lane 0's acquire, then the warp barrier, order every lane's loads after the count
        __syncwarp();
        if (lane == 0) trace_start(a.trace_red, item, SPLITKV_TRACE_REDUCTION);
        const int n = r.n_splits;
        for (int v = it.row_begin; v < it.row_end; ++v) {
            const size_t orow = (size_t)r.q_start * Hq + v;
            const size_t s0 = (size_t)r.state_base + (size_t)v * n;
            float M = -INFINITY;
            for (int q = lane; q < n; q += 32) M = fmaxf(M, __ldcg(a.lse_part + s0 + q));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            float den = 0.f;
            if (M != -INFINITY)
                for (int q = lane; q < n; q += 32) den += expf(__ldcg(a.lse_part + s0 + q) - M);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
            const float inv = (M == -INFINITY) ? 0.f : 1.f / den;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q0 = 0; q0 < n; q0 += 32) {
                float wq = 0.f;
                if (q0 + lane < n && M != -INFINITY) wq = expf(__ldcg(a.lse_part + s0 + q0 + lane) - M) * inv;
                const int cnt = min(32, n - q0);
                // every lane runs every shuffle; lanes past the row's width skip the loads
#pragma unroll 4
                for (int q = 0; q < cnt; ++q) {
                    const float wj = __shfl_sync(0xffffffffu, wq, q);
                    if (c < C::D) {
                        const float4 x = load_part4(a.o_part, a.part_bf16, (s0 + q0 + q) * C::D + c);
                        acc.x = fmaf(wj, x.x, acc.x);
                        acc.y = fmaf(wj, x.y, acc.y);
                        acc.z = fmaf(wj, x.z, acc.z);
                        acc.w = fmaf(wj, x.w, acc.w);
                    }
                }
            }
            if (c < C::D) {
                if (a.out_bf16) {
                    __nv_bfloat162* op = (__nv_bfloat162*)((__nv_bfloat16*)a.out + orow * C::D + c);
                    op[0] = __floats2bfloat162_rn(acc.x, acc.y);
                    op[1] = __floats2bfloat162_rn(acc.z, acc.w);
                } else {
                    *(float4*)((float*)a.out + orow * C::D + c) = acc;
                }
            }
            if (lane == 0 && a.lse_out) a.lse_out[orow] = (M == -INFINITY) ? -INFINITY : M + logf(den);
        }
        __syncwarp();
        if (lane == 0) trace_end(a.trace_red, item);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
gqa_engine_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  KernelArgs a) {
    static_assert(smem_bytes<C>() <= kSmemLimit, "shared memory budget");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // TMA with 128-byte swizzle needs 1024-byte aligned destinations
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char* stages = smem;
    float* comb = (float*)(smem + C::STAGES_BYTES);
    SmemExtra<C>& X = *(SmemExtra<C>*)(smem + C::STAGES_BYTES + C::COMB_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&X.full[s]), 1);
            mbar_init(smem_u32(&X.empty[s]), C::NWC);
        }
        mbar_init(smem_u32(&X.sched_req), 1);
        mbar_init(smem_u32(&X.sched_ready), 32);
        mbar_init(smem_u32(&X.comb_full), C::NWC * 32);
        mbar_init(smem_u32(&X.comb_empty), 32);
        X.abort_flag = 0;
        X.fin_end = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort_flag = &X.abort_flag;

    if (warp == 0) {
        // ============================ producer ============================
        // Streams the pages of the tasks the scheduler hands over into the stage ring;
        // asks for the next task AHEAD pages before the current one ends.
        const uint64_t policy = evict_first_policy();
        uint32_t item = 0, nslot = 0;
        uint32_t had_tma = 0, last_parity = 0;   // per-stage bits (lane 0)
        bool stop = false;
        // returns the stage for the next item after waiting for it to be free
        auto acquire = [&](int& stage) -> bool {
            stage = (int)(item % C::NSTAGE);
            return warp_wait(smem_u32(&X.empty[stage]), ((item / C::NSTAGE) & 1) ^ 1, abort_flag, a.err,
                             SITE_EMPTY_WAIT, lane);
        };
        if (lane == 0) mbar_arrive(smem_u32(&X.sched_req));
        while (!stop) {
            if (!warp_wait(smem_u32(&X.sched_ready), nslot & 1, abort_flag, a.err, SITE_FULL_WAIT, lane)) break;
            ++nslot;
            const int task = X.slot.task;
            if (task >= a.num_tasks) {
                int stage;
                if (!acquire(stage)) break;
                if (lane == 0) {
                    X.hdr[stage].flags = F_END;
                    had_tma &= ~(1u << stage);
                    mbar_arrive(smem_u32(&X.full[stage]));
                }
                ++item;
                break;
            }
            const TaskDesc t = X.slot.t;
            const ReqDesc r = X.slot.r;
            const int pb = X.slot.pb, pe = X.slot.pe, mask_from = X.slot.mask_from;
            int pid = X.slot.ids[lane];
            __syncwarp();
            const int ps = max(1, t.page_stride);
            const int npt = (pe > pb) ? (pe - pb + ps - 1) / ps : 0;   // pages pb + k ps, k < npt
            if (npt == 0) {
                if (lane == 0) mbar_arrive(smem_u32(&X.sched_req));   // the slot has been read
                int stage;
                if (!acquire(stage)) break;
                if (lane == 0) {
                    X.hdr[stage].t = t;
                    X.hdr[stage].r = r;
                    X.hdr[stage].page = pb;
                    X.hdr[stage].npages = 0;
                    X.hdr[stage].task = task;
                    X.hdr[stage].flags = F_FIRST | F_LAST | F_EMPTY;
                    had_tma &= ~(1u << stage);
                    mbar_arrive(smem_u32(&X.full[stage]));
                }
                ++item;
                continue;
            }
            const int k_ask = max(0, npt - C::AHEAD);
            for (int k0 = 0; k0 < npt && !stop; k0 += 32) {
                // page ids of the following 32 pages of the task, loaded a chunk ahead
                int pid_next = 0;
                if (k0 + 32 + lane < npt) pid_next = a.page_table[r.page_row + pb + (k0 + 32 + lane) * ps];
                const int cnt = min(32, npt - k0);
                for (int j = 0; j < cnt; j += C::S) {
                    const int k = k0 + j;                      // the stage's first page: pb + k ps
                    const int p = pb + k * ps;
                    const int np = min(C::S, cnt - j);
                    if (k <= k_ask && k_ask < k + np && lane == 0) mbar_arrive(smem_u32(&X.sched_req));
                    int phys[C::S];
#pragma unroll
                    for (int u = 0; u < C::S; ++u) phys[u] = __shfl_sync(0xffffffffu, pid, min(j + u, 31));
                    int stage;
                    if (!acquire(stage)) { stop = true; break; }
                    if (lane == 0) {
                        StageHdr& hd = X.hdr[stage];
                        hd.t = t;
                        hd.r = r;
                        hd.page = p;
                        hd.npages = np;
                        hd.task = task;
                        int fl = 0;
                        if (k == 0) fl |= F_FIRST;
                        if (k + np == npt) fl |= F_LAST;
                        if ((p + (np - 1) * ps + 1) * C::P > mask_from) fl |= F_MASK;
                        hd.flags = fl;
                        last_parity = (last_parity & ~(1u << stage)) | (((item / C::NSTAGE) & 1u) << stage);
                        const uint32_t full = smem_u32(&X.full[stage]);
                        bool valid = true;
#pragma unroll
                        for (int u = 0; u < C::S; ++u)
                            if (u < np && (phys[u] < 0 || phys[u] >= a.num_pages)) valid = false;
                        if (!valid) {
                            set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
                            had_tma &= ~(1u << stage);
                            mbar_arrive(full);
                        } else {
                            had_tma |= 1u << stage;
                            mbar_arrive_expect_tx(full, np * C::PAGE_BYTES);
#pragma unroll
                            for (int u = 0; u < C::S; ++u) {
                                if (u >= np) break;
                                const int y = (phys[u] * a.num_kv_heads + t.kv_head) * C::P;
                                const uint32_t dk =
                                    smem_u32(stages + (size_t)stage * C::STAGE_BYTES + (size_t)u * C::PAGE_BYTES);
                                const uint32_t dv = dk + C::TILE_BYTES;
#pragma unroll
                                for (int bx = 0; bx < C::BOXES; ++bx) {
                                    tma_load_2d(dk + bx * C::P * 128, &tmap_k, bx * (128 / C::EB), y, full, policy);
                                    tma_load_2d(dv + bx * C::P * 128, &tmap_v, bx * (128 / C::EB), y, full, policy);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    ++item;
                }
                pid = pid_next;
            }
        }
        // make sure no copy issued by this CTA is still landing in shared memory
        if (lane == 0) {
            for (int s = 0; s < C::NSTAGE; ++s) {
                if (((had_tma >> s) & 1u) &&
                    !mbar_wait_bounded(smem_u32(&X.full[s]), (last_parity >> s) & 1u, abort_flag, false))
                    set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == C::W_SCHED) {
        // ============================ scheduler ===========================
        // On each request: claim the next task (plan order), load its descriptors and
        // first 32 page ids, publish them in the slot.  Stops after handing over the
        // end marker (a task index past the queue).
        for (uint32_t n = 0; a.inject != 1; ++n) {   // (test hook: hand nothing over)
            if (!warp_wait(smem_u32(&X.sched_req), n & 1, abort_flag, a.err, SITE_EMPTY_WAIT, lane)) break;
            int task = 0;
            if (lane == 0) task = atomicAdd(&a.ctrl->queue_head, 1);
            task = __shfl_sync(0xffffffffu, task, 0);
            if (task < a.num_tasks && lane == 0) trace_start(a.trace, task, SPLITKV_TRACE_ATTENTION);
            if (task < a.num_tasks) {
                const TaskDesc t = a.tasks[task];
                const ReqDesc r = a.reqs[t.b];
                const int g = a.group;
                const int i_first = t.row_begin / g;
                const int i_last = (t.row_end - 1) / g;
                const int hi_key = min(t.key_end, r.seq_len - r.q_len + i_last + 1);   // exclusive
                const int pb = t.key_begin / C::P;
                const int pe = (hi_key > t.key_begin) ? (hi_key + C::P - 1) / C::P : pb;
                // the task's pages: pb, pb + ps, ... below pe (ps = 1: a contiguous range)
                const int ps = max(1, t.page_stride);
                const int npt = (pe > pb) ? (pe - pb + ps - 1) / ps : 0;
                X.slot.ids[lane] = (lane < npt) ? a.page_table[r.page_row + pb + lane * ps] : 0;
                if (lane == 0) {
                    X.slot.t = t;
                    X.slot.r = r;
                    X.slot.pb = pb;
                    X.slot.pe = pe;
                    X.slot.mask_from = min(t.key_end, r.seq_len - r.q_len + i_first + 1);
                }
            }
            if (lane == 0) X.slot.task = task;
            mbar_arrive(smem_u32(&X.sched_ready));
            if (task >= a.num_tasks) break;
        }
    } else if (warp == C::W_FIN) {
        // ============================ finaliser ===========================
        // For each finished task: combine the consumer warps' states of every row (one
        // slot per warp: narrow blocks hold the same 16 rows in every slot, wide blocks
        // 16 different rows per slot), write the partial state -- or, for an unsplit
        // request in fused mode, the output -- release the buffer, and in fused mode
        // count the task in for its request's reduction.
        const bool fused = a.fused != 0;
        const int g = a.group;
        for (uint32_t k = 0;; ++k) {
            if (!warp_wait(smem_u32(&X.comb_full), k & 1, abort_flag, a.err, SITE_FULL_WAIT, lane)) break;
            if (X.fin_end) break;
            const TaskDesc t = X.fin_t;
            const ReqDesc r = X.fin_r;
            const int fin_task = X.fin_task;
            const int nrows = t.row_end - t.row_begin;
            const bool wide = nrows > 16;
            const bool unsplit = r.n_splits == 1;
            for (int rr = 0; rr < nrows; ++rr) {
                const int src0 = wide ? (rr >> 4) : 0, nsrc = wide ? 1 : C::NWC;
                const int sr = wide ? (rr & 15) : rr;
                float M = -INFINITY;
#pragma unroll
                for (int u = 0; u < C::NWC; ++u)
                    if (u < nsrc) M = fmaxf(M, X.comb_m[src0 + u][sr]);
                float L = 0.f;
                float f[C::NWC];
#pragma unroll
                for (int u = 0; u < C::NWC; ++u) {
                    f[u] = (u >= nsrc || M == -INFINITY) ? 0.f : exp2f(X.comb_m[src0 + u][sr] - M);
                    if (u < nsrc) L += X.comb_l[src0 + u][sr] * f[u];
                }
                const bool empty = !(L > 0.f);
                const float inv = empty ? 0.f : a.v_scale / L;   // (E4M3 values: times their scale)
                const float lse = empty ? -INFINITY : (M + log2f(L)) * 0.69314718055994531f;
                const int row = t.row_begin + rr;
                const int i = row / g;
                const int h = t.kv_head * g + row % g;
                const size_t orow = (size_t)(r.q_start + i) * a.num_q_heads + h;
                const size_t st = (size_t)r.state_base + ((size_t)i * a.num_q_heads + h) * r.n_splits + t.split;
                const int c = lane * 4;
                if (c < C::D) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < C::NWC; ++u) {
                        if (u >= nsrc) break;
                        const float4 v = *(const float4*)(comb + (size_t)(src0 + u) * 16 * C::D + comb_idx<C>(sr, c));
                        acc.x = fmaf(f[u], v.x, acc.x);
                        acc.y = fmaf(f[u], v.y, acc.y);
                        acc.z = fmaf(f[u], v.z, acc.z);
                        acc.w = fmaf(f[u], v.w, acc.w);
                    }
                    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
                    if (fused && unsplit) {
                        if (a.out_bf16) {
                            __nv_bfloat162* op = (__nv_bfloat162*)((__nv_bfloat16*)a.out + orow * C::D + c);
                            op[0] = __floats2bfloat162_rn(acc.x, acc.y);
                            op[1] = __floats2bfloat162_rn(acc.z, acc.w);
                        } else {
                            *(float4*)((float*)a.out + orow * C::D + c) = acc;
                        }
                    } else {
                        store_part4(a.o_part, a.part_bf16, st * C::D + c, acc);
                    }
                }
                if (lane == 0) {
                    if (fused && unsplit) {
                        if (a.lse_out) a.lse_out[orow] = lse;
                    } else {
                        __stcg(a.lse_part + st, lse);
                    }
                }
            }
            // the combine buffer is free for the consumers' next task
            mbar_arrive(smem_u32(&X.comb_empty));
            if (lane == 0) trace_end(a.trace, fin_task);   // (the lanes' stores precede their arrives)
            if (fused && !unsplit) {
                // publish the states, then count the task in for the request's reduction:
                // the warp barrier orders every lane's stores before lane 0's fence, whose
                // cumulativity carries them ahead of the count
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(&a.counters[t.b], 1);
                }
            }
        }
    } else {
        // ============================ consumers ===========================
        const int w = warp - 1;
        const int qr = lane >> 2;        // fragment row (and row + 8)
        const int qc = (lane & 3) * 2;   // fragment column pair
        uint32_t qa[C::KT][4];
        float o[C::DT][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int lim0 = 0, lim1 = 0;          // last key index visible to rows qr, qr + 8
        uint32_t item = 0, nfin = 0;
        while (true) {
            const int stage = (int)(item % C::NSTAGE);
            if (!warp_wait(smem_u32(&X.full[stage]), (item / C::NSTAGE) & 1, abort_flag, a.err, SITE_FULL_WAIT, lane))
                break;
            const int flags = X.hdr[stage].flags;
            if (flags & F_END) {
                // tell the finaliser to stop, once it has taken the last task's states
                if (!warp_wait(smem_u32(&X.comb_empty), (nfin & 1) ^ 1, abort_flag, a.err, SITE_EMPTY_WAIT, lane))
                    break;
                if (w == 0 && lane == 0) X.fin_end = 1;
                __syncwarp();
                mbar_arrive(smem_u32(&X.comb_full));
                break;
            }
            const TaskDesc t = X.hdr[stage].t;
            const ReqDesc r = X.hdr[stage].r;
            const int page = X.hdr[stage].page;
            const int task_id = X.hdr[stage].task;
            const int g = a.group;
            const int nrows = t.row_end - t.row_begin;
            // Row blocks of more than 16 rows (chunked prefill) run "wide": warp w owns rows
            // 16w .. 16w+15 and walks every key of the page; 16-row blocks (decode) split the
            // page's keys across the warps instead.
            const bool wide = nrows > 16;
            const int wrow0 = wide ? w * 16 : 0;
            if constexpr (C::T8) {
                if (flags & F_FIRST) {
                    // Q^T fragments: query row qr, dims 16 kk + qc, + 1 (and + 8); limits of the
                    // rows this thread keeps the state of, qc and qc + 1
                    const bool valid = qr < nrows;
                    const int row = t.row_begin + qr;
                    const int i = valid ? row / g : 0;
                    const int h = t.kv_head * g + (valid ? row % g : 0);
                    const __nv_bfloat16* qp =
                        (const __nv_bfloat16*)a.q + ((size_t)(r.q_start + i) * a.num_q_heads + h) * C::D;
#pragma unroll
                    for (int kk = 0; kk < C::KT; ++kk) {
                        qa[kk][0] = valid ? *(const uint32_t*)(qp + kk * 16 + qc) : 0u;
                        qa[kk][1] = valid ? *(const uint32_t*)(qp + kk * 16 + 8 + qc) : 0u;
                    }
                    lim0 = qc < nrows ? r.seq_len - r.q_len + (t.row_begin + qc) / g : -1;
                    lim1 = qc + 1 < nrows ? r.seq_len - r.q_len + (t.row_begin + qc + 1) / g : -1;
#pragma unroll
                    for (int n = 0; n < C::DT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
                    m0 = m1 = -INFINITY;
                    l0 = l1 = 0.f;
                }
            } else if (flags & F_FIRST) {
                // load this warp's Q fragments (rows qr, qr + 8 of its 16-row tile)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int rr = wrow0 + qr + half * 8;
                    const bool valid = rr < nrows;
                    const int row = t.row_begin + rr;
                    const int i = valid ? row / g : 0;
                    const int h = t.kv_head * g + (valid ? row % g : 0);
                    const __nv_bfloat16* qp =
                        (const __nv_bfloat16*)a.q + ((size_t)(r.q_start + i) * a.num_q_heads + h) * C::D;
#pragma unroll
                    for (int kk = 0; kk < C::KT; ++kk) {
                        uint32_t lo = 0, hi = 0;
                        if (valid) {
                            if (C::F8) {
                                // f16, dims 16kk + 4t, +1 (k-slots 2t, 2t+1) and + 2, + 3 (2t+8, 2t+9)
                                const uint2 w = *(const uint2*)(qp + kk * 16 + 2 * qc);
                                const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
                                const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
                                lo = pack_f16(x.x, x.y);
                                hi = pack_f16(y.x, y.y);
                            } else {
                                lo = *(const uint32_t*)(qp + kk * 16 + qc);
                                hi = *(const uint32_t*)(qp + kk * 16 + 8 + qc);
                            }
                        }
                        qa[kk][half] = lo;        // a0a1 (row qr) / a2a3 (row qr+8)
                        qa[kk][2 + half] = hi;    // a4a5 / a6a7
                    }
                    const int lim = valid ? (r.seq_len - r.q_len + i) : -1;
                    if (half == 0) lim0 = lim; else lim1 = lim;
                }
#pragma unroll
                for (int n = 0; n < C::DT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
            }
            if (!(flags & F_EMPTY)) {
                const unsigned char* sbase = stages + (size_t)stage * C::STAGE_BYTES;
                const int npages = C::S == 1 ? 1 : X.hdr[stage].npages;
                // chunk ch: keys ch * KPW .. of the stage, which lie in page (ch * KPW) / P
                auto attend_chunk = [&](int ch) {
                    const int u = (ch * C::KPW) / C::P;
                    if (u >= npages) return;
                    const uint32_t kbase = smem_u32(sbase + (size_t)u * C::PAGE_BYTES);
                    const int kw0 = (ch * C::KPW) % C::P;
                    const int key_page = (page + u * max(1, t.page_stride)) * C::P;
                    if constexpr (C::F8) {
                        if (flags & F_MASK)
                            attend_keys_f8<C, true>(kbase, kw0, key_page, t.key_end, lim0, lim1, a.scale_log2, qa, o,
                                                    m0, m1, l0, l1, lane);
                        else
                            attend_keys_f8<C, false>(kbase, kw0, key_page, t.key_end, lim0, lim1, a.scale_log2, qa, o,
                                                     m0, m1, l0, l1, lane);
                    } else if constexpr (C::T8) {
                        if (flags & F_MASK)
                            attend_keys_t<C, true>(kbase, kw0, key_page, t.key_end, lim0, lim1, a.scale_log2, qa, o,
                                                   m0, m1, l0, l1, lane);
                        else
                            attend_keys_t<C, false>(kbase, kw0, key_page, t.key_end, lim0, lim1, a.scale_log2, qa, o,
                                                    m0, m1, l0, l1, lane);
                    } else if (flags & F_MASK) {
                        attend_keys<C, true>(kbase, kw0, key_page, t.key_end, lim0, lim1, a.scale_log2, qa, o, m0,
                                             m1, l0, l1, lane);
                    } else {
                        attend_keys<C, false>(kbase, kw0, key_page, t.key_end, lim0, lim1, a.scale_log2, qa, o, m0,
                                              m1, l0, l1, lane);
                    }
                };
                if (C::T8 || !wide) {
                    attend_chunk(w);
                } else {
                    for (int ch = 0; ch < C::NWC; ++ch) attend_chunk(ch);
                }
            }
            // release the stage to the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&X.empty[stage]));
            ++item;

            if (C::T8 && (flags & F_LAST)) {
                // ---- the same for a transposed block: rows qc, qc + 1; O^T dims 16 md + qr, + 8 ----
                float lt0 = l0, lt1 = l1;
#pragma unroll
                for (int x = 4; x < 32; x <<= 1) {
                    lt0 += __shfl_xor_sync(0xffffffffu, lt0, x);
                    lt1 += __shfl_xor_sync(0xffffffffu, lt1, x);
                }
                if (!warp_wait(smem_u32(&X.comb_empty), (nfin & 1) ^ 1, abort_flag, a.err, SITE_EMPTY_WAIT, lane))
                    break;
                ++nfin;
                float* cw = comb + (size_t)w * 16 * C::D;
#pragma unroll
                for (int md = 0; md < C::D / 16; ++md) {
                    cw[comb_idx<C>(qc, md * 16 + qr)] = o[md][0];
                    cw[comb_idx<C>(qc + 1, md * 16 + qr)] = o[md][1];
                    cw[comb_idx<C>(qc, md * 16 + qr + 8)] = o[md][2];
                    cw[comb_idx<C>(qc + 1, md * 16 + qr + 8)] = o[md][3];
                }
                if (qr == 0) {
                    X.comb_m[w][qc] = m0;
                    X.comb_m[w][qc + 1] = m1;
                    X.comb_l[w][qc] = lt0;
                    X.comb_l[w][qc + 1] = lt1;
                }
                if (w == 0 && lane == 0) {
                    X.fin_t = t;
                    X.fin_r = r;
                    X.fin_task = task_id;
                }
                mbar_arrive(smem_u32(&X.comb_full));
            } else if (!C::T8 && (flags & F_LAST)) {
                // ---- hand this warp's state of the task to the finaliser ----
                float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
                lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
                float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
                lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
                if (!warp_wait(smem_u32(&X.comb_empty), (nfin & 1) ^ 1, abort_flag, a.err, SITE_EMPTY_WAIT, lane))
                    break;
                ++nfin;
                float* cw = comb + (size_t)w * 16 * C::D;
                if (C::F8) {
                    // tiles 2c / 2c + 1 hold dims 16c + 2j / 16c + 2j + 1: this lane's four dims
                    // 16c + 2qc .. + 3 are (even j=qc, odd j=qc, even j=qc+1, odd j=qc+1)
#pragma unroll
                    for (int c = 0; c < C::DT / 2; ++c) {
                        *(float4*)(cw + comb_idx<C>(qr, 16 * c + 2 * qc)) =
                            make_float4(o[2 * c][0], o[2 * c + 1][0], o[2 * c][1], o[2 * c + 1][1]);
                        *(float4*)(cw + comb_idx<C>(qr + 8, 16 * c + 2 * qc)) =
                            make_float4(o[2 * c][2], o[2 * c + 1][2], o[2 * c][3], o[2 * c + 1][3]);
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < C::DT; ++n) {
                        *(float2*)(cw + comb_idx<C>(qr, n * 8 + qc)) = make_float2(o[n][0], o[n][1]);
                        *(float2*)(cw + comb_idx<C>(qr + 8, n * 8 + qc)) = make_float2(o[n][2], o[n][3]);
                    }
                }
                if ((lane & 3) == 0) {
                    X.comb_m[w][qr] = m0;
                    X.comb_m[w][qr + 8] = m1;
                    X.comb_l[w][qr] = lt0;
                    X.comb_l[w][qr + 8] = lt1;
                }
                if (w == 0 && lane == 0) {
                    X.fin_t = t;
                    X.fin_r = r;
                    X.fin_task = task_id;
                }
                mbar_arrive(smem_u32(&X.comb_full));
            }
        }
    }

    // fused mode: every warp, once its attention role is done, takes reduction items
    if (a.fused && !*abort_flag) reduce_items<C>(a, abort_flag, lane);

    // every warp leaves its loops (all waits are bounded); the last CTA to leave resets
    // the queues and the per-request task counters for the next launch
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        X.exit_last = (atomicAdd(&a.ctrl->exit_count, 1) == (int)gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (X.exit_last) {
        for (int b = threadIdx.x; b < a.num_reqs; b += blockDim.x) a.counters[b] = 0;
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicExch(&a.ctrl->queue_head, 0);
            atomicExch(&a.ctrl->red_head, 0);
            atomicExch(&a.ctrl->exit_count, 0);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
        else
            cudaGetLastError();
    });
    return fn;
}

// 2D view of a cache: rows = num_pages * Hkv * P, D elements per row (bf16, or E4M3 bytes);
// 128-byte x P boxes, 128B swizzle
cudaError_t make_map(CUtensorMap* map, const void* base, int D, int P, long long rows, bool f8) {
    auto enc = get_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int eb = f8 ? 1 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * eb};
    cuuint32_t box[2] = {(cuuint32_t)(128 / eb), (cuuint32_t)P};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int P, int S, bool F8 = false, bool T8 = false>
cudaError_t launch_cfg(const KernelArgs& a, int num_pages_total, cudaStream_t s) {
    using C = Cfg<D, P, S, F8, T8>;
    const long long rows = (long long)num_pages_total * a.num_kv_heads * P;
    if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
    if ((((uintptr_t)a.k_cache) & 15) || (((uintptr_t)a.v_cache) & 15)) return cudaErrorMisalignedAddress;
    CUtensorMap mk, mv;
    cudaError_t e = make_map(&mk, a.k_cache, D, P, rows, F8);
    if (e != cudaSuccess) return e;
    if ((e = make_map(&mv, a.v_cache, D, P, rows, F8)) != cudaSuccess) return e;
    auto kern = gqa_engine_kernel<C>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&]() {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<C>());
    });
    if (attr_err != cudaSuccess) return attr_err;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int grid = gqa_engine_ctas(dev);
    if (grid <= 0) return cudaErrorUnknown;
    if (a.max_ctas > 0) grid = std::min(grid, a.max_ctas);
    // enough CTAs for the tasks, or (a reduction-only launch) for the reduction items
    const long long work = std::max<long long>(a.num_tasks, a.fused ? (a.num_red + C::THREADS / 32 - 1) / (C::THREADS / 32) : 0);
    grid = (int)std::min<long long>(grid, std::max<long long>(1, work));
    {
        ProfileScope ps(SPLITKV_KERNEL_GQA_ENGINE, s);
        kern<<<grid, C::THREADS, smem_bytes<C>(), s>>>(mk, mv, a);
    }
    return cudaGetLastError();
}

}  // namespace

bool gqa_engine_supports_fp8(int head_dim, int page_size) {
    return head_dim == 128 && (page_size == 64 || page_size == 128);
}

bool gqa_engine_supports(int head_dim, int page_size) {
    return (head_dim == 128 || head_dim == 64) && (page_size == 16 || page_size == 64 || page_size == 128);
}

int gqa_engine_ctas(int device) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;   // one persistent CTA per SM
}

cudaError_t launch_gqa_engine(const KernelArgs& a, int num_pages_total, int rows8, cudaStream_t s) {
    // nothing to attend and (fused) nothing to reduce: no launch
    if (a.num_tasks <= 0 && !(a.fused && a.num_red > 0)) return cudaSuccess;
    const int D = a.head_dim_qk, P = a.page_size;
    if (a.kv_fp8) {
        // E4M3 codes: 128 keys (16 KiB of K and of V) per stage, six stages
        if (D == 128 && P == 64) return launch_cfg<128, 64, 4, true>(a, num_pages_total, s);
        if (D == 128 && P == 128) return launch_cfg<128, 128, 2, true>(a, num_pages_total, s);
        return cudaErrorNotSupported;
    }
    // every task of at most 8 rows (decode with up to 8 query heads per KV head): the
    // transposed products, without padded MMA rows
    if (rows8 && D == 128 && P == 64) return launch_cfg<128, 64, 2, false, true>(a, num_pages_total, s);
    if (rows8 && D == 128 && P == 128) return launch_cfg<128, 128, 1, false, true>(a, num_pages_total, s);
    // 64-token pages go two to a stage: 128 keys per pipeline step, as with 128-token pages
    if (D == 128 && P == 64) return launch_cfg<128, 64, 2>(a, num_pages_total, s);
    if (D == 128 && P == 128) return launch_cfg<128, 128, 1>(a, num_pages_total, s);
    if (D == 128 && P == 16) return launch_cfg<128, 16, 1>(a, num_pages_total, s);
    if (D == 64 && P == 64) return launch_cfg<64, 64, 2>(a, num_pages_total, s);
    if (D == 64 && P == 128) return launch_cfg<64, 128, 1>(a, num_pages_total, s);
    if (D == 64 && P == 16) return launch_cfg<64, 16, 1>(a, num_pages_total, s);
    return cudaErrorNotSupported;
}

}  // namespace skv
