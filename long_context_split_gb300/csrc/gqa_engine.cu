// Persistent split-KV engine for bf16 GQA attention on sm_103a.
//
// What it computes (Helix Parallelism, "Attention-Phase Configuration" steps
// 2-3; LiquidCP Section 3 Eq. 1): for every task -- query rows of one
// (request, KV head) over one split of the history -- the split's partial
// state (output normalised over the split, natural-log LSE); in fused mode
// the last task to finish for a (request, KV head, row block) merges that
// block's splits in split order and writes the final output.
//
// How (LiquidCP Section 6: a persistent GPU-resident engine dispatching
// host-prepared task descriptors):
//  * one CTA per SM; warp 0 produces, warps 1..NWC consume;
//  * the producer claims tasks from a device queue (atomic head, plan
//    order), reads the task's page ids with one warp-wide load, and streams
//    each (page, KV head) K and V block into a ring of NSTAGE shared-memory
//    stages with TMA bulk-tensor copies (128-byte swizzle), completion on an
//    mbarrier per stage; it runs ahead across task boundaries;
//  * consumer warps split each page's keys; each keeps a 16-row online
//    softmax state (base-2 exponent, scale folded in), computes S = Q K^T and
//    O += P V with bf16 m16n8k16 tensor-core MMA (fp32 accumulate), reading
//    K and V from the swizzled stages with ldmatrix; P enters the MMA as a
//    bf16 high part plus a bf16 residual, so rows that see few keys keep
//    float-like weight precision;
//  * at a task's last page the consumer warps combine their states through
//    shared memory and write the partial state (or, for an unsplit request in
//    fused mode, the output); the completion counter of the row block elects
//    the last writer, which merges.
// Every wait is bounded (globaltimer); on expiry the kernel records an error
// word, stops, waits for its own copies in flight and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

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

// (x, y) -> bf16 pair hi = round(x, y) and residual pair lo = round((x, y) - hi):
// hi + lo carries about 16 significant bits of each probability
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

// ---------------------------------------------------------------------------
// configuration
// ---------------------------------------------------------------------------
template <int D_, int P_>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int P = P_;
    static constexpr int NWC = (P == 16) ? 1 : 4;        // consumer warps
    static constexpr int KPW = P / NWC;                  // keys per consumer warp per page
    static constexpr int NT = KPW / 8;                   // score n-tiles per warp
    static constexpr int KSTEP_PV = KPW / 16;            // PV k-steps per warp
    static constexpr int TILE_BYTES = P * D * 2;         // one (page, KV head) block
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K + V
    static constexpr int NSTAGE = (STAGE_BYTES >= 65536) ? 3 : (STAGE_BYTES >= 32768 ? 5 : 8);
    static constexpr int BOXES = D / 64;                 // 128-byte-wide TMA boxes per row
    static constexpr int DT = D / 8;                     // output n-tiles
    static constexpr int KT = D / 16;                    // QK k-steps
    static constexpr int COMB_STRIDE = D + 4;            // floats per combine row
    static constexpr int THREADS = (NWC + 1) * 32;
    static constexpr size_t STAGES_BYTES = (size_t)NSTAGE * STAGE_BYTES;
    static constexpr size_t COMB_BYTES = (size_t)NWC * 16 * COMB_STRIDE * 4;
    static_assert(KPW % 16 == 0, "keys per warp must be a multiple of 16");
};

// Stage header written by the producer before it arrives on the stage's full barrier.
enum : int { F_FIRST = 1, F_LAST = 2, F_EMPTY = 4, F_END = 8, F_MASK = 16 };
struct StageHdr {
    TaskDesc t;
    ReqDesc r;
    int page;     // page index within the request
    int flags;
    int pad[6];
};
static_assert(sizeof(StageHdr) == 96, "StageHdr");

template <class C>
struct SmemExtra {
    StageHdr hdr[C::NSTAGE];
    unsigned long long full[C::NSTAGE];
    unsigned long long empty[C::NSTAGE];
    float comb_m[C::NWC][16];
    float comb_l[C::NWC][16];
    int abort_flag;
    int is_last;
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

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
gqa_engine_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  KernelArgs a) {
    static_assert(smem_bytes<C>() <= 227 * 1024, "shared memory budget");
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
        X.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort_flag = &X.abort_flag;

    if (warp == 0) {
        // ============================ producer ============================
        const uint64_t policy = evict_first_policy();
        uint32_t item = 0;
        int last_parity[C::NSTAGE];
        bool had_tma[C::NSTAGE];
#pragma unroll
        for (int s = 0; s < C::NSTAGE; ++s) { last_parity[s] = 0; had_tma[s] = false; }
        bool stop = false;
        // returns the stage for the next item after waiting for it to be free
        auto acquire = [&](int& stage) -> bool {
            stage = (int)(item % C::NSTAGE);
            const uint32_t round = item / C::NSTAGE;
            int okw = 1;
            if (lane == 0) {
                okw = mbar_wait_bounded(smem_u32(&X.empty[stage]), (round & 1) ^ 1, abort_flag, true) ? 1 : 0;
                if (!okw && !*abort_flag) {
                    set_error(a.err, ERR_TIMEOUT | SITE_EMPTY_WAIT);
                    *abort_flag = 1;
                }
            }
            return __shfl_sync(0xffffffffu, okw, 0) != 0;
        };
        while (!stop) {
            int task = 0;
            if (lane == 0) task = atomicAdd(&a.ctrl->queue_head, 1);
            task = __shfl_sync(0xffffffffu, task, 0);
            if (task >= a.num_tasks) {
                int stage;
                if (!acquire(stage)) break;
                if (lane == 0) {
                    X.hdr[stage].flags = F_END;
                    had_tma[stage] = false;
                    mbar_arrive(smem_u32(&X.full[stage]));
                }
                ++item;
                break;
            }
            const TaskDesc t = a.tasks[task];
            const ReqDesc r = a.reqs[t.b];
            const int g = a.group;
            const int i_first = t.row_begin / g;
            const int i_last = (t.row_end - 1) / g;
            const int hi_key = min(t.key_end, r.seq_len - r.q_len + i_last + 1);   // exclusive
            const int mask_from = min(t.key_end, r.seq_len - r.q_len + i_first + 1);
            const int pb = t.key_begin / C::P;
            const int pe = (hi_key > t.key_begin) ? (hi_key + C::P - 1) / C::P : pb;
            if (pe <= pb) {
                int stage;
                if (!acquire(stage)) break;
                if (lane == 0) {
                    X.hdr[stage].t = t;
                    X.hdr[stage].r = r;
                    X.hdr[stage].page = pb;
                    X.hdr[stage].flags = F_FIRST | F_LAST | F_EMPTY;
                    had_tma[stage] = false;
                    mbar_arrive(smem_u32(&X.full[stage]));
                }
                ++item;
                continue;
            }
            for (int c0 = pb; c0 < pe && !stop; c0 += 32) {
                int pid = 0;
                if (c0 + lane < pe) pid = a.page_table[r.page_row + c0 + lane];
                const int cnt = min(32, pe - c0);
                for (int j = 0; j < cnt; ++j) {
                    const int p = c0 + j;
                    const int phys = __shfl_sync(0xffffffffu, pid, j);
                    int stage;
                    if (!acquire(stage)) { stop = true; break; }
                    if (lane == 0) {
                        StageHdr& hd = X.hdr[stage];
                        hd.t = t;
                        hd.r = r;
                        hd.page = p;
                        int fl = 0;
                        if (p == pb) fl |= F_FIRST;
                        if (p == pe - 1) fl |= F_LAST;
                        if ((p + 1) * C::P > mask_from) fl |= F_MASK;
                        hd.flags = fl;
                        last_parity[stage] = (int)((item / C::NSTAGE) & 1);
                        const uint32_t full = smem_u32(&X.full[stage]);
                        if (phys < 0 || phys >= a.num_pages) {
                            set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
                            had_tma[stage] = false;
                            mbar_arrive(full);
                        } else {
                            had_tma[stage] = true;
                            mbar_arrive_expect_tx(full, C::STAGE_BYTES);
                            const int y = (phys * a.num_kv_heads + t.kv_head) * C::P;
                            const uint32_t dk = smem_u32(stages + (size_t)stage * C::STAGE_BYTES);
                            const uint32_t dv = dk + C::TILE_BYTES;
#pragma unroll
                            for (int bx = 0; bx < C::BOXES; ++bx) {
                                tma_load_2d(dk + bx * C::P * 128, &tmap_k, bx * 64, y, full, policy);
                                tma_load_2d(dv + bx * C::P * 128, &tmap_v, bx * 64, y, full, policy);
                            }
                        }
                    }
                    __syncwarp();
                    ++item;
                }
            }
        }
        // make sure no copy issued by this CTA is still landing in shared memory
        if (lane == 0) {
            for (int s = 0; s < C::NSTAGE; ++s) {
                if (had_tma[s] &&
                    !mbar_wait_bounded(smem_u32(&X.full[s]), (uint32_t)last_parity[s], abort_flag, false))
                    set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
            }
        }
        __syncwarp();
    } else {
        // ============================ consumers ===========================
        const int w = warp - 1;
        const int qr = lane >> 2;        // fragment row (and row + 8)
        const int qc = (lane & 3) * 2;   // fragment column pair
        uint32_t qa[C::KT][4];
        float o[C::DT][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int lim0 = 0, lim1 = 0;          // last key index visible to rows qr, qr + 8
        uint32_t item = 0;
        while (true) {
            const int stage = (int)(item % C::NSTAGE);
            const uint32_t round = item / C::NSTAGE;
            int okw = 1;
            if (lane == 0) {
                okw = mbar_wait_bounded(smem_u32(&X.full[stage]), round & 1, abort_flag, true) ? 1 : 0;
                if (!okw && !*abort_flag) {
                    set_error(a.err, ERR_TIMEOUT | SITE_FULL_WAIT);
                    *abort_flag = 1;
                }
            }
            if (!__shfl_sync(0xffffffffu, okw, 0)) break;
            // the phase is complete (lane 0 saw it and it cannot advance before this warp
            // releases the stage); one more test gives every lane acquire ordering
            (void)mbar_try_wait(smem_u32(&X.full[stage]), round & 1);
            const int flags = X.hdr[stage].flags;
            if (flags & F_END) break;
            const TaskDesc t = X.hdr[stage].t;
            const ReqDesc r = X.hdr[stage].r;
            const int page = X.hdr[stage].page;
            const int g = a.group;
            const int nrows = t.row_end - t.row_begin;
            // Row blocks of more than 16 rows (chunked prefill) run "wide": warp w owns rows
            // 16w .. 16w+15 and walks every key of the page; 16-row blocks (decode) split the
            // page's keys across the warps instead.
            const bool wide = nrows > 16;
            const int wrow0 = wide ? w * 16 : 0;
            if (flags & F_FIRST) {
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
                            lo = *(const uint32_t*)(qp + kk * 16 + qc);
                            hi = *(const uint32_t*)(qp + kk * 16 + 8 + qc);
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
            const int nchunks = (flags & F_EMPTY) ? 0 : (wide ? C::NWC : 1);
            for (int ch = 0; ch < nchunks; ++ch) {
                const uint32_t kbase = smem_u32(stages + (size_t)stage * C::STAGE_BYTES);
                const uint32_t vbase = kbase + C::TILE_BYTES;
                const int kw0 = (wide ? ch : w) * C::KPW;
                // ---- S = Q K^T over this warp's KPW keys ----
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
                // ---- scale, mask, online softmax (base 2) ----
                const int key0 = page * C::P + kw0;
                const bool need_mask = (flags & F_MASK) != 0;
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int n = 0; n < C::NT; ++n) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kidx = key0 + n * 8 + qc + e;
                        float v0 = s[n][e] * a.scale_log2;
                        float v1 = s[n][2 + e] * a.scale_log2;
                        if (need_mask) {
                            if (kidx > lim0 || kidx >= t.key_end) v0 = -INFINITY;
                            if (kidx > lim1 || kidx >= t.key_end) v1 = -INFINITY;
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
                    s[n][0] = exp2f(s[n][0] - b0s);
                    s[n][1] = exp2f(s[n][1] - b0s);
                    s[n][2] = exp2f(s[n][2] - b1s);
                    s[n][3] = exp2f(s[n][3] - b1s);
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
                // ---- O += P V, with P = P_hi + P_lo (two bf16 terms, ~16-bit weights) ----
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
                        mma_bf16(o[nd], ph, b0, b1);
                        mma_bf16(o[nd + 1], ph, b2, b3);
                        mma_bf16(o[nd], pl, b0, b1);
                        mma_bf16(o[nd + 1], pl, b2, b3);
                    }
                }
            }
            // release the stage to the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&X.empty[stage]));
            ++item;

            if (flags & F_LAST) {
                // ---- combine the NWC warp states of this task ----
                float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
                lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
                float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
                lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
                float* cw = comb + (size_t)w * 16 * C::COMB_STRIDE;
#pragma unroll
                for (int n = 0; n < C::DT; ++n) {
                    *(float2*)(cw + qr * C::COMB_STRIDE + n * 8 + qc) = make_float2(o[n][0], o[n][1]);
                    *(float2*)(cw + (qr + 8) * C::COMB_STRIDE + n * 8 + qc) = make_float2(o[n][2], o[n][3]);
                }
                if ((lane & 3) == 0) {
                    X.comb_m[w][qr] = m0;
                    X.comb_m[w][qr + 8] = m1;
                    X.comb_l[w][qr] = lt0;
                    X.comb_l[w][qr + 8] = lt1;
                }
                if (C::NWC > 1) named_bar_sync(1, C::NWC * 32); else __syncwarp();
                // Finalise: narrow blocks merge the NWC warps' states of each row (each warp
                // takes 16 / NWC rows); in wide blocks every warp finalises its own 16 rows
                // from its own slot.  Lanes cover a row with float4.
                constexpr int RPW = 16 / C::NWC;
                const bool fused = a.fused != 0;
                const bool unsplit = r.n_splits == 1;
                const int src0 = wide ? w : 0, nsrc = wide ? 1 : C::NWC;
                const int rbeg = wide ? 0 : w * RPW, rend = wide ? 16 : (w + 1) * RPW;
                for (int rr = rbeg; rr < rend; ++rr) {
                    if (wrow0 + rr >= nrows) break;
                    float M = -INFINITY;
#pragma unroll
                    for (int u = 0; u < C::NWC; ++u)
                        if (u < nsrc) M = fmaxf(M, X.comb_m[src0 + u][rr]);
                    float L = 0.f;
                    float f[C::NWC];
#pragma unroll
                    for (int u = 0; u < C::NWC; ++u) {
                        f[u] = (u >= nsrc || M == -INFINITY) ? 0.f : exp2f(X.comb_m[src0 + u][rr] - M);
                        if (u < nsrc) L += X.comb_l[src0 + u][rr] * f[u];
                    }
                    const bool empty = !(L > 0.f);
                    const float inv = empty ? 0.f : 1.f / L;
                    const float lse = empty ? -INFINITY : (M + log2f(L)) * 0.69314718055994531f;
                    const int row = t.row_begin + wrow0 + rr;
                    const int i = row / g;
                    const int h = t.kv_head * g + row % g;
                    const size_t orow = (size_t)(r.q_start + i) * a.num_q_heads + h;
                    const size_t st = (size_t)r.state_base + ((size_t)i * a.num_q_heads + h) * r.n_splits + t.split;
                    for (int c = lane * 4; c < C::D; c += 128) {
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int u = 0; u < C::NWC; ++u) {
                            if (u >= nsrc) break;
                            const float4 v =
                                *(const float4*)(comb + ((size_t)(src0 + u) * 16 + rr) * C::COMB_STRIDE + c);
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
                            __stcg((float4*)(a.o_part + st * C::D + c), acc);
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
                if (fused && !unsplit) {
                    // publish, then let the last writer of this row block merge
                    __threadfence();
                    if (C::NWC > 1) named_bar_sync(1, C::NWC * 32); else __syncwarp();
                    if (w == 0 && lane == 0) {
                        const int prev = atomicAdd(&a.counters[t.merge_slot], 1);
                        X.is_last = (prev == r.n_splits - 1) ? 1 : 0;
                    }
                    if (C::NWC > 1) named_bar_sync(1, C::NWC * 32); else __syncwarp();
                    if (X.is_last) {
                        __threadfence();
                        const int n = r.n_splits;
                        for (int rr = rbeg; rr < rend; ++rr) {
                            if (wrow0 + rr >= nrows) break;
                            const int row = t.row_begin + wrow0 + rr;
                            const int i = row / g;
                            const int h = t.kv_head * g + row % g;
                            const size_t orow = (size_t)(r.q_start + i) * a.num_q_heads + h;
                            const size_t s0 = (size_t)r.state_base + ((size_t)i * a.num_q_heads + h) * n;
                            float M = -INFINITY;
                            for (int q = lane; q < n; q += 32) M = fmaxf(M, __ldcg(a.lse_part + s0 + q));
#pragma unroll
                            for (int off = 16; off > 0; off >>= 1)
                                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                            float den = 0.f;
                            if (M != -INFINITY)
                                for (int q = lane; q < n; q += 32) den += expf(__ldcg(a.lse_part + s0 + q) - M);
#pragma unroll
                            for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
                            const float inv = (M == -INFINITY) ? 0.f : 1.f / den;
                            // every lane runs every shuffle; lanes past the row's width skip the loads
                            constexpr int C4 = (C::D + 127) / 128;   // float4 columns per lane
                            float4 acc[C4];
#pragma unroll
                            for (int u = 0; u < C4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int q0 = 0; q0 < n; q0 += 32) {
                                float wq = 0.f;
                                if (q0 + lane < n && M != -INFINITY)
                                    wq = expf(__ldcg(a.lse_part + s0 + q0 + lane) - M) * inv;
                                const int cnt = min(32, n - q0);
                                for (int q = 0; q < cnt; ++q) {
                                    const float wj = __shfl_sync(0xffffffffu, wq, q);
#pragma unroll
                                    for (int u = 0; u < C4; ++u) {
                                        const int c = lane * 4 + u * 128;
                                        if (c < C::D) {
                                            const float4 v =
                                                __ldcg((const float4*)(a.o_part + (s0 + q0 + q) * C::D + c));
                                            acc[u].x = fmaf(wj, v.x, acc[u].x);
                                            acc[u].y = fmaf(wj, v.y, acc[u].y);
                                            acc[u].z = fmaf(wj, v.z, acc[u].z);
                                            acc[u].w = fmaf(wj, v.w, acc[u].w);
                                        }
                                    }
                                }
                            }
#pragma unroll
                            for (int u = 0; u < C4; ++u) {
                                const int c = lane * 4 + u * 128;
                                if (c >= C::D) continue;
                                const float4 accu = acc[u];
                                if (a.out_bf16) {
                                    __nv_bfloat162* op = (__nv_bfloat162*)((__nv_bfloat16*)a.out + orow * C::D + c);
                                    op[0] = __floats2bfloat162_rn(accu.x, accu.y);
                                    op[1] = __floats2bfloat162_rn(accu.z, accu.w);
                                } else {
                                    *(float4*)((float*)a.out + orow * C::D + c) = accu;
                                }
                            }
                            if (lane == 0 && a.lse_out)
                                a.lse_out[orow] = (M == -INFINITY) ? -INFINITY : M + logf(den);
                        }
                        if (w == 0 && lane == 0) atomicExch(&a.counters[t.merge_slot], 0);
                    }
                }
                // the combine buffer is reused by the next task
                if (C::NWC > 1) named_bar_sync(1, C::NWC * 32); else __syncwarp();
            }
        }
    }

    // every warp leaves its loop (all waits are bounded); the last CTA resets the queue
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(&a.ctrl->exit_count, 1);
        if (prev == (int)gridDim.x - 1) {
            atomicExch(&a.ctrl->queue_head, 0);
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

// 2D view of a cache: rows = num_pages * Hkv * P, D bf16 per row; 64 x P boxes, 128B swizzle
cudaError_t make_map(CUtensorMap* map, const void* base, int D, int P, long long rows) {
    auto enc = get_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)P};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int P>
cudaError_t launch_cfg(const KernelArgs& a, int num_pages_total, cudaStream_t s) {
    using C = Cfg<D, P>;
    const long long rows = (long long)num_pages_total * a.num_kv_heads * P;
    if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
    if ((((uintptr_t)a.k_cache) & 15) || (((uintptr_t)a.v_cache) & 15)) return cudaErrorMisalignedAddress;
    CUtensorMap mk, mv;
    cudaError_t e = make_map(&mk, a.k_cache, D, P, rows);
    if (e != cudaSuccess) return e;
    if ((e = make_map(&mv, a.v_cache, D, P, rows)) != cudaSuccess) return e;
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
    grid = (int)std::min<long long>(grid, std::max(1, a.num_tasks));
    kern<<<grid, C::THREADS, smem_bytes<C>(), s>>>(mk, mv, a);
    return cudaGetLastError();
}

}  // namespace

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

cudaError_t launch_gqa_engine(const KernelArgs& a, int num_pages_total, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    const int D = a.head_dim_qk, P = a.page_size;
    if (D == 128 && P == 64) return launch_cfg<128, 64>(a, num_pages_total, s);
    if (D == 128 && P == 128) return launch_cfg<128, 128>(a, num_pages_total, s);
    if (D == 128 && P == 16) return launch_cfg<128, 16>(a, num_pages_total, s);
    if (D == 64 && P == 64) return launch_cfg<64, 64>(a, num_pages_total, s);
    if (D == 64 && P == 128) return launch_cfg<64, 128>(a, num_pages_total, s);
    if (D == 64 && P == 16) return launch_cfg<64, 16>(a, num_pages_total, s);
    return cudaErrorNotSupported;
}

}  // namespace skv
