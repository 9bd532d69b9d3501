// Absorbed-MLA partial attention on sm_103a with tcgen05 tensor cores.
//
// What it computes (SPLASH Section 2 Eq. 1 and Appendix A; Helix Parallelism,
// "Attention-Phase Configuration" step 2): for one query token of request b,
// all 128 heads attend one split of the request's latent cache; keys are the
// 576-wide latent rows (d_c = 512 plus d_r = 64 rotary columns), values
// their first 512 columns.  Output: per head the split's normalised O
// (float32, 512 wide) and natural-log LSE.
//
// How: the per-head output accumulator (128 x 512 float32) fills a whole
// SM's tensor memory and the 128 x 576 query most of its shared memory, so
// one task runs on a cluster of two CTAs (two SMs):
//   CTA 0 holds query/key columns [0, 256) and output columns [0, 256);
//   CTA 1 holds query/key columns [256, 576) and output columns [256, 512).
// The history is streamed one 64-token page ("unit") at a time.  Per unit
// each CTA TMA-loads its columns (128-byte swizzle) into one of three stages
// (pages four units ahead are prefetched into L2 so the loads find them
// there), one thread computes a split-K partial score tile S_c = Q_c K_c^T
// into tensor memory (tcgen05.mma, M=128 heads, N=64 keys; the query's first
// 256 columns of the CTA are an A operand in tensor memory, CTA 1's last 64
// in shared memory), the softmax threads (one per head)
// read it back, send it to the peer through distributed shared memory and
// add the peer's: both CTAs then hold the same S (fp32 addition commutes)
// and run the same online softmax (base 2, scale folded in after the row
// max, lazy rescaling of O when a row's running max grows by more than
// 2^8).  P is written over its S in tensor memory as a bf16 high part plus
// a bf16 residual, and the MMA thread accumulates O_c += P_hi V_c + P_lo V_c
// with A = P from tensor memory and V_c as an MN-major shared-memory operand
// (M=128, N=256).  Tensor memory per CTA: O (256 columns), two S/P buffers
// (64 columns each), the query (128 columns).  The MMA thread follows a
// fixed order -- S of unit u + 1, then P V of unit u once its P is in -- and
// waits only on softmax and copy events, never on its own products (MMA
// issue runs at the pace of the tensor pipe).  Products run in issue order,
// so S of unit u + 2 overwrites P of unit u only after P V of unit u has
// read it, and a softmax thread that sees S of unit u knows that P V of
// unit u - 2 (the last reader of that buffer) and every S of the task
// before it are done.
//
// Warp roles per CTA: warp 0 TMA producer, warp 1 MMA thread and
// tensor-memory owner, warps 2..5 softmax/epilogue (thread = head row; each
// also writes its head's query row into tensor memory when a task starts,
// once the last S of the previous task is done).  Rank
// 0's producer claims tasks in plan order from the workspace queue and
// publishes each id to a small ring in both CTAs, so both CTAs and all roles
// follow the same sequence.  Every wait is bounded (%globaltimer); on expiry
// the CTA records the error word and drains its own copies and MMAs before
// leaving.
#include "splitkv.h"
#include "tc_common.cuh"

namespace skv {
namespace {

constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPage = 64;
constexpr int kUnit = 64;                           // tokens per unit (one page)
constexpr int kHalfV = 256;                         // output columns per CTA
constexpr int kBoxes0 = 4;                          // 64-column boxes held by CTA 0 (columns 0..255)
constexpr int kBoxes1 = 5;                          // CTA 1: columns 256..575
constexpr int kQBox = kHeads * 128;                 // one 64-column box of Q: 128 rows x 128 B
constexpr int kKBox = kUnit * 128;                  // one 64-column box of a unit: 64 rows x 128 B
constexpr int kNS = 3;                              // unit stages
constexpr int kPrefetch = 4;                        // pages brought into L2 ahead of their load
constexpr int kQTmemBoxes = 4;                      // query boxes held in tensor memory (columns 0..255 of the CTA)
constexpr int kQBytes = kQBox;                      // 16 KB: CTA 1's fifth query box (shared memory)
constexpr int kStageBytes = kBoxes1 * kKBox;        // 40 KB
constexpr int kXBytes = kHeads * kUnit * 4;         // 32 KB of fp32 partial scores (the peer's)
constexpr int kThreads = 6 * 32;
constexpr int kTmemCols = 512;
constexpr int kColO = 0, kColS = 256, kColQ = 384;  // O: 256 columns; S/P: two 64-column buffers; Q: 128
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr int kTR = 4;                              // task ring slots
constexpr int kTaskConsumers = 5 + 6;               // rank 0: MMA + 4 softmax warps; rank 1: + producer

struct Bars {
    unsigned long long task_full[kTR], task_empty[kTR];
    int task_slot[kTR];
    unsigned long long stage_full[kNS], stage_empty[kNS];
    unsigned long long q_full, q4_full, q_empty;   // query in tensor memory / fifth box copied / free
    unsigned long long s_full[2];
    unsigned long long x_full[2][4];     // per buffer and softmax warp: 8 KB of the peer warp's st.async
    unsigned long long p_full[2], pv_done[2];
    unsigned long long o_full, o_empty;
    unsigned long long drain;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = 1024 + kQBytes + kNS * kStageBytes + 2 * kXBytes + sizeof(Bars);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// arrive on a barrier of the peer CTA (address already mapped to shared::cluster)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Task ring: rank 0's producer claims tasks from the workspace queue and
// publishes each task id (or -1 at the end) to both CTAs; every other role of
// both CTAs reads the ids in order and releases the slot on rank 0.
struct TaskRing {
    uint32_t n = 0;
    // Next task id for a consumer role; -2 when the wait gave up.  With
    // whole_warp every lane of the warp calls this together (one release per
    // warp); otherwise a single thread does.
    __device__ __forceinline__ int next(Bars& B, volatile int* abort_flag, int lane, uint32_t crank, bool whole_warp) {
        const int slot = (int)(n % kTR);
        const uint32_t par = (n / kTR) & 1;
        int ok = 1;
        if (lane == 0) ok = wait_bar(smem_u32(&B.task_full[slot]), par, abort_flag, true, crank != 0) ? 1 : 0;
        if (whole_warp) ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return -2;
        (void)mbar_try(smem_u32(&B.task_full[slot]), par, crank != 0);
        const int id = ((volatile int*)B.task_slot)[slot];
        if (whole_warp) __syncwarp();
        if (lane == 0) {
            const uint32_t bar = smem_u32(&B.task_empty[slot]);
            if (crank == 0) mbar_arrive(bar); else mbar_arrive_remote(mapa(bar, 0));
        }
        ++n;
        return id;
    }
};

// per-task facts every role derives from the descriptor
struct TaskInfo {
    int b, i, split, n_units, pb, kend, empty;
    ReqDesc r;
};

__device__ __forceinline__ TaskInfo task_info(const KernelArgs& a, int task) {
    TaskInfo ti;
    const TaskDesc t = a.tasks[task];
    ti.r = a.reqs[t.b];
    ti.b = t.b;
    ti.i = t.row_begin / kHeads;
    ti.split = t.split;
    ti.kend = min(t.key_end, ti.r.seq_len - ti.r.q_len + ti.i + 1);
    ti.pb = t.key_begin / kPage;
    ti.empty = ti.kend <= t.key_begin;
    ti.n_units = ti.empty ? 0 : (ti.kend - ti.pb * kPage + kUnit - 1) / kUnit;
    return ti;
}

// ---------------------------------------------------------------- kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_partial_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kv,
                   KernelArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char* sQ = smem;
    unsigned char* sStage = sQ + kQBytes;
    unsigned char* sX = sStage + kNS * kStageBytes;       // 2 buffers: the peer's partial scores land here
    Bars& B = *(Bars*)(sX + 2 * kXBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_rank();
    const uint32_t peer = crank ^ 1u;
    const int nboxes = crank == 0 ? kBoxes0 : kBoxes1;
    const int col0 = crank == 0 ? 0 : 256;                // first latent column held here

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTR; ++s) {
            mbar_init(smem_u32(&B.task_full[s]), 1);
            mbar_init(smem_u32(&B.task_empty[s]), kTaskConsumers);
        }
        for (int s = 0; s < kNS; ++s) {
            mbar_init(smem_u32(&B.stage_full[s]), 1);
            mbar_init(smem_u32(&B.stage_empty[s]), 1);
        }
        // q_full: the four softmax warps wrote the query to tensor memory; q4_full: rank 1's
        // fifth query box landed in shared memory
        mbar_init(smem_u32(&B.q_full), 4);
        mbar_init(smem_u32(&B.q4_full), 1);
        mbar_init(smem_u32(&B.q_empty), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&B.s_full[s]), 1);
            for (int w = 0; w < 4; ++w) mbar_init(smem_u32(&B.x_full[s][w]), 1);
            mbar_init(smem_u32(&B.p_full[s]), 4);
            mbar_init(smem_u32(&B.pv_done[s]), 1);
        }
        mbar_init(smem_u32(&B.o_full), 1);
        mbar_init(smem_u32(&B.o_empty), 4);
        mbar_init(smem_u32(&B.drain), 1);
        B.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&B.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = B.tmem_base;
    volatile int* abort_flag = &B.abort_flag;

    auto give_up = [&](int site) {
        if (!*abort_flag) {
            set_error(a.err, ERR_TIMEOUT | site);
            *abort_flag = 1;
        }
    };

    if (warp == 0) {
        // ===================== producer (lane 0) =====================
        if (lane == 0) {
            uint32_t item = 0, qn = 0;
            uint32_t had_tma = 0, last_par = 0;   // per-stage bits
            bool q_tma = false;
            uint32_t q_par = 0;
            bool ok = true;
            TaskRing ring;
            uint32_t claimed = 0;
            const uint32_t peer_slots = mapa(smem_u32(&B.task_slot[0]), peer);
            const uint32_t peer_full = mapa(smem_u32(&B.task_full[0]), peer);
            if (crank == 0 && a.inject == 1) ok = false;   // (test hook: publish nothing)
            while (ok) {
                int task;
                if (crank == 0) {
                    // claim the next task and publish it to both CTAs
                    const int slot = (int)(claimed % kTR);
                    if (!wait_bar(smem_u32(&B.task_empty[slot]), ((claimed / kTR) & 1) ^ 1, abort_flag, true, true)) {
                        give_up(SITE_EMPTY_WAIT); ok = false; break;
                    }
                    task = atomicAdd(&a.ctrl->queue_head, 1);
                    if (task >= a.num_tasks) task = -1;
                    ((volatile int*)B.task_slot)[slot] = task;
                    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(peer_slots + 4u * slot), "r"(task) : "memory");
                    mbar_arrive(smem_u32(&B.task_full[slot]));
                    mbar_arrive_remote(peer_full + 8u * slot);
                    ++claimed;
                } else {
                    task = ring.next(B, abort_flag, 0, crank, false);
                    if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
                }
                if (task < 0) break;
                const TaskInfo ti = task_info(a, task);
                if (ti.empty) continue;
                // rank 1: the query's last 64 columns for token (q_start + i), rows tok*128 ..
                // +127, once the previous task's last S product has read them
                if (crank == 1) {
                    if (!wait_bar(smem_u32(&B.q_empty), (qn & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                    mbar_expect_tx(smem_u32(&B.q4_full), kQBox);
                    const int qrow = (ti.r.q_start + ti.i) * kHeads;
                    tma_2d(smem_u32(sQ), &tmap_q, col0 + 64 * kQTmemBoxes, qrow, smem_u32(&B.q4_full));
                    q_tma = true;
                    q_par = qn & 1;
                }
                ++qn;
                // the stage ring holds two pages; the pages kPrefetch ahead are brought into L2
                // so each stage load finds its data there
                auto prefetch = [&](int u) {
                    const int ph = a.page_table[ti.r.page_row + ti.pb + u];
                    if (ph < 0 || ph >= a.num_pages) return;
                    for (int j = 0; j < nboxes; ++j) tma_prefetch_2d(&tmap_kv, col0 + 64 * j, ph * kPage);
                };
                for (int u = 1; u < kPrefetch && u < ti.n_units; ++u) prefetch(u);
                for (int u = 0; u < ti.n_units; ++u) {
                    if (u + kPrefetch < ti.n_units) prefetch(u + kPrefetch);
                    const int s = (int)(item % kNS);
                    const uint32_t round = item / kNS;
                    if (!wait_bar(smem_u32(&B.stage_empty[s]), (round & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                    const int phys = a.page_table[ti.r.page_row + ti.pb + u];
                    const uint32_t full = smem_u32(&B.stage_full[s]);
                    last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
                    if (phys < 0 || phys >= a.num_pages) {
                        set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
                        had_tma &= ~(1u << s);
                        mbar_arrive(full);
                    } else {
                        had_tma |= 1u << s;
                        mbar_expect_tx(full, nboxes * kKBox);
                        for (int j = 0; j < nboxes; ++j)
                            tma_2d(smem_u32(sStage + s * kStageBytes + j * kKBox), &tmap_kv, col0 + 64 * j, phys * kPage, full);
                    }
                    ++item;
                }
            }
            // no copy may still be landing when the CTA leaves
            for (int s = 0; s < kNS; ++s)
                if (((had_tma >> s) & 1u) && !wait_bar(smem_u32(&B.stage_full[s]), (last_par >> s) & 1u, abort_flag, false))
                    set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
            if (q_tma && !wait_bar(smem_u32(&B.q4_full), q_par, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ===================== MMA thread (lane 0) =====================
        // Fixed order per task: S of unit 0; then for each unit u, S of unit u + 1 (stage
        // loaded), then P V of unit u (its P in).  S of unit u + 1 reuses the buffer of
        // unit u - 1, whose P V product was issued before it.  Bounded hardware waits;
        // descriptors precomputed, k-steps unrolled.
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kHeads, kUnit, 0);
            const uint32_t id_o = idesc_bf16(kHeads, kHalfV, 1);
            const uint64_t qd = desc_sw128(smem_u32(sQ), 16, 1024);
            uint32_t item = 0, qn = 0, tn = 0;
            bool ok = true;
            TaskRing ring;
            while (ok) {
                const int task = ring.next(B, abort_flag, 0, crank, false);
                if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
                if (task < 0) break;
                const TaskInfo ti = task_info(a, task);
                if (ti.empty) continue;
                if (!wait_bar(smem_u32(&B.q_full), qn & 1, abort_flag, true)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                if (crank == 1 && !wait_bar(smem_u32(&B.q4_full), qn & 1, abort_flag, true)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++qn;
                tc_fence_after();
                const uint32_t item0 = item;     // units so far: stage, S and P buffers and phases
                auto issue_s = [&](int u) -> bool {
                    const uint32_t gi = item0 + u;
                    const int stage = (int)(gi % kNS);
                    if (!wait_bar(smem_u32(&B.stage_full[stage]), (gi / kNS) & 1, abort_flag, true)) return false;
                    tc_fence_after();
                    const uint64_t kd = desc_sw128(smem_u32(sStage + stage * kStageBytes), 16, 1024);
                    const uint32_t dcol = tmem + kColS + kUnit * (gi & 1);
#pragma unroll
                    for (int kk = 0; kk < 4 * kBoxes1; ++kk) {
                        if (kk >= 4 * nboxes) break;
                        const uint64_t bd = kd + (uint64_t)((((kk >> 2) * kKBox) + (kk & 3) * 32) >> 4);
                        if (kk < 4 * kQTmemBoxes)   // query columns 16 kk .. 16 kk + 15: tensor-memory columns 8 kk ..
                            mma_f16_ts(dcol, tmem + kColQ + 8 * kk, bd, id_s, kk > 0 ? 1u : 0u);
                        else
                            mma_f16(dcol, qd + (uint64_t)(((kk & 3) * 32) >> 4), bd, id_s, 1u);
                    }
                    mma_commit(smem_u32(&B.s_full[gi & 1]));
                    if (u == ti.n_units - 1) mma_commit(smem_u32(&B.q_empty));
                    return true;
                };
                auto issue_pv = [&](int u) -> bool {
                    const uint32_t gp = item0 + u;
                    if (u == 0 && !wait_bar(smem_u32(&B.o_empty), (tn & 1) ^ 1, abort_flag, true)) return false;
                    if (!wait_bar(smem_u32(&B.p_full[gp & 1]), (gp >> 1) & 1, abort_flag, true)) return false;
                    tc_fence_after();
                    const int stage = (int)(gp % kNS);
                    const uint64_t vd = desc_sw128(smem_u32(sStage + stage * kStageBytes), kKBox, 1024);
                    const uint32_t pcol = tmem + kColS + kUnit * (gp & 1);
                    // k-steps 0..3: bf16 high parts (P columns 0..31); 4..7: residuals (32..63)
                    mma_f16_ts(tmem + kColO, pcol, vd, id_o, u > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < 8; ++kk)
                        mma_f16_ts(tmem + kColO, pcol + (kk >> 2) * 32 + (kk & 3) * 8,
                                   vd + (uint64_t)(((kk & 3) * 2048) >> 4), id_o, 1u);
                    mma_commit(smem_u32(&B.pv_done[gp & 1]));
                    mma_commit(smem_u32(&B.stage_empty[stage]));
                    return true;
                };
                if (!issue_s(0)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                for (int u = 0; u < ti.n_units; ++u) {
                    if (u + 1 < ti.n_units && !issue_s(u + 1)) { ok = false; break; }
                    if (!issue_pv(u)) { ok = false; break; }
                }
                if (!ok) { give_up(SITE_FULL_WAIT); break; }
                mma_commit(smem_u32(&B.o_full));
                item += ti.n_units;
                ++tn;
            }
            // every MMA issued here completes before tensor memory is released: a final
            // commit tracks all of this thread's earlier tcgen05 operations
            mma_commit(smem_u32(&B.drain));
            if (!wait_bar(smem_u32(&B.drain), 0, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else {
        // ===================== softmax + epilogue (thread = head row) =====================
        const int wq = warp & 3;                                  // tensor-memory lane quadrant
        const int row = (wq << 5) + lane;                         // head
        const uint32_t lane_addr = tmem + ((uint32_t)(wq << 5) << 16);
        const uint32_t x_remote = mapa(smem_u32(sX), peer);
        const uint32_t xfull_remote = mapa(smem_u32(&B.x_full[0][wq]), peer);
        const float c2 = a.scale_log2;
        uint32_t sn = 0, on = 0;
        bool ok = true;
        TaskRing ring;
        // This head's query columns col0 .. col0 + 255 of the task's token into tensor memory
        // (bf16 pairs, lower column in the low half: the MMA's K-major A layout), then the
        // warp's arrive on q_full.  Called once every S product of earlier tasks is done.
        auto load_q = [&](const TaskInfo& tq) {
            const uint4* src = (const uint4*)((const __nv_bfloat16*)a.q +
                                              ((size_t)(tq.r.q_start + tq.i) * kHeads + row) * kDqk + col0);
#pragma unroll
            for (int j = 0; j < kQTmemBoxes; j += 2) {
                uint32_t r0[32], r1[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v0 = __ldg(src + 8 * j + c);
                    const uint4 v1 = __ldg(src + 8 * (j + 1) + c);
                    r0[4 * c] = v0.x; r0[4 * c + 1] = v0.y; r0[4 * c + 2] = v0.z; r0[4 * c + 3] = v0.w;
                    r1[4 * c] = v1.x; r1[4 * c + 1] = v1.y; r1[4 * c + 2] = v1.z; r1[4 * c + 3] = v1.w;
                }
                SKV_ST32(lane_addr + kColQ + 32 * j, r0);
                SKV_ST32(lane_addr + kColQ + 32 * (j + 1), r1);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&B.q_full));
        };
        int task = ring.next(B, abort_flag, lane, crank, true);
        if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; }
        TaskInfo ti{};
        if (ok && task >= 0) {
            ti = task_info(a, task);
            if (!ti.empty) load_q(ti);
        }
        while (ok && task >= 0) {
            const int h = row;
            const size_t st = (size_t)ti.r.state_base + ((size_t)ti.i * kHeads + h) * ti.r.n_splits + ti.split;
            float m = -INFINITY, l = 0.f;
            if (ti.empty) {
                for (int c = 0; c < kHalfV; c += 4)
                    __stcg((float4*)(a.o_part + st * kDv + col0 + c), make_float4(0.f, 0.f, 0.f, 0.f));
                if (crank == 0) __stcg(a.lse_part + st, -INFINITY);
            }
            for (int u = 0; u < ti.n_units; ++u) {
                const uint32_t gi = sn;           // unit index: stage gi % kNS, buffers gi & 1
                const int b2 = (int)(gi & 1);
                const uint32_t par = (gi >> 1) & 1;
                // ---- this CTA's partial scores from tensor memory ----
                if (!warp_wait(smem_u32(&B.s_full[b2]), par, abort_flag, lane, false, false)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                tc_fence_after();
                uint32_t sr[64];
                SKV_LD32(lane_addr + kColS + kUnit * b2, sr);
                SKV_LD32(lane_addr + kColS + kUnit * b2 + 32, (sr + 32));
                tc_wait_ld();
                // ---- exchange with the peer (fp32 rows, 16-byte chunks rotated by row) ----
                // Asynchronous remote stores that complete transaction bytes on the peer warp's
                // barrier; this warp's barrier expects the peer's 32 rows x 256 B.  Buffer b2 of
                // the peer held its copy of unit gi - 2; the peer read it before sending unit
                // gi - 1, which this warp has already received, so it is free.
                if (lane == 0) mbar_expect_tx(smem_u32(&B.x_full[b2][wq]), 32 * 256);
                const uint32_t xoff = (uint32_t)(b2 * kXBytes + row * 256);
                const uint32_t xbar = xfull_remote + 8u * (uint32_t)(b2 * 4);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t dst = x_remote + xoff + (uint32_t)((c ^ (row & 15)) << 4);
                    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                                 ::"r"(dst), "r"(sr[4 * c]), "r"(sr[4 * c + 1]), "r"(sr[4 * c + 2]), "r"(sr[4 * c + 3]),
                                 "r"(xbar)
                                 : "memory");
                }
                if (!warp_wait(smem_u32(&B.x_full[b2][wq]), par, abort_flag, lane, true, false)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                const unsigned char* xrow = sX + xoff;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 v = *(const float4*)(xrow + ((c ^ (row & 15)) << 4));
                    sr[4 * c + 0] = __float_as_uint(__uint_as_float(sr[4 * c + 0]) + v.x);
                    sr[4 * c + 1] = __float_as_uint(__uint_as_float(sr[4 * c + 1]) + v.y);
                    sr[4 * c + 2] = __float_as_uint(__uint_as_float(sr[4 * c + 2]) + v.z);
                    sr[4 * c + 3] = __float_as_uint(__uint_as_float(sr[4 * c + 3]) + v.w);
                }
                // these reads come before the peer's asynchronous stores of unit gi + 2 into the
                // same rows (which follow this warp's next send)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                ++sn;
                // ---- online softmax in base 2 (keys >= kend masked; the same for every head) ----
                const int key0 = (ti.pb + u) * kPage;
                const bool unmasked = key0 + kUnit <= ti.kend;
                float mxr = -INFINITY;
                if (unmasked) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) mxr = fmaxf(mxr, __uint_as_float(sr[j]));
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        if (key0 + j < ti.kend) mxr = fmaxf(mxr, __uint_as_float(sr[j]));
                }
                const float mx = mxr * c2;
                // Slots of the unit past the task's last key (the unused tail of the last page)
                // may hold anything; their weight is 0, but 0 * NaN is not, so their value rows
                // (boxes 0..3 of the stage) are zeroed before the P V product.  The score
                // product of this unit has completed, and the fence before the p_full arrive
                // orders these stores before the tensor-core reads.
                if (!unmasked) {
                    const int r0 = ti.kend - key0;
                    unsigned char* vst = sStage + (gi % kNS) * kStageBytes;
                    for (int idx = row; idx < (kUnit - r0) * 32; idx += kHeads) {
                        const int rr = r0 + (idx >> 5), bx = (idx >> 3) & 3, ch = idx & 7;
                        *(uint4*)(vst + bx * kKBox + rr * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // lazy rescale: a row whose max grew by more than 2^8 rescales its O and l.  The
                // tensor-memory loads and stores are warp-collective, so the whole warp takes the
                // branch when any of its rows needs it (scale 1 for the others), after every P V
                // product issued so far (unit gi - 1) has completed.
                float scale_o = 1.f;
                bool need = false;
                if (m == -INFINITY) {
                    m = mx;
                } else if (mx > m + kRescaleThreshold) {
                    scale_o = exp2f(m - mx);
                    m = mx;
                    need = true;
                }
                if (__any_sync(0xffffffffu, need)) {
                    if (u > 0) {
                        const uint32_t gq = gi - 1;
                        if (!warp_wait(smem_u32(&B.pv_done[gq & 1]), (gq >> 1) & 1, abort_flag, lane, false, false)) {
                            give_up(SITE_EMPTY_WAIT); ok = false; break;
                        }
                        tc_fence_after();
                    }
                    l *= scale_o;
                    for (int c = 0; c < kHalfV; c += 32) {
                        uint32_t o[32];
                        SKV_LD32(lane_addr + kColO + c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * scale_o);
                        SKV_ST32(lane_addr + kColO + c, o);
                    }
                }
                // P over this unit's S (read above); the buffer's previous P was read by the P V
                // product of unit gi - 2, issued before S of this unit and so already done
                const float base = (m == -INFINITY) ? 0.f : m;
                const uint32_t pcol = lane_addr + kColS + kUnit * b2;
                l += unmasked ? write_p<false>(sr, c2, base, key0, ti.kend - 1, pcol)
                              : write_p<true>(sr, c2, base, key0, ti.kend - 1, pcol);
                tc_wait_st();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.p_full[b2]));
            }
            if (!ok) break;
            // ---- the next task's query: every S product of this task is done ----
            const int next = ring.next(B, abort_flag, lane, crank, true);
            if (next == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
            TaskInfo tn{};
            if (next >= 0) {
                tn = task_info(a, next);
                if (!tn.empty) load_q(tn);
            }
            if (!ti.empty) {
                // ---- epilogue: O / l to the partial state ----
                if (!warp_wait(smem_u32(&B.o_full), on & 1, abort_flag, lane, false, false)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++on;
                tc_fence_after();
                const bool empty_row = !(l > 0.f);
                const float inv = empty_row ? 0.f : 1.f / l;
                for (int c = 0; c < kHalfV; c += 32) {
                    uint32_t o[32];
                    SKV_LD32(lane_addr + kColO + c, o);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        __stcg((float4*)(a.o_part + st * kDv + col0 + c + j),
                               make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                           __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv));
                }
                if (crank == 0) __stcg(a.lse_part + st, empty_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.o_empty));
            }
            task = next;
            ti = tn;
        }
    }

    // leave together: no remote write or arrive may target a CTA that has gone
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(&a.ctrl->exit_count, 1);
        if (prev == (int)gridDim.x - 1) {
            atomicExch(&a.ctrl->queue_head, 0);
            atomicExch(&a.ctrl->exit_count, 0);
        }
    }
}

// ---------------------------------------------------------------- host
// 2D bf16 view [rows][576] with 64-column x box_rows boxes, 128-byte swizzle
cudaError_t map_576(CUtensorMap* m, const void* base, long long rows, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kDqk * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool mla_tc_supports(int kind_mla, int bf16, int num_q_heads, int dqk, int dv, int page_size) {
    return kind_mla && bf16 && num_q_heads == kHeads && dqk == kDqk && dv == kDv && page_size == kPage;
}

int mla_tc_clusters(int device) {
    static int cached[64] = {0};
    if (device < 0 || device >= 64) return 0;
    if (cached[device] > 0) return cached[device];
    cudaError_t e = cudaFuncSetAttribute(mla_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) { cudaGetLastError(); return 0; }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, mla_partial_kernel, &cfg);
    if (e != cudaSuccess) { cudaGetLastError(); return 0; }
    cached[device] = n;
    return n;
}

cudaError_t launch_mla_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    if ((((uintptr_t)a.q) & 15) || (((uintptr_t)a.k_cache) & 15)) return cudaErrorMisalignedAddress;
    const long long qrows = total_q * kHeads, kvrows = (long long)num_pages_total * kPage;
    if (qrows >= (1LL << 31) || kvrows >= (1LL << 31)) return cudaErrorInvalidValue;
    CUtensorMap mq, mkv;
    cudaError_t e = map_576(&mq, a.q, qrows, kHeads);
    if (e != cudaSuccess) return e;
    if ((e = map_576(&mkv, a.k_cache, kvrows, kUnit)) != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    const int ncl = mla_tc_clusters(dev);
    if (ncl <= 0) return cudaErrorNotSupported;
    const int clusters = std::min(ncl, a.num_tasks);
    {
        ProfileScope ps(SPLITKV_KERNEL_MLA, s);
        mla_partial_kernel<<<dim3(2 * clusters), dim3(kThreads), kSmemBytes, s>>>(mq, mkv, a);
    }
    return cudaGetLastError();
}

}  // namespace skv
