// Absorbed-MLA partial attention on sm_103a with tcgen05 tensor cores.
//
// What it computes (SPLASH Section 2 Eq. 1 and Appendix A; Helix Parallelism,
// "Attention-Phase Configuration" step 2): for one query token of request b,
// all 128 heads attend one split of the request's latent cache; keys are the
// 576-wide latent rows (d_c = 512 plus d_r = 64 rotary columns), values
// their first 512 columns.  Output: per head the split's normalised O
// (float32, 512 wide) and natural-log LSE.
//
// How: the per-head output accumulator (128 x 512 float32) would fill a whole
// SM's tensor memory, so each task runs as two work items on two CTAs; item
// h produces output columns [256 h, 256 h + 256).  Both items compute the
// task's full score tiles -- the same products in the same order, so the
// same P and LSE bit for bit -- which doubles the score work but needs no
// exchange between SMs, and 128-key tiles keep every score MMA at N = 128.
// The history is streamed in units of 128 keys (two 64-token pages) through
// a ring of nine 16 KB shared-memory slots, in the order the MMA thread reads
// them: the unit's nine key boxes (128 keys x 64 latent columns), then its
// value slots (32 keys x the item's 256 value columns, read again from L2).
// Load latency, not bandwidth, bounds this stream, so the ring is made as
// deep as shared memory allows: the query's first 256 columns live in tensor
// memory (the score MMA's A operand from tensor memory), its last 320 in
// shared memory (80 KB), which leaves one S/P buffer in tensor memory.
// Per unit, in order: one thread issues S = Q K^T (M = 128 heads, N = 128
// keys, 36 k-steps); eight softmax warps (two per tensor-memory lane quadrant,
// each head's row max taken over all 128 keys by both, the exponentials split
// between them by key halves) run the online softmax in base 2 (scale folded
// in after the row max; lazy rescaling of O when a row's running max grows by
// more than 2^8) and write P over its S as a bf16 high part plus a bf16
// residual; the MMA thread then accumulates O += P_hi V + P_lo V (A = P from
// tensor memory, V an MN-major shared-memory operand, N = 256).  Products
// run in issue order, so S of unit u + 1 overwrites P of unit u only after
// P V of unit u has read it, and the softmax of unit u + 1 (which waits for
// its S) may rescale O without further waits.
// Tensor memory: O (256 columns), S/P (128), query (128).
//
// Warp roles: warp 0 TMA producer and work-item claimer (from the workspace
// queue, in plan order: both halves of a task are claimed one after the
// other, so they run side by side and the second reads the pages from L2),
// warp 1 MMA thread and tensor-memory owner, warps 2..9 softmax/epilogue.
// Every wait is bounded (%globaltimer); on expiry the CTA records the error
// word and drains its own copies and MMAs before leaving.
#include "splitkv.h"
#include "tc_common.cuh"
#include "partial_io.cuh"
#include "trace.cuh"

namespace skv {
namespace {

constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPage = 64;
constexpr int kUnit = 128;                          // keys per unit (two pages)
constexpr int kHalfV = 256;                         // output columns per work item
constexpr int kBoxes = 9;                           // 64-column boxes of a query / key row
constexpr int kQTmem = 4;                           // query boxes held in tensor memory (columns 0..255)
constexpr int kQSmem = kBoxes - kQTmem;             // the rest, in shared memory
constexpr int kSlot = 16384;                        // 128 rows x 128 B
constexpr int kPageBox = kPage * 128;               // one page's rows of one 64-column box: 8 KB
constexpr int kVRows = 32;                          // keys per value slot
constexpr int kVBox = kVRows * 128;                 // 32 keys x 64 value columns: 4 KB (four per slot)
constexpr int kNS = 9;                              // ring slots
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (2 + kSoftmaxWarps) * 32;
constexpr int kTmemCols = 512;
constexpr int kColO = 0, kColS = 256, kColQ = 384;  // O: 256 columns; S/P: 128; query: 128
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr int kTR = 4;                              // work-item ring slots
constexpr int kItemConsumers = 1 + kSoftmaxWarps;   // MMA thread + softmax warps

struct Bars {
    unsigned long long item_full[kTR], item_empty[kTR];
    int item_slot[kTR];
    unsigned long long slot_full[kNS], slot_empty[kNS];
    unsigned long long qt_full, qs_full, q_empty;   // query in tensor memory / in shared memory / free
    unsigned long long s_full, p_full;
    unsigned long long o_full, o_empty;
    unsigned long long drain;
    unsigned long long pair[4];                      // per lane quadrant: both softmax warps posted to `xch`
    uint32_t tmem_base;
    int abort_flag;
    float xch[2][kHeads];                            // per key half: the row's max of a unit, or its l at the end
};

constexpr size_t kSmemBytes = 1024 + (size_t)kQSmem * kSlot + (size_t)kNS * kSlot + sizeof(Bars);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Work-item ring: the producer claims items from the workspace queue and
// publishes each id (or -1 at the end); the MMA thread and the softmax warps
// read the ids in order and release the slot.
struct ItemRing {
    uint32_t n = 0;
    // next item id; -2 when the wait gave up.  With whole_warp every lane of the
    // warp calls this together (one release per warp); otherwise a single thread does.
    __device__ __forceinline__ int next(Bars& B, volatile int* abort_flag, int lane, bool whole_warp) {
        const int slot = (int)(n % kTR);
        const uint32_t par = (n / kTR) & 1;
        int ok = 1;
        if (lane == 0) ok = wait_bar(smem_u32(&B.item_full[slot]), par, abort_flag, true) ? 1 : 0;
        if (whole_warp) ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return -2;
        (void)mbar_try(smem_u32(&B.item_full[slot]), par);
        const int id = ((volatile int*)B.item_slot)[slot];
        if (whole_warp) __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&B.item_empty[slot]));
        ++n;
        return id;
    }
};

// per-item facts every role derives from the task descriptor.  The item's keys are those
// of its pages pb, pb + ps, pb + 2 ps, ... (ps = 1: a contiguous range; ps = the split count:
// Helix's round-robin interleaved layout) below the token's causal limit, taken in that
// order: the k-th 64-key page of this dense sequence holds dense keys 64 k .. 64 k + 63.
// Keys rise with the dense index, so the causal cut leaves a dense prefix of nkeys keys.
struct ItemInfo {
    int h, i, split, n_units, pb, ps, nkeys, empty;
    ReqDesc r;
};

__device__ __forceinline__ ItemInfo item_info(const KernelArgs& a, int item) {
    ItemInfo ti;
    const TaskDesc t = a.tasks[item >> 1];
    ti.h = item & 1;
    ti.r = a.reqs[t.b];
    ti.i = t.row_begin / kHeads;
    ti.split = t.split;
    const int kend = min(t.key_end, ti.r.seq_len - ti.r.q_len + ti.i + 1);   // one past the last key
    ti.pb = t.key_begin / kPage;   // splits start on a page boundary
    ti.ps = max(1, t.page_stride);
    const int pe = (kend + kPage - 1) / kPage;                                 // pages holding keys < kend
    const int np = kend > t.key_begin ? (pe - ti.pb + ti.ps - 1) / ti.ps : 0;
    ti.nkeys = np > 0 ? (np - 1) * kPage + min(kPage, kend - (ti.pb + (np - 1) * ti.ps) * kPage) : 0;
    ti.empty = ti.nkeys <= 0;
    ti.n_units = ti.empty ? 0 : (ti.nkeys + kUnit - 1) / kUnit;
    return ti;
}

// keys of unit u that exist (1..128; only the last unit can hold fewer than 128)
__device__ __forceinline__ int unit_keys(const ItemInfo& ti, int u) {
    return min(kUnit, ti.nkeys - u * kUnit);
}

__device__ __forceinline__ int value_slots(int keys) { return (keys + kVRows - 1) / kVRows; }

// ring slots an item passes through: nine key boxes per unit, four value slots per
// full unit and value_slots(keys) for the last one
__device__ __forceinline__ uint32_t item_slots(const ItemInfo& ti) {
    if (ti.n_units == 0) return 0;
    return (uint32_t)(kBoxes * ti.n_units + 4 * (ti.n_units - 1) + value_slots(unit_keys(ti, ti.n_units - 1)));
}

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(kThreads, 1)
mla_partial_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, KernelArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char* sQ = smem;                          // query boxes kQTmem .. 8
    unsigned char* sRing = sQ + kQSmem * kSlot;
    Bars& B = *(Bars*)(sRing + kNS * kSlot);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTR; ++s) {
            mbar_init(smem_u32(&B.item_full[s]), 1);
            mbar_init(smem_u32(&B.item_empty[s]), kItemConsumers);
        }
        for (int s = 0; s < kNS; ++s) {
            mbar_init(smem_u32(&B.slot_full[s]), 1);
            mbar_init(smem_u32(&B.slot_empty[s]), 1);
        }
        mbar_init(smem_u32(&B.qt_full), kSoftmaxWarps);
        mbar_init(smem_u32(&B.qs_full), 1);
        mbar_init(smem_u32(&B.q_empty), 1);
        mbar_init(smem_u32(&B.s_full), 1);
        mbar_init(smem_u32(&B.p_full), kSoftmaxWarps);
        mbar_init(smem_u32(&B.o_full), 1);
        mbar_init(smem_u32(&B.o_empty), kSoftmaxWarps);
        mbar_init(smem_u32(&B.drain), 1);
        for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&B.pair[q]), 64);
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
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B.tmem_base;
    volatile int* abort_flag = &B.abort_flag;

    auto give_up = [&](int site) {
        if (!*abort_flag) {
            set_error(a.err, ERR_TIMEOUT | site);
            *abort_flag = 1;
        }
    };
    // the page (or, over an E4M3 cache, the bf16 copy's slot) of the item's k-th page
    auto page_of = [&](const ItemInfo& ti, int k) -> int {
        const int j = ti.pb + k * ti.ps;
        return a.lat_copy ? ti.r.vh_base + j : a.page_table[ti.r.page_row + j];
    };
    auto page_ok = [&](int ph) { return ph >= 0 && ph < (a.lat_copy ? a.num_vh_pages : a.num_pages); };

    if (warp == 0) {
        // ===================== producer (lane 0) =====================
        if (lane == 0) {
            uint32_t sc = 0, qn = 0, claimed = 0;
            uint32_t had_tma = 0, last_par = 0;   // per ring slot: its last fill had copies, at this parity
            bool q_tma = false;
            uint32_t q_par = 0;
            bool ok = a.inject != 1;              // (test hook: publish nothing)
            // next ring slot, once the MMA thread has released it; -1 when the wait gave up
            auto acquire = [&]() -> int {
                const int s = (int)(sc % kNS);
                if (!wait_bar(smem_u32(&B.slot_empty[s]), ((sc / kNS) & 1) ^ 1, abort_flag, true)) return -1;
                last_par = (last_par & ~(1u << s)) | (((sc / kNS) & 1u) << s);
                ++sc;
                return s;
            };
            // arm slot s for `bytes` of copies (or complete it at once when there are none)
            auto arm = [&](int s, uint32_t bytes) {
                const uint32_t full = smem_u32(&B.slot_full[s]);
                if (bytes) {
                    had_tma |= 1u << s;
                    mbar_expect_tx(full, bytes);
                } else {
                    had_tma &= ~(1u << s);
                    mbar_arrive(full);
                }
            };
            while (ok) {
                const int rs = (int)(claimed % kTR);
                if (!wait_bar(smem_u32(&B.item_empty[rs]), ((claimed / kTR) & 1) ^ 1, abort_flag, true)) {
                    give_up(SITE_EMPTY_WAIT); ok = false; break;
                }
                int item = atomicAdd(&a.ctrl->queue_head, 1);
                if (item >= 2 * a.num_tasks) item = -1;
                ((volatile int*)B.item_slot)[rs] = item;
                mbar_arrive(smem_u32(&B.item_full[rs]));
                ++claimed;
                if (item < 0) break;
                trace_start(a.trace, item, SPLITKV_TRACE_MLA_ITEM);
                const ItemInfo ti = item_info(a, item);
                if (ti.empty) {
                    trace_end(a.trace, item);
                    continue;
                }
                // the query's last five boxes (latent columns 256..575) of token (q_start + i),
                // once the previous item's last score product has read the old ones
                if (!wait_bar(smem_u32(&B.q_empty), (qn & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                {
                    const uint32_t qf = smem_u32(&B.qs_full);
                    mbar_expect_tx(qf, kQSmem * kSlot);
                    const int qrow = (ti.r.q_start + ti.i) * kHeads;
                    for (int c = 0; c < kQSmem; ++c) tma_2d(smem_u32(sQ + c * kSlot), &tmap_q, 64 * (kQTmem + c), qrow, qf);
                    q_tma = true;
                    q_par = qn & 1;
                    ++qn;
                }
                // unit u's nine key boxes (one or two pages of 64 rows each), then its value
                // slots (32 keys x this item's 256 value columns: four boxes)
                for (int u = 0; u < ti.n_units && ok; ++u) {
                    const int keys = unit_keys(ti, u);
                    const int np = keys > kPage ? 2 : 1;
                    int ph[2] = {-1, -1};
                    for (int p = 0; p < np; ++p) {
                        ph[p] = page_of(ti, 2 * u + p);
                        if (!page_ok(ph[p])) { set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE); ph[p] = -1; }
                    }
                    const uint32_t kbytes = (uint32_t)((ph[0] >= 0) + (ph[1] >= 0)) * kPageBox;
                    for (int c = 0; c < kBoxes; ++c) {
                        const int s = acquire();
                        if (s < 0) { ok = false; break; }
                        arm(s, kbytes);
                        const uint32_t dst = smem_u32(sRing + s * kSlot), full = smem_u32(&B.slot_full[s]);
                        for (int p = 0; p < 2; ++p)
                            if (ph[p] >= 0) tma_2d(dst + p * kPageBox, &tmap_k, 64 * c, ph[p] * kPage, full);
                    }
                    const int nv = value_slots(keys);
                    for (int j = 0; j < nv && ok; ++j) {
                        const int pv = ph[j >> 1];
                        const int s = acquire();
                        if (s < 0) { ok = false; break; }
                        arm(s, pv >= 0 ? 4u * kVBox : 0u);
                        if (pv < 0) continue;
                        const uint32_t dst = smem_u32(sRing + s * kSlot), full = smem_u32(&B.slot_full[s]);
                        const int row = pv * kPage + (j & 1) * kVRows;
                        for (int bx = 0; bx < 4; ++bx) tma_2d(dst + bx * kVBox, &tmap_v, kHalfV * ti.h + 64 * bx, row, full);
                    }
                }
                if (!ok) { give_up(SITE_EMPTY_WAIT); break; }
            }
            // no copy may still be landing when the CTA leaves
            for (int s = 0; s < kNS; ++s)
                if (((had_tma >> s) & 1u) && !wait_bar(smem_u32(&B.slot_full[s]), (last_par >> s) & 1u, abort_flag, false))
                    set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
            if (q_tma && !wait_bar(smem_u32(&B.qs_full), q_par, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ===================== MMA thread (lane 0) =====================
        // Per unit: S (nine key boxes), then P V (the value slots) once its P is in.  Ring
        // slots are read in the producer's order.  A full unit's issue code is straight-line
        // (boxes and k-steps unrolled, operand sources and accumulate flags compile-time):
        // tcgen05 issue from one thread queues only a few MMAs, and run-time loops and branches
        // between them left the tensor pipe idle (measured: 2,507 cycles for the score
        // product's 36 MMAs unrolled against 6,052 in a loop over boxes).
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(kHeads, kUnit, 0);
            constexpr uint32_t id_o = idesc_bf16(kHeads, kHalfV, 1);
            const uint64_t kdesc0 = desc_sw128(smem_u32(sRing), 16, 1024);     // + 1024 per slot (16 KB >> 4)
            const uint64_t vdesc0 = desc_sw128(smem_u32(sRing), kVBox, 1024);
            const uint64_t qdesc0 = desc_sw128(smem_u32(sQ), 16, 1024);
            const uint32_t full0 = smem_u32(&B.slot_full[0]), empty0 = smem_u32(&B.slot_empty[0]);
            const uint32_t dcol = tmem + kColS;
            uint32_t rs = 0, rph = 0;                 // next ring slot to read and its phase parity
            uint32_t gi = 0, qn = 0, tn = 0;
            bool ok = true;
            ItemRing ring;
            // one value slot's P V MMAs (keys 32 j .. 32 j + 31 of the unit): high parts at
            // column 64 (kk / 4) + 8 (kk % 4) of the S/P buffer, residuals 32 further
            auto pv_slot = [&](int j, uint32_t first_acc) {
                const uint64_t vd = vdesc0 + ((uint64_t)rs << 10);
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int kk = 2 * j + ks;
                    const uint32_t hi = dcol + (uint32_t)(64 * (kk >> 2) + 8 * (kk & 3));
                    const uint64_t bd = vd + (uint64_t)((ks * 2048) >> 4);
                    if (ks == 0) mma_f16_ts(tmem + kColO, hi, bd, id_o, first_acc);
                    else mma_f16_tsc<1>(tmem + kColO, hi, bd, id_o);
                    mma_f16_tsc<1>(tmem + kColO, hi + 32, bd, id_o);
                }
            };
            auto slot_done = [&]() {
                mma_commit(empty0 + 8u * rs);
                rs = rs == kNS - 1 ? 0u : rs + 1u;
                rph ^= rs == 0u ? 1u : 0u;
            };
            while (ok) {
                const int item = ring.next(B, abort_flag, 0, false);
                if (item == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
                if (item < 0) break;
                const ItemInfo ti = item_info(a, item);
                if (ti.empty) continue;
                if (!wait_bar(smem_u32(&B.qt_full), qn & 1, abort_flag, true) ||
                    !wait_bar(smem_u32(&B.qs_full), qn & 1, abort_flag, true)) {
                    give_up(SITE_FULL_WAIT); ok = false; break;
                }
                ++qn;
                tc_fence_after();
                for (int u = 0; u < ti.n_units && ok; ++u) {
                    // ---- S = Q K^T over the nine key boxes ----
#pragma unroll
                    for (int c = 0; c < kBoxes; ++c) {
                        if (!wait_bar(full0 + 8u * rs, rph, abort_flag, true)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t kd = kdesc0 + ((uint64_t)rs << 10);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {   // 16 latent columns per k-step: 32 bytes
                            if (c < kQTmem) {               // query columns 64 c + 16 kk ..: tensor-memory column 32 c + 8 kk
                                if (c == 0 && kk == 0) mma_f16_tsc<0>(dcol, tmem + kColQ, kd, id_s);
                                else mma_f16_tsc<1>(dcol, tmem + kColQ + 32 * c + 8 * kk, kd + (uint64_t)(2 * kk), id_s);
                            } else {
                                mma_f16c<1>(dcol, qdesc0 + (uint64_t)(((c - kQTmem) * kSlot) >> 4) + (uint64_t)(2 * kk),
                                            kd + (uint64_t)(2 * kk), id_s);
                            }
                        }
                        slot_done();
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&B.s_full));
                    mma_commit_if(smem_u32(&B.q_empty), u == ti.n_units - 1);
                    // ---- O += P V once P is in ----
                    const uint32_t g = gi + u;
                    if (u == 0 && !wait_bar(smem_u32(&B.o_empty), (tn & 1) ^ 1, abort_flag, true)) { ok = false; break; }
                    if (!wait_bar(smem_u32(&B.p_full), g & 1, abort_flag, true)) { ok = false; break; }
                    tc_fence_after();
                    const int nv = value_slots(unit_keys(ti, u));
                    if (nv == 4) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (!wait_bar(full0 + 8u * rs, rph, abort_flag, true)) { ok = false; break; }
                            tc_fence_after();
                            pv_slot(j, (u > 0 || j > 0) ? 1u : 0u);
                            slot_done();
                        }
                    } else {   // the item's last unit, 1..3 value slots
                        for (int j = 0; j < nv; ++j) {
                            if (!wait_bar(full0 + 8u * rs, rph, abort_flag, true)) { ok = false; break; }
                            tc_fence_after();
                            pv_slot(j, (u > 0 || j > 0) ? 1u : 0u);
                            slot_done();
                        }
                    }
                }
                if (!ok) { give_up(SITE_FULL_WAIT); break; }
                mma_commit(smem_u32(&B.o_full));
                gi += ti.n_units;
                ++tn;
            }
            // every MMA issued here completes before tensor memory is released: a final
            // commit tracks all of this thread's earlier tcgen05 operations
            mma_commit(smem_u32(&B.drain));
            if (!wait_bar(smem_u32(&B.drain), 0, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else {
        // ===================== softmax + epilogue =====================
        // Thread = head row of its lane quadrant; the quadrant's two warps split each
        // unit's keys (kh = 0: keys 0..63, kh = 1: 64..127) and the item's output columns.
        const int wq = warp & 3;                                  // tensor-memory lane quadrant
        const int kh = (warp - 2) >> 2;                           // key half
        const int row = (wq << 5) + lane;                         // head
        const int stid = (warp - 2) * 32 + lane;                  // 0..255
        const uint32_t lane_addr = tmem + ((uint32_t)(wq << 5) << 16);
        const float c2 = a.scale_log2;
        uint32_t gi = 0, on = 0, sbase = 0;                       // units, epilogues, ring slots so far
        bool ok = true;
        ItemRing ring;
        // This head's query columns 128 kh .. 128 kh + 127 of the item's token into tensor
        // memory (bf16 pairs, lower column in the low half: the MMA's K-major A layout),
        // then the warp's arrive on qt_full.  Called once every S product of earlier items
        // is done.
        auto load_q = [&](const ItemInfo& tq) {
            const uint4* src = (const uint4*)((const __nv_bfloat16*)a.q +
                                              ((size_t)(tq.r.q_start + tq.i) * kHeads + row) * kDqk + 128 * kh);
            uint32_t r0[32], r1[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v0 = __ldg(src + c);
                const uint4 v1 = __ldg(src + 8 + c);
                r0[4 * c] = v0.x; r0[4 * c + 1] = v0.y; r0[4 * c + 2] = v0.z; r0[4 * c + 3] = v0.w;
                r1[4 * c] = v1.x; r1[4 * c + 1] = v1.y; r1[4 * c + 2] = v1.z; r1[4 * c + 3] = v1.w;
            }
            SKV_ST32(lane_addr + kColQ + 64 * kh, r0);
            SKV_ST32(lane_addr + kColQ + 64 * kh + 32, r1);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&B.qt_full));
        };
        // Post v for the partner warp of this lane quadrant and take its value.  The
        // single slot per key half is reused: the partner has read this warp's previous
        // value before this warp posts again (a unit's P is in, from all eight warps,
        // before the next unit's S exists; the item's last P before its l is posted;
        // the next item's query, loaded after the l swap, before its first S).
        uint32_t xn = 0;
        auto swap = [&](float v, float& partner) -> bool {
            B.xch[kh][row] = v;
            mbar_arrive(smem_u32(&B.pair[wq]));
            if (!warp_wait(smem_u32(&B.pair[wq]), xn & 1, abort_flag, lane)) return false;
            ++xn;
            partner = B.xch[kh ^ 1][row];
            return true;
        };
        int item = ring.next(B, abort_flag, lane, true);
        if (item == -2) { give_up(SITE_FULL_WAIT); ok = false; }
        ItemInfo ti{};
        if (ok && item >= 0) {
            ti = item_info(a, item);
            if (!ti.empty) load_q(ti);
        }
        while (ok && item >= 0) {
            const int col0 = kHalfV * ti.h + 128 * kh;              // this warp's output columns
            const size_t st = (size_t)ti.r.state_base + ((size_t)ti.i * kHeads + row) * ti.r.n_splits + ti.split;
            float m = -INFINITY, l = 0.f;
            if (ti.empty) {
                for (int c = 0; c < 128; c += 4)
                    store_part4(a.o_part, a.part_bf16, st * kDv + col0 + c, make_float4(0.f, 0.f, 0.f, 0.f));
                if (ti.h == 0 && kh == 0) __stcg(a.lse_part + st, -INFINITY);
            }
            for (int u = 0; u < ti.n_units; ++u) {
                const uint32_t g = gi;
                if (!warp_wait(smem_u32(&B.s_full), g & 1, abort_flag, lane)) {
                    give_up(SITE_FULL_WAIT); ok = false; break;
                }
                tc_fence_after();
                ++gi;
                const int keys = unit_keys(ti, u);
                const int key0 = u * kUnit;                                  // dense index of the unit's first key
                const bool unmasked = keys == kUnit;
                // this warp's 64 scores (it reads and later overwrites only its own columns);
                // the row max over all 128 keys from its half's max and the partner warp's
                uint32_t sr[64];
                SKV_LD32(lane_addr + kColS + 64 * kh, sr);
                SKV_LD32(lane_addr + kColS + 64 * kh + 32, (sr + 32));
                tc_wait_ld();
                const float mxr = unmasked ? row_max64<false>(sr, 64) : row_max64<true>(sr, keys - 64 * kh);
                float other;
                if (!swap(mxr, other)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                const float mx = fmaxf(mxr, other) * c2;
                // lazy rescale: a row whose max grew by more than 2^8 rescales its O and l.  The
                // tensor-memory loads and stores are warp-collective, so the whole warp takes the
                // branch when any of its rows needs it (scale 1 for the others).  P V of the
                // previous unit is done: S of this unit was issued after it.
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
                    l *= scale_o;
                    for (int c = 0; c < 128; c += 32) {
                        uint32_t o[32];
                        SKV_LD32(lane_addr + kColO + 128 * kh + c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * scale_o);
                        SKV_ST32(lane_addr + kColO + 128 * kh + c, o);
                    }
                }
                // The last unit's value rows past the task's last key (the unused tail of its
                // last page) may hold anything; their weight is 0, but 0 * NaN is not, so they
                // are zeroed once the slot has landed (the item's last value slot; the MMA
                // thread reads it only after this unit's P is in).  The slot's previous fill,
                // nine slots back, is a key box of this unit, so its phase is complete and the
                // parity wait below cannot match it.
                if (!unmasked) {
                    const int nv = value_slots(keys);
                    const int r0 = keys - kVRows * (nv - 1);
                    if (r0 < kVRows) {
                        const uint32_t q = sbase + item_slots(ti) - 1;
                        const int s = (int)(q % kNS);
                        if (!warp_wait(smem_u32(&B.slot_full[s]), (q / kNS) & 1, abort_flag, lane)) {
                            give_up(SITE_FULL_WAIT); ok = false; break;
                        }
                        unsigned char* vs = sRing + s * kSlot;
                        for (int idx = stid; idx < (kVRows - r0) * 32; idx += 32 * kSoftmaxWarps) {
                            const int rr = r0 + (idx >> 5), bx = (idx >> 3) & 3, ch = idx & 7;
                            *(uint4*)(vs + bx * kVBox + rr * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                // P of this warp's 64 keys over their S: high parts at columns 64 kh .. + 31,
                // residuals at 64 kh + 32 ..
                const float base = (m == -INFINITY) ? 0.f : m;
                const uint32_t pcol = lane_addr + kColS + 64 * kh;
                l += unmasked ? write_p<false>(sr, c2, base, key0 + 64 * kh, ti.nkeys - 1, pcol)
                              : write_p<true>(sr, c2, base, key0 + 64 * kh, ti.nkeys - 1, pcol);
                tc_wait_st();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.p_full));
            }
            if (!ok) break;
            sbase += item_slots(ti);
            // ---- l summed over both key halves: once the item's last P is in from all
            // eight warps (so the partner has read this warp's last row max) ----
            float lt = l;
            if (!ti.empty) {
                if (!warp_wait(smem_u32(&B.p_full), (gi - 1) & 1, abort_flag, lane)) {
                    give_up(SITE_FULL_WAIT); ok = false; break;
                }
                float lp;
                if (!swap(l, lp)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                lt = l + lp;
            }
            // ---- the next item's query: every S product of this item is done ----
            const int next = ring.next(B, abort_flag, lane, true);
            if (next == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
            ItemInfo tn{};
            if (next >= 0) {
                tn = item_info(a, next);
                if (!tn.empty) load_q(tn);
            }
            if (!ti.empty) {
                // ---- epilogue: O / l to the partial state ----
                if (!warp_wait(smem_u32(&B.o_full), on & 1, abort_flag, lane)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++on;
                tc_fence_after();
                const bool empty_row = !(lt > 0.f);
                const float inv = empty_row ? 0.f : a.v_scale / lt;   // v_scale: the E4M3 latent's scale, else 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t o[32];
                    SKV_LD32(lane_addr + kColO + 128 * kh + c, o);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        store_part4(a.o_part, a.part_bf16, st * kDv + col0 + c + j,
                                    make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                                __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv));
                }
                if (ti.h == 0 && kh == 0)
                    __stcg(a.lse_part + st, empty_row ? -INFINITY : (m + log2f(lt)) * 0.69314718055994531f);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.o_empty));
                if (lane == 0) trace_end(a.trace, item);
            }
            item = next;
            ti = tn;
        }
    }

    tc_fence_before();
    __syncthreads();
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

// The bf16 copy of the batch's E4M3 latent pages that the kernel reads when the cache
// holds codes: slot s is page vh_pages[s].j of request vh_pages[s].b (64 rows x 576).
// E4M3 values are exact in bf16, so the copy holds the codes' values; the key scale is
// folded into the score scale and the value scale into the normalisation.  Rows past a
// request's last key are zeros; page ids outside the pool are reported (DEVICE_CHECK) and
// their slots zeroed.
__global__ void __launch_bounds__(256) mla_latent_convert_kernel(KernelArgs a) {
    constexpr int kChunks = kDqk / 16;                                   // 16 codes per chunk
    const uint8_t* codes = (const uint8_t*)a.k_cache;
    __nv_bfloat16* dst = (__nv_bfloat16*)a.v_half;
    // one slot per CTA iteration: its page and key count read once
    for (int s = blockIdx.x; s < a.num_vh_pages; s += gridDim.x) {
        const VhPage vp = a.vh_pages[s];
        const ReqDesc r = a.reqs[vp.b];
        const int rows = min(kPage, r.seq_len - vp.j * kPage);           // rows holding keys
        int page = a.page_table[r.page_row + vp.j];
        if (page < 0 || page >= a.num_pages) {
            if (threadIdx.x == 0) atomicCAS(a.err, 0, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
            page = -1;
        }
        const uint8_t* src = codes + (size_t)max(page, 0) * kPage * kDqk;
        __nv_bfloat16* out = dst + (size_t)s * kPage * kDqk;
        for (int c = threadIdx.x; c < kPage * kChunks; c += blockDim.x) {
            const int row = c / kChunks;
            uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (row < rows && page >= 0) {
                const uint4 v = *(const uint4*)(src + (size_t)c * 16);
                const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t f16x2;
                    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
                        : "=r"(f16x2) : "r"(cw[k >> 1] >> (16 * (k & 1))));
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f16x2));
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x, f.y);
                    w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                }
            }
            uint4* o = (uint4*)(out + (size_t)c * 16);
            o[0] = make_uint4(w[0], w[1], w[2], w[3]);
            o[1] = make_uint4(w[4], w[5], w[6], w[7]);
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

int mla_tc_ctas(int device) {
    static int cached[64] = {0};
    if (device < 0 || device >= 64) return 0;
    if (cached[device] > 0) return cached[device];
    cudaError_t e = cudaFuncSetAttribute(mla_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) { cudaGetLastError(); return 0; }
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mla_partial_kernel, kThreads, kSmemBytes);
    if (e != cudaSuccess) { cudaGetLastError(); return 0; }
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) { cudaGetLastError(); return 0; }
    // one CTA per SM: each allocates all 512 tensor-memory columns
    cached[device] = std::min(per_sm, 1) * sms;
    return cached[device];
}

cudaError_t launch_mla_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    if ((((uintptr_t)a.q) & 15) || (((uintptr_t)a.k_cache) & 15)) return cudaErrorMisalignedAddress;
    // over an E4M3 cache the kernel reads the bf16 copy, written first
    const void* lat = a.lat_copy ? a.v_half : a.k_cache;
    const long long qrows = total_q * kHeads;
    const long long kvrows = (long long)(a.lat_copy ? a.num_vh_pages : num_pages_total) * kPage;
    if (qrows >= (1LL << 31) || kvrows >= (1LL << 31)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (a.lat_copy) {
        if (!a.v_half || a.num_vh_pages <= 0 || (((uintptr_t)a.v_half) & 15)) return cudaErrorInvalidValue;
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        const long long blocks = std::min<long long>((long long)sms * 8, a.num_vh_pages);
        {
            ProfileScope ps(SPLITKV_KERNEL_MLA_LATENT, s);
            mla_latent_convert_kernel<<<(int)blocks, 256, 0, s>>>(a);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    CUtensorMap mq, mk, mv;
    if ((e = map_576(&mq, a.q, qrows, kHeads)) != cudaSuccess) return e;
    if ((e = map_576(&mk, lat, kvrows, kPage)) != cudaSuccess) return e;
    if ((e = map_576(&mv, lat, kvrows, kVRows)) != cudaSuccess) return e;
    const int nctas = mla_tc_ctas(dev);
    if (nctas <= 0) return cudaErrorNotSupported;
    const int grid = (int)std::min<long long>(nctas, 2LL * a.num_tasks);
    {
        ProfileScope ps(SPLITKV_KERNEL_MLA, s);
        mla_partial_kernel<<<dim3(grid), dim3(kThreads), kSmemBytes, s>>>(mq, mk, mv, a);
    }
    return cudaGetLastError();
}

}  // namespace skv
