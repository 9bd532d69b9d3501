// Paired row blocks of GQA attention on sm_103a with tcgen05 tensor cores.
//
// What it computes (LiquidCP Section 3 Eq. 1 and Section 7.1: decode steps
// with several query tokens per request -- one target and up to fifteen
// drafts -- and short appended chunks; Helix Parallelism, "Attention-Phase
// Configuration" step 2 for the split state): for a block of 33..128 query
// rows of one (request, KV head) -- row = token * g + head-in-group -- over
// one split of the request's history, each row's partial state (output
// normalised over the keys it sees in the split, natural-log LSE).  Token i
// of a request with q_len appended tokens sees keys [0, seq_len - q_len + i].
//
// How: such a block is too small for the chunk tiles' two-tile tasks (which
// share every K/V unit between 256 rows of one (request, KV head)) and too
// large for the decode engine's warp-level products, so each CTA runs two
// independent blocks side by side, one per 128-row tensor-memory tile: the
// two blocks may belong to different requests, KV heads and splits.  Per
// 64-key unit one producer TMA-loads both tiles' K (128-byte swizzle) into a
// key slot and another both tiles' V into a value slot: a key slot is free
// again once the score products have read it, a value slot once the P V
// products have, so key loads run several units ahead of the products and
// value loads one unit behind them.  Per tile one thread issues S = Q K^T
// (M=128, N=64) into a tensor-memory S/P buffer, the tile's four softmax
// warps (one thread per row) apply the causal mask and the online softmax
// (base 2, lazy rescaling of O when a row's running max grows by more than
// 2^8), write P over S in f16 and convert the tile's values of the unit to
// f16 in place in shared memory (each unit is read by one block only, so a
// copy of the cache in f16 would cost more HBM traffic than it saves); the
// MMA thread then accumulates O += P V as one f16 product.  Per tile, tensor memory holds O and two
// S/P buffers; each tile's MMA thread issues S of unit u + 1 into the other
// buffer, then P V of unit u; products run in issue order, so the softmax
// writes P without waiting on them.  The two tiles' products interleave on
// the tensor pipe and their softmax work on every scheduler.
//
// Warp roles: warp 0 task claimer and producer of Q and K, warp 1 tile 0's
// MMA thread and the tensor-memory owner, warps 2..5 softmax/epilogue of tile
// 0, warps 6..9 of tile 1, warp 10 tile 1's MMA thread, warp 11 producer of
// V.  A task is a pair of
// block descriptors (the second may be empty); tasks come from the
// workspace queue in plan order (pairs of similar length, longest first)
// through a small ring.  In fused mode each softmax warp of a split
// request's block counts itself in once its rows are written, for the
// request's reduction, which the decode engine's reduction phase performs.
// Every wait is bounded (%globaltimer); on expiry the CTA records the error
// word and drains its own copies and MMAs before leaving.
#include "splitkv.h"
#include "tc_common.cuh"
#include "partial_io.cuh"
#include "trace.cuh"

namespace skv {
namespace {

constexpr int kRows = 128;                          // query rows per tile (tensor-memory lanes)
constexpr int kTiles = 2;                           // independent blocks per CTA
constexpr int kKeys = 64;                           // keys per unit
constexpr int kTR = 4;                              // task ring slots
constexpr int kSoftWarps = 4 * kTiles;
constexpr int kTaskConsumers = kTiles + kSoftWarps + 1;   // per tile an MMA thread and 4 softmax
                                                          // warps; the value producer
constexpr int kIssuerWarp1 = 2 + kSoftWarps;        // tile 1's MMA warp (tile 0's is warp 1)
constexpr int kValueWarp = 3 + kSoftWarps;          // the value producer
constexpr int kThreads = (kValueWarp + 1) * 32;
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr size_t kSmemLimit = 232448;
constexpr int kTmemTile = 256;                      // tensor-memory columns per tile: O | S/P | S/P
constexpr int kColS = 128;                          // S/P buffer b at kColS + 64 b: 64 fp32 columns of S,
                                                    // then P as 32 columns of bf16 high parts and 32 of residuals
constexpr int kTmemCols = kTiles * kTmemTile;

template <int D>
struct PairCfg {
    static constexpr int BOXES = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int Q_BOX = kRows * 128;            // 128 rows x 128 B
    static constexpr int KV_BOX = kKeys * 128;           // 64 keys x 128 B
    static constexpr int Q_TILE = BOXES * Q_BOX;
    static constexpr int Q_BYTES = kTiles * Q_TILE;
    static constexpr int TILE_BYTES = BOXES * KV_BOX;    // K (or V) of one unit of one tile
    static constexpr int SLOT_BYTES = kTiles * TILE_BYTES;   // a key (or value) slot: both tiles
    static constexpr int SLOTS_FIT = (int)((kSmemLimit - 1024 - Q_BYTES - 1024) / SLOT_BYTES);
    static constexpr int NK_FIT = (SLOTS_FIT + 1) / 2;
    static constexpr int NK = NK_FIT < 8 ? NK_FIT : 8;           // key slots
    static constexpr int NV = SLOTS_FIT - NK < 8 ? SLOTS_FIT - NK : 8;   // value slots
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(D <= kColS && kColS + 2 * kKeys <= kTmemTile, "tensor memory budget");
    static_assert(NK >= 2 && NV >= 2, "slot rings");
};

template <int NK, int NV>
struct PairBars {
    unsigned long long task_full[kTR], task_empty[kTR];
    int task_slot[kTR];
    unsigned long long k_full[NK], k_empty[NK];
    unsigned long long v_full[NV], v_empty[NV];
    unsigned long long q_full, q_empty;
    unsigned long long s_full[kTiles][2], p_full[kTiles][2], pv_done[kTiles];   // [tile][S/P buffer]
    unsigned long long o_full[kTiles], o_empty[kTiles];
    unsigned long long drain[kTiles];
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
constexpr size_t pair_smem_bytes() {
    using C = PairCfg<D>;
    return 1024 + C::Q_BYTES + (size_t)(C::NK + C::NV) * C::SLOT_BYTES + sizeof(PairBars<C::NK, C::NV>);
}

// one block of a task, as every role derives it from its descriptor
struct PairBlock {
    int b, kv, row0, rows, split, kb, kend, nu;   // kend: one past the last key a row may see; nu: units
    ReqDesc r;
};

struct PairTask {
    PairBlock t[kTiles];
    int n_units, empty;
};

__device__ __forceinline__ PairTask pair_task(const KernelArgs& a, int task) {
    PairTask pt;
    pt.n_units = 0;
#pragma unroll
    for (int tt = 0; tt < kTiles; ++tt) {
        const TaskDesc d = a.tasks[2 * task + tt];
        PairBlock& k = pt.t[tt];
        k.r = a.reqs[d.b];
        k.b = d.b;
        k.kv = d.kv_head;
        k.row0 = d.row_begin;
        k.rows = max(0, min(kRows, d.row_end - d.row_begin));
        k.split = d.split;
        k.kb = d.key_begin;
        k.kend = k.kb;
        k.nu = 0;
        if (k.rows > 0) {
            // keys the block's last row may see: the split's range cut by its causal limit
            const int i_last = (d.row_end - 1) / a.group;
            const int ke = min(d.key_end, k.r.seq_len - k.r.q_len + i_last + 1);
            if (ke > k.kb) {
                k.nu = (ke - k.kb + kKeys - 1) / kKeys;
                k.kend = ke;
            }
        }
        pt.n_units = max(pt.n_units, k.nu);
    }
    pt.empty = pt.n_units == 0;
    return pt;
}

template <class Bars>
struct PairRing {
    uint32_t n = 0;
    // next task id (-1: no more) for a consumer role; -2 when the wait gave up
    __device__ __forceinline__ int next(Bars& B, volatile int* abort_flag, int lane, bool whole_warp) {
        const int slot = (int)(n % kTR);
        const uint32_t par = (n / kTR) & 1;
        int ok = 1;
        if (lane == 0) ok = wait_bar(smem_u32(&B.task_full[slot]), par, abort_flag, true) ? 1 : 0;
        if (whole_warp) ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return -2;
        (void)mbar_try(smem_u32(&B.task_full[slot]), par);
        const int id = ((volatile int*)B.task_slot)[slot];
        if (whole_warp) __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&B.task_empty[slot]));
        ++n;
        return id;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
pair_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, KernelArgs a) {
    using C = PairCfg<D>;
    constexpr int NK = C::NK, NV = C::NV;
    using Bars = PairBars<NK, NV>;
    static_assert(pair_smem_bytes<D>() <= kSmemLimit, "shared memory budget");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char* sQ = smem;                              // tile t at t * Q_TILE
    unsigned char* sK = sQ + C::Q_BYTES;                   // key slot j: tile t's boxes at t * TILE_BYTES
    unsigned char* sV = sK + NK * C::SLOT_BYTES;           // value slot j: likewise
    Bars& B = *(Bars*)(sV + NV * C::SLOT_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTR; ++s) {
            mbar_init(smem_u32(&B.task_full[s]), 1);
            mbar_init(smem_u32(&B.task_empty[s]), kTaskConsumers);
        }
        // a slot is released by one commit per tile's product that read it
        for (int s = 0; s < NK; ++s) {
            mbar_init(smem_u32(&B.k_full[s]), 1);
            mbar_init(smem_u32(&B.k_empty[s]), kTiles);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(smem_u32(&B.v_full[s]), 1);
            mbar_init(smem_u32(&B.v_empty[s]), kTiles);
        }
        mbar_init(smem_u32(&B.q_full), 1);
        mbar_init(smem_u32(&B.q_empty), kTiles);            // one per tile's MMA thread
        for (int t = 0; t < kTiles; ++t) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&B.s_full[t][b]), 1);
                mbar_init(smem_u32(&B.p_full[t][b]), 4);
            }
            mbar_init(smem_u32(&B.pv_done[t]), 1);
            mbar_init(smem_u32(&B.o_full[t]), 1);
            mbar_init(smem_u32(&B.o_empty[t]), 4);
            mbar_init(smem_u32(&B.drain[t]), 1);
        }
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
    const int g = a.group;

    auto give_up = [&](int site) {
        if (!*abort_flag) {
            set_error(a.err, ERR_TIMEOUT | site);
            *abort_flag = 1;
        }
    };
    // row of the key/value tensor maps where tile t's unit u starts (-1: no copy for it)
    auto unit_row = [&](const PairTask& pt, int t, int u) -> int {
        if (u >= pt.t[t].nu) return -1;
        const int key0 = pt.t[t].kb + u * kKeys;
        const int phys = a.page_table[pt.t[t].r.page_row + key0 / a.page_size];
        if (phys < 0 || phys >= a.num_pages) {
            set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
            return -1;
        }
        return (phys * a.num_kv_heads + pt.t[t].kv) * a.page_size + key0 % a.page_size;
    };
    // one slot ring of the producers: load both tiles' boxes of every unit of a task
    // (`map`: K or V), releasing nothing; `had`/`last` remember the slots' last copies
    struct SlotRing {
        uint32_t item = 0, had = 0, last = 0;
    };
    auto load_units = [&](SlotRing& rg, const PairTask& pt, int n_slots, unsigned long long* full,
                          unsigned long long* empty, unsigned char* base, const CUtensorMap* map) -> bool {
        for (int u = 0; u < pt.n_units; ++u) {
            const int s = (int)(rg.item % n_slots);
            const uint32_t round = rg.item / n_slots;
            if (!wait_bar(smem_u32(&empty[s]), (round & 1) ^ 1, abort_flag, true)) return false;
            const uint32_t fb = smem_u32(&full[s]);
            rg.last = (rg.last & ~(1u << s)) | ((round & 1u) << s);
            int y[kTiles];
            uint32_t bytes = 0;
#pragma unroll
            for (int t = 0; t < kTiles; ++t) {
                y[t] = unit_row(pt, t, u);
                if (y[t] >= 0) bytes += C::TILE_BYTES;
            }
            if (bytes == 0) {
                rg.had &= ~(1u << s);
                mbar_arrive(fb);
            } else {
                rg.had |= 1u << s;
                mbar_expect_tx(fb, bytes);
                unsigned char* st = base + s * C::SLOT_BYTES;
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    if (y[t] < 0) continue;
                    for (int j = 0; j < C::BOXES; ++j)
                        tma_2d(smem_u32(st + t * C::TILE_BYTES + j * C::KV_BOX), map, 64 * j, y[t], fb);
                }
            }
            ++rg.item;
        }
        return true;
    };
    // no copy of the ring may still be landing when the CTA leaves
    auto drain_ring = [&](const SlotRing& rg, int n_slots, unsigned long long* full) {
        for (int s = 0; s < n_slots; ++s)
            if (((rg.had >> s) & 1u) && !wait_bar(smem_u32(&full[s]), (rg.last >> s) & 1u, abort_flag, false))
                set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
    };

    if (warp == 0) {
        // ===================== task claimer, Q and K producer (lane 0) =====================
        if (lane == 0) {
            SlotRing kr;
            uint32_t qn = 0, claimed = 0;
            bool q_tma = false;
            uint32_t q_par = 0;
            bool ok = a.inject != 1;   // (test hook: publish nothing)
            while (ok) {
                const int slot = (int)(claimed % kTR);
                if (!wait_bar(smem_u32(&B.task_empty[slot]), ((claimed / kTR) & 1) ^ 1, abort_flag, true)) {
                    give_up(SITE_EMPTY_WAIT); ok = false; break;
                }
                int task = atomicAdd(&a.ctrl->pair_head, 1);
                if (task >= a.num_tasks) task = -1;
                ((volatile int*)B.task_slot)[slot] = task;
                mbar_arrive(smem_u32(&B.task_full[slot]));
                ++claimed;
                if (task < 0) break;
                trace_start(a.trace, task, SPLITKV_TRACE_PAIR);
                const PairTask pt = pair_task(a, task);
                if (pt.empty) {
                    trace_end(a.trace, task);
                    continue;
                }
                // each tile's query rows: tokens (row0 / g) .. + 128 / g of the g heads of its KV
                // head (rows past the block read other tokens or the zero fill past the tensor;
                // they are never written back)
                if (!wait_bar(smem_u32(&B.q_empty), (qn & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                mbar_expect_tx(smem_u32(&B.q_full), C::Q_BYTES);
                for (int t = 0; t < kTiles; ++t) {
                    const int tok0 = pt.t[t].r.q_start + pt.t[t].row0 / g;
                    for (int j = 0; j < C::BOXES; ++j)
                        tma_3d(smem_u32(sQ + t * C::Q_TILE + j * C::Q_BOX), &tmap_q, 64 * j, pt.t[t].kv * g, tok0,
                               smem_u32(&B.q_full));
                }
                q_tma = true;
                q_par = qn & 1;
                ++qn;
                if (!load_units(kr, pt, NK, B.k_full, B.k_empty, sK, &tmap_k)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
            }
            drain_ring(kr, NK, B.k_full);
            if (q_tma && !wait_bar(smem_u32(&B.q_full), q_par, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == kValueWarp) {
        // ===================== V producer (lane 0) =====================
        if (lane == 0) {
            SlotRing vr;
            PairRing<Bars> ring;
            while (true) {
                const int task = ring.next(B, abort_flag, 0, false);
                if (task == -2) { give_up(SITE_FULL_WAIT); break; }
                if (task < 0) break;
                const PairTask pt = pair_task(a, task);
                if (!load_units(vr, pt, NV, B.v_full, B.v_empty, sV, &tmap_v)) { give_up(SITE_EMPTY_WAIT); break; }
            }
            drain_ring(vr, NV, B.v_full);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kIssuerWarp1) {
        // ===================== MMA issuer of tile t (lane 0) =====================
        // Fixed schedule per task: S of unit 0; then for each unit u, S of unit u + 1 (once its
        // keys are in) into the other S/P buffer, whose last reader, P V of unit u - 1, was
        // issued before it, then the P V product of unit u (once its probabilities and values
        // are in).  The thread waits only on its softmax and the copies, never on its own
        // products.
        const int t = warp == 1 ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(kRows, kKeys, 0);
            constexpr uint32_t id_o = idesc_f16(kRows, D, 1);
            const uint64_t qd = desc_sw128(smem_u32(sQ + t * C::Q_TILE), 16, 1024);
            const uint32_t bufcol = tmem + t * kTmemTile + kColS;   // S/P buffer b: bufcol + kKeys b
            const uint32_t ocol = tmem + t * kTmemTile;
            uint32_t item = 0, qn = 0;
            uint32_t pc = 0;      // units this tile attended so far (S, P phases)
            uint32_t tn = 0;      // blocks this tile finished (O phases)
            bool ok = true;
            PairRing<Bars> ring;
            while (ok) {
                const int task = ring.next(B, abort_flag, 0, false);
                if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
                if (task < 0) break;
                const PairTask pt = pair_task(a, task);
                if (pt.empty) continue;
                const uint32_t item0 = item;      // slots of unit u: (item0 + u) % NK, % NV
                item += pt.n_units;
                const int nu = pt.t[t].nu;
                const int nu_other = pt.t[t ^ 1].nu;
                if (!wait_bar(smem_u32(&B.q_full), qn & 1, abort_flag, true)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++qn;
                if (nu == 0) {
                    // this tile attends no key of the task: release the query buffer for it
                    mbar_arrive(smem_u32(&B.q_empty));
                    continue;
                }
                tc_fence_after();
                // S = Q K^T of unit u
                auto issue_s = [&](int u) -> bool {
                    const uint32_t gi = item0 + u;
                    const int ks = (int)(gi % NK);
                    if (!wait_bar(smem_u32(&B.k_full[ks]), (gi / NK) & 1, abort_flag, true)) return false;
                    tc_fence_after();
                    const uint32_t gs = pc + u;       // this tile's unit index: buffer gs & 1
                    const uint32_t scol = bufcol + kKeys * (gs & 1);
                    const uint64_t kd = desc_sw128(smem_u32(sK + ks * C::SLOT_BYTES + t * C::TILE_BYTES), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ad = qd + (uint64_t)((((kk >> 2) * C::Q_BOX) + (kk & 3) * 32) >> 4);
                        const uint64_t bd = kd + (uint64_t)((((kk >> 2) * C::KV_BOX) + (kk & 3) * 32) >> 4);
                        if (kk == 0) mma_f16c<0>(scol, ad, bd, id_s);
                        else mma_f16c<1>(scol, ad, bd, id_s);
                    }
                    mma_commit(smem_u32(&B.s_full[t][gs & 1]));
                    mma_commit_if(smem_u32(&B.q_empty), u == nu - 1);
                    // the key slot is free once both tiles' score products of this unit are
                    // done; a unit the other tile does not attend is released for it too
                    mma_commit(smem_u32(&B.k_empty[ks]));
                    mma_commit_if(smem_u32(&B.k_empty[ks]), u >= nu_other);
                    return true;
                };
                // O += P V of unit u (f16 P from tensor memory, f16 V: the softmax converted the
                // tile's values in the slot before it signalled P, so p_full covers both)
                auto issue_pv = [&](int u) -> bool {
                    if (u == 0 && !wait_bar(smem_u32(&B.o_empty[t]), (tn & 1) ^ 1, abort_flag, true)) return false;
                    const uint32_t gp = pc + u;
                    if (!wait_bar(smem_u32(&B.p_full[t][gp & 1]), (gp >> 1) & 1, abort_flag, true)) return false;
                    tc_fence_after();
                    const int vs = (int)((item0 + u) % NV);
                    const uint32_t pcol = bufcol + kKeys * (gp & 1);
                    const uint64_t vd =
                        desc_sw128(smem_u32(sV + vs * C::SLOT_BYTES + t * C::TILE_BYTES), C::KV_BOX, 1024);
                    // k-step kk: keys 16 kk .. 16 kk + 15 (P columns 8 kk .., value rows 16 kk ..)
                    mma_f16_ts(ocol, pcol, vd, id_o, u > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < 4; ++kk)
                        mma_f16_tsc<1>(ocol, pcol + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), id_o);
                    mma_commit(smem_u32(&B.pv_done[t]));
                    // the value slot likewise, after both tiles' P V products
                    mma_commit(smem_u32(&B.v_empty[vs]));
                    mma_commit_if(smem_u32(&B.v_empty[vs]), u >= nu_other);
                    return true;
                };
                if (!issue_s(0)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                for (int u = 0; u < nu; ++u) {
                    if (u + 1 < nu && !issue_s(u + 1)) { ok = false; break; }
                    if (!issue_pv(u)) { ok = false; break; }
                }
                if (!ok) { give_up(SITE_FULL_WAIT); break; }
                mma_commit(smem_u32(&B.o_full[t]));
                pc += nu;
                ++tn;
            }
            // every MMA issued here completes before tensor memory is released
            mma_commit(smem_u32(&B.drain[t]));
            if (!wait_bar(smem_u32(&B.drain[t]), 0, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else {
        // ===================== softmax + epilogue (thread = query row of tile t) =====================
        const int t = (warp - 2) >> 2;
        const int row = ((warp & 3) << 5) + lane;                 // tensor-memory lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) << 5) << 16) + t * kTmemTile;
        const bool fused = a.fused != 0;
        const float c2 = a.scale_log2;
        uint32_t sn = 0, on = 0, item = 0;
        bool ok = true;
        PairRing<Bars> ring;
        while (ok) {
            const int task = ring.next(B, abort_flag, lane, true);
            if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
            if (task < 0) break;
            const PairTask pt = pair_task(a, task);
            const uint32_t item0 = item;                          // value slot of unit u: (item0 + u) % NV
            item += pt.n_units;
            const PairBlock k = pt.t[t];
            const int nu = k.nu;
            if (k.rows == 0) continue;                            // this tile holds no block in the task
            const bool valid = row < k.rows;
            const int grow = k.row0 + row;                        // row in the (request, KV head) group
            const int i = valid ? grow / g : 0;
            const int h = k.kv * g + (valid ? grow % g : 0);
            // last key this row sees in the split (-1: none)
            const int limit = valid ? min(k.kend - 1, k.r.seq_len - k.r.q_len + i) : -1;
            const size_t orow = (size_t)(k.r.q_start + i) * a.num_q_heads + h;
            const size_t st = (size_t)k.r.state_base + ((size_t)i * a.num_q_heads + h) * k.r.n_splits + k.split;
            const bool direct = fused && k.r.n_splits == 1;      // write the final output
            float m = -INFINITY, l = 0.f;
            for (int u = 0; u < nu; ++u) {
                const uint32_t gi = sn;       // this tile's unit index: S/P buffer gi & 1
                const int b2 = (int)(gi & 1);
                if (!warp_wait(smem_u32(&B.s_full[t][b2]), (gi >> 1) & 1, abort_flag, lane)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                tc_fence_after();
                uint32_t sr[64];
                SKV_LD32(lane_addr + kColS + kKeys * b2, sr);
                SKV_LD32(lane_addr + kColS + kKeys * b2 + 32, (sr + 32));
                tc_wait_ld();
                ++sn;
                const int key0 = k.kb + u * kKeys;
                // no key of the unit is masked for any row of this warp; warp-uniform, since
                // the P stores below are warp-collective tensor-memory instructions
                const bool unmasked = __all_sync(0xffffffffu, key0 + kKeys - 1 <= limit);
                // row max of the raw scores (the scale, > 0 on this path, is applied after)
                const float mxr = unmasked ? row_max64<false>(sr, 64) : row_max64<true>(sr, limit - key0 + 1);
                const float mx = mxr * c2;
                // lazy rescale: a row whose max grew by more than 2^8 rescales its O and l, the
                // whole warp when any of its rows needs it, once this tile's P V product of the
                // previous unit has updated O (S of this unit is complete, so P V of unit gi - 2
                // is too: the barrier is at most one phase behind)
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
                    if (gi >= 1) {
                        if (!warp_wait(smem_u32(&B.pv_done[t]), (gi - 1) & 1, abort_flag, lane)) {
                            give_up(SITE_EMPTY_WAIT); ok = false; break;
                        }
                        tc_fence_after();
                    }
                    l *= scale_o;
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        SKV_LD32(lane_addr + c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * scale_o);
                        SKV_ST32(lane_addr + c, o);
                    }
                }
                // P over this unit's S; the buffer's previous P was read by P V of unit gi - 2,
                // issued before S of this unit and so already done
                const float base = (m == -INFINITY) ? 0.f : m;
                const uint32_t pcol = lane_addr + kColS + kKeys * b2;
                l += unmasked ? write_p16<false>(sr, c2, base, key0, limit, pcol)
                              : write_p16<true>(sr, c2, base, key0, limit, pcol);
                // The tile's values of the unit to f16, in place (the 16-byte chunks keep their
                // swizzled positions), once they have landed; the slot is not reloaded before
                // this tile's P V product has read it.  Slots past the block's last key (the
                // unused tail of the last page) may hold anything: their weight is 0, but 0 * NaN
                // is not, so they become zeros.  Bf16 magnitudes of 2^16 and above overflow f16
                // to infinity, which the epilogue reports.
                {
                    const uint32_t vi = item0 + u;
                    if (!warp_wait(smem_u32(&B.v_full[vi % NV]), (vi / NV) & 1, abort_flag, lane)) {
                        give_up(SITE_FULL_WAIT); ok = false; break;
                    }
                    unsigned char* vst = sV + (vi % NV) * C::SLOT_BYTES + t * C::TILE_BYTES;
                    const int r0 = k.kend - key0;          // first key row to clear (>= 64: none)
#pragma unroll
                    for (int i = 0; i < C::TILE_BYTES / 16 / kRows; ++i) {
                        const int c = row + i * kRows;      // 16-byte chunk; its key row within the box
                        uint4* ptr = (uint4*)(vst + c * 16);
                        uint4 w = *ptr;
                        if (((c * 16) % C::KV_BOX) / 128 >= r0) w = make_uint4(0u, 0u, 0u, 0u);
                        *ptr = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z),
                                          bf16x2_to_f16x2(w.w));
                    }
                }
                tc_wait_st();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.p_full[t][b2]));
            }
            if (!ok) break;
            if (nu > 0) {
                // ---- epilogue: O / l ----
                if (!warp_wait(smem_u32(&B.o_full[t]), on & 1, abort_flag, lane)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++on;
                tc_fence_after();
            }
            const bool empty_row = !(l > 0.f);
            const float inv = empty_row ? 0.f : 1.f / l;
            const float lse = empty_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
            bool nonfinite = false;
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                if (nu > 0) {
                    SKV_LD32(lane_addr + c, o);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0u;
                }
                if (!valid) continue;
#pragma unroll
                for (int j = 0; j < 32; ++j) nonfinite |= (o[j] & 0x7F800000u) == 0x7F800000u;
                if (direct) {
                    if (a.out_bf16) {
                        uint4* op = (uint4*)((__nv_bfloat16*)a.out + orow * D + c);
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(o[j + 2 * e]) * inv,
                                                                          __uint_as_float(o[j + 2 * e + 1]) * inv);
                                w[e] = *reinterpret_cast<uint32_t*>(&p2);
                            }
                            op[j / 8] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *(float4*)((float*)a.out + orow * D + c + j) =
                                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        store_part4(a.o_part, a.part_bf16, st * D + c + j,
                                    make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                                __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv));
                }
            }
            if (valid) {
                if (direct) {
                    if (a.lse_out) a.lse_out[orow] = lse;
                } else {
                    __stcg(a.lse_part + st, lse);
                }
                // a value outside the f16 range (or a non-finite input) made the row non-finite
                if (nonfinite) set_error(a.err, ERR_DEVICE_CHECK | SITE_VALUE_RANGE);
            }
            if (nu > 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.o_empty[t]));
            }
            __syncwarp();
            if (lane == 0) trace_end(a.trace, task);
            if (fused && k.r.n_splits > 1) {
                // this warp's 32 row states are written (the warp barrier orders the lanes'
                // stores before lane 0's fence): the warp counts in for the reduction, which
                // waits for 4 counts per block
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(&a.counters[k.b], 1);
                }
            }
        }
    }

    // leave together: tensor memory is released once every MMA has completed
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(&a.ctrl->pair_exit, 1);
        if (prev == (int)gridDim.x - 1) {
            atomicExch(&a.ctrl->pair_head, 0);
            atomicExch(&a.ctrl->pair_exit, 0);
        }
    }
}

// ---------------------------------------------------------------- host
// bf16 tiled map with 128-byte swizzle over `rank` dims (innermost first)
cudaError_t pair_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_pair_d(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
    const int g = a.group;
    // Q as [total_q][Hq][D]: one box = 128 / g tokens x the g heads of a KV head x 64 columns
    cuuint64_t qd[3] = {(cuuint64_t)D, (cuuint64_t)a.num_q_heads, (cuuint64_t)total_q};
    cuuint64_t qs[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_q_heads * D * 2};
    cuuint32_t qb[3] = {64, (cuuint32_t)g, (cuuint32_t)(kRows / g)};
    // K, V as [num_pages * Hkv * P][D]: one box = 64 keys x 64 columns
    const long long kvrows = (long long)num_pages_total * a.num_kv_heads * a.page_size;
    cuuint64_t kd[2] = {(cuuint64_t)D, (cuuint64_t)kvrows};
    cuuint64_t ks[1] = {(cuuint64_t)D * 2};
    cuuint32_t kb[2] = {64, (cuuint32_t)kKeys};
    CUtensorMap mq, mk, mv;
    cudaError_t e = pair_map(&mq, a.q, 3, qd, qs, qb);
    if (e != cudaSuccess) return e;
    if ((e = pair_map(&mk, a.k_cache, 2, kd, ks, kb)) != cudaSuccess) return e;
    if ((e = pair_map(&mv, a.v_cache, 2, kd, ks, kb)) != cudaSuccess) return e;
    constexpr size_t smem = pair_smem_bytes<D>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&]() {
        attr_err = cudaFuncSetAttribute(pair_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int grid = std::min(a.max_ctas > 0 ? std::min(sms, a.max_ctas) : sms, a.num_tasks);
    {
        ProfileScope ps(SPLITKV_KERNEL_PAIR, s);
        pair_tc_kernel<D><<<grid, kThreads, smem, s>>>(mq, mk, mv, a);
    }
    return cudaGetLastError();
}

}  // namespace

bool pair_tc_supports(int bf16, int head_dim, int page_size, int group) {
    return bf16 && (head_dim == 64 || head_dim == 128) && (page_size == 64 || page_size == 128) && group >= 1 &&
           group <= kRows && (kRows % group) == 0;
}

cudaError_t launch_pair_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    if ((((uintptr_t)a.q) & 15) || (((uintptr_t)a.k_cache) & 15) || (((uintptr_t)a.v_cache) & 15))
        return cudaErrorMisalignedAddress;
    if ((long long)num_pages_total * a.num_kv_heads * a.page_size >= (1LL << 31) || total_q >= (1LL << 31))
        return cudaErrorInvalidValue;
    if (a.head_dim_qk == 128) return launch_pair_d<128>(a, total_q, num_pages_total, s);
    if (a.head_dim_qk == 64) return launch_pair_d<64>(a, total_q, num_pages_total, s);
    return cudaErrorNotSupported;
}

}  // namespace skv
