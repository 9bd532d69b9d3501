// Causal chunk tiles of GQA attention on sm_103a with tcgen05 tensor cores.
//
// What it computes (LiquidCP Section 3 Eq. 1 and Section 5: the causal
// chunked-prefill requests of a mixed batch; Helix Parallelism, "Attention-
// Phase Configuration" step 2 for the split state): for up to 256 query rows
// of one (request, KV head) -- row = token * g + head-in-group -- over one
// split of the request's history, each row's partial state (output
// normalised over the keys it sees in the split, natural-log LSE).  Token i
// of a request with q_len appended tokens sees keys [0, seq_len - q_len + i].
//
// How: the contraction is dense (every row of the tile meets every key), so
// it runs on the fifth-generation tensor cores, two 128-row tiles per CTA
// sharing each K/V unit.  Per 64-key unit the producer TMA-loads K and V
// (128-byte swizzle) into a ring of stages; one thread issues, per tile,
// S = Q K^T (M=128, N=64) into a tensor-memory buffer; the tile's four
// softmax warps (one thread per row) read S back, apply the causal mask and
// the online softmax (base 2, lazy rescaling of O when a row's running max
// grows by more than 2^8), and write P over S in tensor memory as f16 (11
// significant bits: a bf16 P, 8 bits, misses the output bound on rows that see
// few keys); the MMA thread then accumulates O += P V (A = P from tensor
// memory, B = V as an MN-major shared-memory operand; M=128, N=D).  The f16
// product needs V in f16 too (one type per product): a streaming pre-pass
// writes an f16 copy of the chunk requests' value pages once per launch (the
// row-block tasks of a (request, KV head) all read the same pages), and the
// producer loads V from that copy.  Per tile, tensor memory holds O and
// two S/P buffers; each tile's MMA thread issues S of unit u + 1 into the
// other buffer, then P V of unit u.  Products run in issue order, so S of unit
// u + 2 overwrites P of unit u only after P V of unit u has read it, and the
// softmax, which has seen S of unit u complete, knows that P V of unit u - 2
// (the buffer's last reader) is done: it writes P without waiting on the
// products.  The two tiles' softmax work interleaves on every scheduler.
// MMA issue runs at the pace of the tensor pipe (its queue is short), so each
// tile has its own MMA thread, which waits only on its softmax and copy
// events, never on its own products.  A tcgen05 commit takes a queue slot like
// an MMA, so a tile makes two per unit: S done (for its softmax) and its own
// release of the unit's stage, which the producer waits for from each tile that
// attended the unit and which also tells the softmax that P V has updated O.
//
// Warp roles: warp 0 TMA producer and task claimer, warp 1 tile 0's MMA
// thread and the tensor-memory owner, warps 2..5 softmax/epilogue of tile 0,
// warps 6..9 of tile 1, warp 10 tile 1's MMA thread.  Tasks come from the workspace queue in plan order
// (longest first) through a small ring, so every role follows the same
// sequence.  In fused mode each softmax warp of a split request's task counts
// itself in once its rows are written, for the request's reduction, which
// the decode engine's reduction phase performs.  Every wait is bounded
// (%globaltimer); on expiry the CTA records the error word and drains its own
// copies and MMAs before leaving.
#include "splitkv.h"
#include <cuda_fp16.h>

#include "tc_common.cuh"
#include "partial_io.cuh"
#include "trace.cuh"

namespace skv {
namespace {

constexpr int kRows = 128;                          // query rows per tile (tensor-memory lanes)
constexpr int kTiles = 2;                           // tiles per task (256 rows)
constexpr int kKeys = 64;                           // keys per unit
constexpr int kTR = 4;                              // task ring slots
constexpr int kSoftWarps = 4 * kTiles;
constexpr int kTaskConsumers = kTiles + kSoftWarps; // per tile an MMA thread and 4 softmax warps
constexpr int kThreads = (1 + kTiles + kSoftWarps) * 32;
constexpr int kIssuerWarp1 = 2 + kSoftWarps;        // tile 1's MMA warp (tile 0's is warp 1)
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr size_t kSmemLimit = 232448;
constexpr int kTmemTile = 256;                      // tensor-memory columns per tile: O | S/P | S/P
constexpr int kColS = 128;                          // S/P buffer b at kColS + 64 b: 64 fp32 columns of S;
                                                    // P over its first 32 columns as f16 pairs (key 2k in
                                                    // the low half of column k)
constexpr int kTmemCols = kTiles * kTmemTile;

template <int D>
struct ChunkCfg {
    static constexpr int BOXES = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int Q_BOX = kRows * 128;            // 128 rows x 128 B
    static constexpr int KV_BOX = kKeys * 128;           // 64 keys x 128 B
    static constexpr int Q_TILE = BOXES * Q_BOX;
    static constexpr int Q_BYTES = kTiles * Q_TILE;
    static constexpr int TILE_BYTES = BOXES * KV_BOX;    // K (or V) of one unit
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int NS_FIT = (int)((kSmemLimit - 1024 - Q_BYTES - 1024) / STAGE_BYTES);
    static constexpr int NS = NS_FIT < 8 ? NS_FIT : 8;
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(D <= kColS && kColS + 2 * kKeys <= kTmemTile, "tensor memory budget");
    static_assert(NS >= 2, "stage ring");
};

template <int NS>
struct ChunkBars {
    unsigned long long task_full[kTR], task_empty[kTR];
    int task_slot[kTR];
    unsigned long long stage_full[NS];
    unsigned long long stage_empty[kTiles][NS];   // per tile: its P V product of the stage's unit is done
    unsigned long long q_full, q_empty;
    unsigned long long s_full[kTiles][2], p_full[kTiles][2];   // [tile][S/P buffer]
    unsigned long long o_full[kTiles], o_empty[kTiles];
    unsigned long long drain[kTiles];
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
constexpr size_t chunk_smem_bytes() {
    using C = ChunkCfg<D>;
    return 1024 + C::Q_BYTES + (size_t)C::NS * C::STAGE_BYTES + sizeof(ChunkBars<C::NS>);
}

// per-task facts every role derives from the descriptor
struct ChunkTask {
    int b, kv, row0, split, kb, kend, n_units, empty;
    int rows[kTiles];     // valid rows of each tile
    int nu[kTiles];       // units each tile attends (0: none)
    ReqDesc r;
};

__device__ __forceinline__ ChunkTask chunk_task(const KernelArgs& a, int task) {
    ChunkTask ct;
    const TaskDesc t = a.tasks[task];
    ct.r = a.reqs[t.b];
    ct.b = t.b;
    ct.kv = t.kv_head;
    ct.row0 = t.row_begin;
    ct.split = t.split;
    ct.kb = t.key_begin;
    ct.kend = ct.kb;
    ct.n_units = 0;
#pragma unroll
    for (int tt = 0; tt < kTiles; ++tt) {
        const int r0 = t.row_begin + tt * kRows;
        ct.rows[tt] = max(0, min(kRows, t.row_end - r0));
        ct.nu[tt] = 0;
        if (ct.rows[tt] > 0) {
            // keys the tile's last row may see: the split's range cut by its causal limit
            const int i_last = (r0 + ct.rows[tt] - 1) / a.group;
            const int ke = min(t.key_end, ct.r.seq_len - ct.r.q_len + i_last + 1);
            if (ke > ct.kb) {
                ct.nu[tt] = (ke - ct.kb + kKeys - 1) / kKeys;
                ct.kend = max(ct.kend, ke);
                ct.n_units = max(ct.n_units, ct.nu[tt]);
            }
        }
    }
    ct.empty = ct.n_units == 0;
    return ct;
}

template <int NS>
struct Ring {
    uint32_t n = 0;
    // next task id (-1: no more) for a consumer role; -2 when the wait gave up
    __device__ __forceinline__ int next(ChunkBars<NS>& B, volatile int* abort_flag, int lane, bool whole_warp) {
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

// The f16 copy of the chunk requests' value pages: slot k holds page vh_pages[k].j of
// request vh_pages[k].b (all KV heads, the cache's layout).  Values are exact in f16 for
// bf16 magnitudes in [2^-14, 65504] (within 2^-25 below); the slots past a request's last
// key are zeros (their weight is 0, but 0 * NaN is not); finite magnitudes above the
// f16 range are reported (DEVICE_CHECK, value range), page ids outside the pool too.
// A CTA takes one slot at a time: the slot's descriptors are read once, and each thread
// keeps four 16-byte loads in flight (a copy at the pace of HBM, not of a chain of
// dependent descriptor reads per 16 bytes).
__global__ void __launch_bounds__(256) chunk_value_convert_kernel(KernelArgs a) {
    constexpr int U = 4;
    const int P = a.page_size;
    const int c8 = a.head_dim_v / 8;                                   // 16-byte chunks per row
    const int per_page = a.num_kv_heads * P * c8;
    const uint4* src = (const uint4*)a.v_cache;
    uint4* dst = (uint4*)a.v_half;
    uint32_t vmax = 0;   // largest used |value| per half, as bf16 magnitude bits
    bool bad_page = false;
    for (int slot = blockIdx.x; slot < a.num_vh_pages; slot += gridDim.x) {
        const VhPage vp = a.vh_pages[slot];
        const ReqDesc r = a.reqs[vp.b];
        const int rows = r.seq_len - vp.j * P;                         // keys of the page in use
        const int phys = a.page_table[r.page_row + vp.j];
        const bool ok = phys >= 0 && phys < a.num_pages;
        if (!ok && rows > 0) bad_page = true;
        const uint4* sp = src + (size_t)(ok ? phys : 0) * per_page;
        uint4* dp = dst + (size_t)slot * per_page;
        for (int i0 = threadIdx.x; i0 < per_page; i0 += U * blockDim.x) {
            uint4 w[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int idx = i0 + k * blockDim.x;
                w[k] = make_uint4(0u, 0u, 0u, 0u);
                if (idx < per_page && ok && (idx / c8) % P < rows) w[k] = __ldcs(sp + idx);   // read once
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int idx = i0 + k * blockDim.x;
                if (idx >= per_page) continue;
                vmax = __vmaxu2(vmax, __vmaxu2(__vmaxu2(w[k].x & 0x7FFF7FFFu, w[k].y & 0x7FFF7FFFu),
                                               __vmaxu2(w[k].z & 0x7FFF7FFFu, w[k].w & 0x7FFF7FFFu)));
                dp[idx] = make_uint4(bf16x2_to_f16x2(w[k].x), bf16x2_to_f16x2(w[k].y), bf16x2_to_f16x2(w[k].z),
                                     bf16x2_to_f16x2(w[k].w));
            }
        }
    }
    // finite bf16 magnitudes from 2^16 up (0x4780 .. 0x7F7F) overflow f16
    const uint32_t lo = vmax & 0xFFFFu, hi = vmax >> 16;
    if ((lo >= 0x4780u && lo < 0x7F80u) || (hi >= 0x4780u && hi < 0x7F80u))
        set_error(a.err, ERR_DEVICE_CHECK | SITE_VALUE_RANGE);
    if (bad_page) set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, KernelArgs a) {
    using C = ChunkCfg<D>;
    constexpr int NS = C::NS;
    static_assert(chunk_smem_bytes<D>() <= kSmemLimit, "shared memory budget");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char* sQ = smem;                              // tile t at t * Q_TILE
    unsigned char* sStage = sQ + C::Q_BYTES;               // stage: K boxes, then V boxes
    ChunkBars<NS>& B = *(ChunkBars<NS>*)(sStage + NS * C::STAGE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTR; ++s) {
            mbar_init(smem_u32(&B.task_full[s]), 1);
            mbar_init(smem_u32(&B.task_empty[s]), kTaskConsumers);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&B.stage_full[s]), 1);
            for (int t = 0; t < kTiles; ++t) mbar_init(smem_u32(&B.stage_empty[t][s]), 1);
        }
        mbar_init(smem_u32(&B.q_full), 1);
        mbar_init(smem_u32(&B.q_empty), kTiles);            // one per tile's MMA thread
        for (int t = 0; t < kTiles; ++t) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&B.s_full[t][b]), 1);
                mbar_init(smem_u32(&B.p_full[t][b]), 4);
            }
            mbar_init(smem_u32(&B.o_full[t]), 1);
            mbar_init(smem_u32(&B.o_empty[t]), 4);
        }
        for (int t = 0; t < kTiles; ++t) mbar_init(smem_u32(&B.drain[t]), 1);
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

    if (warp == 0) {
        // ===================== producer and task claimer (lane 0) =====================
        if (lane == 0) {
            uint32_t item = 0, qn = 0, claimed = 0;
            uint32_t had_tma = 0, last_par = 0;   // per-stage bits
            // per (tile, stage), bit 8 t + s: the stage's unit is one the tile attends (its
            // release is that tile's commit), that commit's phase parity, the next one's
            uint32_t occ = 0, opar = 0, nph = 0;
            bool q_tma = false;
            uint32_t q_par = 0;
            bool ok = a.inject != 1;   // (test hook: publish nothing)
            while (ok) {
                const int slot = (int)(claimed % kTR);
                if (!wait_bar(smem_u32(&B.task_empty[slot]), ((claimed / kTR) & 1) ^ 1, abort_flag, true)) {
                    give_up(SITE_EMPTY_WAIT); ok = false; break;
                }
                int task = atomicAdd(&a.ctrl->chunk_head, 1);
                if (task >= a.num_tasks) task = -1;
                ((volatile int*)B.task_slot)[slot] = task;
                mbar_arrive(smem_u32(&B.task_full[slot]));
                ++claimed;
                if (task < 0) break;
                trace_start(a.trace, task, SPLITKV_TRACE_CHUNK);
                const ChunkTask ct = chunk_task(a, task);
                if (ct.empty) {
                    trace_end(a.trace, task);
                    continue;
                }
                // both tiles' query rows: tile t holds tokens (row0 + 128 t) / g .. + 128 / g of
                // the g heads of the KV head (rows past the request read other tokens or the
                // zero fill past the tensor; they are never written back)
                if (!wait_bar(smem_u32(&B.q_empty), (qn & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                mbar_expect_tx(smem_u32(&B.q_full), C::Q_BYTES);
                for (int t = 0; t < kTiles; ++t) {
                    const int tok0 = ct.r.q_start + (ct.row0 + t * kRows) / g;
                    for (int j = 0; j < C::BOXES; ++j)
                        tma_3d(smem_u32(sQ + t * C::Q_TILE + j * C::Q_BOX), &tmap_q, 64 * j, ct.kv * g, tok0,
                               smem_u32(&B.q_full));
                }
                q_tma = true;
                q_par = qn & 1;
                ++qn;
                for (int u = 0; u < ct.n_units; ++u) {
                    const int s = (int)(item % NS);
                    const uint32_t round = item / NS;
                    // the stage is free once each tile that attended its previous unit is done with it
                    bool freed = true;
                    for (int t = 0; t < kTiles && freed; ++t) {
                        const uint32_t bit = 1u << (8 * t + s);
                        if (occ & bit) freed = wait_bar(smem_u32(&B.stage_empty[t][s]), (opar & bit) ? 1u : 0u, abort_flag, true);
                    }
                    if (!freed) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                    for (int t = 0; t < kTiles; ++t) {
                        const uint32_t bit = 1u << (8 * t + s);
                        if (u < ct.nu[t]) {
                            occ |= bit;
                            opar = (opar & ~bit) | (nph & bit);
                            nph ^= bit;
                        } else {
                            occ &= ~bit;
                        }
                    }
                    const int key0 = ct.kb + u * kKeys;
                    const int phys = a.page_table[ct.r.page_row + key0 / a.page_size];
                    const uint32_t full = smem_u32(&B.stage_full[s]);
                    last_par = (last_par & ~(1u << s)) | ((round & 1u) << s);
                    if (phys < 0 || phys >= a.num_pages) {
                        set_error(a.err, ERR_DEVICE_CHECK | SITE_PAGE_RANGE);
                        had_tma &= ~(1u << s);
                        mbar_arrive(full);
                    } else {
                        had_tma |= 1u << s;
                        mbar_expect_tx(full, C::STAGE_BYTES);
                        const int y = (phys * a.num_kv_heads + ct.kv) * a.page_size + key0 % a.page_size;
                        // values from the f16 copy: slot vh_base + page index of the request
                        const int yv = ((ct.r.vh_base + key0 / a.page_size) * a.num_kv_heads + ct.kv) * a.page_size +
                                       key0 % a.page_size;
                        unsigned char* st = sStage + s * C::STAGE_BYTES;
                        for (int j = 0; j < C::BOXES; ++j) {
                            tma_2d(smem_u32(st + j * C::KV_BOX), &tmap_k, 64 * j, y, full);
                            tma_2d(smem_u32(st + C::TILE_BYTES + j * C::KV_BOX), &tmap_v, 64 * j, yv, full);
                        }
                    }
                    ++item;
                }
            }
            // no copy may still be landing when the CTA leaves
            for (int s = 0; s < NS; ++s)
                if (((had_tma >> s) & 1u) && !wait_bar(smem_u32(&B.stage_full[s]), (last_par >> s) & 1u, abort_flag, false))
                    set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
            if (q_tma && !wait_bar(smem_u32(&B.q_full), q_par, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kIssuerWarp1) {
        // ===================== MMA issuer of tile t (lane 0) =====================
        // Each tile has its own MMA thread, so the two tiles' products interleave on the
        // tensor pipe (MMA issue runs at the pace of the pipe: its queue is short).  Fixed
        // schedule per task: S of unit 0; then for each unit u, S of unit u + 1 (once the
        // stage is loaded) into the other S/P buffer, whose last reader, P V of unit u - 1,
        // was issued before it, then the P V product of unit u (once its probabilities
        // are in).  The thread waits only on its softmax and the copies, never on its own
        // products.  Waits are bounded hardware waits; descriptors are precomputed, the
        // k-steps unrolled to constant offsets.
        const int t = warp == 1 ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(kRows, kKeys, 0);
            constexpr uint32_t id_o = idesc_f16(kRows, D, 1);     // P and V both f16
            const uint64_t qd = desc_sw128(smem_u32(sQ + t * C::Q_TILE), 16, 1024);
            const uint32_t bufcol = tmem + t * kTmemTile + kColS;   // S/P buffer b: bufcol + kKeys b
            const uint32_t ocol = tmem + t * kTmemTile;
            uint32_t item = 0, qn = 0;
            uint32_t pc = 0;      // units this tile attended so far (S, P phases)
            uint32_t tn = 0;      // tasks this tile finished (O phases)
            bool ok = true;
            Ring<NS> ring;
            while (ok) {
                const int task = ring.next(B, abort_flag, 0, false);
                if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
                if (task < 0) break;
                const ChunkTask ct = chunk_task(a, task);
                if (ct.empty) continue;
                const uint32_t item0 = item;      // stage of unit u: (item0 + u) % NS
                item += ct.n_units;
                const int nu = t ? ct.nu[1] : ct.nu[0];
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
                    const int stage = (int)(gi % NS);
                    if (!wait_bar(smem_u32(&B.stage_full[stage]), (gi / NS) & 1, abort_flag, true)) return false;
                    tc_fence_after();
                    const uint32_t gs = pc + u;       // this tile's unit index: buffer gs & 1
                    const uint32_t scol = bufcol + kKeys * (gs & 1);
                    const uint64_t kd = desc_sw128(smem_u32(sStage + stage * C::STAGE_BYTES), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ad = qd + (uint64_t)((((kk >> 2) * C::Q_BOX) + (kk & 3) * 32) >> 4);
                        const uint64_t bd = kd + (uint64_t)((((kk >> 2) * C::KV_BOX) + (kk & 3) * 32) >> 4);
                        if (kk == 0) mma_f16c<0>(scol, ad, bd, id_s);
                        else mma_f16c<1>(scol, ad, bd, id_s);
                    }
                    mma_commit(smem_u32(&B.s_full[t][gs & 1]));
                    return true;
                };
                // O += P V of unit u (P from tensor memory)
                auto issue_pv = [&](int u) -> bool {
                    if (u == 0 && !wait_bar(smem_u32(&B.o_empty[t]), (tn & 1) ^ 1, abort_flag, true)) return false;
                    const uint32_t gp = pc + u;
                    if (!wait_bar(smem_u32(&B.p_full[t][gp & 1]), (gp >> 1) & 1, abort_flag, true)) return false;
                    tc_fence_after();
                    const uint32_t pcol = bufcol + kKeys * (gp & 1);
                    const int stage = (int)((item0 + u) % NS);
                    const uint64_t vd =
                        desc_sw128(smem_u32(sStage + stage * C::STAGE_BYTES + C::TILE_BYTES), C::KV_BOX, 1024);
                    // four k-steps of 16 keys: P columns 8 kk .. 8 kk + 7 (two keys per column)
                    mma_f16_ts(ocol, pcol, vd, id_o, u > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < 4; ++kk)
                        mma_f16_tsc<1>(ocol, pcol + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), id_o);
                    // this tile is done with the stage: one commit, whether or not the other
                    // tile attends the unit (every commit takes a slot in the tensor pipe's short
                    // queue, which sets this kernel's pace, so P V has no barrier of its own)
                    mma_commit(smem_u32(&B.stage_empty[t][stage]));
                    return true;
                };
                if (!issue_s(0)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                for (int u = 0; u + 1 < nu; ++u) {
                    if (!issue_s(u + 1) || !issue_pv(u)) { ok = false; break; }
                }
                // every S of the task is issued: the query buffer is free once they are done
                // (one commit per task, not a predicated one per unit)
                if (ok) mma_commit(smem_u32(&B.q_empty));
                if (ok && !issue_pv(nu - 1)) ok = false;
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
        uint32_t sn = 0, on = 0, item = 0;   // item: ring position of the task's first unit
        uint32_t ph = 0;                     // per stage: phase parity of this tile's next release
        bool ok = true;
        Ring<NS> ring;
        while (ok) {
            const int task = ring.next(B, abort_flag, lane, true);
            if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
            if (task < 0) break;
            const ChunkTask ct = chunk_task(a, task);
            const int trows = t ? ct.rows[1] : ct.rows[0];       // (selects keep ct in registers)
            const int nu = t ? ct.nu[1] : ct.nu[0];
            const uint32_t item0 = item;
            if (!ct.empty) item += ct.n_units;
            if (trows == 0) continue;                             // this tile holds no rows of the task
            const bool valid = row < trows;
            const int grow = ct.row0 + t * kRows + row;           // row in the (request, KV head) group
            const int i = valid ? grow / g : 0;
            const int h = ct.kv * g + (valid ? grow % g : 0);
            // last key this row sees in the split (-1: none)
            const int limit = valid ? min(ct.kend - 1, ct.r.seq_len - ct.r.q_len + i) : -1;
            const size_t orow = (size_t)(ct.r.q_start + i) * a.num_q_heads + h;
            const size_t st = (size_t)ct.r.state_base + ((size_t)i * a.num_q_heads + h) * ct.r.n_splits + ct.split;
            const bool direct = fused && ct.r.n_splits == 1;   // write the final output
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
                const int key0 = ct.kb + u * kKeys;
                // no key of the unit is masked for any row of this warp; warp-uniform, since
                // the P stores below are warp-collective tensor-memory instructions
                const bool unmasked = __all_sync(0xffffffffu, key0 + kKeys - 1 <= limit);
                // row max of the raw scores (the scale, > 0 on this path, is applied after)
                const float mxr = unmasked ? row_max64<false>(sr, 64) : row_max64<true>(sr, limit - key0 + 1);
                const float mx = mxr * c2;
                // lazy rescale: a row whose max grew by more than 2^8 rescales its O and l.
                // The tensor-memory loads and stores are warp-collective, so the whole warp
                // takes the branch when any of its rows needs it (scale 1 for the others),
                // once this tile's P V product of the previous unit has updated O, which the
                // release of that unit's stage shows (below).
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
                    if (u >= 1) {
                        // P V of unit u - 1 has updated O once this tile released that unit's
                        // stage (whose phase bit in ph has flipped once since); the release
                        // barrier moves on only with this tile's next release, which needs this
                        // softmax's next P: it is at most one phase behind
                        const int rs = (int)((item0 + u - 1) % NS);
                        if (!warp_wait(smem_u32(&B.stage_empty[t][rs]), ((ph >> rs) & 1u) ^ 1u, abort_flag, lane)) {
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
                tc_wait_st();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.p_full[t][b2]));
                // the release of this unit's stage will be this tile's next phase on it
                ph ^= 1u << ((item0 + u) % NS);
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
            }
            if (nu > 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.o_empty[t]));
            }
            __syncwarp();
            if (lane == 0) trace_end(a.trace, task);
            if (fused && ct.r.n_splits > 1) {
                // this warp's 32 row states are written (the warp barrier orders the lanes'
                // stores before lane 0's fence): the warp counts in for the reduction, which
                // waits for 4 counts per tile with rows
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(&a.counters[ct.b], 1);
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
        const int prev = atomicAdd(&a.ctrl->chunk_exit, 1);
        if (prev == (int)gridDim.x - 1) {
            atomicExch(&a.ctrl->chunk_head, 0);
            atomicExch(&a.ctrl->chunk_exit, 0);
        }
    }
}

// ---------------------------------------------------------------- host
// bf16 tiled map with 128-byte swizzle over `rank` dims (innermost first)
cudaError_t make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, dtype, rank, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_d(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
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
    cudaError_t e = make_map(&mq, a.q, 3, qd, qs, qb);
    if (e != cudaSuccess) return e;
    if ((e = make_map(&mk, a.k_cache, 2, kd, ks, kb)) != cudaSuccess) return e;
    // V: the f16 copy, [slot * Hkv * P][D]
    cuuint64_t vd[2] = {(cuuint64_t)D, (cuuint64_t)a.num_vh_pages * a.num_kv_heads * a.page_size};
    if ((e = make_map(&mv, a.v_half, 2, vd, ks, kb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != cudaSuccess) return e;
    constexpr size_t smem = chunk_smem_bytes<D>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&]() {
        attr_err = cudaFuncSetAttribute(chunk_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int grid = std::min(a.max_ctas > 0 ? std::min(sms, a.max_ctas) : sms, a.num_tasks);
    {
        ProfileScope ps(SPLITKV_KERNEL_CHUNK, s);
        chunk_tc_kernel<D><<<grid, kThreads, smem, s>>>(mq, mk, mv, a);
    }
    return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supports(int bf16, int head_dim, int page_size, int group) {
    return bf16 && (head_dim == 64 || head_dim == 128) && (page_size == 64 || page_size == 128) && group >= 1 &&
           group <= kRows && (kRows % group) == 0;
}

cudaError_t launch_chunk_value_convert(const KernelArgs& a, cudaStream_t s) {
    if (a.num_vh_pages <= 0) return cudaSuccess;
    if ((((uintptr_t)a.v_cache) & 15) || (((uintptr_t)a.v_half) & 15) || (a.head_dim_v % 8))
        return cudaErrorMisalignedAddress;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int blocks = std::min(sms * 8, a.num_vh_pages);   // one slot per CTA at a time
    {
        ProfileScope ps(SPLITKV_KERNEL_CHUNK_VCONV, s);
        chunk_value_convert_kernel<<<blocks, 256, 0, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    if (!a.v_half || a.num_vh_pages <= 0) return cudaErrorInvalidValue;
    if ((((uintptr_t)a.q) & 15) || (((uintptr_t)a.k_cache) & 15) || (((uintptr_t)a.v_half) & 15))
        return cudaErrorMisalignedAddress;
    if ((long long)num_pages_total * a.num_kv_heads * a.page_size >= (1LL << 31) || total_q >= (1LL << 31))
        return cudaErrorInvalidValue;
    if (a.head_dim_qk == 128) return launch_d<128>(a, total_q, num_pages_total, s);
    if (a.head_dim_qk == 64) return launch_d<64>(a, total_q, num_pages_total, s);
    return cudaErrorNotSupported;
}

}  // namespace skv
