// Causal chunk tiles of GQA attention on sm_103a with tcgen05 tensor cores.
//
// What it computes (LiquidCP Section 3 Eq. 1 and Section 5: the causal
// chunked-prefill requests of a mixed batch; Helix Parallelism, "Attention-
// Phase Configuration" step 2 for the split state): for a tile of 128 query
// rows of one (request, KV head) -- row = token * g + head-in-group -- over
// one split of the request's history, each row's partial state (output
// normalised over the keys it sees in the split, natural-log LSE).  Token i
// of a request with q_len appended tokens sees keys [0, seq_len - q_len + i].
//
// How: the contraction is dense (128 rows share every key), so it runs on
// the fifth-generation tensor cores.  Per 64-key unit the CTA TMA-loads K and
// V (128-byte swizzle) into a ring of stages, one thread issues
// S = Q K^T (M=128, N=64) into tensor memory, the softmax threads (one per
// row) read S back, apply the causal mask and the online softmax (base 2,
// lazy rescaling of O when a row's running max grows by more than 2^8), and
// store P as a bf16 high part plus a bf16 residual, two K-major tiles; the
// MMA thread then accumulates O += P_hi V + P_lo V (M=128, N=D, V as an
// MN-major operand) into tensor memory.  Score and probability tiles are
// double buffered and the MMA thread polls both queues, so the scores of the
// next unit are computed while this unit's softmax runs.
//
// Warp roles: warp 0 TMA producer and task claimer, warp 1 MMA issuer (one
// thread) and tensor-memory owner, warps 2..5 softmax and epilogue.  Tasks
// come from the workspace queue in plan order (longest first) through a
// small ring, so every role follows the same sequence.  In fused mode a task
// of a split request counts itself in for the request's reduction, which the
// decode engine's reduction phase performs.  Every wait is bounded
// (%globaltimer); on expiry the CTA records the error word and drains its own
// copies and MMAs before leaving.
#include "tc_common.cuh"

namespace skv {
namespace {

constexpr int kRows = 128;                          // query rows per tile (tensor-memory lanes)
constexpr int kKeys = 64;                           // keys per unit
constexpr int kTR = 4;                              // task ring slots
constexpr int kTaskConsumers = 5;                   // MMA thread + 4 softmax warps
constexpr int kThreads = 6 * 32;
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr size_t kSmemLimit = 232448;

template <int D>
struct ChunkCfg {
    static constexpr int BOXES = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int Q_BOX = kRows * 128;            // 128 rows x 128 B
    static constexpr int KV_BOX = kKeys * 128;           // 64 keys x 128 B
    static constexpr int Q_BYTES = BOXES * Q_BOX;
    static constexpr int TILE_BYTES = BOXES * KV_BOX;    // K (or V) of one unit
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int P_TILE = kRows * 128;           // 128 rows x 64 keys bf16
    static constexpr int P_BYTES = 2 * P_TILE;           // high part + residual
    static constexpr int NS_FIT = (int)((kSmemLimit - 1024 - Q_BYTES - 2 * P_BYTES - 512) / STAGE_BYTES);
    static constexpr int NS = NS_FIT < 6 ? NS_FIT : 6;
    static constexpr int COL_O = 0, COL_S = D;           // tensor-memory columns: O, then two S buffers
    static constexpr int TMEM_COLS = 256;
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(COL_S + 2 * kKeys <= TMEM_COLS, "tensor memory budget");
    static_assert(NS >= 2, "stage ring");
};

template <int NS>
struct ChunkBars {
    unsigned long long task_full[kTR], task_empty[kTR];
    int task_slot[kTR];
    unsigned long long stage_full[NS], stage_empty[NS];
    unsigned long long q_full, q_empty;
    unsigned long long s_full[2], s_empty[2];
    unsigned long long p_full[2], p_empty[2];
    unsigned long long o_full, o_empty;
    unsigned long long drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
constexpr size_t chunk_smem_bytes() {
    using C = ChunkCfg<D>;
    return 1024 + C::Q_BYTES + (size_t)C::NS * C::STAGE_BYTES + 2 * C::P_BYTES + sizeof(ChunkBars<C::NS>);
}

// per-task facts every role derives from the descriptor
struct ChunkTask {
    int b, kv, row0, nrows, split, kb, kend, n_units, empty;
    ReqDesc r;
};

__device__ __forceinline__ ChunkTask chunk_task(const KernelArgs& a, int task) {
    ChunkTask ct;
    const TaskDesc t = a.tasks[task];
    ct.r = a.reqs[t.b];
    ct.b = t.b;
    ct.kv = t.kv_head;
    ct.row0 = t.row_begin;
    ct.nrows = t.row_end - t.row_begin;
    ct.split = t.split;
    ct.kb = t.key_begin;
    const int i_last = (t.row_end - 1) / a.group;
    // keys any row of the tile may see: the split's range cut by the last row's causal limit
    ct.kend = min(t.key_end, ct.r.seq_len - ct.r.q_len + i_last + 1);
    ct.empty = ct.kend <= ct.kb;
    ct.n_units = ct.empty ? 0 : (ct.kend - ct.kb + kKeys - 1) / kKeys;
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
        (void)mbar_try(smem_u32(&B.task_full[slot]), par, false);
        const int id = ((volatile int*)B.task_slot)[slot];
        if (whole_warp) __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&B.task_empty[slot]));
        ++n;
        return id;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, KernelArgs a) {
    using C = ChunkCfg<D>;
    constexpr int NS = C::NS;
    static_assert(chunk_smem_bytes<D>() <= kSmemLimit, "shared memory budget");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char* sQ = smem;
    unsigned char* sStage = sQ + C::Q_BYTES;
    unsigned char* sP = sStage + NS * C::STAGE_BYTES;     // 2 buffers of [high tile | residual tile]
    ChunkBars<NS>& B = *(ChunkBars<NS>*)(sP + 2 * C::P_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTR; ++s) {
            mbar_init(smem_u32(&B.task_full[s]), 1);
            mbar_init(smem_u32(&B.task_empty[s]), kTaskConsumers);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&B.stage_full[s]), 1);
            mbar_init(smem_u32(&B.stage_empty[s]), 1);
        }
        mbar_init(smem_u32(&B.q_full), 1);
        mbar_init(smem_u32(&B.q_empty), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&B.s_full[s]), 1);
            mbar_init(smem_u32(&B.s_empty[s]), 4);
            mbar_init(smem_u32(&B.p_full[s]), 4);
            mbar_init(smem_u32(&B.p_empty[s]), 1);
        }
        mbar_init(smem_u32(&B.o_full), 1);
        mbar_init(smem_u32(&B.o_empty), 4);
        mbar_init(smem_u32(&B.drain), 1);
        B.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&B.tmem_base)),
                     "r"(C::TMEM_COLS)
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
            bool q_tma = false;
            uint32_t q_par = 0;
            bool ok = true;
            while (ok) {
                const int slot = (int)(claimed % kTR);
                if (!wait_bar(smem_u32(&B.task_empty[slot]), ((claimed / kTR) & 1) ^ 1, abort_flag, true)) {
                    give_up(SITE_EMPTY_WAIT); ok = false; break;
                }
                int task = atomicAdd(&a.ctrl->queue_head, 1);
                if (task >= a.num_tasks) task = -1;
                ((volatile int*)B.task_slot)[slot] = task;
                mbar_arrive(smem_u32(&B.task_full[slot]));
                ++claimed;
                if (task < 0) break;
                const ChunkTask ct = chunk_task(a, task);
                if (ct.empty) continue;
                // the tile's 128 query rows: tokens row0/g .. +128/g, heads kv*g .. +g
                if (!wait_bar(smem_u32(&B.q_empty), (qn & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                mbar_expect_tx(smem_u32(&B.q_full), C::Q_BYTES);
                const int tok0 = ct.r.q_start + ct.row0 / g;
                for (int j = 0; j < C::BOXES; ++j)
                    tma_3d(smem_u32(sQ + j * C::Q_BOX), &tmap_q, 64 * j, ct.kv * g, tok0, smem_u32(&B.q_full));
                q_tma = true;
                q_par = qn & 1;
                ++qn;
                for (int u = 0; u < ct.n_units; ++u) {
                    const int s = (int)(item % NS);
                    const uint32_t round = item / NS;
                    if (!wait_bar(smem_u32(&B.stage_empty[s]), (round & 1) ^ 1, abort_flag, true)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
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
                        unsigned char* st = sStage + s * C::STAGE_BYTES;
                        for (int j = 0; j < C::BOXES; ++j) {
                            tma_2d(smem_u32(st + j * C::KV_BOX), &tmap_k, 64 * j, y, full);
                            tma_2d(smem_u32(st + C::TILE_BYTES + j * C::KV_BOX), &tmap_v, 64 * j, y, full);
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
    } else if (warp == 1) {
        // ===================== MMA issuer (lane 0) =====================
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kRows, kKeys, 0);
            const uint32_t id_o = idesc_bf16(kRows, D, 1);
            uint32_t item = 0, qn = 0, tn = 0;
            bool ok = true;
            Ring<NS> ring;
            while (ok) {
                const int task = ring.next(B, abort_flag, 0, false);
                if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
                if (task < 0) break;
                const ChunkTask ct = chunk_task(a, task);
                if (ct.empty) continue;
                if (!wait_bar(smem_u32(&B.q_full), qn & 1, abort_flag, true)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++qn;
                tc_fence_after();
                const uint32_t item0 = item;
                int s_next = 0, pv_next = 0;
                bool o_free = false;
                unsigned long long t0 = 0;
                uint32_t spins = 0;
                // Poll both queues: the P V product of unit u needs its probabilities; the
                // scores of unit u need its stage and a free score buffer (at most two units
                // ahead of the P V products).  P V goes first when both are ready.
                while (pv_next < ct.n_units) {
                    bool issued = false;
                    if (pv_next < s_next) {
                        const uint32_t gp = item0 + pv_next;
                        if (!o_free) o_free = mbar_test(smem_u32(&B.o_empty), (tn & 1) ^ 1);
                        if (o_free && mbar_test(smem_u32(&B.p_full[gp & 1]), (gp >> 1) & 1)) {
                            tc_fence_after();
                            const int stage = (int)(gp % NS);
                            const uint32_t vbase = smem_u32(sStage + stage * C::STAGE_BYTES + C::TILE_BYTES);
                            const uint32_t pbase = smem_u32(sP + (gp & 1) * C::P_BYTES);
                            for (int kk = 0; kk < 8; ++kk) {
                                // k-steps 0..3: bf16 high part; 4..7: residual (same V rows)
                                const uint64_t ad = desc_sw128(pbase + (kk >> 2) * C::P_TILE + (kk & 3) * 32, 16, 1024);
                                const uint64_t bd = desc_sw128(vbase + (kk & 3) * 2048, C::KV_BOX, 1024);
                                mma_f16(tmem + C::COL_O, ad, bd, id_o, (pv_next > 0 || kk > 0) ? 1u : 0u);
                            }
                            mma_commit(smem_u32(&B.p_empty[gp & 1]));
                            mma_commit(smem_u32(&B.stage_empty[stage]));
                            ++pv_next;
                            issued = true;
                        }
                    }
                    if (!issued && s_next < ct.n_units && s_next < pv_next + 2) {
                        const uint32_t gs = item0 + s_next;
                        const int stage = (int)(gs % NS);
                        if (mbar_test(smem_u32(&B.stage_full[stage]), (gs / NS) & 1) &&
                            mbar_test(smem_u32(&B.s_empty[gs & 1]), ((gs >> 1) & 1) ^ 1)) {
                            tc_fence_after();
                            const uint32_t kbase = smem_u32(sStage + stage * C::STAGE_BYTES);
                            const uint32_t qbase = smem_u32(sQ);
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t ad = desc_sw128(qbase + (kk >> 2) * C::Q_BOX + (kk & 3) * 32, 16, 1024);
                                const uint64_t bd = desc_sw128(kbase + (kk >> 2) * C::KV_BOX + (kk & 3) * 32, 16, 1024);
                                mma_f16(tmem + C::COL_S + kKeys * (gs & 1), ad, bd, id_s, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(smem_u32(&B.s_full[gs & 1]));
                            if (s_next == ct.n_units - 1) mma_commit(smem_u32(&B.q_empty));
                            ++s_next;
                            issued = true;
                        }
                    }
                    if (issued) {
                        spins = 0;
                    } else {
                        // nothing ready: bounded spin
                        if (spins == 0) t0 = gtimer();
                        if ((++spins & 63) == 0) {
                            if (*abort_flag) { ok = false; break; }
                            if (gtimer() - t0 > kWaitLimitNs) { give_up(SITE_FULL_WAIT); ok = false; break; }
                        }
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&B.o_full));
                item += ct.n_units;
                ++tn;
            }
            // every MMA issued here completes before tensor memory is released
            mma_commit(smem_u32(&B.drain));
            if (!wait_bar(smem_u32(&B.drain), 0, abort_flag, false)) set_error(a.err, ERR_TIMEOUT | SITE_DRAIN);
        }
        __syncwarp();
    } else {
        // ===================== softmax + epilogue (thread = query row) =====================
        const int row = ((warp & 3) << 5) + lane;                 // tensor-memory lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) << 5) << 16);
        const bool fused = a.fused != 0;
        uint32_t sn = 0, on = 0;
        bool ok = true;
        Ring<NS> ring;
        while (ok) {
            const int task = ring.next(B, abort_flag, lane, true);
            if (task == -2) { give_up(SITE_FULL_WAIT); ok = false; break; }
            if (task < 0) break;
            const ChunkTask ct = chunk_task(a, task);
            const bool valid = row < ct.nrows;
            const int grow = ct.row0 + row;                       // row in the (request, KV head) group
            const int i = valid ? grow / g : 0;
            const int h = ct.kv * g + (valid ? grow % g : 0);
            // last key this row sees (-1: none)
            const int limit = valid ? min(ct.kend - 1, ct.r.seq_len - ct.r.q_len + i) : -1;
            const size_t orow = (size_t)(ct.r.q_start + i) * a.num_q_heads + h;
            const size_t st = (size_t)ct.r.state_base + ((size_t)i * a.num_q_heads + h) * ct.r.n_splits + ct.split;
            const bool direct = fused && ct.r.n_splits == 1;   // write the final output
            float m = -INFINITY, l = 0.f;
            if (!ct.empty) {
                for (int u = 0; u < ct.n_units; ++u) {
                    const uint32_t gi = sn;       // global unit index: stage gi % NS, buffers gi & 1
                    const int b2 = (int)(gi & 1);
                    const uint32_t par = (gi >> 1) & 1;
                    if (!warp_wait(smem_u32(&B.s_full[b2]), par, abort_flag, lane)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                    tc_fence_after();
                    uint32_t sr[64];
                    SKV_LD32(lane_addr + C::COL_S + kKeys * b2, sr);
                    SKV_LD32(lane_addr + C::COL_S + kKeys * b2 + 32, (sr + 32));
                    tc_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&B.s_empty[b2]));
                    ++sn;
                    const int key0 = ct.kb + u * kKeys;
                    float s[64];
                    float mx = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float v = (key0 + j > limit) ? -INFINITY : __uint_as_float(sr[j]) * a.scale_log2;
                        s[j] = v;
                        mx = fmaxf(mx, v);
                    }
                    // this P buffer was last read by the P V product of unit gi - 2
                    if (gi >= 2) {
                        if (!warp_wait(smem_u32(&B.p_empty[b2]), par ^ 1, abort_flag, lane)) { give_up(SITE_EMPTY_WAIT); ok = false; break; }
                    }
                    // Slots of the unit past the tile's last key (the unused tail of the last
                    // page) may hold anything; their weight is 0, but 0 * NaN is not, so their
                    // value rows are zeroed before the P V product (the score product of this
                    // unit has completed; the fence before the p_full arrive orders the stores).
                    if (key0 + kKeys > ct.kend) {
                        const int r0 = ct.kend - key0;
                        unsigned char* vst = sStage + (gi % NS) * C::STAGE_BYTES + C::TILE_BYTES;
                        for (int idx = row; idx < (kKeys - r0) * 8 * C::BOXES; idx += kRows) {
                            const int rr = r0 + idx / (8 * C::BOXES), rem = idx % (8 * C::BOXES);
                            *(uint4*)(vst + (rem >> 3) * C::KV_BOX + rr * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    // lazy rescale: a row whose max grew by more than 2^8 rescales its O and l.
                    // The tensor-memory loads and stores are warp-collective, so the whole warp
                    // takes the branch when any of its rows needs it (scale 1 for the others),
                    // after every P V product issued so far (unit gi - 1) has completed.
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
                            if (!warp_wait(smem_u32(&B.p_empty[gq & 1]), (gq >> 1) & 1, abort_flag, lane)) {
                                give_up(SITE_EMPTY_WAIT); ok = false; break;
                            }
                            tc_fence_after();
                        }
                        l *= scale_o;
                        for (int c = 0; c < D; c += 32) {
                            uint32_t o[32];
                            SKV_LD32(lane_addr + C::COL_O + c, o);
                            tc_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * scale_o);
                            SKV_ST32(lane_addr + C::COL_O + c, o);
                        }
                        tc_wait_st();
                    }
                    const float base = (m == -INFINITY) ? 0.f : m;
                    unsigned char* phi = sP + b2 * C::P_BYTES + row * 128;
                    unsigned char* plo = phi + C::P_TILE;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = exp2f(s[8 * c + 2 * e] - base);
                            const float x1 = exp2f(s[8 * c + 2 * e + 1] - base);
                            l += x0 + x1;
                            split_bf16(x0, x1, hi[e], lo[e]);
                        }
                        const int sw = (c ^ (row & 7)) << 4;
                        *(uint4*)(phi + sw) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *(uint4*)(plo + sw) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&B.p_full[b2]));
                }
                if (!ok) break;
                // ---- epilogue: O / l ----
                if (!warp_wait(smem_u32(&B.o_full), on & 1, abort_flag, lane)) { give_up(SITE_FULL_WAIT); ok = false; break; }
                ++on;
                tc_fence_after();
            }
            const bool empty_row = !(l > 0.f);
            const float inv = empty_row ? 0.f : 1.f / l;
            const float lse = empty_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                if (!ct.empty) {
                    SKV_LD32(lane_addr + C::COL_O + c, o);
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
                        __stcg((float4*)(a.o_part + st * D + c + j),
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
            if (!ct.empty) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.o_empty));
            }
            if (fused && ct.r.n_splits > 1) {
                // this warp's 32 row states are written (the warp barrier orders the lanes'
                // stores before lane 0's fence): the warp counts in for the reduction, which
                // waits for 4 counts per chunk task
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
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
// bf16 tiled map with 128-byte swizzle over `rank` dims (innermost first)
cudaError_t make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
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
    if ((e = make_map(&mv, a.v_cache, 2, kd, ks, kb)) != cudaSuccess) return e;
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
    const int grid = std::min(sms, a.num_tasks);
    chunk_tc_kernel<D><<<grid, kThreads, smem, s>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supports(int bf16, int head_dim, int page_size, int group) {
    return bf16 && (head_dim == 64 || head_dim == 128) && (page_size == 64 || page_size == 128) && group >= 1 &&
           group <= kRows && (kRows % group) == 0;
}

cudaError_t launch_chunk_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s) {
    if (a.num_tasks <= 0) return cudaSuccess;
    if ((((uintptr_t)a.q) & 15) || (((uintptr_t)a.k_cache) & 15) || (((uintptr_t)a.v_cache) & 15))
        return cudaErrorMisalignedAddress;
    if ((long long)num_pages_total * a.num_kv_heads * a.page_size >= (1LL << 31) || total_q >= (1LL << 31))
        return cudaErrorInvalidValue;
    if (a.head_dim_qk == 128) return launch_d<128>(a, total_q, num_pages_total, s);
    if (a.head_dim_qk == 64) return launch_d<64>(a, total_q, num_pages_total, s);
    return cudaErrorNotSupported;
}

}  // namespace skv
