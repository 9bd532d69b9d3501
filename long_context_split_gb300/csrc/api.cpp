// libsplitkv host side: argument checks, the plan object (split counts, task
// list, partial-state layout, workspace layout) and the C-ABI entry points.
// The arithmetic of the method runs in the CUDA kernels; nothing here
// computes attention.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "splitkv.h"
#include "calibration.h"
#include "internal.h"
#include "planner.h"

using namespace skv;

namespace {

thread_local std::string g_msg;

splitkv_status fail(splitkv_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
splitkv_status fail(splitkv_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_msg = buf;
    return s;
}

splitkv_status ok() {
    g_msg.clear();
    return SPLITKV_OK;
}

splitkv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(SPLITKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

constexpr int kRowsPerTask = 16;
// per-SM rates of this library's kernels, measured on GB300 (CUDA events) with the two
// running side by side: chunk tiles 2.34 TFLOP of causal chunk rows in 2.13 ms on 120 SMs;
// the decode engine 5.2 GB of KV in 2.12 ms on 34 SMs (72 GB/s per SM), in 2.07 ms on 30
// SMs with every task of at most 8 rows (its transposed products: 84 GB/s per SM); the HBM
// copy bandwidth caps the engine
constexpr double kChunkFlopsPerSmUs = 9.1e6;
constexpr double kEngineBytesPerSmUs = 7.1e4;
constexpr double kEngineBytesPerSmUs8 = 8.4e4;
constexpr double kHbmBytesPerUs = 6.7e6;
constexpr int kDefaultSms = 152;   // GB300 SM count, used when no device is visible

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return kDefaultSms; }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return kDefaultSms;
    }
    return n > 0 ? n : kDefaultSms;
}

int engine_ctas_default() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return kDefaultSms; }
    int n = gqa_engine_ctas(dev);
    return n > 0 ? n : device_sms();
}

// the MLA path runs each task as two work items on two CTAs side by side
int mla_units_default() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return kDefaultSms / 2; }
    int n = mla_tc_ctas(dev) / 2;
    return n > 0 ? n : device_sms() / 2;
}

}  // namespace

namespace skv {
void set_last_error_message(const char* msg) { g_msg = msg ? msg : ""; }
}  // namespace skv

struct splitkv_plan_s {
    // problem shape
    int32_t kind = 0, dtype = 0, batch = 0, hq = 0, hkv = 0, group = 0, dqk = 0, dv = 0, page = 0;
    int32_t max_pages = 0;
    int32_t path = 0;
    int32_t interleave = 0;            // splits take pages r, r + n, ... (Helix round-robin)
    int32_t kv_fp8 = 0;                // the plan was made for an E4M3 KV cache
    int32_t part_bf16 = 0;             // partial outputs stored as bf16 (splitkv_plan_params.partial_dtype)
    int32_t lat_copy = 0;              // MLA over an E4M3 cache: the kernel reads a bf16 copy of the pages
    int32_t chunk_ctas = 0, engine_ctas = 0;   // > 0: chunk tiles and engine run side by side on these CTAs
    int32_t gen_max_keys = 0;          // CUDA-core kernel: the most dense key slots of a task
    int32_t engine_rows8 = 0;          // decode engine: every task holds at most 8 rows
    int32_t trace = 0;                 // the workspace holds trace records (splitkv_plan_params.trace)
    size_t off_trace = 0;
    size_t off_vhp = 0, off_vh = 0;    // f16 value copy: its slot list (in the image) and its pages
    int32_t n_trace = 0, trace_red0 = 0, trace_chunk0 = 0, trace_pair0 = 0;   // records; first reduction /
                                                                              // chunk / paired-tile record
    int32_t rows_per_task = kRowsPerTask;
    std::vector<int32_t> seq_len, q_len, qo, n_splits;
    std::vector<TaskDesc> tasks;       // engine (or single-kernel) tasks, queue order
    std::vector<TaskDesc> ctasks;      // GQA chunk-tile tasks (tcgen05 kernel), longest first
    std::vector<TaskDesc> ptasks;      // GQA paired-tile blocks (tcgen05 kernel), longest first; task i =
                                       // blocks 2i and 2i + 1 (an odd count gets an empty last block)
    std::vector<int32_t> is_chunk;     // per request: 1 chunk-tile kernel, 2 paired-tile kernel, else 0
    std::vector<ReqDesc> reqs;
    std::vector<RedItem> red;          // reduction items of the fused engine
    std::vector<VhPage> vh_pages;      // slots of the chunk tiles' f16 value copy
    std::vector<int32_t> state_indptr;
    int64_t num_states = 0;
    int32_t num_rows = 0;
    double scores[4] = {0, 0, 0, 0};
    // workspace layout
    size_t off_tasks = 0, off_ctasks = 0, off_ptasks = 0, off_reqs = 0, off_indptr = 0, off_counters = 0, off_red = 0;
    size_t image_bytes = 0;
    size_t off_opart = 0, off_lse = 0, ws_bytes = 0;
    std::vector<unsigned char> image;   // control + descriptors + zeroed counters
};

namespace {

splitkv_status check_problem_shape(const splitkv_problem* p) {
    if (!p) return fail(SPLITKV_ERR_INVALID_ARG, "problem is NULL");
    if (p->kind != SPLITKV_GQA && p->kind != SPLITKV_MLA)
        return fail(SPLITKV_ERR_INVALID_ARG, "kind %d is not GQA or MLA", p->kind);
    if (p->dtype != SPLITKV_F32 && p->dtype != SPLITKV_BF16)
        return fail(SPLITKV_ERR_INVALID_ARG, "dtype %d is not F32 or BF16", p->dtype);
    if (p->batch < 1) return fail(SPLITKV_ERR_INVALID_ARG, "batch %d < 1", p->batch);
    if (p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_q_heads % p->num_kv_heads)
        return fail(SPLITKV_ERR_INVALID_ARG, "num_q_heads %d must be a positive multiple of num_kv_heads %d",
                    p->num_q_heads, p->num_kv_heads);
    if (p->head_dim_qk < 1 || p->head_dim_v < 1 || p->page_size < 1 || p->num_pages < 1 ||
        p->max_pages_per_req < 1)
        return fail(SPLITKV_ERR_INVALID_ARG, "head dims, page_size, num_pages and max_pages_per_req must be >= 1");
    if (p->kind == SPLITKV_GQA && p->head_dim_qk != p->head_dim_v)
        return fail(SPLITKV_ERR_INVALID_ARG, "GQA needs head_dim_qk == head_dim_v");
    if (p->kind == SPLITKV_MLA) {
        if (p->num_kv_heads != 1) return fail(SPLITKV_ERR_INVALID_ARG, "MLA needs num_kv_heads == 1");
        if (p->head_dim_v > p->head_dim_qk)
            return fail(SPLITKV_ERR_INVALID_ARG, "MLA needs head_dim_v <= head_dim_qk");
    }
    if (!std::isfinite(p->scale)) return fail(SPLITKV_ERR_INVALID_ARG, "scale is not finite");
    if (p->kv_fp8 != 0 && p->kv_fp8 != 1) return fail(SPLITKV_ERR_INVALID_ARG, "kv_fp8 %d", p->kv_fp8);
    if (p->reserved0 != 0) return fail(SPLITKV_ERR_INVALID_ARG, "reserved0 must be 0");
    if (p->kv_fp8 && !(std::isfinite(p->k_scale) && std::isfinite(p->v_scale) && p->k_scale > 0.f &&
                       p->v_scale > 0.f))
        return fail(SPLITKV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
    if (!p->seq_lens_host || !p->qo_indptr_host)
        return fail(SPLITKV_ERR_INVALID_ARG, "seq_lens_host and qo_indptr_host are required");
    if (p->qo_indptr_host[0] != 0) return fail(SPLITKV_ERR_INVALID_ARG, "qo_indptr[0] must be 0");
    for (int b = 0; b < p->batch; ++b) {
        int L = p->seq_lens_host[b];
        int ql = p->qo_indptr_host[b + 1] - p->qo_indptr_host[b];
        if (ql < 0) return fail(SPLITKV_ERR_INVALID_ARG, "qo_indptr decreases at request %d", b);
        if (L < 1) return fail(SPLITKV_ERR_INVALID_ARG, "seq_len[%d] = %d < 1", b, L);
        if (ql > L) return fail(SPLITKV_ERR_INVALID_ARG, "q_len %d > seq_len %d at request %d", ql, L, b);
        long long pages = ((long long)L + p->page_size - 1) / p->page_size;
        if (pages > p->max_pages_per_req)
            return fail(SPLITKV_ERR_INVALID_ARG, "request %d needs %lld pages > max_pages_per_req %d", b,
                        pages, p->max_pages_per_req);
    }
    long long rows = (long long)p->qo_indptr_host[p->batch] * p->num_q_heads;
    if (rows >= (1LL << 30)) return fail(SPLITKV_ERR_INVALID_ARG, "too many output rows");
    return ok();
}

// Which kernel serves the problem; UNSUPPORTED when none does.
splitkv_status choose_path(const splitkv_problem* p, int32_t* path) {
    if (p->kv_fp8) {
        // E4M3 caches: the GQA engine's f16-operand variant where it applies, else the
        // CUDA-core path (16-byte rows of codes, bf16 queries)
        if (p->kind == SPLITKV_GQA && p->dtype == SPLITKV_BF16 && gqa_engine_supports_fp8(p->head_dim_qk, p->page_size)) {
            *path = 1;
            return ok();
        }
        // absorbed MLA of the tcgen05 kernel's shape: that kernel over a bf16 copy of the
        // batch's latent pages (exact), written by a pre-pass
        if (mla_tc_supports(p->kind == SPLITKV_MLA, p->dtype == SPLITKV_BF16, p->num_q_heads, p->head_dim_qk,
                            p->head_dim_v, p->page_size)) {
            *path = 2;
            return ok();
        }
        if (p->dtype == SPLITKV_BF16 && p->head_dim_qk % 16 == 0 && p->head_dim_qk <= 1024 &&
            (p->head_dim_v / 32 == 2 || p->head_dim_v / 32 == 4 || p->head_dim_v / 32 == 16) &&
            p->head_dim_v % 32 == 0) {
            *path = 0;
            return ok();
        }
        return fail(SPLITKV_ERR_UNSUPPORTED,
                    "FP8 KV cache needs bf16 queries, head_dim_qk a multiple of 16 and head_dim_v 64, 128 or 512 "
                    "(kind %d dtype %d head_dim_qk %d head_dim_v %d page_size %d)", p->kind, p->dtype,
                    p->head_dim_qk, p->head_dim_v, p->page_size);
    }
    if (p->kind == SPLITKV_GQA && p->dtype == SPLITKV_BF16 &&
        gqa_engine_supports(p->head_dim_qk, p->page_size)) {
        *path = 1;
        return ok();
    }
    if (mla_tc_supports(p->kind == SPLITKV_MLA, p->dtype == SPLITKV_BF16, p->num_q_heads, p->head_dim_qk,
                        p->head_dim_v, p->page_size)) {
        *path = 2;
        return ok();
    }
    // CUDA-core path: 16-byte key-row loads, 32 lanes over the value columns
    if (p->head_dim_v % 32 == 0 && p->head_dim_qk <= 1024 &&
        p->head_dim_qk % (p->dtype == SPLITKV_BF16 ? 8 : 4) == 0 &&
        (p->head_dim_v / 32 == 2 || p->head_dim_v / 32 == 4 || p->head_dim_v / 32 == 16)) {
        *path = 0;
        return ok();
    }
    return fail(SPLITKV_ERR_UNSUPPORTED,
                "no kernel for kind %d dtype %d head_dim_qk %d head_dim_v %d page_size %d", p->kind,
                p->dtype, p->head_dim_qk, p->head_dim_v, p->page_size);
}

model::Params model_params(const splitkv_plan_params& pp, int hq, int path, int page_size) {
    model::Params m;
    m.num_ctas = pp.num_ctas > 0 ? pp.num_ctas
                                 : (path == 1 ? engine_ctas_default() : path == 2 ? mla_units_default() : device_sms());
    // reduction warps of one scheduling unit of the chosen engine: every warp of a GQA
    // engine CTA (7; 4 with 16-token pages); one per MLA task slot (that path merges in a
    // separate kernel after attention, so its reductions are modelled coarsely: runs of
    // h_q rows); the CUDA-core path's 16
    m.warps_per_cta = pp.warps_per_cta > 0 ? pp.warps_per_cta
                                           : (path == 1 ? (page_size == 16 ? 4 : 7) : path == 2 ? 1 : 16);
    m.q_heads = hq;
    m.decode_qlen_max = pp.decode_qlen_max > 0 ? pp.decode_qlen_max : 16;
    // a negative setting takes the constant fitted on this kind of GPU for the chosen kernel
    const calib::Fit& f = path == 2 ? calib::kMla : path == 1 ? calib::kGqaEngine : calib::kTable2;
    m.rho = pp.rho < 0 ? f.rho : pp.rho;
    m.delta_attn = pp.delta_attn < 0 ? f.delta_attn : pp.delta_attn;
    m.delta_red = pp.delta_red < 0 ? f.delta_red : pp.delta_red;
    m.gamma = pp.gamma < 0 ? f.gamma : pp.gamma;
    m.adopt_margin = pp.adopt_margin;
    return m;
}

splitkv_status check_plan_matches(const splitkv_problem* p, const splitkv_plan_t* pl) {
    if (!pl) return fail(SPLITKV_ERR_INVALID_ARG, "plan is NULL");
    splitkv_status s = check_problem_shape(p);
    if (s) return s;
    if (p->kind != pl->kind || p->dtype != pl->dtype || p->kv_fp8 != pl->kv_fp8 || p->batch != pl->batch ||
        p->num_q_heads != pl->hq || p->num_kv_heads != pl->hkv || p->head_dim_qk != pl->dqk ||
        p->head_dim_v != pl->dv || p->page_size != pl->page)
        return fail(SPLITKV_ERR_INVALID_ARG, "problem shape differs from the plan's");
    for (int b = 0; b < p->batch; ++b)
        if (p->seq_lens_host[b] != pl->seq_len[b] || p->qo_indptr_host[b + 1] != pl->qo[b + 1])
            return fail(SPLITKV_ERR_INVALID_ARG, "lengths of request %d differ from the plan's", b);
    return ok();
}

splitkv_status check_device_ptr(const void* ptr, const char* name, bool allow_null) {
    if (!ptr) {
        if (allow_null) return ok();
        return fail(SPLITKV_ERR_INVALID_ARG, "%s is NULL", name);
    }
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SPLITKV_ERR_INVALID_ARG, "%s: %s", name, cudaGetErrorString(e));
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fail(SPLITKV_ERR_INVALID_ARG, "%s is not device memory", name);
    return ok();
}

splitkv_status check_problem_ptrs(const splitkv_problem* p) {
    splitkv_status s;
    if (((uintptr_t)p->q | (uintptr_t)p->k_cache | (uintptr_t)p->v_cache) & 15)
        return fail(SPLITKV_ERR_INVALID_ARG, "q, k_cache and v_cache must be 16-byte aligned");
    if ((s = check_device_ptr(p->q, "q", false))) return s;
    if ((s = check_device_ptr(p->k_cache, "k_cache", false))) return s;
    if (p->kind == SPLITKV_GQA) {
        if ((s = check_device_ptr(p->v_cache, "v_cache", false))) return s;
    } else if (p->v_cache) {
        return fail(SPLITKV_ERR_INVALID_ARG, "MLA takes values from k_cache; v_cache must be NULL");
    }
    if ((s = check_device_ptr(p->page_table, "page_table", false))) return s;
    if ((s = check_device_ptr(p->seq_lens, "seq_lens", false))) return s;
    if ((s = check_device_ptr(p->qo_indptr, "qo_indptr", false))) return s;
    return ok();
}

splitkv_status check_workspace(const splitkv_plan_t* pl, void* ws, size_t bytes) {
    if (!ws) return fail(SPLITKV_ERR_WORKSPACE, "workspace is NULL");
    if (((uintptr_t)ws) & 255) return fail(SPLITKV_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    if (bytes < pl->ws_bytes)
        return fail(SPLITKV_ERR_WORKSPACE, "workspace has %zu bytes, plan needs %zu", bytes, pl->ws_bytes);
    return check_device_ptr(ws, "workspace", false);
}

}  // namespace

namespace skv {
splitkv_status check_decode_args(const splitkv_problem* prob, const splitkv_plan_t* plan, const void* out,
                                 const float* lse_out, const int32_t* dev_error_word) {
    splitkv_status s = check_plan_matches(prob, plan);
    if (s) return s;
    if ((s = check_problem_ptrs(prob))) return s;
    if ((s = check_device_ptr(out, "out", plan->num_rows == 0))) return s;
    if ((s = check_device_ptr(lse_out, "lse_out", true))) return s;
    return check_device_ptr(dev_error_word, "dev_error_word", true);
}
}  // namespace skv

namespace {

KernelArgs kernel_args(const splitkv_problem* p, const splitkv_plan_t* pl, void* ws) {
    KernelArgs a;
    std::memset(&a, 0, sizeof a);
    unsigned char* base = (unsigned char*)ws;
    a.q = p->q;
    a.k_cache = p->k_cache;
    a.v_cache = p->kind == SPLITKV_MLA ? p->k_cache : p->v_cache;
    a.page_table = p->page_table;
    a.tasks = (const TaskDesc*)(base + pl->off_tasks);
    a.reqs = (const ReqDesc*)(base + pl->off_reqs);
    a.num_tasks = (int32_t)pl->tasks.size();
    a.num_q_heads = p->num_q_heads;
    a.num_kv_heads = p->num_kv_heads;
    a.group = p->num_q_heads / p->num_kv_heads;
    a.head_dim_qk = p->head_dim_qk;
    a.head_dim_v = p->head_dim_v;
    a.page_size = p->page_size;
    a.num_pages = p->num_pages;
    a.kv_row_stride = p->head_dim_qk;
    a.mla = p->kind == SPLITKV_MLA ? 1 : 0;
    // E4M3 caches: the key scale folds into the score scale, the value scale multiplies the
    // normalised partial output
    a.scale_log2 = (float)((double)p->scale * (p->kv_fp8 ? (double)p->k_scale : 1.0) * 1.4426950408889634);
    a.kv_fp8 = p->kv_fp8;
    a.v_scale = p->kv_fp8 ? (p->kind == SPLITKV_MLA ? p->k_scale : p->v_scale) : 1.f;   // MLA values are latent rows
    a.part_bf16 = pl->part_bf16;
    a.v_half = base + pl->off_vh;
    a.vh_pages = (const VhPage*)(base + pl->off_vhp);
    a.num_vh_pages = (int32_t)pl->vh_pages.size();
    a.lat_copy = pl->lat_copy;
    if (pl->trace) {
        a.trace = (splitkv_trace_record*)(base + pl->off_trace);
        a.trace_red = a.trace + pl->trace_red0;
    }
    a.counters = (int32_t*)(base + pl->off_counters);
    a.red_items = (const RedItem*)(base + pl->off_red);
    a.num_red = (int32_t)pl->red.size();
    a.num_reqs = pl->batch;
    a.ctrl = (Control*)base;
    a.err = &((Control*)base)->error_word;
    a.inject = debug_inject();
    return a;
}

// The plan's chunk-tile tasks on the tcgen05 chunk kernel (same arguments as the
// engine's launch, its own task list)
cudaError_t launch_chunk_tiles(const KernelArgs& a, const splitkv_problem* p, const splitkv_plan_t* pl, void* ws,
                               splitkv_stream stream) {
    if (pl->ctasks.empty()) return cudaSuccess;
    KernelArgs c = a;
    c.tasks = (const TaskDesc*)((unsigned char*)ws + pl->off_ctasks);
    if (a.trace) c.trace = a.trace + pl->trace_chunk0;
    c.trace_red = nullptr;
    c.num_tasks = (int32_t)pl->ctasks.size();
    cudaError_t e = launch_chunk_value_convert(c, (cudaStream_t)stream);
    if (e != cudaSuccess) return e;
    return launch_chunk_partial(c, pl->qo[pl->batch], p->num_pages, (cudaStream_t)stream);
}

// The plan's paired-tile tasks on the tcgen05 paired-tile kernel (same arguments as the
// engine's launch, its own block list)
cudaError_t launch_pair_tiles(const KernelArgs& a, const splitkv_problem* p, const splitkv_plan_t* pl, void* ws,
                              splitkv_stream stream) {
    if (pl->ptasks.empty()) return cudaSuccess;
    KernelArgs c = a;
    c.tasks = (const TaskDesc*)((unsigned char*)ws + pl->off_ptasks);
    if (a.trace) c.trace = a.trace + pl->trace_pair0;
    c.trace_red = nullptr;
    c.num_tasks = (int32_t)(pl->ptasks.size() / 2);
    return launch_pair_partial(c, pl->qo[pl->batch], p->num_pages, (cudaStream_t)stream);
}

// A second stream per device (with a fork and a join event) for running the chunk tiles
// beside the engine; created on the first such launch on that device and kept.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mutex;
SideStream g_side[128];

cudaError_t side_stream(SideStream** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    SideStream& ss = g_side[dev];
    if (!ss.s) {
        if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &ss;
    return cudaSuccess;
}

// The GQA path: chunk tiles and paired tiles (if any) and the engine.  One after the other
// on `stream` (the tile kernels count their split requests in for the engine's reduction
// phase), or, when the plan chose a partition (chunk tiles, no paired tiles), side by side
// on disjoint SMs: the chunk tiles on the side stream, forked from and joined back into
// `stream`; neither kernel waits on the other.
cudaError_t launch_gqa_path(const KernelArgs& a, const splitkv_problem* p, const splitkv_plan_t* pl, void* ws,
                            splitkv_stream stream) {
    cudaError_t e;
    if (pl->chunk_ctas <= 0 || pl->ctasks.empty()) {
        if ((e = launch_chunk_tiles(a, p, pl, ws, stream)) != cudaSuccess) return e;
        if ((e = launch_pair_tiles(a, p, pl, ws, stream)) != cudaSuccess) return e;
        return launch_gqa_engine(a, p->num_pages, pl->engine_rows8, (cudaStream_t)stream);
    }
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStream* ss = nullptr;
    if ((e = side_stream(&ss)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ss->fork, (cudaStream_t)stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess) return e;
    KernelArgs c = a;
    c.max_ctas = pl->chunk_ctas;
    cudaError_t ec = launch_chunk_tiles(c, p, pl, ws, ss->s);
    if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return e;
    KernelArgs g = a;
    g.max_ctas = pl->engine_ctas;
    const cudaError_t eg = ec == cudaSuccess ? launch_gqa_engine(g, p->num_pages, pl->engine_rows8, (cudaStream_t)stream) : ec;
    // the caller's stream resumes only after the side stream's work
    if ((e = cudaStreamWaitEvent((cudaStream_t)stream, ss->join, 0)) != cudaSuccess) return e;
    return eg;
}

}  // namespace

namespace skv {
namespace {
std::atomic<int32_t> g_inject{0};
}
int32_t debug_inject() { return g_inject.load(std::memory_order_relaxed); }
}  // namespace skv

extern "C" {

splitkv_status splitkv_debug_set_inject(int32_t mode) {
    if (mode != 0 && mode != 1) return fail(SPLITKV_ERR_INVALID_ARG, "inject mode %d is not 0 or 1", mode);
    skv::g_inject.store(mode, std::memory_order_relaxed);
    return ok();
}

int32_t splitkv_abi_version(void) { return SPLITKV_ABI_VERSION; }

const char* splitkv_last_error_message(void) { return g_msg.c_str(); }

const char* splitkv_status_string(splitkv_status s) {
    switch (s) {
        case SPLITKV_OK: return "ok";
        case SPLITKV_ERR_INVALID_ARG: return "invalid argument";
        case SPLITKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case SPLITKV_ERR_WORKSPACE: return "workspace too small or misaligned";
        case SPLITKV_ERR_CUDA: return "CUDA error";
        case SPLITKV_ERR_TIMEOUT: return "device wait timed out";
        case SPLITKV_ERR_DEVICE_CHECK: return "device range check failed";
    }
    return "unknown status";
}

void splitkv_plan_params_default(splitkv_plan_params* p) {
    if (!p) return;
    std::memset(p, 0, sizeof *p);
    p->mode = SPLITKV_PLAN_CRITICAL_WAVE;
    p->uniform_splits = 1;
    p->min_splits = 1;
    p->max_splits = 64;
    p->num_ctas = 0;
    p->warps_per_cta = 0;
    p->tile_tokens = 0;
    p->decode_qlen_max = 16;
    // negative: the calibrated constants of the kernel the plan targets (calibration.h)
    p->rho = -1.0;
    p->delta_attn = -1.0;
    p->delta_red = -1.0;
    p->gamma = -1.0;
    p->adopt_margin = 0.10;
}

splitkv_status splitkv_plan(const splitkv_problem* prob, const splitkv_plan_params* params,
                            splitkv_plan_t** out) {
    if (!out) return fail(SPLITKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    splitkv_status s = check_problem_shape(prob);
    if (s) return s;
    splitkv_plan_params pp;
    if (params) pp = *params; else splitkv_plan_params_default(&pp);
    if (pp.mode != SPLITKV_PLAN_UNIFORM && pp.mode != SPLITKV_PLAN_CRITICAL_WAVE)
        return fail(SPLITKV_ERR_INVALID_ARG, "plan mode %d", pp.mode);
    if (pp.mode == SPLITKV_PLAN_UNIFORM && (pp.uniform_splits < 1 || pp.uniform_splits > 4096))
        return fail(SPLITKV_ERR_INVALID_ARG, "uniform_splits %d outside [1, 4096]", pp.uniform_splits);
    if (pp.mode == SPLITKV_PLAN_CRITICAL_WAVE &&
        (pp.min_splits < 1 || pp.max_splits < pp.min_splits || pp.max_splits > 4096))
        return fail(SPLITKV_ERR_INVALID_ARG, "split bounds [%d, %d]", pp.min_splits, pp.max_splits);
    if (pp.mode == SPLITKV_PLAN_CRITICAL_WAVE &&
        !((pp.rho > 0 || pp.rho < 0) && std::isfinite(pp.rho) && std::isfinite(pp.delta_attn) &&
          std::isfinite(pp.delta_red) && std::isfinite(pp.gamma) && pp.adopt_margin >= 0 && pp.adopt_margin < 1))
        return fail(SPLITKV_ERR_INVALID_ARG, "model parameters out of range");
    if (pp.interleave != 0 && pp.interleave != 1) return fail(SPLITKV_ERR_INVALID_ARG, "interleave %d", pp.interleave);
    if (pp.trace != 0 && pp.trace != 1) return fail(SPLITKV_ERR_INVALID_ARG, "trace %d is not 0 or 1", pp.trace);
    if (pp.reserved != 0) return fail(SPLITKV_ERR_INVALID_ARG, "reserved must be 0");
    if (pp.partial_dtype != SPLITKV_F32 && pp.partial_dtype != SPLITKV_BF16)
        return fail(SPLITKV_ERR_INVALID_ARG, "partial_dtype %d is not F32 or BF16", pp.partial_dtype);

    splitkv_plan_t* pl = new splitkv_plan_t();
    pl->interleave = pp.interleave;
    pl->part_bf16 = pp.partial_dtype == SPLITKV_BF16 ? 1 : 0;
    pl->kind = prob->kind;
    pl->dtype = prob->dtype;
    pl->kv_fp8 = prob->kv_fp8;
    pl->batch = prob->batch;
    pl->hq = prob->num_q_heads;
    pl->hkv = prob->num_kv_heads;
    pl->group = prob->num_q_heads / prob->num_kv_heads;
    pl->dqk = prob->head_dim_qk;
    pl->dv = prob->head_dim_v;
    pl->page = prob->page_size;
    pl->max_pages = prob->max_pages_per_req;
    if ((s = choose_path(prob, &pl->path))) { delete pl; return s; }
    if (pl->path == 2) pl->rows_per_task = prob->num_q_heads;   // one query token, all heads, per task
    const int B = prob->batch, P = prob->page_size, g = pl->group;
    pl->seq_len.assign(prob->seq_lens_host, prob->seq_lens_host + B);
    pl->qo.assign(prob->qo_indptr_host, prob->qo_indptr_host + B + 1);
    pl->q_len.resize(B);
    for (int b = 0; b < B; ++b) pl->q_len[b] = pl->qo[b + 1] - pl->qo[b];

    // model view of the batch
    const int tile = pp.tile_tokens > 0 ? pp.tile_tokens : P;
    std::vector<model::Seq> seqs(B);
    std::vector<int> row_blocks(B);
    // rows per task: 16 (decode tile); on the GQA path where the tcgen05 kernels apply,
    // 256 rows (two 128-row tiles of the chunk kernel) for requests with more than 128
    // query rows per KV head and one block of all of them (one 128-row tile of the
    // paired-tile kernel) for 33..128 rows; otherwise 64 rows (the engine's wide prefill
    // mode) above 16; all heads of one token on the MLA path
    // (the tile kernels fold the scale into the exponent after the row max: scale > 0)
    const bool chunk_ok = pl->path == 1 && prob->scale > 0.f && !pl->interleave && !prob->kv_fp8 &&
                          chunk_tc_supports(prob->dtype == SPLITKV_BF16, prob->head_dim_qk, P, g);
    const bool pair_ok = pl->path == 1 && prob->scale > 0.f && !pl->interleave && !prob->kv_fp8 &&
                         pair_tc_supports(prob->dtype == SPLITKV_BF16, prob->head_dim_qk, P, g);
    std::vector<int> rpt(B);
    std::vector<int32_t>& is_chunk = pl->is_chunk;
    is_chunk.assign(B, 0);
    for (int b = 0; b < B; ++b) {
        long long rows = (long long)pl->q_len[b] * g;
        rpt[b] = pl->rows_per_task;
        if (pl->path == 1 && P >= 64 && rows > 16) rpt[b] = 64;
        if (chunk_ok && rows > 128) {
            rpt[b] = 256;
            is_chunk[b] = 1;
        } else if (pair_ok && rows > 32) {
            rpt[b] = 128;
            is_chunk[b] = 2;
        }
        row_blocks[b] = (int)((rows + rpt[b] - 1) / rpt[b]);
        seqs[b].tiles = (pl->seq_len[b] + tile - 1) / tile;
        seqs[b].tasks_per_split = prob->num_kv_heads * row_blocks[b];
        seqs[b].vectors = pl->q_len[b] * prob->num_q_heads;
        seqs[b].q_len = pl->q_len[b];
    }
    model::Params mp = model_params(pp, prob->num_q_heads, pl->path, P);
    // Chunk tiles beside the engine: when every chunk request stays unsplit (its tiles write
    // the final rows, so the engine's reduction phase needs nothing from them) and no request
    // runs on the paired tiles, the two kernels run at once on disjoint SMs, split in
    // proportion to their work (chunk flops against engine KV bytes, at the per-SM rates
    // measured for these kernels on GB300).
    {
        long long n_chunk = 0, n_eng = 0, n_pair = 0;
        bool unsplit = true, rows8 = true;   // rows8: every engine task of at most 8 rows
        double flops = 0.0, kv_bytes = 0.0;
        for (int b = 0; b < B; ++b) {
            const int cs = pp.mode == SPLITKV_PLAN_UNIFORM ? pp.uniform_splits
                                                            : std::max(1, std::min(pp.min_splits, seqs[b].tiles));
            if (is_chunk[b] == 2) {
                ++n_pair;
            } else if (is_chunk[b]) {
                ++n_chunk;
                if (cs != 1) unsplit = false;
                const double L = pl->seq_len[b], ql = pl->q_len[b];
                flops += 2.0 * (prob->head_dim_qk + prob->head_dim_v) * prob->num_q_heads *
                         (ql * (L - ql) + ql * (ql + 1) / 2);
            } else {
                ++n_eng;
                if ((long long)pl->q_len[b] * g > 8) rows8 = false;
                kv_bytes += (double)pl->seq_len[b] * prob->num_kv_heads * (prob->head_dim_qk + prob->head_dim_v) * 2.0;
            }
        }
        const int sms = device_sms();
        if (n_chunk > 0 && n_eng > 0 && n_pair == 0 && unsplit && sms >= 4) {
            const double wc = flops / kChunkFlopsPerSmUs;          // SM-microseconds
            const double we = kv_bytes / (rows8 ? kEngineBytesPerSmUs8 : kEngineBytesPerSmUs);
            const double t_serial = wc / sms + std::max(we / sms, kv_bytes / kHbmBytesPerUs);
            int best_e = 0;
            double best_t = t_serial;
            for (int e = 1; e < sms; ++e) {
                const double t = std::max(wc / (sms - e), std::max(we / e, kv_bytes / kHbmBytesPerUs));
                if (t < best_t) { best_t = t; best_e = e; }
            }
            if (best_e > 0 && best_t < 0.95 * t_serial) {
                pl->engine_ctas = best_e;
                pl->chunk_ctas = sms - best_e;
                if (pp.num_ctas <= 0) mp.num_ctas = best_e;   // the engine's scheduling units
            }
        }
    }
    std::vector<int> splits(B, 1);
    if (pp.mode == SPLITKV_PLAN_UNIFORM) {
        std::fill(splits.begin(), splits.end(), pp.uniform_splits);
    } else {
        // The tile kernels run their own queues ahead of the engine, so the model plans the
        // engine's requests alone; chunk requests (hundreds of tile tasks each) keep the
        // minimum split count; the paired-tile requests are planned as a batch of their own
        // on K = two blocks per SM (each CTA runs two blocks side by side).  The scores
        // reported are the engine's, else the paired tiles'.
        std::vector<int> eng, pair;
        for (int b = 0; b < B; ++b) {
            if (is_chunk[b] == 1) splits[b] = std::max(1, std::min(pp.min_splits, seqs[b].tiles));
            else if (is_chunk[b] == 2) pair.push_back(b);
            else eng.push_back(b);
        }
        for (int part = 0; part < 2; ++part) {
            const std::vector<int>& idx = part == 0 ? pair : eng;
            if (idx.empty()) continue;
            model::Params m = mp;
            if (part == 0) m.num_ctas = 2 * (pp.num_ctas > 0 ? pp.num_ctas : device_sms());
            std::vector<model::Seq> es;
            for (int b : idx) es.push_back(seqs[b]);
            model::PlanResult r = model::plan_with_uniform(es, m, pp.min_splits, pp.max_splits);
            for (size_t k = 0; k < idx.size(); ++k) splits[idx[k]] = r.splits[k];
            pl->scores[0] = r.base_score;
            pl->scores[1] = r.score;
            pl->scores[2] = r.search_score;
            pl->scores[3] = r.reference_score;
        }
    }
    pl->n_splits.assign(splits.begin(), splits.end());

    // partial-state layout
    long long base = 0;
    pl->reqs.resize(B);
    for (int b = 0; b < B; ++b) {
        ReqDesc& r = pl->reqs[b];
        std::memset(&r, 0, sizeof r);
        r.seq_len = pl->seq_len[b];
        r.q_len = pl->q_len[b];
        r.q_start = pl->qo[b];
        r.n_splits = splits[b];
        r.state_base = (int32_t)base;
        r.page_row = b * prob->max_pages_per_req;
        r.vh_base = -1;
        // completion counts: one per engine task; four per 128-row tile holding rows of a
        // chunk task or per paired-tile block (one per softmax warp)
        long long counts = (long long)splits[b] * prob->num_kv_heads * row_blocks[b];
        if (is_chunk[b]) counts = (long long)splits[b] * prob->num_kv_heads * 4 * ((pl->q_len[b] * g + 127) / 128);
        r.n_tasks = (int32_t)counts;
        base += (long long)pl->q_len[b] * prob->num_q_heads * splits[b];
        if (base >= (1LL << 31) - 1) { delete pl; return fail(SPLITKV_ERR_INVALID_ARG, "too many partial states"); }
    }
    pl->num_states = base;
    pl->num_rows = pl->qo[B] * prob->num_q_heads;
    pl->state_indptr.resize((size_t)pl->num_rows + 1);
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < pl->q_len[b]; ++i)
            for (int h = 0; h < prob->num_q_heads; ++h)
                pl->state_indptr[(size_t)(pl->qo[b] + i) * prob->num_q_heads + h] =
                    pl->reqs[b].state_base + (i * prob->num_q_heads + h) * splits[b];
    pl->state_indptr[pl->num_rows] = (int32_t)base;

    // tasks, in model queue order
    // The engine's queue and the tile kernels' are separate: each is the model's queue
    // over its own requests (so a decode-only engine batch keeps its longest-first order).
    std::vector<model::QTask> queue;
    for (int part = 0; part < 3; ++part) {
        std::vector<int> idx;
        for (int b = 0; b < B; ++b)
            if (is_chunk[b] == part) idx.push_back(b);
        if (idx.empty()) continue;
        std::vector<model::Seq> ps;
        std::vector<int> psplits;
        for (int b : idx) {
            ps.push_back(seqs[b]);
            psplits.push_back(splits[b]);
        }
        for (model::QTask q : model::attention_queue(ps, psplits, mp)) {
            q.seq = idx[q.seq];
            queue.push_back(q);
        }
    }
    pl->tasks.reserve(queue.size());
    for (const model::QTask& q : queue) {
        const int b = q.seq;
        const int n_pages = (pl->seq_len[b] + P - 1) / P;
        const int per = n_pages / splits[b], extra = n_pages % splits[b];
        int p0 = q.split * per + std::min(q.split, extra);
        int cnt = per + (q.split < extra ? 1 : 0);
        TaskDesc t;
        t.page_stride = 1;
        if (pl->interleave) {
            // pages q.split, q.split + n, ...: the task's key window runs from its first page to
            // the end of the history, and the kernels visit every n-th page of it
            p0 = q.split;
            cnt = std::max(0, n_pages - p0);
            t.page_stride = splits[b];
        }
        t.b = b;
        t.kv_head = q.sub / row_blocks[b];
        int rb = q.sub % row_blocks[b];
        t.row_begin = rb * rpt[b];
        t.row_end = std::min(pl->q_len[b] * g, t.row_begin + rpt[b]);
        t.key_begin = std::min(p0 * P, pl->seq_len[b]);
        t.key_end = std::min((p0 + cnt) * P, pl->seq_len[b]);
        if (t.key_end < t.key_begin) t.key_end = t.key_begin;
        t.split = q.split;
        (is_chunk[b] == 1 ? pl->ctasks : is_chunk[b] == 2 ? pl->ptasks : pl->tasks).push_back(t);
    }
    // the decode engine computes tasks of at most 8 rows transposed (no padded MMA rows)
    pl->engine_rows8 = 1;
    for (const TaskDesc& t : pl->tasks)
        if (t.row_end - t.row_begin > 8) pl->engine_rows8 = 0;
    // the CUDA-core kernel stages a split's rows in shared memory when its largest task fits:
    // a task's dense key slots are its pages' (pages key_begin / P + k * page_stride)
    for (const TaskDesc& t : pl->tasks) {
        const int ps = std::max(1, t.page_stride), pb = t.key_begin / P, pe = (t.key_end + P - 1) / P;
        const int slots = t.key_end > t.key_begin ? ((pe - pb + ps - 1) / ps) * P : 0;
        pl->gen_max_keys = std::max(pl->gen_max_keys, slots);
    }
    // keys a tile's last row sees in its split
    auto tile_keys = [&](const TaskDesc& t) {
        const int i_last = (t.row_end - 1) / g;
        const int kend = std::min(t.key_end, pl->seq_len[t.b] - pl->q_len[t.b] + i_last + 1);
        return std::max(0, kend - t.key_begin);
    };
    // Chunk tiles by (request, KV head, split) group, the group with the longest tile first,
    // longest first within a group: the tiles of a group read the same key/value units, so
    // running them together keeps those units in L2 (longest first over all tiles interleaves
    // every group, whose units together exceed L2 on long chunks and are re-read from DRAM).
    {
        auto group_of = [&](const TaskDesc& t) {
            return ((long long)t.b * prob->num_kv_heads + t.kv_head) * 4096 + t.split;
        };
        std::map<long long, int> longest;
        for (const TaskDesc& t : pl->ctasks) {
            int& v = longest[group_of(t)];
            v = std::max(v, tile_keys(t));
        }
        std::stable_sort(pl->ctasks.begin(), pl->ctasks.end(), [&](const TaskDesc& x, const TaskDesc& y) {
            const long long gx = group_of(x), gy = group_of(y);
            if (gx != gy) {
                const int lx = longest[gx], ly = longest[gy];
                return lx != ly ? lx > ly : gx < gy;
            }
            return tile_keys(x) > tile_keys(y);
        });
    }
    // paired tiles: blocks longest first, consecutive blocks paired (a CTA's time is its
    // longer block's), an empty block after an odd last one
    std::stable_sort(pl->ptasks.begin(), pl->ptasks.end(),
                     [&](const TaskDesc& x, const TaskDesc& y) { return tile_keys(x) > tile_keys(y); });
    if (pl->ptasks.size() % 2) {
        TaskDesc e = pl->ptasks.back();
        e.row_begin = e.row_end = 0;
        e.key_begin = e.key_end = 0;
        e.split = 0;
        pl->ptasks.push_back(e);
    }

    // reduction items (fused engine): the rows of every split request in runs of R,
    // requests in order (the model's reduction queue).  R follows the model's run-length
    // rule over the requests that are reduced here (unsplit ones write their output
    // directly, they need no reduction).
    std::vector<model::Seq> red_seqs;
    for (int b = 0; b < B; ++b)
        if (splits[b] > 1) red_seqs.push_back(seqs[b]);
    const int R = red_seqs.empty() ? 1 : std::max(1, model::run_length(red_seqs, mp));
    for (int b = 0; b < B; ++b) {
        if (splits[b] <= 1) continue;
        const int rows = pl->q_len[b] * prob->num_q_heads;
        for (int v = 0; v < rows; v += R) pl->red.push_back(RedItem{b, v, std::min(rows, v + R), 0});
    }

    // MLA over an E4M3 cache on the tcgen05 kernel: every page of every request gets a slot in
    // a bf16 copy of the latent cache, written by a pre-pass before the kernel
    if (pl->path == 2 && prob->kv_fp8) {
        pl->lat_copy = 1;
        for (int b = 0; b < B; ++b) {
            pl->reqs[b].vh_base = (int32_t)pl->vh_pages.size();
            const int n_pages = (pl->seq_len[b] + P - 1) / P;
            for (int j = 0; j < n_pages; ++j) pl->vh_pages.push_back(VhPage{b, j});
        }
    }
    // the chunk tiles multiply f16 values: every page of a chunk request gets a slot in an
    // f16 copy of the value cache, written by a pre-pass before the chunk kernel
    if (!pl->ctasks.empty()) {
        for (int b = 0; b < B; ++b) {
            if (is_chunk[b] != 1) continue;
            pl->reqs[b].vh_base = (int32_t)pl->vh_pages.size();
            const int n_pages = (pl->seq_len[b] + P - 1) / P;
            for (int j = 0; j < n_pages; ++j) pl->vh_pages.push_back(VhPage{b, j});
        }
    }

    // workspace layout and upload image
    size_t off = sizeof(Control);
    pl->off_tasks = off;
    off = align256(off + pl->tasks.size() * sizeof(TaskDesc));
    pl->off_ctasks = off;
    off = align256(off + pl->ctasks.size() * sizeof(TaskDesc));
    pl->off_ptasks = off;
    off = align256(off + pl->ptasks.size() * sizeof(TaskDesc));
    pl->off_reqs = off;
    off = align256(off + (size_t)B * sizeof(ReqDesc));
    pl->off_indptr = off;
    off = align256(off + pl->state_indptr.size() * sizeof(int32_t));
    pl->off_counters = off;
    off = align256(off + (size_t)B * sizeof(int32_t));
    pl->off_red = off;
    off = align256(off + std::max<size_t>(1, pl->red.size()) * sizeof(RedItem));
    pl->off_vhp = off;
    off = align256(off + pl->vh_pages.size() * sizeof(VhPage));
    pl->image_bytes = off;
    pl->off_opart = off;
    off = align256(off + (size_t)pl->num_states * pl->dv * (pl->part_bf16 ? 2 : 4));
    pl->off_lse = off;
    off = align256(off + (size_t)pl->num_states * sizeof(float));
    // trace records: engine tasks (MLA: work items, two per task), reduction items, chunk tasks,
    // paired-tile tasks; the CUDA-core path records nothing
    if (pp.trace && pl->path != 0) {
        pl->trace = 1;
        const size_t units = pl->tasks.size() * (pl->path == 2 ? 2 : 1);
        const size_t reds = pl->path == 1 ? pl->red.size() : 0;   // the engine's reduction phase
        pl->trace_red0 = (int32_t)units;
        pl->trace_chunk0 = (int32_t)(units + reds);
        pl->trace_pair0 = (int32_t)(units + reds + pl->ctasks.size());
        pl->n_trace = (int32_t)(units + reds + pl->ctasks.size() + pl->ptasks.size() / 2);
        pl->off_trace = off;
        off = align256(off + (size_t)pl->n_trace * sizeof(splitkv_trace_record));
    }
    pl->off_vh = off;
    off = align256(off + pl->vh_pages.size() * (size_t)P *
                             (pl->lat_copy ? (size_t)prob->head_dim_qk : (size_t)prob->num_kv_heads * prob->head_dim_v) * 2);
    pl->ws_bytes = off;
    pl->image.assign(pl->image_bytes, 0);
    std::memcpy(pl->image.data() + pl->off_tasks, pl->tasks.data(), pl->tasks.size() * sizeof(TaskDesc));
    if (!pl->ctasks.empty())
        std::memcpy(pl->image.data() + pl->off_ctasks, pl->ctasks.data(), pl->ctasks.size() * sizeof(TaskDesc));
    if (!pl->ptasks.empty())
        std::memcpy(pl->image.data() + pl->off_ptasks, pl->ptasks.data(), pl->ptasks.size() * sizeof(TaskDesc));
    std::memcpy(pl->image.data() + pl->off_reqs, pl->reqs.data(), (size_t)B * sizeof(ReqDesc));
    std::memcpy(pl->image.data() + pl->off_indptr, pl->state_indptr.data(),
                pl->state_indptr.size() * sizeof(int32_t));
    if (!pl->red.empty())
        std::memcpy(pl->image.data() + pl->off_red, pl->red.data(), pl->red.size() * sizeof(RedItem));
    if (!pl->vh_pages.empty())
        std::memcpy(pl->image.data() + pl->off_vhp, pl->vh_pages.data(), pl->vh_pages.size() * sizeof(VhPage));
    *out = pl;
    return ok();
}

void splitkv_plan_destroy(splitkv_plan_t* plan) { delete plan; }

int32_t splitkv_plan_num_tasks(const splitkv_plan_t* plan) {
    return plan ? (int32_t)(plan->tasks.size() + plan->ctasks.size() + plan->ptasks.size() / 2) : -1;
}

int32_t splitkv_plan_num_pair_tasks(const splitkv_plan_t* plan) {
    return plan ? (int32_t)(plan->ptasks.size() / 2) : -1;
}

int32_t splitkv_plan_num_chunk_tasks(const splitkv_plan_t* plan) {
    return plan ? (int32_t)plan->ctasks.size() : -1;
}

splitkv_status splitkv_plan_chunk_requests(const splitkv_plan_t* plan, int32_t* flags) {
    if (!plan || !flags) return fail(SPLITKV_ERR_INVALID_ARG, "plan or flags is NULL");
    for (int b = 0; b < plan->batch; ++b) flags[b] = plan->is_chunk[b];
    return ok();
}

int64_t splitkv_plan_num_states(const splitkv_plan_t* plan) { return plan ? plan->num_states : -1; }

int32_t splitkv_plan_num_rows(const splitkv_plan_t* plan) { return plan ? plan->num_rows : -1; }

int32_t splitkv_plan_kernel_path(const splitkv_plan_t* plan) { return plan ? plan->path : -1; }

splitkv_status splitkv_plan_splits(const splitkv_plan_t* plan, int32_t* n_splits) {
    if (!plan || !n_splits) return fail(SPLITKV_ERR_INVALID_ARG, "NULL argument");
    std::copy(plan->n_splits.begin(), plan->n_splits.end(), n_splits);
    return ok();
}

splitkv_status splitkv_plan_state_indptr(const splitkv_plan_t* plan, int32_t* indptr) {
    if (!plan || !indptr) return fail(SPLITKV_ERR_INVALID_ARG, "NULL argument");
    std::copy(plan->state_indptr.begin(), plan->state_indptr.end(), indptr);
    return ok();
}

splitkv_status splitkv_plan_split_ranges(const splitkv_plan_t* plan, int32_t b, int32_t* be) {
    if (!plan || !be) return fail(SPLITKV_ERR_INVALID_ARG, "NULL argument");
    if (b < 0 || b >= plan->batch) return fail(SPLITKV_ERR_INVALID_ARG, "request %d out of range", b);
    if (plan->interleave) return fail(SPLITKV_ERR_UNSUPPORTED, "an interleaved plan's splits are not key ranges");
    const int P = plan->page, n = plan->n_splits[b], L = plan->seq_len[b];
    const int n_pages = (L + P - 1) / P, per = n_pages / n, extra = n_pages % n;
    for (int r = 0; r < n; ++r) {
        int p0 = r * per + std::min(r, extra);
        int cnt = per + (r < extra ? 1 : 0);
        int kb = std::min(p0 * P, L), ke = std::min((p0 + cnt) * P, L);
        be[2 * r] = kb;
        be[2 * r + 1] = std::max(kb, ke);
    }
    return ok();
}

int32_t splitkv_plan_interleaved(const splitkv_plan_t* plan) { return plan ? plan->interleave : 0; }

int32_t splitkv_plan_trace_records(const splitkv_plan_t* plan) { return plan ? plan->n_trace : 0; }

int32_t splitkv_plan_overlap_ctas(const splitkv_plan_t* plan) { return plan ? plan->chunk_ctas : -1; }

splitkv_status splitkv_trace_read(const splitkv_plan_t* plan, const void* workspace, size_t ws_bytes,
                                  splitkv_trace_record* out, splitkv_stream stream) {
    if (!plan || !out) return fail(SPLITKV_ERR_INVALID_ARG, "plan or out is NULL");
    if (!plan->trace) return fail(SPLITKV_ERR_INVALID_ARG, "the plan was made without trace");
    splitkv_status s = check_workspace(plan, const_cast<void*>(workspace), ws_bytes);
    if (s) return s;
    cudaError_t e = cudaMemcpyAsync(out, (const unsigned char*)workspace + plan->off_trace,
                                    (size_t)plan->n_trace * sizeof(splitkv_trace_record), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the trace");
    return ok();
}

splitkv_status splitkv_trace_tail_idle(const splitkv_trace_record* recs, int32_t n, int32_t kind_mask,
                                       int32_t num_sms, splitkv_trace_stats* out) {
    if (!recs || !out || n < 0 || num_sms < 0) return fail(SPLITKV_ERR_INVALID_ARG, "bad arguments");
    // the stage: every selected record; per SM, the last end
    uint64_t begin = UINT64_MAX, end = 0;
    std::vector<int32_t> sm_ids;
    std::vector<uint64_t> last;
    int32_t count = 0;
    for (int32_t k = 0; k < n; ++k) {
        const splitkv_trace_record& r = recs[k];
        if (r.kind < 0 || r.kind > 30 || !((kind_mask >> r.kind) & 1)) continue;
        if (r.end_ns < r.start_ns) return fail(SPLITKV_ERR_INVALID_ARG, "record %d ends before it starts", k);
        if (r.sm < 0 || (num_sms > 0 && r.sm >= num_sms))
            return fail(SPLITKV_ERR_INVALID_ARG, "record %d: SM %d outside [0, %d)", k, r.sm, num_sms);
        ++count;
        begin = std::min<uint64_t>(begin, r.start_ns);
        end = std::max<uint64_t>(end, r.end_ns);
        if ((size_t)r.sm >= last.size()) last.resize((size_t)r.sm + 1, 0);
        if (last[r.sm] == 0) sm_ids.push_back(r.sm);
        last[r.sm] = std::max<uint64_t>(last[r.sm], std::max<uint64_t>(r.end_ns, 1));
    }
    if (count == 0) return fail(SPLITKV_ERR_INVALID_ARG, "no record of the selected kinds");
    const int32_t sms = num_sms > 0 ? num_sms : (int32_t)sm_ids.size();
    double tail = 0.0;
    for (int32_t sm : sm_ids) tail += (double)(end - last[sm]);
    // SMs that ran nothing of the stage wait for all of it
    tail += (double)(sms - (int32_t)sm_ids.size()) * (double)(end - begin);
    out->records = count;
    out->sms = sms;
    out->begin_ns = (double)begin;
    out->end_ns = (double)end;
    out->tail_idle_sm_ns = tail;
    out->tail_idle_frac = end > begin ? tail / ((double)sms * (double)(end - begin)) : 0.0;
    return ok();
}

int32_t splitkv_plan_partial_dtype(const splitkv_plan_t* plan) {
    return plan ? (plan->part_bf16 ? SPLITKV_BF16 : SPLITKV_F32) : -1;
}

splitkv_status splitkv_plan_scores(const splitkv_plan_t* plan, double* scores4) {
    if (!plan || !scores4) return fail(SPLITKV_ERR_INVALID_ARG, "NULL argument");
    for (int i = 0; i < 4; ++i) scores4[i] = plan->scores[i];
    return ok();
}

size_t splitkv_workspace_bytes(const splitkv_plan_t* plan) { return plan ? plan->ws_bytes : 0; }

splitkv_status splitkv_plan_upload(const splitkv_plan_t* plan, void* workspace, size_t ws_bytes,
                                   splitkv_stream stream) {
    if (!plan) return fail(SPLITKV_ERR_INVALID_ARG, "plan is NULL");
    splitkv_status s = check_workspace(plan, workspace, ws_bytes);
    if (s) return s;
    cudaError_t e = cudaMemcpyAsync(workspace, plan->image.data(), plan->image_bytes,
                                    cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    return ok();
}

splitkv_status splitkv_partial(const splitkv_problem* prob, const splitkv_plan_t* plan, void* workspace,
                               size_t ws_bytes, void* o_part, float* lse_part, int32_t* dev_error_word,
                               splitkv_stream stream) {
    splitkv_status s = check_plan_matches(prob, plan);
    if (s) return s;
    if ((s = check_workspace(plan, workspace, ws_bytes))) return s;
    if ((s = check_problem_ptrs(prob))) return s;
    if ((s = check_device_ptr(o_part, "o_part", plan->num_states == 0))) return s;
    if (((uintptr_t)o_part) & (plan->part_bf16 ? 7 : 15))
        return fail(SPLITKV_ERR_INVALID_ARG, "o_part must be %d-byte aligned", plan->part_bf16 ? 8 : 16);
    if ((s = check_device_ptr(lse_part, "lse_part", plan->num_states == 0))) return s;
    if ((s = check_device_ptr(dev_error_word, "dev_error_word", true))) return s;
    if (plan->tasks.empty() && plan->ctasks.empty() && plan->ptasks.empty()) return ok();
    KernelArgs a = kernel_args(prob, plan, workspace);
    a.o_part = (float*)o_part;   // bf16 elements when the plan stores bf16 partials
    a.lse_part = lse_part;
    if (dev_error_word) a.err = dev_error_word;
    a.fused = 0;
    cudaError_t e;
    if (plan->path == 1)
        e = launch_gqa_path(a, prob, plan, workspace, stream);
    else if (plan->path == 2)
        e = launch_mla_partial(a, plan->qo[plan->batch], prob->num_pages, (cudaStream_t)stream);
    else
        e = launch_generic_partial(a, prob->dtype == SPLITKV_BF16, plan->gen_max_keys, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "partial attention launch");
    return ok();
}

splitkv_status merge_states(const float* o_part, const float* lse_part, const int32_t* state_indptr,
                            int32_t num_rows, int32_t head_dim, void* out, int32_t out_dtype,
                            float* lse_out, splitkv_stream stream) {
    return merge_states_typed(o_part, SPLITKV_F32, lse_part, state_indptr, num_rows, head_dim, out, out_dtype,
                              lse_out, stream);
}

splitkv_status merge_states_typed(const void* o_part, int32_t o_part_dtype, const float* lse_part,
                                  const int32_t* state_indptr, int32_t num_rows, int32_t head_dim, void* out,
                                  int32_t out_dtype, float* lse_out, splitkv_stream stream) {
    if (o_part_dtype != SPLITKV_F32 && o_part_dtype != SPLITKV_BF16)
        return fail(SPLITKV_ERR_INVALID_ARG, "o_part_dtype %d", o_part_dtype);
    if (num_rows < 0) return fail(SPLITKV_ERR_INVALID_ARG, "num_rows %d < 0", num_rows);
    if (head_dim < 4 || head_dim % 4 || head_dim > 1024)
        return fail(SPLITKV_ERR_UNSUPPORTED, "head_dim %d: need a multiple of 4 in [4, 1024]", head_dim);
    if (out_dtype != SPLITKV_F32 && out_dtype != SPLITKV_BF16)
        return fail(SPLITKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (num_rows == 0) return ok();
    splitkv_status s;
    if ((s = check_device_ptr(o_part, "o_part", false))) return s;
    if ((s = check_device_ptr(lse_part, "lse_part", false))) return s;
    if ((s = check_device_ptr(state_indptr, "state_indptr", false))) return s;
    if ((s = check_device_ptr(out, "out", false))) return s;
    if ((s = check_device_ptr(lse_out, "lse_out", true))) return s;
    if (((uintptr_t)o_part) & (o_part_dtype == SPLITKV_BF16 ? 7 : 15))
        return fail(SPLITKV_ERR_INVALID_ARG, "o_part must be %d-byte aligned", o_part_dtype == SPLITKV_BF16 ? 8 : 16);
    cudaError_t e = launch_merge(o_part, o_part_dtype == SPLITKV_BF16, lse_part, state_indptr, num_rows, head_dim,
                                 out, out_dtype == SPLITKV_BF16, lse_out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return ok();
}

splitkv_status splitkv_decode(const splitkv_problem* prob, const splitkv_plan_t* plan, void* workspace,
                              size_t ws_bytes, void* out, float* lse_out, int32_t* dev_error_word,
                              splitkv_stream stream) {
    splitkv_status s = skv::check_decode_args(prob, plan, out, lse_out, dev_error_word);
    if (s) return s;
    if ((s = check_workspace(plan, workspace, ws_bytes))) return s;
    if (plan->tasks.empty() && plan->ctasks.empty() && plan->ptasks.empty()) return ok();
    KernelArgs a = kernel_args(prob, plan, workspace);
    unsigned char* base = (unsigned char*)workspace;
    a.o_part = (float*)(base + plan->off_opart);
    a.lse_part = (float*)(base + plan->off_lse);
    if (dev_error_word) a.err = dev_error_word;
    a.out = out;
    a.lse_out = lse_out;
    a.out_bf16 = prob->dtype == SPLITKV_BF16;
    cudaError_t e;
    if (plan->path == 1) {
        // chunk and paired tiles first (their split requests count in), then the engine:
        // its tasks, then the reduction phase for every split request
        a.fused = 1;
        e = launch_gqa_path(a, prob, plan, workspace, stream);
        if (e != cudaSuccess) return cuda_fail(e, "chunk tile / paired tile / decode engine launch");
    } else if (plan->path == 0) {
        // CUDA-core kernel: each request's last task merges the request's splits
        a.fused = 1;
        e = launch_generic_partial(a, prob->dtype == SPLITKV_BF16, plan->gen_max_keys, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "partial attention launch");
    } else {
        a.fused = 0;
        e = launch_mla_partial(a, plan->qo[plan->batch], prob->num_pages, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "partial attention launch");
        e = launch_merge(a.o_part, a.part_bf16, a.lse_part, (const int32_t*)(base + plan->off_indptr), plan->num_rows,
                         plan->dv, out, a.out_bf16, lse_out, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    }
    return ok();
}

splitkv_status splitkv_read_device_error(int32_t* dev_error_word, void* workspace, int32_t clear,
                                         int32_t* raw, splitkv_stream stream) {
    int32_t* word = dev_error_word;
    if (!word) {
        if (!workspace) return fail(SPLITKV_ERR_INVALID_ARG, "need dev_error_word or workspace");
        word = &((Control*)workspace)->error_word;
    }
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (clear && v) {
        e = cudaMemsetAsync(word, 0, sizeof v, (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    }
    if (raw) *raw = v;
    if (v == 0) return ok();
    int code = v & 0xff;
    if (code == ERR_TIMEOUT) return fail(SPLITKV_ERR_TIMEOUT, "device wait timed out (word 0x%x)", v);
    return fail(SPLITKV_ERR_DEVICE_CHECK, "device check failed (word 0x%x)", v);
}

splitkv_status splitkv_model_simulate(const splitkv_seq_model* seqs, int32_t nseq, const int32_t* splits,
                                      const splitkv_model_params* params, double* score, double* attn_end) {
    if (!seqs || !splits || !params || nseq < 1) return fail(SPLITKV_ERR_INVALID_ARG, "bad arguments");
    if (params->num_ctas < 1 || params->warps_per_cta < 1)
        return fail(SPLITKV_ERR_INVALID_ARG, "num_ctas and warps_per_cta must be >= 1");
    std::vector<model::Seq> sq(nseq);
    std::vector<int> sp(splits, splits + nseq);
    for (int b = 0; b < nseq; ++b) {
        if (seqs[b].tiles < 1 || seqs[b].tasks_per_split < 1 || seqs[b].vectors < 0 || sp[b] < 1)
            return fail(SPLITKV_ERR_INVALID_ARG, "sequence %d: bad model fields", b);
        sq[b].tiles = seqs[b].tiles;
        sq[b].tasks_per_split = seqs[b].tasks_per_split;
        sq[b].vectors = seqs[b].vectors;
        sq[b].q_len = seqs[b].q_len;
    }
    model::Params p;
    p.num_ctas = params->num_ctas;
    p.warps_per_cta = params->warps_per_cta;
    p.q_heads = std::max(1, params->q_heads);
    p.decode_qlen_max = params->decode_qlen_max > 0 ? params->decode_qlen_max : 16;
    p.rho = params->rho;
    p.delta_attn = params->delta_attn;
    p.delta_red = params->delta_red;
    p.gamma = params->gamma;
    p.adopt_margin = params->adopt_margin;
    model::SimResult r = model::simulate(sq, sp, p);
    if (score) *score = r.score;
    if (attn_end) *attn_end = r.attn_end;
    return ok();
}

splitkv_status splitkv_model_plan(const splitkv_seq_model* seqs, int32_t nseq,
                                  const splitkv_model_params* params, int32_t min_splits,
                                  int32_t max_splits, int32_t* splits_out, double* scores_out) {
    if (!seqs || !params || !splits_out || nseq < 1) return fail(SPLITKV_ERR_INVALID_ARG, "bad arguments");
    if (params->num_ctas < 1 || params->warps_per_cta < 1 || min_splits < 1 || max_splits < min_splits)
        return fail(SPLITKV_ERR_INVALID_ARG, "bad model parameters");
    std::vector<model::Seq> sq(nseq);
    for (int b = 0; b < nseq; ++b) {
        if (seqs[b].tiles < 1 || seqs[b].tasks_per_split < 1 || seqs[b].vectors < 0)
            return fail(SPLITKV_ERR_INVALID_ARG, "sequence %d: bad model fields", b);
        sq[b].tiles = seqs[b].tiles;
        sq[b].tasks_per_split = seqs[b].tasks_per_split;
        sq[b].vectors = seqs[b].vectors;
        sq[b].q_len = seqs[b].q_len;
    }
    model::Params p;
    p.num_ctas = params->num_ctas;
    p.warps_per_cta = params->warps_per_cta;
    p.q_heads = std::max(1, params->q_heads);
    p.decode_qlen_max = params->decode_qlen_max > 0 ? params->decode_qlen_max : 16;
    p.rho = params->rho;
    p.delta_attn = params->delta_attn;
    p.delta_red = params->delta_red;
    p.gamma = params->gamma;
    p.adopt_margin = params->adopt_margin;
    model::PlanResult r = model::plan(sq, p, min_splits, max_splits);
    std::copy(r.splits.begin(), r.splits.end(), splits_out);
    if (scores_out) {
        scores_out[0] = r.base_score;
        scores_out[1] = r.score;
        scores_out[2] = r.search_score;
        scores_out[3] = r.reference_score;
    }
    return ok();
}

}  // extern "C"
