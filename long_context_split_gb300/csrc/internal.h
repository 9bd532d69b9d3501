// Internal types shared by the host library and the CUDA kernels of
// libsplitkv.  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "splitkv.h"

namespace skv {

// One attention task: the partial state of query rows [row_begin, row_end)
// of (request b, KV head kv_head) over the keys of split `split`,
// [key_begin, key_end) cut by each row's causal limit.  Rows index the
// (query token, head-in-group) pairs of the group: row = i * g + h_local.
struct TaskDesc {
    int32_t b;
    int32_t kv_head;
    int32_t row_begin;
    int32_t row_end;
    int32_t key_begin;
    int32_t key_end;
    int32_t split;
    int32_t page_stride;   // the task's pages: key_begin / P + k * page_stride below key_end (1: contiguous)
};
static_assert(sizeof(TaskDesc) == 32, "TaskDesc layout");

// Per-request table.  Partial state of token i, head h, split r of request b
// is state_base + (i * Hq + h) * n_splits + r.
struct ReqDesc {
    int32_t seq_len;
    int32_t q_len;
    int32_t q_start;
    int32_t n_splits;
    int32_t state_base;
    int32_t page_row;     // b * max_pages_per_req (offset of the request's page-table row)
    int32_t n_tasks;      // completion counts the fused reduction waits for: one per engine
                          // task, four per 128-row tile of a chunk task or per block of a
                          // paired-tile task (one per softmax warp)
    int32_t vh_base;      // chunk-tile requests: slot of their first page in the f16 value copy
                          // (-1: the request has none)
};
static_assert(sizeof(ReqDesc) == 32, "ReqDesc layout");

// One reduction item of the fused engine: merge the splits of rows
// [row_begin, row_end) of request b (row v = token i * Hq + head h).  Items
// run in plan order on warps that have no attention work left, once every
// attention task of the request has finished (LiquidCP Section 5.2).
struct RedItem {
    int32_t b;
    int32_t row_begin;
    int32_t row_end;
    int32_t pad;
};
static_assert(sizeof(RedItem) == 16, "RedItem layout");

// One page of a chunk-tile request in the f16 value copy: page j of request b.
struct VhPage {
    int32_t b;
    int32_t j;
};
static_assert(sizeof(VhPage) == 8, "VhPage layout");

// Workspace control block (first 256 bytes of the workspace).
struct Control {
    int32_t queue_head;   // next task index to claim
    int32_t exit_count;   // CTAs that finished (the last one resets the block)
    int32_t error_word;   // device error (0 = none)
    int32_t red_head;     // next reduction item to claim
    int32_t chunk_head;   // chunk-tile kernel: next task to claim (its own queue, so it can run
    int32_t chunk_exit;   //   beside the engine); CTAs that finished
    int32_t pair_head;    // paired-tile kernel: next task to claim; CTAs that finished
    int32_t pair_exit;
    int32_t pad[56];
};
static_assert(sizeof(Control) == 256, "Control layout");

// Device error word: low 8 bits = splitkv_status, next bits = site.
enum : int32_t {
    ERR_TIMEOUT = 5,
    ERR_DEVICE_CHECK = 6,
};
enum : int32_t {
    SITE_FULL_WAIT = 1 << 8,
    SITE_EMPTY_WAIT = 2 << 8,
    SITE_PAGE_RANGE = 3 << 8,
    SITE_DRAIN = 4 << 8,
    SITE_REDUCE_WAIT = 5 << 8,
    SITE_VALUE_RANGE = 6 << 8,   // a bf16 value outside the f16 range met an f16 product
};

// Bounded waits give up after this long (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct KernelArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;       // GQA V cache; MLA: same as k_cache
    const int32_t* page_table;
    const TaskDesc* tasks;
    const ReqDesc* reqs;
    int32_t num_tasks;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;             // num_q_heads / num_kv_heads (MLA: num_q_heads)
    int32_t head_dim_qk;
    int32_t head_dim_v;
    int32_t page_size;
    int32_t num_pages;
    int32_t kv_row_stride;     // elements between consecutive tokens of one KV head in a page
    int32_t mla;               // 1: V is the first head_dim_v columns of the K rows
    float scale_log2;          // scale * log2(e)
    float* o_part;             // [num_states][head_dim_v]
    float* lse_part;           // [num_states]
    int32_t* counters;         // fused engine: finished attention tasks per request
    const RedItem* red_items;  // fused engine: reduction items, plan order
    int32_t num_red;
    int32_t num_reqs;
    Control* ctrl;
    int32_t* err;              // device error word
    void* out;                 // fused mode: [rows][head_dim_v] (bf16 or f32)
    float* lse_out;            // fused mode, may be null
    int32_t out_bf16;
    int32_t fused;             // 1: the launch also produces the merged output
    int32_t inject;            // test hook (splitkv_debug_set_inject): 1 = the task claimer
                               // withholds every task, so the kernel's bounded waits expire
    int32_t kv_fp8;            // 1: k_cache / v_cache hold E4M3 codes (GQA engine only)
    float v_scale;             // value of a V code = e4m3 value * v_scale (1 otherwise; the key
                               // scale is folded into scale_log2)
    int32_t part_bf16;         // 1: o_part holds bf16 partial outputs (LSE stays float32)
    splitkv_trace_record* trace;       // per-task trace records of this launch, or null
    splitkv_trace_record* trace_red;   // fused engine: reduction-item records, or null
    void* v_half;              // chunk tiles: f16 copy of the chunk requests' value pages,
                               // [slot][num_kv_heads][page_size][head_dim]; MLA over an E4M3
                               // cache: bf16 copy of the batch's latent pages [slot][page_size][576]
    const VhPage* vh_pages;    // the copy's slots
    int32_t num_vh_pages;
    int32_t lat_copy;          // MLA: 1 when the kernel reads the bf16 latent copy (slot =
                               // vh_base of the request + its page index)
    int32_t max_ctas;          // persistent kernels: at most this many CTAs (0: one per SM)
};

// Brackets one kernel launch with events on its stream while the launch
// profiler is on (splitkv_profile_begin / splitkv_profile_end); no-op otherwise.
class ProfileScope {
  public:
    ProfileScope(int kernel, cudaStream_t s);
    ~ProfileScope();
    ProfileScope(const ProfileScope&) = delete;
    ProfileScope& operator=(const ProfileScope&) = delete;

  private:
    int kernel_;
    cudaStream_t stream_;
    cudaEvent_t start_, stop_;
};

// Current value of the test hook set by splitkv_debug_set_inject.
int32_t debug_inject();

// Sets the message returned by splitkv_last_error_message on this thread.
void set_last_error_message(const char* msg);

// Host-side argument checks of the fused decode (everything but the workspace):
// the plan matches the problem, every device pointer is device memory.  Enqueues
// nothing.
splitkv_status check_decode_args(const splitkv_problem* prob, const splitkv_plan_t* plan, const void* out,
                                 const float* lse_out, const int32_t* dev_error_word);

// ---- kernel launchers (defined in the .cu files) --------------------------
// max_keys: the most dense key slots of any task (its pages' slots); > 0 lets splits whose
// rows fit in shared memory be staged there first
cudaError_t launch_generic_partial(const KernelArgs& a, int bf16, int max_keys, cudaStream_t s);
// o_part: float32, or bf16 when part_bf16
cudaError_t launch_merge(const void* o_part, int part_bf16, const float* lse_part, const int32_t* indptr,
                         int32_t rows, int32_t dim, void* out, int out_bf16, float* lse_out,
                         cudaStream_t s);
// GQA bf16 tensor-core engine; returns cudaErrorNotSupported for shapes it lacks
// rows8: every attention task holds at most 8 rows (selects the transposed products)
cudaError_t launch_gqa_engine(const KernelArgs& a, int num_pages_total, int rows8, cudaStream_t s);
bool gqa_engine_supports(int head_dim, int page_size);
bool gqa_engine_supports_fp8(int head_dim, int page_size);   // E4M3 K/V caches
// bf16 absorbed-MLA tcgen05 path (128 heads, 576/512, page 64): each task runs as two
// work items (output column halves) on two CTAs
bool mla_tc_supports(int kind_mla, int bf16, int num_q_heads, int dqk, int dv, int page_size);
int mla_tc_ctas(int device);   // co-resident CTAs on `device`, one per SM (0 if unavailable)
cudaError_t launch_mla_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s);
int gqa_engine_ctas(int device);   // persistent CTAs on `device`
// bf16 GQA causal chunk tiles on tcgen05 (two 128-row tiles per task, 64-key units)
bool chunk_tc_supports(int bf16, int head_dim, int page_size, int group);
// f16 copy of the chunk requests' value pages (the chunk tiles' P V operand); run before
// launch_chunk_partial on the same stream
cudaError_t launch_chunk_value_convert(const KernelArgs& a, cudaStream_t s);
cudaError_t launch_chunk_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s);
// Paired 128-row tiles (33..128 query rows of one (request, KV head) per block, two
// independent blocks per CTA): which shapes the kernel takes, and its launch (task i =
// block descriptors 2i and 2i + 1 of a.tasks; a.num_tasks pairs)
bool pair_tc_supports(int bf16, int head_dim, int page_size, int group);
cudaError_t launch_pair_partial(const KernelArgs& a, long long total_q, int num_pages_total, cudaStream_t s);

}  // namespace skv
