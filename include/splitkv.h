/*
 * splitkv.h -- C ABI of libsplitkv: split-KV decode attention with an exact
 * LSE-weighted merge of partial states, on one GB300 (sm_103a).
 *
 * The method (LiquidCP Section 2.1 and Section 3, Eq. 1; Helix Parallelism,
 * "Attention-Phase Configuration", steps 2-3): the KV history of each
 * request is cut into independent ranges ("splits"); each split yields a
 * partial attention state -- an output normalised over the split and the
 * log-sum-exp (LSE) of its scores -- and the partial states of a query row
 * are merged exactly,
 *      o = sum_r exp(lse_r) o_r / sum_r exp(lse_r),  lse = log sum_r exp(lse_r).
 * On one GPU the splits play the role of the KV-parallel ranks: they are
 * regions of the same HBM, processed by different SMs.
 *
 * Conventions shared by every entry point
 *  - Memory: pointers documented "device" must be device (or managed)
 *    memory of the current CUDA device; "host" pointers are ordinary host
 *    memory.  The caller allocates and frees every buffer; the library
 *    allocates only the host-side plan object, freed by splitkv_plan_destroy.
 *  - Streams: every call that touches the GPU is asynchronous on the given
 *    stream (0 = legacy default stream).  Argument errors are detected on the
 *    host and returned synchronously before anything is enqueued.
 *  - Device-side errors (a page id outside the pool, a bounded wait that ran
 *    out) are written to a caller-visible 32-bit error word; read it with
 *    splitkv_read_device_error after the stream has been synchronised.  The
 *    library never aborts the process and its kernels never trap or assert.
 *  - Threads: all functions are thread-safe except that one plan object must
 *    not be destroyed while another thread uses it.  splitkv_last_error_message
 *    is per thread.
 *  - Query rows: request b owns tokens qo_indptr[b] .. qo_indptr[b+1]-1 of q;
 *    its q_len = qo_indptr[b+1] - qo_indptr[b] appended tokens are the last
 *    q_len of its seq_len cached tokens, and its query row i (0-based) sees
 *    keys 0 .. seq_len - q_len + i (causal over the appended chunk; a decode
 *    row with q_len 1 sees the whole history).
 *  - GQA head map: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - Output rows: out and lse_out hold total_q * num_q_heads rows, row
 *    x = token * num_q_heads + head, out row width head_dim_v.
 */
#ifndef SPLITKV_H
#define SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPLITKV_ABI_VERSION 1

/* a cudaStream_t, passed as an opaque handle so this header needs no CUDA headers */
typedef void *splitkv_stream;

typedef enum {
    SPLITKV_OK = 0,
    SPLITKV_ERR_INVALID_ARG = 1,   /* a pointer, size or length is invalid */
    SPLITKV_ERR_UNSUPPORTED = 2,   /* valid, but no kernel covers this shape/dtype */
    SPLITKV_ERR_WORKSPACE = 3,     /* workspace too small or misaligned */
    SPLITKV_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    SPLITKV_ERR_TIMEOUT = 5,       /* (device) a bounded wait ran out */
    SPLITKV_ERR_DEVICE_CHECK = 6,  /* (device) a page id or index failed its range check */
} splitkv_status;

typedef enum { SPLITKV_GQA = 0, SPLITKV_MLA = 1 } splitkv_kind;
typedef enum { SPLITKV_F32 = 0, SPLITKV_BF16 = 1 } splitkv_dtype;

/*
 * One batch of attention over a paged KV cache (LiquidCP Section 2.1,
 * decode and mixed batches; paged KV as in SPLASH Appendix F.1).
 *
 * kind SPLITKV_GQA: q [total_q][num_q_heads][head_dim_qk]; k_cache and
 *   v_cache [num_pages][num_kv_heads][page_size][head_dim] ("HND": each
 *   (page, KV head) block of page_size x head_dim elements is contiguous);
 *   head_dim_qk == head_dim_v.
 * kind SPLITKV_MLA (absorbed MLA, SPLASH Section 2 Eq. 1 and Appendix A:
 *   one latent row of d_c + d_r = 512 + 64 per token shared by all heads):
 *   q [total_q][num_q_heads][576]; k_cache [num_pages][page_size][576];
 *   v_cache NULL -- values are the first head_dim_v = 512 columns of k_cache;
 *   num_kv_heads == 1.
 * page_table [batch][max_pages_per_req]: token j of request b is at page
 *   page_table[b][j / page_size], offset j % page_size.  Entries past a
 *   request's last page are never read.
 * dtype: storage type of q, k_cache and v_cache (SPLITKV_F32 or SPLITKV_BF16);
 *   arithmetic is float32 with float32 accumulation either way.
 * scale: multiplies q.k (e.g. 1/sqrt(head_dim)); the exported LSE is the
 *   natural log of sum exp(scale * q.k).
 * seq_lens_host / qo_indptr_host: host copies of seq_lens / qo_indptr, read
 *   by the planner (splitkv_plan) and by argument checks; the device copies
 *   are read by the kernels.  Both must hold the same values.
 */
typedef struct {
    int32_t kind;                    /* splitkv_kind */
    int32_t dtype;                   /* splitkv_dtype */
    int32_t batch;                   /* >= 1 */
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim_qk;
    int32_t head_dim_v;
    int32_t page_size;
    int32_t num_pages;               /* pages in the pool; page ids must be < num_pages */
    int32_t max_pages_per_req;       /* row stride of page_table */
    float scale;
    const void *q;                   /* device */
    const void *k_cache;             /* device */
    const void *v_cache;             /* device, NULL for MLA */
    const int32_t *page_table;       /* device */
    const int32_t *seq_lens;         /* device [batch], 1 <= seq_len, q_len <= seq_len */
    const int32_t *qo_indptr;        /* device [batch + 1], qo_indptr[0] == 0, non-decreasing */
    const int32_t *seq_lens_host;    /* host [batch] */
    const int32_t *qo_indptr_host;   /* host [batch + 1] */
    int32_t kv_fp8;                  /* 0: k_cache / v_cache hold `dtype` values.  1: they hold
                                        8-bit E4M3 codes (OCP FP8, the variant without
                                        infinities), the value of code c being e4m3(c) * k_scale
                                        in k_cache and e4m3(c) * v_scale in v_cache: an FP8 KV
                                        cache with one scale per tensor (SPLASH Appendix C.1).
                                        For MLA the latent rows are keys and values, so both
                                        take k_scale (v_scale is checked, not used).  Needs dtype
                                        BF16 (q and outputs).  GQA with head_dim 128 and
                                        page_size 64 or 128 runs on the GQA engine, which
                                        multiplies f16 operands, so query entries must lie
                                        within the f16 range (|q| <= 65504).  MLA of the tcgen05
                                        kernel's shape (128 heads, 576 / 512, page 64, contiguous
                                        splits) runs on that kernel over a bf16 copy of the
                                        batch's latent pages (exact), written into the workspace
                                        by a pre-pass: the workspace grows by 73,728 bytes per
                                        page of the batch.  Other shapes with head_dim_qk a
                                        multiple of 16 and head_dim_v 64, 128 or 512 run on the
                                        CUDA-core path in float32.  Other problems with
                                        kv_fp8 = 1 are UNSUPPORTED. */
    float k_scale;                   /* kv_fp8: finite, > 0 */
    float v_scale;                   /* kv_fp8: finite, > 0 */
    int32_t reserved0;               /* 0 */
} splitkv_problem;

typedef enum { SPLITKV_PLAN_UNIFORM = 0, SPLITKV_PLAN_CRITICAL_WAVE = 1 } splitkv_plan_mode;

/*
 * Planner settings.  Critical-wave model of LiquidCP Section 5.2 (Eq. 5:
 * tau(k) = max(rho, k/K); Eq. 6: c_red = delta_red + gamma * v_u * s_u;
 * c_attn = n_t + delta_attn).  A negative rho, delta_attn, delta_red or
 * gamma takes the constant calibrated on GB300 for the kernel the plan
 * targets (LiquidCP Appendix A.2 "Calibration", redone for this library's
 * kernels; LiquidCP Table 2's H100 values where no fit exists).
 */
typedef struct {
    int32_t mode;             /* splitkv_plan_mode */
    int32_t uniform_splits;   /* UNIFORM: splits per request; a history with fewer pages gets empty splits */
    int32_t min_splits;       /* CRITICAL_WAVE: lower bound per request (>= 1) */
    int32_t max_splits;       /* CRITICAL_WAVE: upper bound per request */
    int32_t num_ctas;         /* K of the model; 0 = the engine's CTA count on the current device */
    int32_t warps_per_cta;    /* reduction warps per scheduling unit in the model; 0 = the engine's own
                                 (GQA engine 7, or 4 with 16-token pages; MLA task slot 1,
                                 its merge being a separate kernel; CUDA-core path 16) */
    int32_t tile_tokens;      /* tokens per model KV tile; 0 = page_size */
    int32_t decode_qlen_max;  /* requests with q_len <= this are decode requests; 0 = 16 */
    double rho;               /* per-tile time floor; < 0: calibrated */
    double delta_attn;        /* fixed work per attention task, in tile units; < 0: calibrated */
    double delta_red;         /* fixed cost per reduction task; < 0: calibrated */
    double gamma;             /* cost per merged partial vector; < 0: calibrated */
    double adopt_margin;      /* adopt a split plan only if >= this fraction below NoSplit */
    int32_t interleave;       /* 0: split r of a request is a contiguous page range (the cut of
                                 LiquidCP Figure 8).  1: split r takes the request's pages r,
                                 r + n, r + 2n, ... (n = its split count): Helix Parallelism's
                                 staggered round-robin KV layout (Section 2.3, step 4), one page
                                 per round-robin block (16-token pages give the paper's 16-token
                                 blocks).  Split sizes are the same as with contiguous ranges.
                                 Interleaved plans run on the GQA engine (row blocks of up to 64
                                 rows: no chunk or paired tiles), on the MLA tcgen05 kernel and
                                 on the CUDA-core path. */
    int32_t partial_dtype;    /* storage type of the partial outputs o_r (splitkv_dtype):
                                 SPLITKV_F32 (default; SGLang's exchange precision) or
                                 SPLITKV_BF16 -- each o_r rounded to nearest even once, the
                                 precision vLLM and MegaDCP exchange partial states in
                                 (LiquidCP Section 7); half the partial-state bytes.  The
                                 LSE of every partial state stays float32.  Applies to the
                                 workspace of splitkv_decode and to splitkv_partial's o_part. */
    int32_t trace;            /* 1: the workspace gets a trace region and the persistent kernels
                                 record every task (see splitkv_trace_read); 0: off */
    int32_t reserved;         /* 0 */
} splitkv_plan_params;

/* Fill *p with the defaults: critical-wave mode, min 1 / max 64 splits, K =
 * engine scheduling units, the engine's reduction warps, tile = page, model
 * constants calibrated for the target kernel (negative values), margin 0.10
 * (LiquidCP Section 5.2). */
void splitkv_plan_params_default(splitkv_plan_params *p);

/* Opaque host-side plan: per-request split counts, the ordered task list and
 * the partial-state layout.  Built once per batch and reusable by every layer
 * that shares the batch's lengths (LiquidCP Section 7, planner runs once per
 * decoding step). */
typedef struct splitkv_plan_s splitkv_plan_t;

/*
 * splitkv_plan -- choose splits and build the task list (host only, no GPU
 * work; LiquidCP Section 5.2 "Plan selection" and "Task ordering", Appendix
 * A.2 "Split planning").
 *  prob:   problem; only shapes, seq_lens_host and qo_indptr_host are read.
 *  params: NULL for defaults.
 *  out:    receives a new plan; free with splitkv_plan_destroy.
 * Splits are contiguous, page-aligned ranges: with N pages and n splits,
 * split r holds floor(N/n) pages, plus one for r < N mod n (LiquidCP
 * Figure 8 cuts 176 tiles as 59/59/58).  Errors: INVALID_ARG (bad lengths,
 * shapes), UNSUPPORTED (no kernel for the shape).
 */
splitkv_status splitkv_plan(const splitkv_problem *prob, const splitkv_plan_params *params,
                            splitkv_plan_t **out);

void splitkv_plan_destroy(splitkv_plan_t *plan);

/* Plan queries (host). */
int32_t splitkv_plan_num_tasks(const splitkv_plan_t *plan);
/* Tasks that run on the tcgen05 chunk-tile kernel (up to 256 query rows each, as two
 * 128-row tiles): GQA bf16 requests with more than 128 query rows per KV head, D 64/128,
 * page 64/128, group size dividing 128, scale > 0, contiguous splits, bf16 cache.
 * Included in splitkv_plan_num_tasks.  -1 on NULL. */
int32_t splitkv_plan_num_chunk_tasks(const splitkv_plan_t *plan);
/* Tasks that run on the tcgen05 paired-tile kernel: GQA requests of the same shapes
 * with 33..128 query rows per KV head (speculative decode blocks, short appended
 * chunks).  Each of the request's (KV head, split) pairs is one block of up to 128 rows;
 * a task is two blocks, run side by side on one CTA (each in its own 128-row
 * tensor-memory tile), paired longest first.  Included in splitkv_plan_num_tasks.
 * -1 on NULL. */
int32_t splitkv_plan_num_pair_tasks(const splitkv_plan_t *plan);
/* flags[b] = 1 when request b runs on the chunk-tile kernel, 2 when on the paired-tile
 * kernel, else 0 (the decode engine or the CUDA-core path); INVALID_ARG on NULL. */
splitkv_status splitkv_plan_chunk_requests(const splitkv_plan_t *plan, int32_t *flags);
int64_t splitkv_plan_num_states(const splitkv_plan_t *plan);     /* partial states (rows of o_part) */
int32_t splitkv_plan_num_rows(const splitkv_plan_t *plan);       /* total_q * num_q_heads */
/* n_splits[b] for every request; returns INVALID_ARG on NULL. */
splitkv_status splitkv_plan_splits(const splitkv_plan_t *plan, int32_t *n_splits);
/* state_indptr[x], x = 0 .. num_rows: partial states of output row x are
 * rows state_indptr[x] .. state_indptr[x+1]-1 of o_part / lse_part, split r
 * at state_indptr[x] + r. */
splitkv_status splitkv_plan_state_indptr(const splitkv_plan_t *plan, int32_t *state_indptr);
/* key ranges [begin, end) of each split of request b (n_splits[b] pairs);
 * UNSUPPORTED for an interleaved plan, whose splits are not ranges: split r
 * holds the keys of pages r, r + n, r + 2n, ... below seq_len. */
splitkv_status splitkv_plan_split_ranges(const splitkv_plan_t *plan, int32_t b, int32_t *begin_end);
/* 1 if the plan's splits are page-interleaved (splitkv_plan_params.interleave), else 0. */
int32_t splitkv_plan_interleaved(const splitkv_plan_t *plan);
/* splitkv_dtype of the plan's partial outputs (splitkv_plan_params.partial_dtype); -1 on NULL. */
int32_t splitkv_plan_partial_dtype(const splitkv_plan_t *plan);
/* model scores: [0] NoSplit (or min-split) baseline, [1] chosen plan,
 * [2] search result, [3] reference plan (all 0 in uniform mode). */
splitkv_status splitkv_plan_scores(const splitkv_plan_t *plan, double *scores4);
/* Which kernel the plan targets: 0 CUDA-core float32 path, 1 bf16 GQA
 * tensor-core engine, 2 bf16 MLA tcgen05 path. */
int32_t splitkv_plan_kernel_path(const splitkv_plan_t *plan);

/*
 * Device workspace needed by splitkv_partial / splitkv_decode for this plan:
 * the task descriptors, request table, state_indptr, completion counters and
 * (for splitkv_decode) the float32 partial states.  Must be 256-byte aligned.
 */
size_t splitkv_workspace_bytes(const splitkv_plan_t *plan);

/*
 * splitkv_plan_upload -- copy the plan's descriptors into the workspace and
 * zero its counters (asynchronous on stream; the plan must outlive the copy).
 * Call once per plan and workspace before splitkv_partial / splitkv_decode;
 * again after any call that returned a device error.
 */
splitkv_status splitkv_plan_upload(const splitkv_plan_t *plan, void *workspace, size_t ws_bytes,
                                   splitkv_stream stream);

/*
 * splitkv_partial -- partial attention states of every split (Helix step 2:
 * attention of each query row over its local KV range, producing the
 * normalised output and the LSE; LiquidCP Section 3 "Attention Regions").
 *  o_part:   device [num_states][head_dim_v] (output): float32, 16-byte aligned,
 *            or bf16, 8-byte aligned, when the plan's partial_dtype is BF16
 *  lse_part: device float32 [num_states] (output; natural log)
 *  state layout: see splitkv_plan_state_indptr.  A split that holds no key a
 *  row may see (empty split, or entirely past the row's causal limit) writes
 *  o = 0 and lse = -inf.
 *  dev_error_word: device int32, or NULL to use the workspace's own word.
 */
splitkv_status splitkv_partial(const splitkv_problem *prob, const splitkv_plan_t *plan,
                               void *workspace, size_t ws_bytes, void *o_part, float *lse_part,
                               int32_t *dev_error_word, splitkv_stream stream);

/*
 * merge_states -- LSE-weighted merge of partial states (LiquidCP Eq. 1;
 * Helix step 3: rescale each partial by exp(lse_r - lse) and sum).
 *  o_part [num_states][head_dim] float32, lse_part [num_states] float32,
 *  state_indptr [num_rows + 1] int32: all device.
 *  out [num_rows][head_dim] of out_dtype (float32, or bf16 rounded to nearest
 *  even once at the end); lse_out [num_rows] float32 (may be NULL).
 *  Partials with lse = -inf contribute nothing; a row with none finite gets
 *  o = 0, lse = -inf.  Splits are combined in index order, so results do not
 *  depend on timing.  head_dim must be a multiple of 4 and <= 1024.
 */
splitkv_status merge_states(const float *o_part, const float *lse_part, const int32_t *state_indptr,
                            int32_t num_rows, int32_t head_dim, void *out, int32_t out_dtype,
                            float *lse_out, splitkv_stream stream);

/*
 * merge_states_typed -- merge_states over partial outputs stored as
 * o_part_dtype: SPLITKV_F32 (16-byte aligned; the same as merge_states) or
 * SPLITKV_BF16 (8-byte aligned: the bf16 partial states of a plan made with
 * partial_dtype BF16, LiquidCP Section 7).  The weights, the sum and the
 * LSE are float32 either way.  Errors as merge_states, plus INVALID_ARG for
 * another dtype or a misaligned o_part.
 */
splitkv_status merge_states_typed(const void *o_part, int32_t o_part_dtype, const float *lse_part,
                                  const int32_t *state_indptr, int32_t num_rows, int32_t head_dim, void *out,
                                  int32_t out_dtype, float *lse_out, splitkv_stream stream);

/*
 * splitkv_decode -- the fused path: one persistent kernel claims the plan's
 * tasks from a device queue in plan order, computes each split's partial
 * state into the workspace, and the last task to finish for a (request, KV
 * head, row block) merges its splits in index order and writes out/lse_out
 * (LiquidCP Section 6.2: attention tasks publish partial results, the
 * dependent reduction runs as soon as its inputs are complete).  The
 * CUDA-core path (kernel path 0) works the same way in one launch: each
 * request's last task to finish merges the request's splits.  The tcgen05 MLA
 * path (kernel path 2) runs its partial kernel, then the merge kernel.
 *  out: device [total_q][num_q_heads][head_dim_v], bf16 for bf16 problems,
 *  float32 for float32 problems.  lse_out: device float32 [total_q *
 *  num_q_heads] (may be NULL).
 * Requires splitkv_plan_upload on this workspace first.  Calls on the same
 * workspace must be stream-ordered (they share the counters).
 * When splitkv_plan_overlap_ctas(plan) > 0 the chunk tiles run on a second
 * stream of the library's own (one per device, created with its fork and join
 * events by the first such call on the device and kept until exit), forked from
 * `stream` and joined back into it: work enqueued on `stream` afterwards still
 * follows the whole call.  The same holds for splitkv_partial.
 */
splitkv_status splitkv_decode(const splitkv_problem *prob, const splitkv_plan_t *plan,
                              void *workspace, size_t ws_bytes, void *out, float *lse_out,
                              int32_t *dev_error_word, splitkv_stream stream);

/*
 * splitkv_decode_static -- splitkv_decode without a caller-provided
 * workspace, for callers that cannot allocate device memory: code that runs
 * where the GPU's memory is already fully reserved by another allocator (a
 * serving framework's caching pool, where an extra cudaMalloc fails or
 * fragments it), latency-critical loops in which cudaMalloc / cudaFree would
 * synchronise the device, and plugin or foreign-language callers that have no
 * access to the host framework's allocator.  The pages describe no such
 * variant; it exists only for these callers.
 *
 * Scratch: a fixed device array of SPLITKV_STATIC_SCRATCH_BYTES inside the
 * library (file-scope device storage).  Every GPU on which the library's
 * device code is loaded holds this array until the process exits.  The call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *  - Size limit: plans with splitkv_workspace_bytes(plan) above
 *    SPLITKV_STATIC_SCRATCH_BYTES are rejected with SPLITKV_ERR_WORKSPACE
 *    before anything is enqueued; use splitkv_decode with your own workspace
 *    for them.
 *  - Set-up: the first call on a device (with that device current) looks up
 *    the array's device address once.
 *  - No stream capture: every call copies the plan's descriptors from the
 *    plan's own (pageable) host memory with cudaMemcpyAsync, which a CUDA graph
 *    could not replay once the plan is gone; call it outside capture (to put a
 *    decode in a graph, use splitkv_plan_upload once and splitkv_decode).
 *  - Sharing: every call uses the same array and it keeps the last call's
 *    contents.  Each call re-uploads its plan's descriptors and zeroes the
 *    counters and error word it needs (asynchronously, on `stream`), so calls
 *    ordered on the GPU are independent; calls that overlap on the GPU (other
 *    streams, other threads) race on the array and give undefined results.
 *  - Arguments and results are those of splitkv_decode.  Every argument is
 *    checked on the host before anything is written to the array, so a call
 *    that returns an argument error has queued nothing.  With dev_error_word
 *    NULL, device errors go to the array's own error word: read it with
 *    splitkv_read_static_device_error before the next call, which clears it.
 */
#define SPLITKV_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
splitkv_status splitkv_decode_static(const splitkv_problem *prob, const splitkv_plan_t *plan, void *out,
                                     float *lse_out, int32_t *dev_error_word, splitkv_stream stream);

/*
 * Read the error word of the static array used by splitkv_decode_static
 * calls made with dev_error_word NULL on the current device: synchronises
 * `stream`, then behaves as splitkv_read_device_error (status, raw word,
 * optional clear).  Allocates nothing.
 */
splitkv_status splitkv_read_static_device_error(int32_t clear, int32_t *raw, splitkv_stream stream);

/*
 * Read the device error word (dev_error_word, or the workspace's own word
 * when dev_error_word is NULL and workspace is given): synchronises the
 * stream, returns SPLITKV_OK, SPLITKV_ERR_TIMEOUT or SPLITKV_ERR_DEVICE_CHECK,
 * and stores the raw word in *raw if raw is non-NULL.  clear != 0 zeroes it.
 */
splitkv_status splitkv_read_device_error(int32_t *dev_error_word, void *workspace, int32_t clear,
                                         int32_t *raw, splitkv_stream stream);

/* Message for the last error returned on the calling thread. */
const char *splitkv_last_error_message(void);
const char *splitkv_status_string(splitkv_status s);
int32_t splitkv_abi_version(void);

/*
 * Critical-wave model entry points (host only), exposed for calibration and
 * tests.  A sequence has `tiles` KV tiles, `tasks_per_split` attention tasks
 * per split, `vectors` output vectors and `q_len` query tokens.
 */
typedef struct {
    int32_t tiles;
    int32_t tasks_per_split;
    int32_t vectors;
    int32_t q_len;
} splitkv_seq_model;

typedef struct {
    int32_t num_ctas;         /* K */
    int32_t warps_per_cta;
    int32_t q_heads;          /* h_q for the reduction run-length rule */
    int32_t decode_qlen_max;
    double rho, delta_attn, delta_red, gamma, adopt_margin;
} splitkv_model_params;

/* Simulated completion (score) and attention completion of one split plan
 * (LiquidCP Section 5.2, Eqs. 5-6). */
splitkv_status splitkv_model_simulate(const splitkv_seq_model *seqs, int32_t nseq,
                                      const int32_t *splits, const splitkv_model_params *params,
                                      double *score, double *attn_end);

/* Plan search and selection (LiquidCP Section 5.2 "Plan selection", Appendix
 * A.2); splits_out [nseq]; scores_out [4] as in splitkv_plan_scores. */
splitkv_status splitkv_model_plan(const splitkv_seq_model *seqs, int32_t nseq,
                                  const splitkv_model_params *params, int32_t min_splits,
                                  int32_t max_splits, int32_t *splits_out, double *scores_out);

/*
 * Task trace (a measurement aid; LiquidCP Section 3 and Section 7 measure
 * per-SM stage timelines and tail idle the same way).  With
 * splitkv_plan_params.trace = 1 the plan's workspace holds one record per
 * traced unit of work and every splitkv_decode / splitkv_partial launch of the
 * plan rewrites them: the claimer stamps start_ns (%globaltimer), sm (%smid)
 * and cta when it takes the unit from the device queue; end_ns is the last
 * moment a role finished its part of it (its outputs written).  Records, in
 * order:
 *   GQA plans: one per engine task (kind ATTENTION), one per reduction item of
 *   the fused engine (kind REDUCTION; start after its inputs were complete),
 *   one per chunk-tile task (kind CHUNK), one per paired-tile task (kind PAIR);
 *   MLA tcgen05 plans: one per work item, two per task (kind MLA_ITEM);
 *   CUDA-core plans: none.
 * Units a launch did not reach (an error) keep the previous launch's values.
 */
typedef struct {
    uint64_t start_ns;
    uint64_t end_ns;
    int32_t id;       /* index of the unit within its kind */
    int32_t sm;
    int32_t kind;     /* splitkv_trace_kind */
    int32_t cta;
} splitkv_trace_record;

typedef enum {
    SPLITKV_TRACE_ATTENTION = 0,
    SPLITKV_TRACE_REDUCTION = 1,
    SPLITKV_TRACE_CHUNK = 2,
    SPLITKV_TRACE_MLA_ITEM = 3,
    SPLITKV_TRACE_PAIR = 4
} splitkv_trace_kind;

/* CTAs of the chunk-tile kernel when the plan runs it beside the engine on disjoint SMs
 * (0: the two run one after the other; -1 on NULL).  Chosen by splitkv_plan for GQA plans
 * whose chunk-tile requests are all unsplit -- their tiles write final rows, so the
 * engine's reduction phase needs nothing from them -- in proportion to the two kernels'
 * work, when that is expected to save at least 5 %; the engine then gets the other SMs
 * (and the critical-wave model plans its requests over that many units). */
int32_t splitkv_plan_overlap_ctas(const splitkv_plan_t *plan);

/* Records of the plan's trace region (0 when the plan was made without trace). */
int32_t splitkv_plan_trace_records(const splitkv_plan_t *plan);

/* Copy the trace records out of `workspace` into host memory `out`
 * [splitkv_plan_trace_records(plan)]; synchronises `stream`.  Errors:
 * INVALID_ARG (NULL, plan without trace), WORKSPACE, CUDA. */
splitkv_status splitkv_trace_read(const splitkv_plan_t *plan, const void *workspace, size_t ws_bytes,
                                  splitkv_trace_record *out, splitkv_stream stream);

typedef struct {
    int32_t records;          /* records of the selected kinds */
    int32_t sms;              /* SMs counted */
    double begin_ns;          /* first start of the selected records */
    double end_ns;            /* last end: the stage's finish */
    double tail_idle_sm_ns;   /* sum over SMs of (end_ns - the SM's last end) */
    double tail_idle_frac;    /* tail_idle_sm_ns / (sms * (end_ns - begin_ns)) */
} splitkv_trace_stats;

/*
 * Tail idle of one stage (host arithmetic only; LiquidCP Section 3: an SM's
 * wait after its last task in the stage until the stage finishes; the
 * fraction is summed tail idle over total SM-time).  The stage is made of the
 * records whose kind bit is set in kind_mask (bit k = kind k).  num_sms > 0
 * counts that many SMs, those with no record of the stage idle for all of it;
 * num_sms = 0 counts the SMs that appear in the records.  Errors: INVALID_ARG
 * (NULL, no selected record, a record with end < start or an SM id outside
 * [0, num_sms)).
 */
splitkv_status splitkv_trace_tail_idle(const splitkv_trace_record *recs, int32_t n, int32_t kind_mask,
                                       int32_t num_sms, splitkv_trace_stats *out);

/*
 * Launch profiler (host).  The pages describe no such facility: it is a
 * measurement aid.  Between splitkv_profile_begin and splitkv_profile_end,
 * every kernel launch of the library is bracketed by CUDA events recorded on
 * the launching stream (a few microseconds of host time per launch).
 * splitkv_profile_end waits for the recorded events, fills out[k] for each
 * kernel k (launch count, summed device time in ms; NULL to discard) and
 * turns the profiler off.  Process-wide; safe to call from several threads.
 * Errors: CUDA when an event could not be read (that launch is skipped).
 */
typedef enum {
    SPLITKV_KERNEL_GENERIC = 0,      /* CUDA-core float32/bf16 partial attention */
    SPLITKV_KERNEL_GQA_ENGINE = 1,   /* persistent bf16 GQA engine */
    SPLITKV_KERNEL_MLA = 2,          /* tcgen05 absorbed-MLA partial attention */
    SPLITKV_KERNEL_CHUNK = 3,        /* tcgen05 GQA chunk tiles */
    SPLITKV_KERNEL_MERGE = 4,        /* merge_states */
    SPLITKV_KERNEL_CHUNK_VCONV = 5,  /* f16 copy of the chunk requests' value pages (before the chunk tiles) */
    SPLITKV_KERNEL_PAIR = 6,         /* tcgen05 paired row blocks (33..128 rows per KV head) */
    SPLITKV_KERNEL_MLA_LATENT = 7,   /* bf16 copy of an E4M3 latent cache's pages (before the MLA kernel) */
    SPLITKV_KERNEL_COUNT = 8
} splitkv_kernel;

typedef struct {
    int32_t launches;
    int32_t pad;
    double total_ms;
} splitkv_kernel_time;

splitkv_status splitkv_profile_begin(void);
splitkv_status splitkv_profile_end(splitkv_kernel_time *out /* [SPLITKV_KERNEL_COUNT] */);

/*
 * Test hook (host; no counterpart on the pages).  mode 1 makes every
 * persistent kernel launched afterwards (GQA engine, chunk tiles, MLA)
 * withhold its tasks from its own roles: nothing ever signals them, so their
 * bounded waits expire after about 2 s each, the launch records
 * SPLITKV_ERR_TIMEOUT in its device error word and returns normally (no
 * fault, the context stays usable, outputs are not written).  mode 0 (the
 * default) restores normal operation.  Process-wide.  Errors: INVALID_ARG
 * for other modes.
 */
splitkv_status splitkv_debug_set_inject(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_H */
