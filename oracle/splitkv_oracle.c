/*
 * Float64 CPU oracle for split-KV decode attention and the LSE-weighted
 * merge of partial attention states.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA path never calls
 * it and shares no code, header or table with it.
 *
 * What it computes (plain definitions, no blocking, no online rescaling):
 *
 *  Partial attention state -- LiquidCP, Section 3 "Attention Regions" and
 *  Helix Parallelism, "Attention-Phase Configuration" step 2: for a query
 *  row q and a subset S of its valid key positions,
 *      s_j   = scale * <q, k_j>                    j in S
 *      lse_S = log sum_{j in S} exp(s_j)            (natural log)
 *      o_S   = sum_{j in S} exp(s_j - lse_S) * v_j  (locally normalised)
 *  An empty S gives o_S = 0 and lse_S = -inf.
 *
 *  Merge -- LiquidCP Eq. (1) and Helix step 3: for disjoint subsets S_r
 *      o   = sum_r exp(lse_r) o_r / sum_r exp(lse_r)
 *      lse = log sum_r exp(lse_r)
 *  (evaluated with the maximum lse subtracted first, which changes nothing
 *  mathematically; terms with lse_r = -inf contribute nothing).
 *
 *  Valid keys of a row: request b holds seq_len_b cached tokens, the last
 *  q_len_b of which are the appended queries; query row i (0-based) sits at
 *  position seq_len_b - q_len_b + i and sees keys 0 .. that position
 *  (LiquidCP Section 2.1: chunk attention over appended KV is causal; a
 *  decode row with q_len 1 sees every cached token).
 *
 *  GQA (LiquidCP Section 2.1; Helix "Why TP_A <= K"): query head h reads
 *  KV head h / (Hq / Hkv).  MLA (SPLASH Section 2, Eq. 1): one latent cache
 *  row of width d_c + d_r per token shared by all heads; keys are the whole
 *  row and values its first d_c columns.
 *
 *  Paged cache: token j of request b lives on physical page
 *  page_table[b][j / P] at offset j % P.
 *
 * Inputs stored as bf16 are widened exactly to double; float32 likewise.
 * K/V caches may instead hold 8-bit E4M3 codes with one scale per tensor
 * (the FP8 KV cache SPLASH serves with, Appendix C.1): the value of a code c
 * is e4m3(c) * k_scale (keys; MLA latent rows) or * v_scale (GQA values).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t kind;             /* 0 = GQA (separate K and V caches), 1 = MLA (one latent cache) */
    int32_t dtype;            /* query storage: 0 = float32, 1 = bf16 bit patterns */
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;     /* 1 for MLA */
    int32_t head_dim_qk;
    int32_t head_dim_v;
    int32_t page_size;
    int32_t num_pages;
    int32_t max_pages_per_req;
    double scale;
    const void *q;            /* [total_q][Hq][D_qk] */
    const void *k_cache;      /* GQA [num_pages][Hkv][P][D_qk]; MLA [num_pages][P][D_qk] */
    const void *v_cache;      /* GQA [num_pages][Hkv][P][D_v];  MLA unused */
    const int32_t *page_table;/* [batch][max_pages_per_req] */
    const int32_t *seq_lens;  /* [batch] */
    const int32_t *qo_indptr; /* [batch + 1] */
    int32_t kv_dtype;         /* K/V storage: 0 = float32, 1 = bf16, 2 = E4M3 codes */
    int32_t pad0;
    double k_scale;           /* value of a key (MLA: latent) element = stored value * k_scale */
    double v_scale;           /* value of a GQA value element = stored value * v_scale */
} oracle_problem;

enum { ORC_OK = 0, ORC_BAD_ROW = -1, ORC_BAD_PAGE = -2, ORC_NOMEM = -3, ORC_BAD_SHAPE = -4 };

/*
 * OCP 8-bit floating point, E4M3 (the variant without infinities): sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
 * subnormals m/8 * 2^-6; S.1111.111 is NaN.  Every other code is
 * (-1)^S (1 + m/8) 2^(e - 7).
 */
static double e4m3_value(uint8_t c)
{
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

static double widen(const void *base, int dtype, size_t idx)
{
    if (dtype == 2)
        return e4m3_value(((const uint8_t *)base)[idx]);
    if (dtype == 0)
        return (double)((const float *)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* element offset of key/value component d of token j of request b */
static int kv_offset(const oracle_problem *p, int b, int j, int kv_head, int width, int d,
                     size_t *out)
{
    int page = p->page_table[(size_t)b * p->max_pages_per_req + j / p->page_size];
    if (page < 0 || page >= p->num_pages)
        return ORC_BAD_PAGE;
    int off = j % p->page_size;
    if (p->kind == 0)
        *out = (((size_t)page * p->num_kv_heads + kv_head) * p->page_size + off) * width + d;
    else
        *out = ((size_t)page * p->page_size + off) * p->head_dim_qk + d;
    return ORC_OK;
}

/*
 * Partial state of one query row over keys [key_begin, key_end) intersected
 * with the row's causal range.  `scores` must hold key_end - key_begin doubles.
 */
static int partial_row(const oracle_problem *p, int b, int i, int h, int key_begin, int key_end,
                       double *o, double *lse, double *scores)
{
    if (b < 0 || b >= p->batch)
        return ORC_BAD_ROW;
    int q_len = p->qo_indptr[b + 1] - p->qo_indptr[b];
    int L = p->seq_lens[b];
    if (i < 0 || i >= q_len || h < 0 || h >= p->num_q_heads || q_len > L)
        return ORC_BAD_ROW;
    int pos = L - q_len + i;
    int j0 = key_begin < 0 ? 0 : key_begin;
    int j1 = key_end < pos + 1 ? key_end : pos + 1;
    for (int d = 0; d < p->head_dim_v; ++d)
        o[d] = 0.0;
    if (j1 <= j0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    int group = p->num_q_heads / p->num_kv_heads;
    int kv_head = (p->kind == 0) ? h / group : 0;
    size_t qrow = ((size_t)(p->qo_indptr[b] + i) * p->num_q_heads + h) * p->head_dim_qk;

    /* s_j = scale * <q, k_j> */
    for (int j = j0; j < j1; ++j) {
        size_t ko;
        int rc = kv_offset(p, b, j, kv_head, p->head_dim_qk, 0, &ko);
        if (rc)
            return rc;
        double dot = 0.0;
        for (int d = 0; d < p->head_dim_qk; ++d)
            dot += widen(p->q, p->dtype, qrow + d) * (widen(p->k_cache, p->kv_dtype, ko + d) * p->k_scale);
        scores[j - j0] = p->scale * dot;
    }
    /* lse = log sum exp(s_j) */
    double m = -INFINITY;
    for (int j = j0; j < j1; ++j)
        if (scores[j - j0] > m)
            m = scores[j - j0];
    double sum = 0.0;
    for (int j = j0; j < j1; ++j)
        sum += exp(scores[j - j0] - m);
    double l = m + log(sum);
    /* o = sum exp(s_j - lse) v_j */
    const void *vbase = (p->kind == 0) ? p->v_cache : p->k_cache;
    double vscale = (p->kind == 0) ? p->v_scale : p->k_scale;
    int vwidth = (p->kind == 0) ? p->head_dim_v : p->head_dim_qk;
    for (int j = j0; j < j1; ++j) {
        double w = exp(scores[j - j0] - l);
        size_t vo;
        int rc = kv_offset(p, b, j, kv_head, vwidth, 0, &vo);
        if (rc)
            return rc;
        for (int d = 0; d < p->head_dim_v; ++d)
            o[d] += w * (widen(vbase, p->kv_dtype, vo + d) * vscale);
    }
    *lse = l;
    return ORC_OK;
}

/*
 * Partial state of one query row over an explicit key set (Helix Parallelism,
 * Section 2.3 step 4: under the staggered round-robin placement a KV shard is
 * not one range of the history).  keys: nkeys distinct key indices of request
 * b; those past the row's causal limit (or past seq_len) are left out.  The
 * same definition as partial_row: s_j = scale <q, k_j>, lse = log sum exp s_j,
 * o = sum exp(s_j - lse) v_j over the kept keys; none kept: o = 0, lse = -inf.
 * `scores` and `kept` must hold nkeys entries.
 */
static int partial_row_keys(const oracle_problem *p, int b, int i, int h, const int32_t *keys, int nkeys,
                            double *o, double *lse, double *scores, int32_t *kept)
{
    if (b < 0 || b >= p->batch)
        return ORC_BAD_ROW;
    const int q_len = p->qo_indptr[b + 1] - p->qo_indptr[b];
    const int seq_len = p->seq_lens[b];
    if (i < 0 || i >= q_len || h < 0 || h >= p->num_q_heads || q_len > seq_len)
        return ORC_BAD_ROW;
    const int last_visible = seq_len - q_len + i;     /* causal limit of row i */
    int nkept = 0;
    for (int t = 0; t < nkeys; ++t)
        if (keys[t] >= 0 && keys[t] <= last_visible)
            kept[nkept++] = keys[t];
    for (int d = 0; d < p->head_dim_v; ++d)
        o[d] = 0.0;
    if (nkept == 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    const int kvh = (p->kind == 0) ? h / (p->num_q_heads / p->num_kv_heads) : 0;
    const size_t qbase = ((size_t)(p->qo_indptr[b] + i) * p->num_q_heads + h) * p->head_dim_qk;
    double smax = -INFINITY;
    for (int t = 0; t < nkept; ++t) {
        size_t kbase;
        int rc = kv_offset(p, b, kept[t], kvh, p->head_dim_qk, 0, &kbase);
        if (rc)
            return rc;
        double qk = 0.0;
        for (int d = 0; d < p->head_dim_qk; ++d)
            qk += widen(p->q, p->dtype, qbase + d) * (widen(p->k_cache, p->kv_dtype, kbase + d) * p->k_scale);
        scores[t] = qk * p->scale;
        smax = scores[t] > smax ? scores[t] : smax;
    }
    double denom = 0.0;
    for (int t = 0; t < nkept; ++t)
        denom += exp(scores[t] - smax);
    const double lse_keys = smax + log(denom);
    const void *vsrc = (p->kind == 0) ? p->v_cache : p->k_cache;
    const double vmul = (p->kind == 0) ? p->v_scale : p->k_scale;
    const int vrow = (p->kind == 0) ? p->head_dim_v : p->head_dim_qk;
    for (int t = 0; t < nkept; ++t) {
        const double wt = exp(scores[t] - lse_keys);
        size_t vbase_off;
        int rc = kv_offset(p, b, kept[t], kvh, vrow, 0, &vbase_off);
        if (rc)
            return rc;
        for (int d = 0; d < p->head_dim_v; ++d)
            o[d] += wt * (widen(vsrc, p->kv_dtype, vbase_off + d) * vmul);
    }
    *lse = lse_keys;
    return ORC_OK;
}

/*
 * Partial states of n rows over key sets: rows[3*r .. 3*r+2] = (b, i, h), its keys
 * keys[key_indptr[r] .. key_indptr[r+1]).  o is [n][D_v], lse is [n].
 */
int oracle_partial_keysets(const oracle_problem *p, int n, const int32_t *rows, const int32_t *key_indptr,
                           const int32_t *keys, double *o, double *lse)
{
    if (p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads || p->page_size <= 0)
        return ORC_BAD_SHAPE;
    int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        const int32_t *rw = rows + 3 * (size_t)r;
        int nk = key_indptr[r + 1] - key_indptr[r];
        double *scores = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        int32_t *kept = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nk > 0 ? nk : 1));
        int rc = (scores && kept) ? partial_row_keys(p, rw[0], rw[1], rw[2], keys + key_indptr[r], nk,
                                                     o + (size_t)r * p->head_dim_v, lse + r, scores, kept)
                                  : ORC_NOMEM;
        free(scores);
        free(kept);
        if (rc) {
#pragma omp atomic write
            status = rc;
        }
    }
    return status;
}

/*
 * Partial states of n rows.  rows[5*r .. 5*r+4] = (b, i, h, key_begin, key_end):
 * request b, query row i within the request, query head h, key range.
 * o is [n][D_v], lse is [n].  Returns 0 or the first error code met.
 */
int oracle_partial_rows(const oracle_problem *p, int n, const int32_t *rows, double *o, double *lse)
{
    if (p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads || p->page_size <= 0)
        return ORC_BAD_SHAPE;
    int maxlen = 1;
    for (int b = 0; b < p->batch; ++b)
        if (p->seq_lens[b] > maxlen)
            maxlen = p->seq_lens[b];
    int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        const int32_t *rw = rows + 5 * (size_t)r;
        int kb = rw[3], ke = rw[4];
        if (kb < 0) kb = 0;
        if (ke > maxlen) ke = maxlen;
        double *scores = (double *)malloc(sizeof(double) * (size_t)(ke > kb ? ke - kb : 1));
        int rc = scores ? partial_row(p, rw[0], rw[1], rw[2], kb, ke,
                                      o + (size_t)r * p->head_dim_v, lse + r, scores)
                        : ORC_NOMEM;
        free(scores);
        if (rc) {
#pragma omp atomic write
            status = rc;
        }
    }
    return status;
}

/*
 * Full (unsplit) attention of n rows: rows[3*r .. 3*r+2] = (b, i, h).
 * The key range is all of [0, seq_len_b), cut by the causal rule.
 */
int oracle_attention_rows(const oracle_problem *p, int n, const int32_t *rows, double *o,
                          double *lse)
{
    int32_t *r5 = (int32_t *)malloc(sizeof(int32_t) * 5 * (size_t)(n > 0 ? n : 1));
    if (!r5)
        return ORC_NOMEM;
    for (int r = 0; r < n; ++r) {
        int b = rows[3 * r];
        r5[5 * r + 0] = b;
        r5[5 * r + 1] = rows[3 * r + 1];
        r5[5 * r + 2] = rows[3 * r + 2];
        r5[5 * r + 3] = 0;
        r5[5 * r + 4] = (b >= 0 && b < p->batch) ? p->seq_lens[b] : 0;
    }
    int rc = oracle_partial_rows(p, n, r5, o, lse);
    free(r5);
    return rc;
}

/*
 * Merge n partial states of width d (LiquidCP Eq. 1):
 *   o = sum_r exp(lse_r) o_r / sum_r exp(lse_r),  lse = log sum_r exp(lse_r).
 * o_parts is [n][d], lse_parts [n].  With no finite lse_r the result is
 * o = 0, lse = -inf.
 */
void oracle_merge(int n, int d, const double *o_parts, const double *lse_parts, double *o,
                  double *lse)
{
    double m = -INFINITY;
    for (int r = 0; r < n; ++r)
        if (lse_parts[r] > m)
            m = lse_parts[r];
    for (int k = 0; k < d; ++k)
        o[k] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double denom = 0.0;
    for (int r = 0; r < n; ++r)
        if (lse_parts[r] != -INFINITY)
            denom += exp(lse_parts[r] - m);
    for (int r = 0; r < n; ++r) {
        if (lse_parts[r] == -INFINITY)
            continue;
        double w = exp(lse_parts[r] - m) / denom;
        for (int k = 0; k < d; ++k)
            o[k] += w * o_parts[(size_t)r * d + k];
    }
    *lse = m + log(denom);
}

/* Batched merge: rows x of width d, states state_indptr[x] .. state_indptr[x+1]-1. */
void oracle_merge_rows(int nrows, int d, const int32_t *state_indptr, const double *o_parts,
                       const double *lse_parts, double *o, double *lse)
{
#pragma omp parallel for schedule(static)
    for (int x = 0; x < nrows; ++x) {
        int s0 = state_indptr[x], s1 = state_indptr[x + 1];
        oracle_merge(s1 - s0, d, o_parts + (size_t)s0 * d, lse_parts + s0, o + (size_t)x * d,
                     lse + x);
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* e4m3 value of each of n codes (the decoder the attention uses) */
void oracle_e4m3_values(int n, const uint8_t *codes, double *out)
{
    for (int i = 0; i < n; ++i)
        out[i] = e4m3_value(codes[i]);
}
