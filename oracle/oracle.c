/*
 * oracle.c -- plain, slow float64 CPU oracle for Multi-Segment Attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What is computed (the method's result has a plain definition, so the
 * oracle is that definition written out):
 *
 *   The method is exact attention over a paged KV cache whose live blocks
 *   are scattered; its output must equal ordinary attention over the whole
 *   logical sequence (AsymCache explainer, "一句话结论" and "核心方法 1.
 *   Multi-Segment Attention"; MSA paper abstract: lossless management keeps
 *   outputs exact).  For a sequence s with L_s cached tokens, a query row at
 *   logical position p and query head h (GQA: kv head g = h / G, G = Hq/Hkv):
 *
 *       visible keys  j = 0 .. min(p, L_s - 1)
 *       t_j   = scale * sum_d q[p,h,d] * K_s[j,g,d]
 *       m     = max_j t_j
 *       lse   = m + ln sum_j exp(t_j - m)
 *       out   = sum_j exp(t_j - lse) * V_s[j,g,:]
 *
 *   A row with no visible key (only possible when L_s = 0) gets out = 0,
 *   lse = -inf.
 *
 *   oracle_dense_attention() evaluates that directly on the LOGICAL K/V
 *   (never the paged pool), one row at a time, in double precision.
 *
 *   oracle_segmented_attention() computes the same result the way MSA
 *   organises it (AsymCache explainer, "核心方法 1": the live blocks of a
 *   sequence are split into physically contiguous segments, each segment is
 *   attended on its own, and the per-segment results are combined; MSA paper
 *   abstract: the outputs stay exact).  Segment r gives a softmax partial, its
 *   normalised output o_r and log-sum-exp lse_r over the visible keys it
 *   holds, and the partials are merged by log-sum-exp, the combination
 *   under which the result is exact:
 *       LSE = ln sum_r exp(lse_r),   out = sum_r exp(lse_r - LSE) * o_r
 *   Segments are maximal runs of logical blocks i..j whose block-table
 *   entries rise by exactly one per block (logically AND physically
 *   contiguous), found left to right.  This path reads the paged pool
 *   through the block table and so checks the indexing independently.
 *
 * bf16 inputs are given as raw 16-bit patterns and widened exactly to double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_TABLE (-2)
#define ORACLE_ERR_NOMEM (-3)

/* bf16 -> double: a bf16 value is the top half of an IEEE binary32, so the
 * widening is exact. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_bf16_to_double(uint16_t b) { return bf16_to_double(b); }

/* Index of the sequence that owns packed query row r (q_indptr is
 * non-decreasing, q_indptr[0] = 0, q_indptr[num_seqs] = n_q). */
static int32_t seq_of_row(const int64_t* q_indptr, int32_t num_seqs, int64_t r) {
    int32_t lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (q_indptr[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* ---------------------------------------------------------------- dense -- */

typedef struct {
    int32_t num_seqs, hq, hkv, d;
    double scale;
    const int64_t* kv_indptr;
    const uint16_t* k;
    const uint16_t* v;
    const int64_t* q_indptr;
    const int32_t* q_pos;
    const uint16_t* q;
    const int64_t* rows;
    int64_t n_rows;
    double* out;
    double* lse;
    int64_t begin, end; /* slice of the output-row list handled by a thread */
    int status;
} dense_job;

static void* dense_worker(void* arg) {
    dense_job* jb = (dense_job*)arg;
    const int32_t d = jb->d, hq = jb->hq, hkv = jb->hkv;
    const int32_t group = hq / hkv;
    int64_t max_len = 0;
    for (int32_t s = 0; s < jb->num_seqs; ++s) {
        int64_t len = jb->kv_indptr[s + 1] - jb->kv_indptr[s];
        if (len > max_len) max_len = len;
    }
    double* t = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)d);
    if (!t || !qv) { free(t); free(qv); jb->status = ORACLE_ERR_NOMEM; return NULL; }

    /* work units are (output row, head) pairs: unit u = i * hq + h */
    for (int64_t u = jb->begin; u < jb->end; ++u) {
        const int64_t i = u / hq;
        const int32_t h = (int32_t)(u % hq);
        const int64_t r = jb->rows ? jb->rows[i] : i;
        const int32_t s = seq_of_row(jb->q_indptr, jb->num_seqs, r);
        const int64_t kv0 = jb->kv_indptr[s];
        const int64_t len = jb->kv_indptr[s + 1] - kv0;
        const int64_t p = jb->q_pos[r];
        int64_t n_vis = p + 1 < len ? p + 1 : len; /* keys j <= p and j < L_s */
        if (n_vis < 0) n_vis = 0;
        {
            const int32_t g = h / group;
            double* o = jb->out + (i * hq + h) * (int64_t)d;
            for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
            if (n_vis == 0) {
                jb->lse[i * hq + h] = -INFINITY;
                continue;
            }
            for (int32_t c = 0; c < d; ++c)
                qv[c] = bf16_to_double(jb->q[(r * hq + h) * (int64_t)d + c]);
            double m = -INFINITY;
            for (int64_t j = 0; j < n_vis; ++j) {
                const uint16_t* kj = jb->k + ((kv0 + j) * hkv + g) * (int64_t)d;
                double acc = 0.0;
                for (int32_t c = 0; c < d; ++c) acc += qv[c] * bf16_to_double(kj[c]);
                t[j] = jb->scale * acc;
                if (t[j] > m) m = t[j];
            }
            double sum = 0.0;
            for (int64_t j = 0; j < n_vis; ++j) sum += exp(t[j] - m);
            const double l = m + log(sum);
            jb->lse[i * hq + h] = l;
            for (int64_t j = 0; j < n_vis; ++j) {
                const double w = exp(t[j] - l);
                const uint16_t* vj = jb->v + ((kv0 + j) * hkv + g) * (int64_t)d;
                for (int32_t c = 0; c < d; ++c) o[c] += w * bf16_to_double(vj[c]);
            }
        }
    }
    free(t);
    free(qv);
    jb->status = ORACLE_OK;
    return NULL;
}

static int run_jobs(void* (*fn)(void*), void* jobs, size_t job_size, int32_t n) {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n);
    if (!th) return ORACLE_ERR_NOMEM;
    int32_t started = 0;
    for (int32_t i = 1; i < n; ++i) {
        if (pthread_create(&th[i], NULL, fn, (char*)jobs + job_size * (size_t)i) != 0) break;
        started = i;
    }
    fn(jobs); /* job 0 on the calling thread */
    for (int32_t i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    /* jobs that failed to start run here, serially */
    for (int32_t i = started + 1; i < n; ++i) fn((char*)jobs + job_size * (size_t)i);
    free(th);
    return ORACLE_OK;
}

/*
 * Dense float64 attention over logical K/V.
 *   kv_indptr [num_seqs+1]  token offsets of each sequence in k / v
 *   k, v      bf16 bits [total_tokens, hkv, d]   (logical order)
 *   q_indptr  [num_seqs+1]  packed query-row offsets of each sequence
 *   q_pos     [n_q]         logical position of each packed row
 *   q         bf16 bits [n_q, hq, d]
 *   rows      optional list of packed rows to evaluate (NULL = all n_q)
 *   out       [n_out, hq, d] double; lse [n_out, hq] double (natural log)
 */
int oracle_dense_attention(int32_t num_seqs, int32_t hq, int32_t hkv, int32_t d, double scale,
                           const int64_t* kv_indptr, const uint16_t* k, const uint16_t* v,
                           const int64_t* q_indptr, const int32_t* q_pos, const uint16_t* q,
                           const int64_t* rows, int64_t n_rows, double* out, double* lse,
                           int32_t num_threads) {
    if (num_seqs <= 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0) return ORACLE_ERR_ARG;
    if (!kv_indptr || !q_indptr || !q_pos || !out || !lse) return ORACLE_ERR_ARG;
    const int64_t n_out = rows ? n_rows : q_indptr[num_seqs];
    if (n_out <= 0) return ORACLE_OK;
    const int64_t n_units = n_out * hq;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > n_units) num_threads = (int32_t)n_units;
    dense_job* jobs = (dense_job*)calloc((size_t)num_threads, sizeof(dense_job));
    if (!jobs) return ORACLE_ERR_NOMEM;
    for (int32_t i = 0; i < num_threads; ++i) {
        dense_job* jb = &jobs[i];
        jb->num_seqs = num_seqs; jb->hq = hq; jb->hkv = hkv; jb->d = d; jb->scale = scale;
        jb->kv_indptr = kv_indptr; jb->k = k; jb->v = v;
        jb->q_indptr = q_indptr; jb->q_pos = q_pos; jb->q = q;
        jb->rows = rows; jb->n_rows = n_rows; jb->out = out; jb->lse = lse;
        jb->begin = n_units * i / num_threads;
        jb->end = n_units * (i + 1) / num_threads;
    }
    int rc = run_jobs(dense_worker, jobs, sizeof(dense_job), num_threads);
    for (int32_t i = 0; rc == ORACLE_OK && i < num_threads; ++i) rc = jobs[i].status;
    free(jobs);
    return rc;
}

/* ------------------------------------------------------------ segments -- */

/*
 * Segments of one sequence: maximal runs of logical blocks i..j with
 * table[b+1] == table[b] + 1, scanned left to right over the first
 * n_blocks entries.  runs[3*r + 0..2] = (first logical block, first
 * physical block, number of blocks).  Returns ORACLE_ERR_TABLE when a
 * needed entry is negative (a missing block).
 */
int oracle_segment_runs(int32_t n_blocks, const int32_t* table, int32_t* runs, int32_t* n_runs) {
    int32_t n = 0;
    int32_t b = 0;
    while (b < n_blocks) {
        if (table[b] < 0) return ORACLE_ERR_TABLE;
        int32_t e = b + 1;
        while (e < n_blocks && table[e] >= 0 && table[e] == table[e - 1] + 1) ++e;
        runs[3 * n + 0] = b;
        runs[3 * n + 1] = table[b];
        runs[3 * n + 2] = e - b;
        ++n;
        b = e;
    }
    *n_runs = n;
    return ORACLE_OK;
}

typedef struct {
    int32_t num_seqs, hq, hkv, d, block_size, max_blocks;
    double scale;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const uint16_t* k_pool;
    const uint16_t* v_pool;
    const int64_t* q_indptr;
    const int32_t* q_pos;
    const uint16_t* q;
    const int64_t* rows;
    double* out;
    double* lse;
    int64_t begin, end;
    int status;
} seg_job;

static void* seg_worker(void* arg) {
    seg_job* jb = (seg_job*)arg;
    const int32_t d = jb->d, hq = jb->hq, hkv = jb->hkv, B = jb->block_size;
    const int32_t group = hq / hkv;
    int32_t* runs = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)(jb->max_blocks > 0 ? jb->max_blocks : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)d);
    double* o_seg = (double*)malloc(sizeof(double) * (size_t)d);
    double* o_acc = (double*)malloc(sizeof(double) * (size_t)d);
    double* t = (double*)malloc(sizeof(double) * (size_t)B * (size_t)(jb->max_blocks > 0 ? jb->max_blocks : 1));
    /* per-run partials: lse_r and o_r for every run of the sequence */
    double* lse_r = (double*)malloc(sizeof(double) * (size_t)(jb->max_blocks > 0 ? jb->max_blocks : 1));
    double* o_r = (double*)malloc(sizeof(double) * (size_t)d * (size_t)(jb->max_blocks > 0 ? jb->max_blocks : 1));
    if (!runs || !qv || !o_seg || !o_acc || !t || !lse_r || !o_r) {
        jb->status = ORACLE_ERR_NOMEM;
        goto done;
    }
    jb->status = ORACLE_OK;
    for (int64_t i = jb->begin; i < jb->end; ++i) {
        const int64_t r = jb->rows ? jb->rows[i] : i;
        const int32_t s = seq_of_row(jb->q_indptr, jb->num_seqs, r);
        const int64_t len = jb->seq_lens[s];
        const int64_t p = jb->q_pos[r];
        const int32_t n_blocks = (int32_t)((len + B - 1) / B);
        int32_t n_runs = 0;
        if (oracle_segment_runs(n_blocks, jb->block_table + (int64_t)s * jb->max_blocks, runs, &n_runs) != ORACLE_OK) {
            jb->status = ORACLE_ERR_TABLE;
            goto done;
        }
        for (int32_t h = 0; h < hq; ++h) {
            const int32_t g = h / group;
            for (int32_t c = 0; c < d; ++c) qv[c] = bf16_to_double(jb->q[(r * hq + h) * (int64_t)d + c]);
            /* attention inside each segment on its own */
            int32_t n_part = 0;
            for (int32_t rr = 0; rr < n_runs; ++rr) {
                const int64_t log0 = (int64_t)runs[3 * rr + 0] * B;  /* first logical token */
                const int64_t phys0 = (int64_t)runs[3 * rr + 1] * B; /* first pool row */
                int64_t log1 = log0 + (int64_t)runs[3 * rr + 2] * B; /* one past the last */
                if (log1 > len) log1 = len;
                if (log1 > p + 1) log1 = p + 1;
                if (log1 <= log0) continue; /* nothing visible in this segment */
                double m = -INFINITY;
                for (int64_t j = log0; j < log1; ++j) {
                    const uint16_t* kj = jb->k_pool + ((phys0 + (j - log0)) * hkv + g) * (int64_t)d;
                    double acc = 0.0;
                    for (int32_t c = 0; c < d; ++c) acc += qv[c] * bf16_to_double(kj[c]);
                    t[j - log0] = jb->scale * acc;
                    if (t[j - log0] > m) m = t[j - log0];
                }
                double sum = 0.0;
                for (int64_t j = log0; j < log1; ++j) sum += exp(t[j - log0] - m);
                const double l = m + log(sum);
                for (int32_t c = 0; c < d; ++c) o_seg[c] = 0.0;
                for (int64_t j = log0; j < log1; ++j) {
                    const double w = exp(t[j - log0] - l);
                    const uint16_t* vj = jb->v_pool + ((phys0 + (j - log0)) * hkv + g) * (int64_t)d;
                    for (int32_t c = 0; c < d; ++c) o_seg[c] += w * bf16_to_double(vj[c]);
                }
                lse_r[n_part] = l;
                memcpy(o_r + (int64_t)n_part * d, o_seg, sizeof(double) * (size_t)d);
                ++n_part;
            }
            /* log-sum-exp merge of the segment partials */
            double* o = jb->out + (i * hq + h) * (int64_t)d;
            if (n_part == 0) {
                for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
                jb->lse[i * hq + h] = -INFINITY;
                continue;
            }
            double mx = -INFINITY;
            for (int32_t k = 0; k < n_part; ++k) if (lse_r[k] > mx) mx = lse_r[k];
            double sum = 0.0;
            for (int32_t k = 0; k < n_part; ++k) sum += exp(lse_r[k] - mx);
            const double LSE = mx + log(sum);
            for (int32_t c = 0; c < d; ++c) o_acc[c] = 0.0;
            for (int32_t k = 0; k < n_part; ++k) {
                const double w = exp(lse_r[k] - LSE);
                for (int32_t c = 0; c < d; ++c) o_acc[c] += w * o_r[(int64_t)k * d + c];
            }
            memcpy(o, o_acc, sizeof(double) * (size_t)d);
            jb->lse[i * hq + h] = LSE;
        }
    }
done:
    free(runs); free(qv); free(o_seg); free(o_acc); free(t); free(lse_r); free(o_r);
    return NULL;
}

/*
 * Segmented float64 attention read through the block table from the pool.
 *   block_table [num_seqs][max_blocks] int32 physical block ids (-1 = none)
 *   seq_lens    [num_seqs]             cached tokens per sequence
 *   k_pool, v_pool bf16 bits [pool_tokens, hkv, d]; pool row = block * B + offset
 * Other arguments as for oracle_dense_attention.
 */
int oracle_segmented_attention(int32_t num_seqs, int32_t hq, int32_t hkv, int32_t d,
                               int32_t block_size, double scale, int32_t max_blocks,
                               const int32_t* block_table, const int32_t* seq_lens,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               const int64_t* q_indptr, const int32_t* q_pos, const uint16_t* q,
                               const int64_t* rows, int64_t n_rows, double* out, double* lse,
                               int32_t num_threads) {
    if (num_seqs <= 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0 || block_size <= 0)
        return ORACLE_ERR_ARG;
    if (!block_table || !seq_lens || !q_indptr || !q_pos || !out || !lse) return ORACLE_ERR_ARG;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (seq_lens[s] < 0 || (seq_lens[s] + block_size - 1) / block_size > max_blocks) return ORACLE_ERR_ARG;
    const int64_t n_out = rows ? n_rows : q_indptr[num_seqs];
    if (n_out <= 0) return ORACLE_OK;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > n_out) num_threads = (int32_t)n_out;
    seg_job* jobs = (seg_job*)calloc((size_t)num_threads, sizeof(seg_job));
    if (!jobs) return ORACLE_ERR_NOMEM;
    for (int32_t i = 0; i < num_threads; ++i) {
        seg_job* jb = &jobs[i];
        jb->num_seqs = num_seqs; jb->hq = hq; jb->hkv = hkv; jb->d = d;
        jb->block_size = block_size; jb->max_blocks = max_blocks; jb->scale = scale;
        jb->block_table = block_table; jb->seq_lens = seq_lens;
        jb->k_pool = k_pool; jb->v_pool = v_pool;
        jb->q_indptr = q_indptr; jb->q_pos = q_pos; jb->q = q;
        jb->rows = rows; jb->out = out; jb->lse = lse;
        jb->begin = n_out * i / num_threads;
        jb->end = n_out * (i + 1) / num_threads;
    }
    int rc = run_jobs(seg_worker, jobs, sizeof(seg_job), num_threads);
    for (int32_t i = 0; rc == ORACLE_OK && i < num_threads; ++i) rc = jobs[i].status;
    free(jobs);
    return rc;
}

/* Scatter reference: pool[slot[t]] = rows[t] for every t with slot[t] >= 0
 * (what writing new or recomputed K/V into the paged pool means). */
int oracle_scatter_rows(int64_t n, int64_t row_elems, const uint16_t* src, const int64_t* slot,
                        uint16_t* pool, int64_t pool_rows) {
    for (int64_t t = 0; t < n; ++t) {
        if (slot[t] < 0) continue;
        if (slot[t] >= pool_rows) return ORACLE_ERR_ARG;
        memcpy(pool + slot[t] * row_elems, src + t * row_elems, sizeof(uint16_t) * (size_t)row_elems);
    }
    return ORACLE_OK;
}
