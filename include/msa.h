/*
 * msa.h -- C ABI of libmsa: Multi-Segment Attention (MSA) on GB300 (sm_103a).
 *
 * MSA is exact attention over a paged KV cache whose live blocks form several
 * disjoint, physically contiguous segments (AsymCache explainer, "核心方法
 * 1. Multi-Segment Attention": the live blocks are split by physical
 * contiguity, each segment is attended with a contiguous kernel and the
 * per-segment results are combined; MSA paper abstract: lossless KV
 * management must keep outputs exact, and MSA is the component that makes
 * non-contiguous context efficient).  Evicted blocks are rebuilt on demand,
 * so the queried positions can themselves be several disjoint ranges
 * (recomputed holes plus a new turn).  The result equals dense causal
 * attention over the full logical sequence:
 *
 *   for sequence s (L_s cached tokens), query row at position p, head h,
 *   kv head g = h / (Hq/Hkv), visible keys j <= min(p, L_s - 1):
 *     t_j = scale * q.K_s[j,g];  lse = ln sum_j exp(t_j);
 *     out = sum_j exp(t_j - lse) * V_s[j,g]
 *
 * Three calls make up the path:
 *   msa_plan_create / msa_plan_upload   block table + query ranges -> segment
 *                                       runs and a work list balanced over
 *                                       the SMs (host planner, one copy up)
 *   msa_append_kv                       new / recomputed K,V -> paged pool
 *   msa_attention                       one persistent launch over all
 *                                       segments of all sequences, decode
 *                                       and prefill/recompute rows alike,
 *                                       with the log-sum-exp merge fused
 *
 * Conventions
 *   - Every function returns MSA_OK (0) or a negative msa_status; no
 *     exception crosses the ABI.  msa_status_string() names a code.
 *   - Device pointers are caller-owned (e.g. torch tensors); the library
 *     never allocates device memory.  The plan is a library-owned host
 *     object; the workspace it needs is caller-allocated device memory.
 *   - Device work is asynchronous on the given stream (a cudaStream_t; NULL
 *     is the legacy default stream) and keeps stream order.  msa_append_kv
 *     and decode-only attention launches use programmatic dependent launch:
 *     such a kernel may be scheduled while the kernel before it in the stream
 *     is still running, but touches no memory until that one has completed,
 *     so stream order holds for the caller as with plain launches.
 *   - bf16 means IEEE bfloat16 (2 bytes).  Layouts are row-major, C order.
 *   - Pool layout ("NHD"): K and V pools are bf16 [pool_tokens, Hkv, D];
 *     pool row = physical_block * block_size + offset_in_block.  A segment of
 *     n blocks starting at physical block b is pool rows [b*B, (b+n)*B).
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t / CUstream without pulling in CUDA headers. */
typedef struct CUstream_st* msa_stream_t;

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad enum      */
    MSA_ERR_BAD_BLOCK_ID = -2,      /* block id >= 2^27 or past pool_tokens        */
    MSA_ERR_MISSING_BLOCK = -3,     /* negative table entry inside [0, L_s)        */
    MSA_ERR_BAD_Q_RANGE = -4,       /* empty, unsorted, overlapping, p<0 or p>L_s  */
    MSA_ERR_WORKSPACE_TOO_SMALL = -5,
    MSA_ERR_UNSUPPORTED_DIMS = -6,  /* D not in {64,128}, B != 16, Hq % Hkv != 0,  */
                                    /* Hq/Hkv > 16, non-finite or <= 0 scale       */
    MSA_ERR_CUDA = -7,              /* a CUDA runtime / driver call failed         */
    MSA_ERR_DEVICE_CHECK = -8,      /* a kernel recorded an error (see below)      */
    MSA_ERR_NOT_UPLOADED = -9       /* msa_attention before msa_plan_upload        */
} msa_status;

typedef enum { MSA_OUT_BF16 = 0, MSA_OUT_FP32 = 1 } msa_out_dtype;

/* Attention shape.  block_size must be 16; head_dim 64 or 128;
 * num_q_heads a multiple of num_kv_heads with at most 16 query heads per kv
 * head (consecutive query heads share a kv head: g = h / (Hq/Hkv)). */
typedef struct {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    float softmax_scale; /* usually 1/sqrt(head_dim) */
} msa_dims;

typedef struct msa_plan_s* msa_plan_t;

/* Summary of a plan (sizes and the algorithmic work it describes). */
typedef struct {
    int32_t num_seqs;
    int32_t num_q_rows;          /* packed query rows                            */
    int32_t num_runs;            /* segments over all sequences                  */
    int32_t num_groups;          /* output groups (merge units)                  */
    int32_t num_items;           /* work items                                   */
    int32_t num_decode_items;
    int32_t num_prefill_items;
    int32_t num_decode_rows;     /* rows served by the decode (GQA-packed) path  */
    int32_t num_prefill_rows;    /* rows served by the 128-row tile path         */
    int32_t grid;                /* CTAs of the persistent launch                */
    int64_t decode_kv_bytes;     /* K+V bytes the decode rows must read          */
    int64_t decode_qo_bytes;     /* q in + bf16 out + fp32 lse of decode rows    */
    double prefill_flops;        /* 4*D*sum over prefill (row, head) of n_vis(p) */
    int64_t max_pool_row;        /* highest pool row the plan reads, plus one    */
    double host_plan_us;         /* time msa_plan_create spent                   */
    double decode_split;         /* split factors the work items were cut with   */
    double prefill_split;        /* (see msa_plan_options)                       */
    int64_t counters_offset;     /* byte range in the workspace of the merge     */
    int64_t counters_bytes;      /* counters and the work-queue head: zero       */
                                 /* before and after every clean launch          */
} msa_plan_info;

/*
 * Build a plan (host only, no CUDA call except a device-attribute query when
 * num_sms == 0).
 *
 *   dims             attention shape (see msa_dims)
 *   num_seqs         S >= 0
 *   max_blocks_per_seq  row stride of block_table; >= ceil(L_s / 16) for all s
 *   block_table      host int32 [S][max_blocks_per_seq]: physical block of
 *                    each logical block; entries past ceil(L_s/16) ignored
 *                    (use -1); a negative entry inside [0, L_s) is
 *                    MSA_ERR_MISSING_BLOCK (evicted blocks must be recomputed
 *                    into fresh blocks before attention)
 *   seq_lens         host int32 [S]: cached tokens L_s (>= 0); only the
 *                    last logical block of a sequence may be partial
 *   q_range_indptr   host int32 [S+1]: ranges of sequence s are
 *                    q_ranges[q_range_indptr[s] .. q_range_indptr[s+1])
 *   q_ranges         host int32 [n][2]: half-open logical position ranges
 *                    [start, end), sorted and non-overlapping within a
 *                    sequence, 0 <= start < end <= L_s + 1.  A row at
 *                    p < L_s is a prefill/recompute row whose own K/V is
 *                    already in the pool (it sees keys 0..p); a row at
 *                    p == L_s is a decode row (it sees all L_s keys).
 *                    Query rows are packed in (sequence, range, position)
 *                    order: that is the row order of q, out and lse.
 *   num_sms          SMs to balance over; 0 = query the current device
 *   out              receives the plan (NULL on error)
 *
 * Segments are maximal runs of logical blocks whose physical ids rise by one
 * per block (AsymCache explainer, "核心方法 1": split the live blocks into
 * physically contiguous segments; holes break them).  The block table is
 * copied: the caller may free or change it afterwards, but a plan is only
 * valid for the table it was built from.
 */
int msa_plan_create(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                    const int32_t* block_table, const int32_t* seq_lens,
                    const int32_t* q_range_indptr, const int32_t* q_ranges, int32_t num_sms,
                    msa_plan_t* out);

/* Device workspace bytes the plan needs (work list, runs, row positions,
 * merge counters, partial-result slots).  256-byte aligned. */
int msa_plan_workspace_bytes(msa_plan_t plan, size_t* bytes);

/* Copy the plan into `workspace` (caller device memory of at least
 * msa_plan_workspace_bytes(), 256-byte aligned) on `stream` and zero its
 * counters and error word.  The plan remembers the workspace: it must stay
 * allocated, and must not be shared with another plan's upload, while
 * msa_attention calls with this plan may run.  Host memory of the plan may
 * be reused as soon as the call returns. */
int msa_plan_upload(msa_plan_t plan, void* workspace, size_t bytes, msa_stream_t stream);

/* Test / tooling introspection of the planner's segments of sequence `seq`:
 * runs[3*i + 0..2] = (first logical block, first physical block, n_blocks).
 * With runs == NULL only *n_runs is written. */
int msa_plan_get_runs(msa_plan_t plan, int32_t seq, int32_t* runs, int32_t* n_runs);

int msa_plan_get_info(msa_plan_t plan, msa_plan_info* info);

/* Host copy of the work list, for tests: items[9*i + 0..8] =
 * (kind 0=decode 1=prefill, seq, head (kv head for decode, first query
 * head for prefill), query heads covered (G for decode; for prefill 2
 * consecutive heads over at most 128 rows, or, when Hq/Hkv is odd, 1 head
 * over at most 256 rows), first packed row, number of rows, key begin, key
 * end, part).  With items == NULL only *n_items is written. */
int msa_plan_get_items(msa_plan_t plan, int32_t* items, int32_t* n_items);

/* The plan's processing order: order[q] = index (into the msa_plan_get_items
 * list) of the q-th item the persistent launch hands out.  With order ==
 * NULL only *n_items is written.  For tests and the cost model's checks. */
int msa_plan_get_order(msa_plan_t plan, int32_t* order, int32_t* n_items);

/*
 * Expected-latency model of one msa_attention launch.  AsymCache's eviction
 * and chunking decisions weigh recompute cost against hit rate using the
 * expected latency of the attention kernel (MSA paper abstract; AsymCache
 * explainer, "核心方法 2/3"); this is that model for this kernel.
 *
 * Each work item runs two phases on the CTA that takes it:
 *   fixed phase (time):
 *     decode : dec_item_us            prefill: pre_item_us + tile_us * tiles * qtiles
 *     + box_us * extra_boxes + dec_merge_us / pre_merge_us (if its group is
 *       split into parts: a decode part's partial is 16 rows, a prefill
 *       part's 128 rows x 1 or 2 heads, and the last part merges them all)
 *   stream phase (decode items only, bytes): tiles * 128 keys * D * 2 B * 2
 *     (K and V); every CTA in a stream phase progresses at
 *     min(dec_cta_gbs, dec_gbs / number of CTAs in a stream phase), so the
 *     CTAs share HBM and the last ones run faster.
 * tiles = 128-key windows the item walks; qtiles = the prefill item's query
 * tiles of 128 rows x one head (1 or 2: two heads of one kv head, or for an
 * odd Hq/Hkv one head over two consecutive row tiles); tile_us = pre_tile_us *
 * (1 - pre_tile_dfrac + pre_tile_dfrac * D / 128), the time of one (key tile x
 * query tile) at head dim D: pre_tile_us is its time at D = 128, and the share
 * pre_tile_dfrac of it (the MMAs, the K/V loads) scales with D while the rest
 * (the softmax over 128 x 128 scores) does not; extra_boxes = TMA boxes beyond one per tile (a tile that is
 * not a full 128-key window inside one segment is fetched per segment piece,
 * a piece's whole 16-key blocks in boxes of 4, 2 and 1 blocks).  Items are
 * handed out in the plan's order to `grid` CTAs, a
 * CTA taking the next one when it becomes free (several freed at once take
 * in CTA order), as the kernel's queue does.  The replay is event by event:
 * time_us = launch_us + the time the last CTA finishes.  Parameters fitted
 * on this GPU ship with the Python package
 * (kv_cache_segment_gb300/cost_params_gb300.json).
 */
typedef struct {
    double launch_us;
    double dec_item_us;
    double dec_gbs;      /* HBM bandwidth the decode streams share (GB/s)   */
    double dec_cta_gbs;  /* most one CTA streams on its own (GB/s)          */
    double pre_item_us;
    double pre_tile_us;  /* (key tile x query tile) at head dim 128 (us)       */
    double box_us;
    double dec_merge_us;
    double pre_merge_us;
    double pre_tile_dfrac; /* share of pre_tile_us proportional to D, in [0, 1] */
} msa_cost_params;

typedef struct {
    double time_us;          /* launch_us + makespan_us                       */
    double makespan_us;      /* finish time of the last CTA                   */
    double fixed_us;         /* sum of all items' fixed phases                */
    int64_t n_items;
    int64_t n_split_items;   /* items of groups split into several parts      */
    int64_t decode_tiles;    /* sum over decode items of their tiles          */
    int64_t prefill_tile_heads; /* sum over prefill items of tiles * qtiles   */
    int64_t extra_boxes;     /* see above                                     */
    int64_t stream_bytes;    /* sum of the decode items' stream phases        */
    int64_t decode_kv_bytes; /* as msa_plan_info                              */
    double prefill_flops;    /* as msa_plan_info                              */
} msa_cost_estimate;

/* Fill *est for the plan under the given parameters (host only). */
int msa_plan_estimate(msa_plan_t plan, const msa_cost_params* params, msa_cost_estimate* est);

/*
 * Kernel-aware eviction choice for one sequence (AsymCache explainer,
 * "核心方法 2": evict the blocks whose score is lowest, the score weighing
 * the block's future hit probability against its position-aware recompute
 * cost, with weights alpha and beta set from the batch and the hardware).
 * For the sequence's n_blocks = ceil(seq_len / 16) cached blocks:
 *
 *   hole(b)    = tile_us * Hq * (sum over b's positions p of
 *                min(p + 1, seq_len)) / (128 * 128)
 *     the attention work of recomputing block b's own rows (4*D*Hq*sum
 *     min(p+1, L) flops: each row attends to every earlier key) in units of
 *     one 128x128 tile of one head, at the latency model's prefill rate
 *     (tile_us as in msa_plan_estimate, at dims->head_dim).
 *
 * The page holds two views of that cost, and the mode picks one:
 *   - hole reading (default): cost_us(b) = hole(b).  Only the evicted block
 *     is rebuilt, so cost grows with position: mid- and late-sequence blocks
 *     are dear to recompute, early ones cheap (the page: recompute cost
 *     depends strongly on where the block sits).
 *   - prefix reading (mode | MSA_EVICT_PREFIX_COST): cost_us(b) = sum over
 *     b' >= b of hole(b'): a block's cache is only usable with its whole
 *     prefix, so evicting b leaves every block from b to the end to be
 *     recomputed.  Cost then falls with position and the tail blocks are the
 *     cheapest to give up (the page: tail blocks are cheap and should yield
 *     first).
 * The score is
 *   score(b)   = alpha * hit_prob[b] + beta * cost_us(b) / max_b cost_us(b)
 * or, with mode | MSA_EVICT_EXPECTED_COST,
 *   score(b)   = hit_prob[b] * cost_us(b)
 * the block's expected recompute time (alpha and beta unused): in the hole
 * reading, for a fixed number of evictions, the lowest such scores give the
 * least expected recompute time, which the pages' linear score only
 * approximates; in the prefix reading it is a per-block ranking.
 * The n_evict blocks of lowest score are written to evicted[0 .. n_evict)
 * in ascending block order; of equal scores the lower block index goes
 * first.
 *   mode       MSA_EVICT_LINEAR or MSA_EVICT_EXPECTED_COST, optionally ORed
 *              with MSA_EVICT_PREFIX_COST
 *   hit_prob   host float [n_blocks], each in [0, 1]
 *   params     latency-model constants (pre_tile_us and pre_tile_dfrac are used)
 *   evicted    host int32 [n_evict]
 *   cost_us    host double [n_blocks] or NULL: receives cost_us(b)
 * Returns MSA_ERR_INVALID_ARG for an unknown mode bit, n_evict outside [0,
 * n_blocks], a probability outside [0, 1], negative or non-finite
 * weights, or a pre_tile_dfrac outside [0, 1].
 */
typedef enum {
    MSA_EVICT_LINEAR = 0,
    MSA_EVICT_EXPECTED_COST = 1,
    MSA_EVICT_PREFIX_COST = 2
} msa_evict_mode;

int msa_select_evictions(const msa_dims* dims, int32_t seq_len, const float* hit_prob, int32_t mode, double alpha,
                         double beta, const msa_cost_params* params, int32_t n_evict, int32_t* evicted,
                         double* cost_us);

/*
 * msa_plan_create with options.  Work items: a group (decode rows of one kv
 * head, or a 128-row tile of one or two query heads) whose key range is
 * long is cut into parts of about (the launch's work per CTA) / split tiles;
 * each part is an item, and the parts are merged by log-sum-exp.  Parts
 * balance the CTAs but each costs a partial write, a merge share and a
 * pipeline start.  Adaptive chunking (AsymCache explainer, "核心方法 3"):
 * with choose_with set, the planner tries decode_split in {1, 1.5, 2, 3, 4}
 * (prefill_split held at its given or default value), then, with the best
 * of those, prefill_split in {1, 2, 4}, and keeps the plan with the lowest
 * msa_plan_estimate time under those parameters (a factor is searched only
 * when the plan has items of that kind).  msa_plan_info reports the factors
 * used.
 */
typedef struct {
    int32_t num_sms;        /* CTAs of the launch; 0 = the current device's SMs   */
    double decode_split;    /* > 0: split factor for decode groups; 0 = default 3  */
    double prefill_split;   /* > 0: split factor for prefill groups; 0 = default 4 */
    const msa_cost_params* choose_with;  /* non-NULL: choose the factors (above) */
} msa_plan_options;

int msa_plan_create_ex(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                       const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                       const int32_t* q_ranges, const msa_plan_options* opts, msa_plan_t* out);

/*
 * Adaptive prefill chunk size (AsymCache explainer, "核心方法 3": the
 * scheduler cuts pending prefill work into chunks and sizes them from how
 * busy the kernel keeps the GPU: chunks too small and launch and per-chunk
 * overheads dominate, too large and a step (and every decode request riding
 * on it) takes too long; MSA paper, methodology: a dynamic chunking
 * scheduler adapts prefill sizes to maximise hardware utilisation).
 *
 * A serving step runs the batch's other query rows (for example one decode
 * row per running sequence) together with the next c positions of every
 * pending prefill.  For each candidate c the step's plan is built with
 * msa_plan_create_ex(opts) and msa_plan_estimate(params) predicts its
 * launch time T(c); the call returns the c with the lowest predicted time
 * per prefill token, T(c) / tokens(c), among the candidates with
 * T(c) <= budget_us (budget_us <= 0: no budget).  Equal costs go to the
 * larger c; with no candidate inside the budget the smallest candidate is
 * returned and choice->within_budget is 0.
 *
 *   dims .. q_ranges   the step's batch as for msa_plan_create: block tables
 *                      and lengths of every sequence, and the query ranges of
 *                      the rows that run besides the prefill chunks.  A
 *                      pending sequence has no ranges there; its seq_lens
 *                      entry is ignored, and its block table must already
 *                      map every position below its `end`.
 *   pending[n_pending] the pending prefills: rows [start, end) of sequence
 *                      seq still to run (their K/V is appended before the
 *                      step's attention, so a chunk of c rows runs with
 *                      seq_len = start + c and rows [start, start + c)); at
 *                      most one entry per sequence
 *   opts               plan options of the step (num_sms, split factors, or
 *                      NULL for the defaults)
 *   params             latency-model constants
 *   granularity        candidate spacing in tokens (0 = 128, one query tile)
 *   max_chunk          largest chunk to consider (0 = no cap)
 *   choice             receives the chosen chunk and its prediction
 *   cand_chunk, cand_time_us   NULL, or arrays of at least 64 entries that
 *                      receive every candidate (ascending) and its T(c)
 * Candidates: the multiples of the granularity up to C = min(max_chunk,
 * largest end - start), thinned to every k-th multiple, k = ceil(multiples /
 * 63), when there are more than 63, then C itself if it is not the last
 * one; a chunk larger than a sequence's remainder runs the remainder.
 * Host only; each candidate costs one msa_plan_create_ex and one
 * msa_plan_estimate, and the candidates are evaluated on up to 8 host
 * threads (the result does not depend on how many; opts->num_sms = 0 is
 * resolved on the calling thread's current device first).  Errors: MSA_ERR_INVALID_ARG (a null pointer, a
 * sequence index out of range or listed twice, a pending sequence with rows
 * of its own, bad params), MSA_ERR_BAD_Q_RANGE (start < 0 or end <= start),
 * and whatever msa_plan_create_ex returns for a candidate's batch.
 */
typedef struct {
    int32_t seq;    /* sequence with a pending prefill                    */
    int32_t start;  /* first position still to run                        */
    int32_t end;    /* end of the pending positions (exclusive), > start  */
} msa_pending_prefill;

typedef struct {
    int32_t chunk;          /* chosen chunk size (positions per pending prefill) */
    int32_t tokens;         /* prefill rows the step runs with it                */
    double time_us;         /* predicted launch time of the step                  */
    double us_per_token;    /* time_us / tokens                                   */
    int32_t within_budget;  /* 1 if time_us <= budget_us (or no budget), else 0   */
    int32_t n_candidates;   /* candidates evaluated (<= 64)                       */
} msa_chunk_choice;

int msa_choose_prefill_chunk(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                             const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                             const int32_t* q_ranges, const msa_pending_prefill* pending, int32_t n_pending,
                             const msa_plan_options* opts, const msa_cost_params* params, double budget_us,
                             int32_t granularity, int32_t max_chunk, msa_chunk_choice* choice, int32_t* cand_chunk,
                             double* cand_time_us);

/* Free a plan (NULL is a no-op).  The host memory of up to two destroyed
 * plans is kept per calling thread and reused by that thread's next
 * msa_plan_create(_ex): a loop that plans every step then works in memory
 * it has already touched.  The workspace is the caller's and is not
 * touched. */
int msa_plan_destroy(msa_plan_t plan);

/*
 * Scatter new or recomputed K/V rows into the paged pools (evicted blocks
 * are rebuilt on demand: AsymCache explainer, "核心方法 2" and "一句话结论";
 * MSA paper abstract).  For t in [0, n):
 *     if slot_mapping[t] >= 0:  k_pool[slot_mapping[t]] = k_new[t]
 *                               v_pool[slot_mapping[t]] = v_new[t]
 * A bit copy.  Rows with slot -1 are skipped.
 *
 *   k_new, v_new    device bf16 [n, Hkv, D] (16-byte aligned)
 *   slot_mapping    device int64 [n]: pool row (block*16 + offset) or -1
 *   k_pool, v_pool  device bf16 [pool_tokens, Hkv, D] (16-byte aligned)
 * Rows move as 16-byte words: a misaligned k_new, v_new or pool pointer
 * returns MSA_ERR_INVALID_ARG before anything is launched; n == 0 is a
 * no-op.  A slot >= pool_tokens is not written; the kernel ORs MSA_DEVERR_SLOT into
 * `error_word` (device int32, may be NULL) instead.
 * Duplicate slots in one call race (one of the rows wins).
 */
int msa_append_kv(const void* k_new, const void* v_new, const int64_t* slot_mapping, int32_t n,
                  void* k_pool, void* v_pool, int64_t pool_tokens, const msa_dims* dims,
                  int32_t* error_word, msa_stream_t stream);

/*
 * Self-check of the bounded waits (for tests; the paper has no counterpart).
 * Every wait in the attention kernel gives up after a time limit, records a
 * bit in the error word, raises the CTA's abort flag (so the CTA's other
 * waiters leave at once) and returns, leaving the context usable.  This
 * launches one CTA that does exactly that on an mbarrier nothing arrives
 * at: a first waiter gives up after limit_ns (1 ns .. 10 s) and ORs
 * MSA_DEVERR_TIMEOUT_COMPUTE into device_words[0]; a second waiter, with a
 * limit 64 times longer, must leave through the abort flag and sets
 * device_words[1] = 1.  device_words: device int32 [2], zeroed by the
 * caller.
 */
int msa_selftest_wait_timeout(uint64_t limit_ns, int32_t* device_words, msa_stream_t stream);

/*
 * Gather K/V rows out of the paged pools (the transpose of msa_append_kv):
 * for t in [0, n), if 0 <= slot_mapping[t] < pool_tokens,
 *     k_out[t] = k_pool[slot_mapping[t]],  v_out[t] = v_pool[slot_mapping[t]]
 * (rows of Hkv*D bf16); slot -1 leaves row t untouched.  This is the first
 * half of the "gather + attention" path that MSA makes unnecessary
 * (AsymCache explainer, "核心方法 1"); the bench times that path against
 * msa_attention on the segmented layout.
 *   k_pool, v_pool  device bf16 [pool_tokens, Hkv, D] (16-byte aligned)
 *   slot_mapping    device int64 [n]
 *   k_out, v_out    device bf16 [n, Hkv, D] (16-byte aligned, caller-owned)
 * A slot >= pool_tokens is skipped; the kernel ORs MSA_DEVERR_SLOT into
 * `error_word` (device int32, may be NULL).
 */
int msa_gather_kv(const void* k_pool, const void* v_pool, int64_t pool_tokens, const int64_t* slot_mapping,
                  int32_t n, void* k_out, void* v_out, const msa_dims* dims, int32_t* error_word,
                  msa_stream_t stream);

/*
 * Attention of every query row of the plan, one persistent launch.
 *
 *   q            device bf16 [n_q, Hq, D], rows in the plan's packed order
 *                (16-byte aligned)
 *   k_pool, v_pool  device bf16 [pool_tokens, Hkv, D] (16-byte aligned)
 *   pool_tokens  rows in each pool: below the highest row the plan reads
 *                returns MSA_ERR_BAD_BLOCK_ID, above 2^31 - 1 (the TMA's
 *                32-bit row coordinate) MSA_ERR_INVALID_ARG
 *   plan         an uploaded plan
 *   out          device [n_q, Hq, D], bf16 or fp32 per out_dtype (16-byte
 *                aligned); a misaligned q, pool or out pointer returns
 *                MSA_ERR_INVALID_ARG before anything is launched
 *   lse          device fp32 [n_q, Hq] (natural log of the sum of
 *                exp(scaled scores)), or NULL
 *   stream       CUDA stream
 *
 * Decode rows (a sequence's trailing rows when they number at most 16/G)
 * are served GQA-packed: one work item reads a K/V chunk of one kv head
 * once for all G query heads.  Other rows go in tiles of 128 rows per
 * query head on the tensor cores, two tiles sharing each K/V chunk (two
 * heads of a kv head, or for odd Hq/Hkv two row tiles of one head).  Items whose sequence was split for SM
 * balance write partial (output, lse) pairs to the workspace; the last item
 * of a group to finish merges them by log-sum-exp and writes out/lse.
 * A kernel that hits an internal time limit or a bad index records a code
 * in the workspace's error word and returns; msa_plan_check_device() reads
 * it.  Calls with the same plan/workspace must not overlap on the GPU.
 */
int msa_attention(const void* q, const void* k_pool, const void* v_pool, int64_t pool_tokens,
                  msa_plan_t plan, void* out, int32_t out_dtype, float* lse, msa_stream_t stream);

/*
 * msa_attention for callers that cannot allocate device memory.  The paper
 * has no counterpart; this is a deployment convenience.  Some callers may not
 * call cudaMalloc or an allocator at all: code that runs inside a
 * pre-planned memory budget (a serving engine whose device memory is fully
 * carved up at start-up), a host thread that must not synchronise with the
 * device the way a first allocation can, or a plug-in that has no handle on
 * the host framework's allocator.  This entry point needs no workspace from
 * them.
 *
 * Same arguments, results and error codes as msa_attention, except that the
 * plan does not have to be uploaded: each call copies the plan's work list
 * into a library-owned device array of 32 MiB (held by every GPU that loads
 * the library, until the process exits) and zeroes its counters there, in
 * stream order, then launches the same kernel.  A plan whose workspace
 * (msa_plan_workspace_bytes) exceeds 32 MiB is rejected with
 * MSA_ERR_WORKSPACE_TOO_SMALL.  No device memory is allocated or freed.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array: calls that overlap on the GPU
 * (other streams, other host threads) race and corrupt each other's results;
 * serialise them.  The kernel's error word (timeouts, bad indices) lives in
 * the same array: msa_plan_check_device does not see it;
 * msa_no_alloc_check_device does.
 */
int msa_attention_no_alloc(const void* q, const void* k_pool, const void* v_pool, int64_t pool_tokens,
                           msa_plan_t plan, void* out, int32_t out_dtype, float* lse, msa_stream_t stream);

/*
 * The error check of msa_attention_no_alloc (the paper has no counterpart).
 * Synchronises `stream`, reads the error word of the library-owned array
 * (the MSA_DEVERR_* bits a kernel of the last msa_attention_no_alloc call on
 * this device recorded) into `detail` (may be NULL), and returns
 * MSA_ERR_DEVICE_CHECK after clearing it if it is nonzero, else MSA_OK.  Call
 * it after the no-alloc call it should check and before the next one: every
 * call starts by clearing the word.  Allocates nothing.
 */
int msa_no_alloc_check_device(msa_stream_t stream, int32_t* detail);

/*
 * For tests of msa_no_alloc_check_device: ORs `bits` into that error word on
 * `stream` (a one-thread kernel), as a kernel that gave up would.
 */
int msa_no_alloc_inject_error(int32_t bits, msa_stream_t stream);

/* Bits of a device error word (msa_plan_check_device's `detail`, the
 * error_word of msa_append_kv / msa_gather_kv): a wait in a role of the
 * attention kernel ran out of time (producer, MMA, compute), a plan index
 * out of range, a slot past the pool, a failed TMEM allocation. */
enum {
    MSA_DEVERR_TIMEOUT_PRODUCER = 1 << 0,
    MSA_DEVERR_TIMEOUT_MMA = 1 << 1,
    MSA_DEVERR_TIMEOUT_COMPUTE = 1 << 2,
    MSA_DEVERR_BAD_INDEX = 1 << 3,
    MSA_DEVERR_SLOT = 1 << 4,
    MSA_DEVERR_TMEM_ALLOC = 1 << 5
};

/* Synchronise `stream`, read the workspace's error word and return
 * MSA_ERR_DEVICE_CHECK if a kernel recorded an error, else MSA_OK.  `detail`
 * (may be NULL) receives the raw error word.  On an error the word is
 * cleared, and so are the merge counters and the work-queue head: a launch
 * that gave up can leave them mid-count, and the next msa_attention with this
 * plan would otherwise merge split groups wrongly.  After MSA_OK nothing is
 * written (the kernel leaves them zeroed itself). */
int msa_plan_check_device(msa_plan_t plan, msa_stream_t stream, int32_t* detail);

const char* msa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
