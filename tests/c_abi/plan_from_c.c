/* A plain C11 caller of libmsa (no C++, no torch): host-only calls of the
 * ABI in include/msa.h.  Prints one line of results for the Python test to
 * check; exits non-zero on any unexpected status. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "msa.h"

#define CHECK(x)                                                            \
    do {                                                                    \
        int rc_ = (x);                                                      \
        if (rc_ != MSA_OK) {                                                \
            fprintf(stderr, "%s -> %s\n", #x, msa_status_string(rc_));      \
            return 1;                                                       \
        }                                                                   \
    } while (0)

int main(void) {
    /* two sequences: 40 tokens in segments of blocks {0,1} and {7}; 20
     * tokens in block {3}; queries: rows [30, 41) of seq 0, a decode row of seq 1 */
    const msa_dims dims = {8, 2, 128, 16, 0.08838834764831845f};
    const int32_t table[2][3] = {{10, 11, 17}, {3, 4, -1}};
    const int32_t lens[2] = {40, 20};
    const int32_t indptr[3] = {0, 1, 2};
    const int32_t ranges[2][2] = {{30, 41}, {20, 21}};
    msa_plan_t plan = NULL;
    CHECK(msa_plan_create(&dims, 2, 3, &table[0][0], lens, indptr, &ranges[0][0], 4, &plan));
    msa_plan_info info;
    memset(&info, 0, sizeof info);
    CHECK(msa_plan_get_info(plan, &info));
    int32_t runs[3 * 8], n_runs = 0;
    CHECK(msa_plan_get_runs(plan, 0, runs, &n_runs));
    int32_t n_items = 0;
    CHECK(msa_plan_get_items(plan, NULL, &n_items));
    size_t ws = 0;
    CHECK(msa_plan_workspace_bytes(plan, &ws));
    /* the last field, the share of a tile's time proportional to the head dim,
     * changes nothing at D = 128 */
    const msa_cost_params prm = {10.0, 2.0, 6000.0, 50.0, 5.0, 1.0, 0.0, 1.0, 40.0, 0.5};
    msa_cost_estimate est;
    CHECK(msa_plan_estimate(plan, &prm, &est));
    const float hit[3] = {0.9f, 0.1f, 0.5f};
    int32_t evicted[1] = {-1};
    double cost[3];
    CHECK(msa_select_evictions(&dims, 40, hit, MSA_EVICT_LINEAR, 1.0, 0.0, &prm, 1, evicted, cost));
    /* prefix reading: a block costs its own rows and every row after it */
    int32_t evicted_prefix[1] = {-1};
    double cost_prefix[3];
    CHECK(msa_select_evictions(&dims, 40, hit, MSA_EVICT_LINEAR | MSA_EVICT_PREFIX_COST, 0.0, 1.0, &prm, 1,
                               evicted_prefix, cost_prefix));
    /* chunk size for a step of one decode row (seq 0, 40 tokens) and a
     * pending prefill of positions [0, 300) of seq 1 (19 blocks mapped) */
    static int32_t table2[2][19];
    for (int b = 0; b < 19; ++b) {
        table2[0][b] = b < 3 ? b : -1;
        table2[1][b] = 32 + b;
    }
    const int32_t lens2[2] = {40, 0};
    const int32_t indptr2[3] = {0, 1, 1};
    const int32_t ranges2[1][2] = {{39, 40}};
    const msa_pending_prefill pend = {1, 0, 300};
    const msa_plan_options opts = {152, 0.0, 0.0, NULL};
    msa_chunk_choice ch, ch_tight;
    int32_t cand[64];
    double cand_us[64];
    CHECK(msa_choose_prefill_chunk(&dims, 2, 19, &table2[0][0], lens2, indptr2, &ranges2[0][0], &pend, 1, &opts,
                                   &prm, 0.0, 0, 0, &ch, cand, cand_us));
    CHECK(msa_choose_prefill_chunk(&dims, 2, 19, &table2[0][0], lens2, indptr2, &ranges2[0][0], &pend, 1, &opts,
                                   &prm, 0.5 * cand_us[0], 0, 0, &ch_tight, NULL, NULL));
    /* an attention call before any upload is refused before any device work */
    const int not_up = msa_attention((const void*)0x1000, (const void*)0x1000, (const void*)0x1000, 64, plan,
                                     (void*)0x1000, MSA_OUT_BF16, NULL, NULL);
    CHECK(msa_plan_destroy(plan));
    printf("rows %d runs %d run0 %d %d %d run1 %d %d %d items %d ws_ok %d est_items %lld evict %d cost_rising %d "
           "not_uploaded %s cost %.17g %.17g %.17g\n",
           info.num_q_rows, n_runs, runs[0], runs[1], runs[2], runs[3], runs[4], runs[5], n_items, ws > 0,
           (long long)est.n_items, evicted[0], cost[1] > cost[0], msa_status_string(not_up), cost[0], cost[1],
           cost[2]);
    printf("evict_prefix %d cost_prefix %.17g %.17g %.17g\n", evicted_prefix[0], cost_prefix[0], cost_prefix[1],
           cost_prefix[2]);
    printf("chunk %d tokens %d within %d ncand %d time %.17g upt %.17g tight_chunk %d tight_within %d cands",
           ch.chunk, ch.tokens, ch.within_budget, ch.n_candidates, ch.time_us, ch.us_per_token, ch_tight.chunk,
           ch_tight.within_budget);
    for (int i = 0; i < ch.n_candidates; ++i) printf(" %d %.17g", cand[i], cand_us[i]);
    printf("\n");
    return 0;
}
