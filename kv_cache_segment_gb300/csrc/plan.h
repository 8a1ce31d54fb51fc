// plan.h -- the host plan object behind msa_plan_t and the internal entry
// points between the C ABI, the planner and the kernel launchers.
#pragma once

#include <memory>
#include <vector>

#include "../../include/msa.h"
#include "msa_internal.h"

struct msa_plan_s {
    msa_dims dims{};
    int32_t num_seqs = 0;
    int32_t G = 1;         // query heads per kv head
    int32_t dec_rows = 16; // most rows a decode group can hold (16 / G)
    int32_t grid = 1;
    int64_t max_pool_row = 0;
    int32_t n_dec_slots = 0;
    int32_t n_pre_slots = 0;

    std::vector<int32_t> seq_lens;
    std::vector<int32_t> run_indptr;
    std::vector<msa::Run> runs;
    std::vector<int32_t> row_indptr;
    std::vector<int32_t> pos;
    std::vector<msa::Group> groups;
    std::vector<msa::Item> items;
    std::vector<int32_t> order;  // processing order of the items (longest first)

    msa::WsLayout lay{};
    std::vector<uint8_t> image;  // host copy of the workspace's int sections

    void* workspace = nullptr;   // set by msa_plan_upload
    size_t workspace_bytes = 0;
    msa_plan_info info{};
};

namespace msa {

int plan_create(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks, const int32_t* table,
                const int32_t* seq_lens, const int32_t* q_range_indptr, const int32_t* q_ranges,
                int32_t num_sms, msa_plan_s** out);
void build_image(msa_plan_s* P);
int device_sm_count();

// kernel launchers (defined in the .cu files); return msa_status
int launch_append_kv(const void* k_new, const void* v_new, const int64_t* slot, int32_t n,
                     void* k_pool, void* v_pool, int64_t pool_tokens, int32_t row_elems,
                     int32_t* error_word, msa_stream_t stream);
int launch_attention(const msa_plan_s* P, const void* q, const void* k_pool, const void* v_pool,
                     int64_t pool_tokens, void* out, int32_t out_dtype, float* lse, msa_stream_t stream);
// the same launch with an explicit device workspace holding the plan image
int launch_attention_ws(const msa_plan_s* P, void* workspace, const void* q, const void* k_pool,
                        const void* v_pool, int64_t pool_tokens, void* out, int32_t out_dtype, float* lse,
                        msa_stream_t stream);

}  // namespace msa
