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

    // Back to the state of a new plan, keeping the vectors' storage (see
    // plan_release).  Every field above must be reset here.
    void reset() {
        dims = msa_dims{};
        num_seqs = 0;
        G = 1;
        dec_rows = 16;
        grid = 1;
        max_pool_row = 0;
        n_dec_slots = n_pre_slots = 0;
        seq_lens.clear();
        run_indptr.clear();
        runs.clear();
        row_indptr.clear();
        pos.clear();
        groups.clear();
        items.clear();
        order.clear();
        lay = msa::WsLayout{};
        image.clear();
        workspace = nullptr;
        workspace_bytes = 0;
        info = msa_plan_info{};
    }
};
// A field added to msa_plan_s must also be reset in reset().
static_assert(sizeof(msa_plan_s) == 520, "msa_plan_s changed: update reset()");

namespace msa {

// Default split factors (a part of a split group holds about the work per
// CTA divided by these): measured on GB300, parts of about a third (decode)
// and a quarter (prefill) of a CTA's share beat finer cuts on every bench
// workload; each part costs a partial write and a share of the merge, each
// item a pipeline start and an epilogue.
constexpr double kDefaultDecodeSplit = 3.0;
constexpr double kDefaultPrefillSplit = 4.0;

// Plans are recycled per thread: plan_release keeps a destroyed plan (its
// vectors emptied but their storage kept) for the next plan_alloc on the
// same thread, so a loop that plans every step reuses memory it has already
// touched instead of faulting in fresh pages.
msa_plan_s* plan_alloc();
void plan_release(msa_plan_s* P);

// An output group before its key range is cut into work items.
struct Pending {
    Group g;
    int32_t ke;     // key range [0, ke)
    int64_t tiles;  // 128-key tiles of [0, ke)
};

// Cut every group's key range into parts and order the items (longest
// first).  A part holds about (work per CTA) / split of a group's tiles:
// `dec_split` for decode groups, `pre_split` for prefill groups.  Rebuilds
// P->groups, items, order and the partial-slot counts from scratch.
void split_items(msa_plan_s* P, const std::vector<Pending>& pend, double dec_split, double pre_split);

// Pick the split factors with the lowest expected launch time under the
// latency model (costmodel.cpp); leaves P's items unspecified.
void choose_split(msa_plan_s* P, const std::vector<Pending>& pend, const msa_cost_params& c, double* dec_split,
                  double* pre_split);

int plan_create(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks, const int32_t* table,
                const int32_t* seq_lens, const int32_t* q_range_indptr, const int32_t* q_ranges,
                int32_t num_sms, const msa_plan_options* opts, msa_plan_s** out);
void build_image(msa_plan_s* P);
int device_sm_count();

// kernel launchers (defined in the .cu files); return msa_status
int launch_append_kv(const void* k_new, const void* v_new, const int64_t* slot, int32_t n,
                     void* k_pool, void* v_pool, int64_t pool_tokens, int32_t row_elems,
                     int32_t* error_word, msa_stream_t stream);
int launch_selftest_wait(uint64_t limit_ns, int32_t* word, msa_stream_t stream);
int launch_gather_kv(const void* k_pool, const void* v_pool, int64_t pool_tokens, const int64_t* slot, int32_t n,
                     void* k_out, void* v_out, int32_t row_elems, int32_t* error_word, msa_stream_t stream);
int launch_attention(const msa_plan_s* P, const void* q, const void* k_pool, const void* v_pool,
                     int64_t pool_tokens, void* out, int32_t out_dtype, float* lse, msa_stream_t stream);
// the same launch with an explicit device workspace holding the plan image
int launch_attention_ws(const msa_plan_s* P, void* workspace, const void* q, const void* k_pool,
                        const void* v_pool, int64_t pool_tokens, void* out, int32_t out_dtype, float* lse,
                        msa_stream_t stream);

}  // namespace msa
