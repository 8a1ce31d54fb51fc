// capi.cpp -- the extern "C" entry points of libmsa (declared in
// include/msa.h): argument checks, plan lifetime, workspace upload, and
// dispatch to the planner and the kernel launchers.
#include <cuda_runtime.h>

#include <cstring>

#include "plan.h"

using msa::WsLayout;

namespace msa {

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

}  // namespace msa

constexpr bool same_bit(int a, int b) { return a == b; }
static_assert(same_bit(msa::kErrTimeoutProducer, MSA_DEVERR_TIMEOUT_PRODUCER) &&
                  same_bit(msa::kErrTimeoutMma, MSA_DEVERR_TIMEOUT_MMA) &&
                  same_bit(msa::kErrTimeoutCompute, MSA_DEVERR_TIMEOUT_COMPUTE) &&
                  same_bit(msa::kErrBadIndex, MSA_DEVERR_BAD_INDEX) && same_bit(msa::kErrAppendSlot, MSA_DEVERR_SLOT) &&
                  same_bit(msa::kErrTmemAlloc, MSA_DEVERR_TMEM_ALLOC),
              "device error bits must match msa.h");

extern "C" {

int msa_plan_create(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                    const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                    const int32_t* q_ranges, int32_t num_sms, msa_plan_t* out) {
    try {
        return msa::plan_create(dims, num_seqs, max_blocks_per_seq, block_table, seq_lens, q_range_indptr,
                                q_ranges, num_sms, nullptr, out);
    } catch (...) {
        if (out) *out = nullptr;
        return MSA_ERR_INVALID_ARG;
    }
}

int msa_plan_create_ex(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                       const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                       const int32_t* q_ranges, const msa_plan_options* opts, msa_plan_t* out) {
    try {
        return msa::plan_create(dims, num_seqs, max_blocks_per_seq, block_table, seq_lens, q_range_indptr,
                                q_ranges, opts ? opts->num_sms : 0, opts, out);
    } catch (...) {
        if (out) *out = nullptr;
        return MSA_ERR_INVALID_ARG;
    }
}

int msa_plan_workspace_bytes(msa_plan_t plan, size_t* bytes) {
    if (!plan || !bytes) return MSA_ERR_INVALID_ARG;
    *bytes = plan->lay.total;
    return MSA_OK;
}

int msa_plan_upload(msa_plan_t plan, void* workspace, size_t bytes, msa_stream_t stream) {
    if (!plan || !workspace) return MSA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MSA_ERR_INVALID_ARG;
    if (bytes < plan->lay.total) return MSA_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const WsLayout& W = plan->lay;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // error word + everything up to the counters: copy the host image, then
    // zero the merge counters.
    if (cudaMemcpyAsync(ws, plan->image.data(), W.image_end, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (W.counters_end > W.counters &&
        cudaMemsetAsync(ws + W.counters, 0, W.counters_end - W.counters, st) != cudaSuccess)
        return MSA_ERR_CUDA;
    plan->workspace = workspace;
    plan->workspace_bytes = bytes;
    return MSA_OK;
}

int msa_plan_get_runs(msa_plan_t plan, int32_t seq, int32_t* runs, int32_t* n_runs) {
    if (!plan || !n_runs || seq < 0 || seq >= plan->num_seqs) return MSA_ERR_INVALID_ARG;
    const int32_t a = plan->run_indptr[seq], b = plan->run_indptr[seq + 1];
    *n_runs = b - a;
    if (runs) {
        for (int32_t i = a; i < b; ++i) {
            const msa::Run& r = plan->runs[i];
            runs[3 * (i - a) + 0] = r.log_start / msa::kBlock;
            runs[3 * (i - a) + 1] = r.phys_row / msa::kBlock;
            runs[3 * (i - a) + 2] = (r.n_tok + msa::kBlock - 1) / msa::kBlock;
        }
    }
    return MSA_OK;
}

int msa_plan_get_info(msa_plan_t plan, msa_plan_info* info) {
    if (!plan || !info) return MSA_ERR_INVALID_ARG;
    *info = plan->info;
    return MSA_OK;
}

int msa_plan_get_items(msa_plan_t plan, int32_t* items, int32_t* n_items) {
    if (!plan || !n_items) return MSA_ERR_INVALID_ARG;
    *n_items = (int32_t)plan->items.size();
    if (items) {
        for (size_t i = 0; i < plan->items.size(); ++i) {
            const msa::Item& it = plan->items[i];
            const msa::Group& g = plan->groups[it.group];
            int32_t* o = items + 9 * i;
            // query heads covered: G (decode); prefill: 2 over <= 128 rows, or
            // 1 over up to 256 rows (the last query head of a kv head, odd G)
            const int32_t heads =
                g.kind == msa::kPrefill && !(g.pad == 2 && g.nrows <= msa::kTileRows) ? 1 : g.pad;
            o[0] = g.kind; o[1] = g.seq; o[2] = g.head; o[3] = heads; o[4] = g.row0;
            o[5] = g.nrows; o[6] = it.kb; o[7] = it.ke; o[8] = it.part;
        }
    }
    return MSA_OK;
}

int msa_plan_destroy(msa_plan_t plan) {
    msa::plan_release(plan);
    return MSA_OK;
}

int msa_append_kv(const void* k_new, const void* v_new, const int64_t* slot_mapping, int32_t n,
                  void* k_pool, void* v_pool, int64_t pool_tokens, const msa_dims* dims,
                  int32_t* error_word, msa_stream_t stream) {
    if (!dims || n < 0 || pool_tokens < 0) return MSA_ERR_INVALID_ARG;
    if (dims->num_kv_heads <= 0 || (dims->head_dim != 64 && dims->head_dim != 128))
        return MSA_ERR_UNSUPPORTED_DIMS;
    if (n == 0) return MSA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return MSA_ERR_INVALID_ARG;
    for (const void* p : {k_new, v_new, (const void*)k_pool, (const void*)v_pool})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return MSA_ERR_INVALID_ARG;
    return msa::launch_append_kv(k_new, v_new, slot_mapping, n, k_pool, v_pool, pool_tokens,
                                 dims->num_kv_heads * dims->head_dim, error_word, stream);
}

int msa_selftest_wait_timeout(uint64_t limit_ns, int32_t* device_words, msa_stream_t stream) {
    if (!device_words || limit_ns == 0 || limit_ns > 10000000000ull) return MSA_ERR_INVALID_ARG;
    return msa::launch_selftest_wait(limit_ns, device_words, stream);
}

int msa_gather_kv(const void* k_pool, const void* v_pool, int64_t pool_tokens, const int64_t* slot_mapping,
                  int32_t n, void* k_out, void* v_out, const msa_dims* dims, int32_t* error_word,
                  msa_stream_t stream) {
    if (!dims || n < 0 || pool_tokens < 0) return MSA_ERR_INVALID_ARG;
    if (dims->num_kv_heads <= 0 || (dims->head_dim != 64 && dims->head_dim != 128))
        return MSA_ERR_UNSUPPORTED_DIMS;
    if (n == 0) return MSA_OK;
    if (!k_out || !v_out || !slot_mapping || !k_pool || !v_pool) return MSA_ERR_INVALID_ARG;
    for (const void* p : {(const void*)k_out, (const void*)v_out, k_pool, v_pool})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return MSA_ERR_INVALID_ARG;
    return msa::launch_gather_kv(k_pool, v_pool, pool_tokens, slot_mapping, n, k_out, v_out,
                                 dims->num_kv_heads * dims->head_dim, error_word, stream);
}

int msa_attention(const void* q, const void* k_pool, const void* v_pool, int64_t pool_tokens,
                  msa_plan_t plan, void* out, int32_t out_dtype, float* lse, msa_stream_t stream) {
    if (!plan) return MSA_ERR_INVALID_ARG;
    if (!plan->workspace) return MSA_ERR_NOT_UPLOADED;
    if (out_dtype != MSA_OUT_BF16 && out_dtype != MSA_OUT_FP32) return MSA_ERR_INVALID_ARG;
    if (plan->info.num_q_rows == 0) return MSA_OK;
    if (!q || !k_pool || !v_pool || !out) return MSA_ERR_INVALID_ARG;
    for (const void* p : {q, k_pool, v_pool, (const void*)out})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return MSA_ERR_INVALID_ARG;
    if (pool_tokens < plan->max_pool_row) return MSA_ERR_BAD_BLOCK_ID;
    if (pool_tokens > (int64_t)INT32_MAX) return MSA_ERR_INVALID_ARG;
    return msa::launch_attention(plan, q, k_pool, v_pool, pool_tokens, out, out_dtype, lse, stream);
}

int msa_plan_check_device(msa_plan_t plan, msa_stream_t stream, int32_t* detail) {
    if (!plan) return MSA_ERR_INVALID_ARG;
    if (!plan->workspace) return MSA_ERR_NOT_UPLOADED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, static_cast<uint8_t*>(plan->workspace) + plan->lay.error, sizeof word,
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (detail) *detail = word;
    if (word != 0) {
        // A launch that gave up may have left merge counters of groups whose
        // parts had only partly arrived (and the queue head) nonzero; the next
        // launch would then pick the wrong last part.  Zero them with the word.
        uint8_t* ws = static_cast<uint8_t*>(plan->workspace);
        const WsLayout& W = plan->lay;
        if (cudaMemset(ws + W.error, 0, sizeof word) != cudaSuccess) return MSA_ERR_CUDA;
        if (W.counters_end > W.counters && cudaMemset(ws + W.counters, 0, W.counters_end - W.counters) != cudaSuccess)
            return MSA_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return MSA_ERR_CUDA;
        return MSA_ERR_DEVICE_CHECK;
    }
    return MSA_OK;
}

const char* msa_status_string(int status) {
    switch (status) {
        case MSA_OK: return "MSA_OK";
        case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
        case MSA_ERR_BAD_BLOCK_ID: return "MSA_ERR_BAD_BLOCK_ID";
        case MSA_ERR_MISSING_BLOCK: return "MSA_ERR_MISSING_BLOCK";
        case MSA_ERR_BAD_Q_RANGE: return "MSA_ERR_BAD_Q_RANGE";
        case MSA_ERR_WORKSPACE_TOO_SMALL: return "MSA_ERR_WORKSPACE_TOO_SMALL";
        case MSA_ERR_UNSUPPORTED_DIMS: return "MSA_ERR_UNSUPPORTED_DIMS";
        case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
        case MSA_ERR_DEVICE_CHECK: return "MSA_ERR_DEVICE_CHECK";
        case MSA_ERR_NOT_UPLOADED: return "MSA_ERR_NOT_UPLOADED";
        default: return "MSA_ERR_UNKNOWN";
    }
}

}  // extern "C"
