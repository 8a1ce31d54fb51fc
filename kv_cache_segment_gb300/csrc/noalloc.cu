// noalloc.cu -- msa_attention_no_alloc: msa_attention for callers that can
// not allocate device memory (see include/msa.h).  The workspace the plan
// needs (work list, segment runs, merge counters, partial-result slots)
// lives in one library-owned device array instead of caller memory.
#include <cuda_runtime.h>

#include <mutex>

#include "plan.h"

namespace msa {
namespace {

// 32 MiB per GPU that loads the library, held until the process exits.
constexpr size_t kNoAllocWorkspaceBytes = size_t(32) << 20;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol: its device address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the first call on each device does it).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_ws) != cudaSuccess || !ptr) return MSA_ERR_CUDA;
        g_addr[dev] = ptr;
    }
    *out = g_addr[dev];
    return MSA_OK;
}

}  // namespace
}  // namespace msa

namespace msa {
namespace {
__global__ void or_error_word_kernel(int32_t* word, int32_t bits) { atomicOr(word, bits); }
}  // namespace
}  // namespace msa

// The planner lays the error word out first (byte 0 of every workspace), so
// it sits at byte 0 of the shared array whichever plan used it last;
// msa_attention_no_alloc refuses a layout where it does not.

extern "C" int msa_no_alloc_check_device(msa_stream_t stream, int32_t* detail) {
    using namespace msa;
    void* ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc != MSA_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
    if (detail) *detail = word;
    if (word == 0) return MSA_OK;
    if (cudaMemset(ws, 0, sizeof word) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return MSA_ERR_CUDA;
    return MSA_ERR_DEVICE_CHECK;
}

extern "C" int msa_no_alloc_inject_error(int32_t bits, msa_stream_t stream) {
    using namespace msa;
    void* ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc != MSA_OK) return rc;
    or_error_word_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int32_t*>(ws), bits);
    return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" int msa_attention_no_alloc(const void* q, const void* k_pool, const void* v_pool, int64_t pool_tokens,
                                      msa_plan_t plan, void* out, int32_t out_dtype, float* lse,
                                      msa_stream_t stream) {
    using namespace msa;
    if (!plan) return MSA_ERR_INVALID_ARG;
    if (out_dtype != MSA_OUT_BF16 && out_dtype != MSA_OUT_FP32) return MSA_ERR_INVALID_ARG;
    if (plan->lay.total > kNoAllocWorkspaceBytes) return MSA_ERR_WORKSPACE_TOO_SMALL;
    if (plan->lay.error != 0) return MSA_ERR_INVALID_ARG;
    if (plan->info.num_q_rows == 0) return MSA_OK;
    if (!q || !k_pool || !v_pool || !out) return MSA_ERR_INVALID_ARG;
    for (const void* p : {q, k_pool, v_pool, (const void*)out})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return MSA_ERR_INVALID_ARG;
    if (pool_tokens < plan->max_pool_row) return MSA_ERR_BAD_BLOCK_ID;
    if (pool_tokens > (int64_t)INT32_MAX) return MSA_ERR_INVALID_ARG;
    void* ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc != MSA_OK) return rc;
    // Every call shares the array and it keeps the previous call's contents:
    // copy this plan's work list in and zero the error word and the merge
    // counters before the launch, all in stream order.
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const WsLayout& W = plan->lay;
    uint8_t* base = static_cast<uint8_t*>(ws);
    if (cudaMemcpyAsync(base, plan->image.data(), W.image_end, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (W.counters_end > W.counters &&
        cudaMemsetAsync(base + W.counters, 0, W.counters_end - W.counters, st) != cudaSuccess)
        return MSA_ERR_CUDA;
    return launch_attention_ws(plan, ws, q, k_pool, v_pool, pool_tokens, out, out_dtype, lse, stream);
}
