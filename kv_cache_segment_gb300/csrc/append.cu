// append.cu -- msa_append_kv: scatter new or recomputed K/V rows into the
// paged pools.  Evicted blocks are rebuilt on demand and written back into
// the pool (AsymCache explainer, "核心方法 2": a hit on an evicted block
// brings it back by recomputation; MSA paper abstract: evicted blocks are
// reconstructed to keep outputs exact), as are a new turn's tokens.
//
// HBM-bound bit copy: one warp per token row (Hkv*D*2 bytes, 128-bit loads
// and stores, fully coalesced on both sides), a grid of whole waves over the
// SMs striding through the rows.
#include <cuda_runtime.h>

#include <cstdint>

#include "msa_internal.h"
#include "plan.h"
#include "ptx.cuh"

namespace msa {

__global__ void __launch_bounds__(256) append_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                                        const int64_t* __restrict__ slot, int32_t n,
                                                        uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                        int64_t pool_tokens, int32_t row_chunks,
                                                        int32_t* error_word) {
    // Launched with programmatic stream serialization: the next kernel (the
    // step's attention launch) may start its launch and set-up now, and this
    // one touches nothing before the kernels ahead of it in the stream have
    // finished.
    ptx::pdl_trigger();
    ptx::pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n; t += warps) {
        const int64_t s = slot[t];
        if (s < 0) continue;
        if (s >= pool_tokens) {
            if (lane == 0 && error_word) atomicOr(error_word, kErrAppendSlot);
            continue;
        }
        const uint4* ks = k_new + t * row_chunks;
        const uint4* vs = v_new + t * row_chunks;
        uint4* kd = k_pool + s * row_chunks;
        uint4* vd = v_pool + s * row_chunks;
        for (int c = lane; c < row_chunks; c += 32) {
            const uint4 a = __ldcs(ks + c);
            const uint4 b = __ldcs(vs + c);
            kd[c] = a;
            vd[c] = b;
        }
    }
}

int launch_append_kv(const void* k_new, const void* v_new, const int64_t* slot, int32_t n, void* k_pool,
                     void* v_pool, int64_t pool_tokens, int32_t row_elems, int32_t* error_word,
                     msa_stream_t stream) {
    static const int sms = device_sm_count();  // grid cap only (thread-safe static)
    if (sms <= 0) return MSA_ERR_CUDA;
    const int32_t row_chunks = row_elems * 2 / 16;  // 16-byte chunks per token row
    const int warps_per_block = 8;
    int64_t blocks = ((int64_t)n + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident blocks of 256 threads per SM
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, append_kv_kernel, static_cast<const uint4*>(k_new),
                                             static_cast<const uint4*>(v_new), slot, n, static_cast<uint4*>(k_pool),
                                             static_cast<uint4*>(v_pool), pool_tokens, row_chunks, error_word);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// The transpose of the scatter: k_out[t] = k_pool[slot[t]] (and V).  It is
// the first half of the "gather + attention" path that MSA replaces
// (AsymCache explainer, "核心方法 1": without MSA, a cache whose live blocks
// are scattered goes through a gather into one contiguous buffer before a
// contiguous attention kernel); the bench times that path against MSA.
__global__ void __launch_bounds__(256) gather_kv_kernel(const uint4* __restrict__ k_pool,
                                                        const uint4* __restrict__ v_pool, int64_t pool_tokens,
                                                        const int64_t* __restrict__ slot, int32_t n,
                                                        uint4* __restrict__ k_out, uint4* __restrict__ v_out,
                                                        int32_t row_chunks, int32_t* error_word) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n; t += warps) {
        const int64_t s = slot[t];
        if (s < 0) continue;
        if (s >= pool_tokens) {
            if (lane == 0 && error_word) atomicOr(error_word, kErrAppendSlot);
            continue;
        }
        const uint4* ks = k_pool + s * row_chunks;
        const uint4* vs = v_pool + s * row_chunks;
        uint4* kd = k_out + t * row_chunks;
        uint4* vd = v_out + t * row_chunks;
        for (int c = lane; c < row_chunks; c += 32) {
            const uint4 a = __ldcs(ks + c);
            const uint4 b = __ldcs(vs + c);
            kd[c] = a;
            vd[c] = b;
        }
    }
}

int launch_gather_kv(const void* k_pool, const void* v_pool, int64_t pool_tokens, const int64_t* slot, int32_t n,
                     void* k_out, void* v_out, int32_t row_elems, int32_t* error_word, msa_stream_t stream) {
    static const int sms = device_sm_count();  // grid cap only (thread-safe static)
    if (sms <= 0) return MSA_ERR_CUDA;
    const int32_t row_chunks = row_elems * 2 / 16;
    const int warps_per_block = 8;
    int64_t blocks = ((int64_t)n + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    gather_kv_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_pool), static_cast<const uint4*>(v_pool), pool_tokens, slot, n,
        static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), row_chunks, error_word);
    return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// Self-check of the bounded waits every role of the attention kernel uses:
// warp 0 waits on an mbarrier that nothing arrives at, gives up after
// limit_ns, records the timeout bit and sets the CTA's abort flag, as a
// role of the attention kernel does; warp 1 waits on the same barrier with
// a far longer limit and must leave on the abort flag.  word[0] = error
// bits, word[1] = 1 if warp 1 left through the abort path.
__global__ void __launch_bounds__(64) selftest_wait_kernel(uint64_t limit_ns, int32_t* word) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns);
        if (!ok && threadIdx.x == 0) {
            atomicOr(word, kErrTimeoutCompute);
            *reinterpret_cast<volatile int*>(&abort_flag) = 1;
        }
    } else {
        const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns * 64);
        if (!ok && threadIdx.x == 32) word[1] = *reinterpret_cast<volatile int*>(&abort_flag) ? 1 : 0;
    }
}

int launch_selftest_wait(uint64_t limit_ns, int32_t* word, msa_stream_t stream) {
    selftest_wait_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, word);
    return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // namespace msa
