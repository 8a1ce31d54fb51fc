// tensor_maps.cpp -- TMA tensor maps of the attention launch (host only):
// the driver's encoder, looked up once, and a per-thread cache of encoded
// maps.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace msa {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (thread-safe static).
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return EncodeTiledFn(nullptr);
    }();
    return fn;
}

// 3-D bf16 map over [rows, heads, D] (innermost D), box = 64 x 1 x box_rows,
// 128-byte swizzle; rows past the end read as zero.
bool encode_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The maps a call needs are usually those of the previous calls (the same
// pools, one of a few q buffers), and encoding five of them is most of the
// host time of a small launch: keep the last few per thread, keyed by every
// input of the encoding, so a hit is the map an encode would give.
struct MapKey {
    const void* base;
    int64_t rows;
    int heads, D, box_rows;
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && heads == o.heads && D == o.D && box_rows == o.box_rows;
    }
};

}  // namespace

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows) {
    constexpr int kSlots = 12;
    thread_local MapKey keys[kSlots];
    thread_local CUtensorMap maps[kSlots];
    thread_local bool used[kSlots] = {};
    thread_local int next = 0;
    const MapKey k{base, rows, heads, D, box_rows};
    for (int i = 0; i < kSlots; ++i)
        if (used[i] && keys[i] == k) {
            *m = maps[i];
            return true;
        }
    if (!encode_map(m, base, rows, heads, D, box_rows)) return false;
    keys[next] = k;
    maps[next] = *m;
    used[next] = true;
    next = (next + 1) % kSlots;
    return true;
}

}  // namespace msa
