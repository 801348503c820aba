// tmap.cu -- TMA tensor-map encoding for the kernels' global operands.
//
// cuTensorMapEncodeTiled is reached through the runtime's driver entry point,
// so the library does not link libcuda directly.  Encoded maps are cached by
// their full description (base address, shape, strides, box, swizzle): a
// decode loop that calls the GEMM with the same weights and activation buffers
// pays the encoding once.  Lookups go first to a small direct-mapped cache
// private to the calling thread (no lock, one hash and one key compare), then
// to the process-wide map under its lock.
#include <array>
#include <map>
#include <mutex>
#include <string.h>

#include "tmap.cuh"

namespace w4a16 {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
        cudaGetLastError();
    });
    return fn;
}

}  // namespace

bool make_tmap(CUtensorMap *out, CUtensorMapDataType dtype, int rank, const void *base,
               const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
               CUtensorMapSwizzle swizzle) {
    if (rank < 1 || rank > 3) return false;
    // cache key: every field of the description, packed into one array
    std::array<uint64_t, 13> key{};
    key[0] = (uintptr_t)base;
    key[1] = ((uint64_t)dtype << 32) | ((uint64_t)rank << 8) | (uint64_t)swizzle;
    for (int i = 0; i < rank; ++i) {
        key[2 + i] = dims[i];
        key[5 + i] = box[i];
        if (i + 1 < rank) key[8 + i] = strides_bytes[i];
    }
    // thread-private direct-mapped front cache
    struct Front {
        std::array<uint64_t, 13> key;
        CUtensorMap map;
        bool valid;
    };
    constexpr int kFront = 64;
    static thread_local Front front[kFront];
    uint64_t h = 0x9E3779B97F4A7C15ull;
    for (uint64_t v : key) h = (h ^ v) * 0x100000001B3ull;
    Front &f = front[(h >> 32) & (kFront - 1)];
    if (f.valid && f.key == key) {
        *out = f.map;
        return true;
    }
    static std::mutex mu;
    static std::map<std::array<uint64_t, 13>, CUtensorMap> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            f.key = key;
            f.map = it->second;
            f.valid = true;
            return true;
        }
    }
    EncodeFn fn = encoder();
    if (!fn) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    CUtensorMap m;
    memset(&m, 0, sizeof m);
    const CUresult r = fn(&m, dtype, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() > 4096) cache.clear();
        cache[key] = m;
    }
    f.key = key;
    f.map = m;
    f.valid = true;
    *out = m;
    return true;
}

bool make_tmap_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    const uint64_t dims[2] = {inner, outer};
    const uint32_t box[2] = {box_inner, box_outer};
    return make_tmap(out, dtype, 2, base, dims, &row_stride_bytes, box, swizzle);
}

}  // namespace w4a16
