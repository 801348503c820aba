// tmap.cu -- TMA tensor-map encoding for the kernels' global operands.
//
// cuTensorMapEncodeTiled is reached through the runtime's driver entry point,
// so the library does not link libcuda directly.  Encoded maps are cached by
// their full description (base address, shape, strides, box, swizzle): a
// decode loop that calls the GEMM with the same weights and activation buffers
// pays the encoding once.
#include <map>
#include <mutex>
#include <string.h>
#include <tuple>

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

using Key = std::tuple<uintptr_t, int, uint64_t, uint64_t, uint64_t, uint32_t, uint32_t, int>;

}  // namespace

bool make_tmap_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    static std::mutex mu;
    static std::map<Key, CUtensorMap> cache;
    const Key key{(uintptr_t)base, (int)dtype, inner, outer, row_stride_bytes, box_inner,
                  box_outer, (int)swizzle};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            return true;
        }
    }
    EncodeFn fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    CUtensorMap m;
    memset(&m, 0, sizeof m);
    const CUresult r = fn(&m, dtype, 2, const_cast<void *>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() > 4096) cache.clear();
    cache[key] = m;
    *out = m;
    return true;
}

}  // namespace w4a16
