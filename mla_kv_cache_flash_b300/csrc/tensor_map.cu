// Host-side TMA descriptor encoding. The driver's cuTensorMapEncodeTiled is fetched through
// the runtime's entry-point query, so the library does not link libcuda and loads on hosts
// without a GPU driver.
#include "tensor_map.cuh"

#include <mutex>

namespace mlakv {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace

cudaError_t encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base,
                              const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                              CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorInitializationError;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, e,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mlakv
