// MLA chunked prefill on the CUDA-core decode kernel (decode_fma.cuh): key [c ‖ kr] of width
// 128 + 48, value c (qqstock MLA article, sections 2, 3 and 6), each packed new-token row a
// decode over its sequence's latent cache up to its own position. Kept in its own translation
// unit so that adding it leaves the GQA instantiations' code as it was.
#include "decode_fma.cuh"

namespace mlakv {

cudaError_t launch_prefill_chunked_mla(const DecodeGqaArgs &a, cudaStream_t s) {
    return a.D == 128 ? launch_d<__nv_bfloat16, __nv_bfloat16, 128, true, true>(a, s) : cudaErrorInvalidValue;
}

}  // namespace mlakv
