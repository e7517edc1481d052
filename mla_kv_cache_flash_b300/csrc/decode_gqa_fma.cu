// The CUDA-core decode kernel's instantiations for GQA decode over fp32 and E4M3 caches and
// for GQA chunked prefill over fp32 and bf16 caches (the kernel itself: decode_fma.cuh). The
// MLA chunked prefill instantiates the same template in its own translation unit.
#include "decode_fma.cuh"

namespace mlakv {

cudaError_t launch_decode_gqa_f32(const DecodeGqaArgs &a, cudaStream_t s) {
    return a.cu_q ? launch_t<float, float, true>(a, s) : launch_t<float, float, false>(a, s);
}
cudaError_t launch_decode_gqa_fp8(const DecodeGqaArgs &a, cudaStream_t s) {
    return launch_t<__nv_bfloat16, uint8_t, false>(a, s);
}
cudaError_t launch_prefill_chunked_bf16(const DecodeGqaArgs &a, cudaStream_t s) {
    return launch_t<__nv_bfloat16, __nv_bfloat16, true>(a, s);
}

}  // namespace mlakv
