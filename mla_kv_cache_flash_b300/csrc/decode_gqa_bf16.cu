// K1 for bf16 caches.
#include "common.cuh"

namespace mlakv {

cudaError_t launch_decode_gqa_fma_bf16(const DecodeGqaArgs &a, cudaStream_t s);

int decode_gqa_bf16_tile_tokens(int, int) { return 128; }

cudaError_t launch_decode_gqa_bf16(const DecodeGqaArgs &a, cudaStream_t s) {
    return launch_decode_gqa_fma_bf16(a, s);
}

}  // namespace mlakv
