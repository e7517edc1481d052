// K4: causal GQA prefill.
#include "common.cuh"

namespace mlakv {

__device__ unsigned g_prefill_status;

cudaError_t launch_prefill(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }

int prefill_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_prefill_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
