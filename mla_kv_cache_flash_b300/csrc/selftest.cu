// attn_selftest_bounded_wait: exercises the library's failure path for a wait that never ends.
//
// Every mbarrier wait in the library's kernels is bounded: when it runs out it records a bit
// in a device status word and the kernel returns, so the GPU context stays usable and
// attn_check_status reports ATTN_ERR_TIMEOUT on the host. This entry point makes such a wait
// run out on purpose, safely: one thread initialises an mbarrier that nothing ever arrives on
// and waits on it with a short, caller-given bound. No memory is touched outside the block's
// shared memory and its own status word, and the kernel always ends.
#include "../../include/mlakv.h"
#include "ptx.cuh"

#include <stdio.h>

namespace mlakv {

__device__ unsigned g_selftest_status;

namespace {

__global__ void bounded_wait_kernel(long long timeout_cycles) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    // phase 0 never completes: the wait gives up after timeout_cycles and records the bit
    mbar_wait_bounded(b, 0, &g_selftest_status, kStatusSelfTest, timeout_cycles);
}

}  // namespace

int selftest_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_selftest_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_selftest_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv

extern "C" __attribute__((visibility("default"))) int attn_selftest_bounded_wait(long long timeout_cycles,
                                                                               mlakv_stream_t stream) {
    using namespace mlakv;
    if (timeout_cycles < 1000 || timeout_cycles > 1000000000LL)
        return report_error(ATTN_ERR_SHAPE, "attn_selftest_bounded_wait: timeout_cycles must lie in [1e3, 1e9]");
    bounded_wait_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(timeout_cycles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "attn_selftest_bounded_wait: kernel launch: %s", cudaGetErrorString(e));
        return report_error(ATTN_ERR_CUDA, msg);
    }
    return ATTN_OK;
}
