// attn_decode_gqa_noalloc: GQA decode for callers that may not allocate device memory.
//
// attn_decode_gqa needs scratch memory for its split partials, and asks the caller for it.
// Some callers cannot provide it on demand: a plugin running inside a host program that
// owns every device allocation, a serving loop that must not call cudaMalloc (which can
// synchronise the whole device and stall other streams), or code that runs where the
// allocator cannot be re-entered. For them this entry point uses a fixed array compiled
// into the library instead, and allocates nothing: no cudaMalloc, no cudaFree, no library
// routine that allocates.
//
// The array is a file-scope __device__ variable of kNoallocScratchBytes, so every GPU that
// loads the library holds it until the process exits. In host code its name only stands in
// for the symbol; its device address is looked up with cudaGetSymbolAddress once per device,
// with that device current, on the first call made on that device. That first call should
// therefore come before any stream capture. The address is kept for the life of the process:
// it assumes the device's primary context (which the CUDA runtime uses) is not destroyed and
// recreated in between (cudaDeviceReset would do that). All calls share the one array. It is
// zero when the library loads. Like every workspace of this library it starts with a fixed
// region that holds only the bf16 kernels' per-segment arrival counters; the split partials
// (written before they are read, so they need no initial value) always lie after it. Every
// call that completes leaves its counters at zero, so calls of any sequence of shapes and
// dtypes find theirs at zero; a call with more counters than the region holds zeroes its own
// (a memset on the caller's stream, which allocates nothing). A call whose kernel gave up a
// bounded wait leaves counters set: attn_check_status, when it reports that timeout, zeroes
// this array's counter region on the current device again. Two calls whose kernels can
// overlap on the GPU (different streams, or different host threads) race on the array and
// must be ordered by the caller.
#include "../../include/mlakv.h"
#include "common.cuh"

#include <mutex>
#include <stdio.h>

namespace mlakv {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the array on the current device; looked up once per device.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "attn_decode_gqa_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return report_error(ATTN_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) return report_error(ATTN_ERR_UNSUPPORTED, "attn_decode_gqa_noalloc: device index above 63");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof(msg), "attn_decode_gqa_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            return report_error(ATTN_ERR_CUDA, msg);
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return ATTN_OK;
}

}  // namespace

// Zeroes the array's counter region on the current device (once a kernel has given up a wait
// and may have left counters set); nothing to do where the array was never used. Synchronous.
int noalloc_clear_counters(cudaStream_t s) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return (int)cudaGetLastError();
    void *p = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        p = g_addr[dev];
    }
    if (!p) return 0;
    cudaError_t e = cudaMemsetAsync(p, 0, kCounterRegionBytes, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv

extern "C" __attribute__((visibility("default"))) size_t attn_decode_gqa_noalloc_max_scratch(void) {
    return mlakv::kNoallocScratchBytes;
}

extern "C" __attribute__((visibility("default"))) int attn_decode_gqa_noalloc(
    const void *q, const void *k_cache, const void *v_cache, const int *seq_lens, float *out, int B, int Hq, int Hkv,
    int D, float scale, int S_max, int max_S, attn_dtype dtype, int n_split, mlakv_stream_t stream) {
    using namespace mlakv;
    // invalid shapes make the size query return 0; attn_decode_gqa then reports them
    const size_t need = attn_decode_gqa_workspace_size(B, Hq, Hkv, D, max_S, dtype, n_split);
    if (need > kNoallocScratchBytes) {
        char msg[320];
        snprintf(msg, sizeof(msg),
                 "attn_decode_gqa_noalloc: these sizes need %zu bytes of split scratch, above the built-in %zu; "
                 "pass a smaller n_split or use attn_decode_gqa with a caller workspace",
                 need, kNoallocScratchBytes);
        return report_error(ATTN_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&scratch);
        if (rc != ATTN_OK) return rc;
    }
    return attn_decode_gqa(q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, D, scale, S_max, max_S, dtype, n_split,
                           scratch, need > 0 ? kNoallocScratchBytes : 0, stream);
}
