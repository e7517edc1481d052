// Device-side checks of the length arrays the entry points trust (off by default).
//
// The lengths, offsets and start positions of a call live in device memory, so the host
// validates only the sizes it is given; the kernels take the arrays as stated (a length above
// the cache capacity would read past the cache). With the checks on (environment variable
// MLAKV_DEVICE_CHECKS=1 when the library loads, or attn_set_device_checks(1)), every entry
// point that takes such an array first runs lengths_check_kernel over it on the call's stream,
// synchronises the stream, and returns ATTN_ERR_INPUT without launching anything else if a
// value lies outside its stated bounds. This costs a launch and a synchronisation per call: a
// debugging aid, not for the hot path, and not usable under stream capture.
#include "common.cuh"
#include "mlakv.h"

#include <stdio.h>
#include <stdlib.h>

namespace mlakv {

namespace {

// Result of the last check: a bit per kind of violation and the smallest offending index.
struct CheckResult {
    unsigned bits;
    int first;
};
__device__ CheckResult g_check;

enum : unsigned {
    kLenNegative = 1u,     // a length or start position below 0
    kLenAboveMax = 2u,     // a length above its bound (max_S, max_seqlen)
    kOffsetStart = 4u,     // offsets[0] != 0
    kOffsetOrder = 8u,     // offsets decrease
    kOffsetEnd = 16u,      // offsets[n] above the row count T
    kChunkEnd = 32u        // start_pos + chunk length above max_kv
};

// mode 0: lens[i] in [0, bound0] for i < n.
// mode 1: offsets (lens) of n sequences: lens[0] == 0, non-decreasing, lens[n] <= bound0 (T),
//         each difference <= bound1 (the longest allowed sequence).
// mode 2: mode 1 with bound1 unused, and start[i] >= 0, start[i] + (lens[i+1] - lens[i]) <= bound2.
__global__ void lengths_check_kernel(const int *lens, const int *start, int n, int mode, int bound0, int bound1,
                                     int bound2) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n + (mode ? 1 : 0); i += gridDim.x * blockDim.x) {
        unsigned bad = 0;
        if (mode == 0) {
            const int v = lens[i];
            if (v < 0) bad |= kLenNegative;
            if (v > bound0) bad |= kLenAboveMax;
        } else {
            const int v = lens[i];
            if (i == 0 && v != 0) bad |= kOffsetStart;
            if (i == n && v > bound0) bad |= kOffsetEnd;
            if (i < n) {
                const int d = lens[i + 1] - v;
                if (d < 0) bad |= kOffsetOrder;
                if (mode == 1 && d > bound1) bad |= kLenAboveMax;
                if (mode == 2) {
                    const int s0 = start[i];
                    if (s0 < 0) bad |= kLenNegative;
                    if ((long long)s0 + d > bound2) bad |= kChunkEnd;
                }
            }
        }
        if (bad) {
            atomicOr(&g_check.bits, bad);
            atomicMin(&g_check.first, i);
        }
    }
}

int g_checks_on = -1;   // -1: not read from the environment yet

int run_check(const int *lens, const int *start, int n, int mode, int b0, int b1, int b2, cudaStream_t s,
              const char *who) {
    const CheckResult clear{0u, 0x7fffffff};
    cudaError_t e = cudaMemcpyToSymbolAsync(g_check, &clear, sizeof(clear), 0, cudaMemcpyHostToDevice, s);
    const int items = n + (mode ? 1 : 0);
    const int blocks = items > 0 ? (items + 255) / 256 < 64 ? (items + 255) / 256 : 64 : 0;
    if (e == cudaSuccess && blocks > 0) {
        lengths_check_kernel<<<blocks, 256, 0, s>>>(lens, start, n, mode, b0, b1, b2);
        e = cudaGetLastError();
    }
    CheckResult got{};
    if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&got, g_check, sizeof(got), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    char what[160];
    if (e != cudaSuccess) {
        snprintf(what, sizeof(what), "%s: device-side input check", who);
        return report_cuda_error(e, what);
    }
    if (got.bits == 0) return ATTN_OK;
    static const char *names[] = {"a negative length or start position", "a length above its bound",
                                  "offsets not starting at 0", "decreasing offsets", "the last offset above T",
                                  "start_pos + chunk length above max_kv"};
    int k = 0;
    while (!(got.bits & (1u << k))) ++k;
    snprintf(what, sizeof(what), "%s: device-side input check: %s (first at index %d)", who, names[k], got.first);
    return report_error(ATTN_ERR_INPUT, what);
}

}  // namespace

bool device_checks_on() {
    if (g_checks_on < 0) {
        const char *v = getenv("MLAKV_DEVICE_CHECKS");
        g_checks_on = (v && v[0] && v[0] != '0') ? 1 : 0;
    }
    return g_checks_on > 0;
}

int set_device_checks(int on) {
    const int prev = device_checks_on() ? 1 : 0;
    g_checks_on = on ? 1 : 0;
    return prev;
}

int check_lengths(const int *lens, int n, int bound, cudaStream_t s, const char *who) {
    return run_check(lens, nullptr, n, 0, bound, 0, 0, s, who);
}

int check_offsets(const int *offsets, int n, int T, int max_len, cudaStream_t s, const char *who) {
    return run_check(offsets, nullptr, n, 1, T, max_len, 0, s, who);
}

int check_chunks(const int *cu, const int *start, int n, int T, int max_kv, cudaStream_t s, const char *who) {
    return run_check(cu, start, n, 2, T, 0, max_kv, s, who);
}

}  // namespace mlakv
