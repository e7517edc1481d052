// K2: log-sum-exp merge of split-KV partials.
//
// Each split of a sequence's cache produced a normalised output o_i and lse_i = ln Σ e^s over
// its tokens. Since e^{lse_i} is the split's softmax denominator, the full softmax output is
//   out = Σ_i e^{lse_i − M} o_i / Σ_i e^{lse_i − M},   M = max_i lse_i,
// which is exact in real arithmetic (the subtraction of M is for range only). Empty splits
// have lse = −inf and weigh nothing; a row with only empty splits is 0.
//
// One warp per output row: the lanes find M and the weight sum over the splits, then each
// lane accumulates 4 consecutive output columns at a time with 16-byte loads. The kernel is
// launched as a programmatic dependent of the decode kernel, so its blocks are resident and
// waiting when the partials are complete instead of paying a full launch after them.
#include "common.cuh"

#include <math.h>

namespace mlakv {
namespace {

__global__ void __launch_bounds__(128) merge_kernel(const float *__restrict__ o_part,
                                                    const float *__restrict__ lse_part,
                                                    float *__restrict__ out, int rows, int n_split,
                                                    int Dv) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    griddep_wait();                 // the partials come from the previous kernel in the stream
    griddep_launch_dependents();
    if (row >= rows) return;
    const float *lse = lse_part + (size_t)row * n_split;
    float M = -INFINITY;
    for (int i = lane; i < n_split; i += 32) M = fmaxf(M, lse[i]);
    M = warp_max(M);
    float4 *dst = reinterpret_cast<float4 *>(out + (size_t)row * Dv);
    if (M == -INFINITY) {
        for (int c = lane; c < Dv / 4; c += 32) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    float W = 0.f;
    for (int i = lane; i < n_split; i += 32) W += expf(lse[i] - M);
    W = warp_sum(W);
    const float inv = 1.f / W;
    const float4 *src = reinterpret_cast<const float4 *>(o_part + (size_t)row * n_split * Dv);
    for (int c = lane; c < Dv / 4; c += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < n_split; ++i) {
            const float w = expf(lse[i] - M);
            if (w == 0.f) continue;
            const float4 x = src[(size_t)i * (Dv / 4) + c];
            acc.x = fmaf(w, x.x, acc.x);
            acc.y = fmaf(w, x.y, acc.y);
            acc.z = fmaf(w, x.z, acc.z);
            acc.w = fmaf(w, x.w, acc.w);
        }
        dst[c] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

}  // namespace

cudaError_t launch_merge(const float *o_part, const float *lse_part, float *out, int rows,
                         int n_split, int Dv, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const cudaError_t e = launch_pdl(merge_kernel, dim3((rows + 3) / 4), dim3(128), 0, s, o_part, lse_part, out,
                                     rows, n_split, Dv);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mlakv
