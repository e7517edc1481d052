// K3: MLA decode with W_UK absorbed into the query (qqstock article on DeepSeek MLA,
// sections 2, 3 and 6): every head attends the same cached latent row [c_t ‖ kr_t]
// (r = 128, dr = 48, so 352 bytes per token in bf16) and averages c_t itself — MQA with key
// width 176 and value width 128, where the value is the first 128 columns of the key row.
//
// One thread block per (sequence, block of 16 heads, split); 4 warps, one token per lane:
// the lane computes the 16 scores of its token from the row in global memory (q in shared
// memory, pre-scaled by scale·log2 e), the warp updates the running max/sum per head, and
// P·c is accumulated with lanes owning 4 of the 128 output columns. Partials (o, lse) go to
// K2 when the sequence is split.
#include "common.cuh"

#include <math.h>

namespace mlakv {
namespace {

constexpr int R = 128;
constexpr int DR = 48;
constexpr int HB = 16;
constexpr int TILE = 128;

__global__ void __launch_bounds__(128) decode_mla_fma_kernel(const DecodeMlaArgs a) {
    constexpr int DPL = R / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h0 = blockIdx.y * HB;
    const int b = blockIdx.z;
    const int split = blockIdx.x;
    const int S = a.seq_lens[b];
    const int t_begin = split * a.split_len;
    const int t_end = min(S, t_begin + a.split_len);

    __shared__ __align__(16) float q_s[HB][R + DR];
    __shared__ float m_s[4][HB];
    __shared__ float l_s[4][HB];
    __shared__ __align__(16) float o_s[4][HB][R];

    const __nv_bfloat16 *ql = static_cast<const __nv_bfloat16 *>(a.q_lat) + ((size_t)b * a.Hq + h0) * R;
    const __nv_bfloat16 *qr = static_cast<const __nv_bfloat16 *>(a.q_rope) + ((size_t)b * a.Hq + h0) * DR;
    for (int i = threadIdx.x; i < HB * R; i += 128) q_s[i / R][i % R] = __bfloat162float(ql[i]) * a.scale_log2;
    for (int i = threadIdx.x; i < HB * DR; i += 128) q_s[i / DR][R + i % DR] = __bfloat162float(qr[i]) * a.scale_log2;
    __syncthreads();

    float m[HB], l[HB], o[HB][DPL];
#pragma unroll
    for (int h = 0; h < HB; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[h][i] = 0.f;
    }
    const __nv_bfloat16 *cb = static_cast<const __nv_bfloat16 *>(a.c) + (size_t)b * a.S_max * R;
    const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(a.kr) + (size_t)b * a.S_max * DR;

    for (int t0 = t_begin + warp * 32; t0 < t_end; t0 += TILE) {
        const int t = t0 + lane;
        const bool valid = t < t_end;
        float s[HB];
#pragma unroll
        for (int h = 0; h < HB; ++h) s[h] = 0.f;
        if (valid) {
            const uint4 *crow = reinterpret_cast<const uint4 *>(cb + (size_t)t * R);
            const uint4 *krow = reinterpret_cast<const uint4 *>(kb + (size_t)t * DR);
            for (int c = 0; c < (R + DR) / 8; ++c) {
                const uint4 w = c < R / 8 ? __ldg(crow + c) : __ldg(krow + (c - R / 8));
                const float x[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                    bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
                for (int h = 0; h < HB; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) s[h] = fmaf(q_s[h][8 * c + e], x[e], s[h]);
            }
        }
        float p[HB];
#pragma unroll
        for (int h = 0; h < HB; ++h) {
            const float mn = fmaxf(m[h], warp_max(valid ? s[h] : -INFINITY));
            const float alpha = exp2f(m[h] - mn);
            p[h] = valid ? exp2f(s[h] - mn) : 0.f;
            l[h] = l[h] * alpha + warp_sum(p[h]);
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[h][i] *= alpha;
            m[h] = mn;
        }
        const int n = min(32, t_end - t0);
        for (int tt = 0; tt < n; ++tt) {
            const uint2 w = __ldg(reinterpret_cast<const uint2 *>(cb + (size_t)(t0 + tt) * R) + lane);
            const float vv[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
#pragma unroll
            for (int h = 0; h < HB; ++h) {
                const float pt = __shfl_sync(0xffffffffu, p[h], tt);
#pragma unroll
                for (int i = 0; i < DPL; ++i) o[h][i] = fmaf(pt, vv[i], o[h][i]);
            }
        }
    }

    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < HB; ++h) {
            m_s[warp][h] = m[h];
            l_s[warp][h] = l[h];
        }
    }
#pragma unroll
    for (int h = 0; h < HB; ++h)
#pragma unroll
        for (int i = 0; i < DPL; ++i) o_s[warp][h][4 * lane + i] = o[h][i];
    __syncthreads();

    for (int idx = threadIdx.x; idx < HB * R; idx += 128) {
        const int h = idx / R;
        const int d = idx % R;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w][h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float f = exp2f(m_s[w][h] - M);
                L = fmaf(l_s[w][h], f, L);
                O = fmaf(o_s[w][h][d], f, O);
            }
        }
        const size_t row = (size_t)b * a.Hq + h0 + h;
        const float val = L > 0.f ? O / L : 0.f;
        if (a.n_split == 1) {
            a.out[row * R + d] = val;
        } else {
            a.o_part[(row * a.n_split + split) * R + d] = val;
            if (d == 0) a.lse_part[row * a.n_split + split] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
}

}  // namespace

int decode_mla_tile_tokens() { return TILE; }

int decode_mla_read_and_clear_status(cudaStream_t, unsigned *flag) {
    *flag = 0;
    return 0;
}

cudaError_t launch_decode_mla(const DecodeMlaArgs &a, cudaStream_t s) {
    const dim3 grid(a.n_split, a.Hq / HB, a.B);
    decode_mla_fma_kernel<<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mlakv
