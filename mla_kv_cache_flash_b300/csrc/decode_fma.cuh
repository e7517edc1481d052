// K1 (CUDA-core form), the kernel template shared by decode_gqa_fma.cu (decode, chunked
// prefill) and prefill_chunked_mla.cu (MLA chunked prefill): split-KV decode for GQA/MHA/MQA over an fp32 cache, or over an
// 8-bit E4M3 cache with one fp32 scale per cached row of K and of V ("MHA, MQA và GQA"
// ebook: fp8 halves every byte of the cache), fp32 FMA. The same kernel runs chunked
// prefill ("模型架构｜MQA & GQA 调研", section "代码": new tokens at start_pos see the cache up
// to their own position): each packed new-token row is a decode over its sequence's cache
// with length start_pos + i + 1, for fp32 and bf16 caches, and for the MLA latent cache
// (qqstock MLA article, sections 2, 3 and 6: key [c ‖ kr] of width 128 + 48, value c).
//
// The fp32 cache stays off the tensor cores, which would round it (TF32 keeps 10 mantissa
// bits) and break the fp32 tolerance; the bf16 decode has its own tensor-core kernels. E4M3
// codes widen exactly to fp32; a row's K scale multiplies its finished dot products and its
// V scale multiplies its softmax weight before P·V (the normaliser takes the unscaled
// weight), so no element is rescaled.
//
// One thread block handles one (query row, KV head j, split, block of HB query heads of j's
// group). The HB heads are stacked so each K/V element is loaded once per block and feeds
// all HB heads (repeat_kv would instead re-read each K/V byte once per query head).
//
// Per 128-token tile each of the 4 warps takes 32 tokens, one token per lane:
//   scores   lane t computes s[h] = (scale·log2 e)·q_h·k_t for its token (q in shared memory,
//            read as broadcasts), so the softmax works in the base-2 domain;
//   softmax  running max m_h and sum l_h per warp (warp-shuffle max/sum), rescale by
//            2^(m_old − m_new) — the online form of the page's fp32 softmax;
//   P·V      lanes own D/32 output columns; p_t is broadcast by shuffle and V rows are read
//            coalesced.
// The four warps' states are merged in shared memory at the end. With one split the block
// writes out = O / l; otherwise it writes the normalised partial and lse = ln Σ e^s for K2.
#pragma once

#include "common.cuh"

#include <cuda_fp8.h>
#include <math.h>

#include <type_traits>

namespace mlakv {
namespace {

__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// eight E4M3 codes (8-byte aligned) → fp32, exactly
__device__ __forceinline__ void load8(const uint8_t *p, float (&x)[8]) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * k)) & 0xffffu), __NV_E4M3);
            const float2 f = __half22float2(__half2(hr));
            x[4 * i + 2 * k] = f.x;
            x[4 * i + 2 * k + 1] = f.y;
        }
    }
}

// eight bf16 (16-byte aligned) → fp32, exactly
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float load1(const float *p) { return __ldg(p); }
__device__ __forceinline__ float load1(const __nv_bfloat16 *p) { return __bfloat162float(p[0]); }
__device__ __forceinline__ float load1(const uint8_t *p) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(__ldg(p)), __NV_E4M3)));
}

constexpr int kMlaRopeWidth = 48;   // MLA: the decoupled RoPE key kr, appended to the key row

// TQ: query type (fp32, or bf16 beside a bf16 or E4M3 cache); T: cache element (fp32, bf16 or
// E4M3 code); kChunk: rows are packed new tokens of chunked prefill (cu_q, start_pos); kMla:
// the key row is [c ‖ kr] (k = c, k2 = kr, q = q_lat, q2 = q_rope) and the value is c (D wide).
template <typename TQ, typename T, int D, int HB, bool kChunk, bool kMla = false>
__global__ void __launch_bounds__(128) decode_gqa_fma_kernel(const DecodeGqaArgs a) {
    constexpr bool kScaled = std::is_same<T, uint8_t>::value;
    constexpr int DPL = D / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.Hq / a.Hkv;
    const int n_hblk = G / HB;
    const int j = blockIdx.y / n_hblk;
    const int h0 = j * G + (blockIdx.y % n_hblk) * HB;
    const int row = blockIdx.z;                 // query / output row
    const int split = blockIdx.x;
    int b = row, S;                             // cache batch index and visible length
    if constexpr (kChunk) {
        // chunked prefill: the sequence whose chunk holds packed row `row` is the b with
        // cu_q[b] <= row < cu_q[b + 1] (cu_q non-decreasing, cu_q[0] = 0, cu_q[n_seq] = rows)
        int lo = 0, hi = a.n_seq;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(a.cu_q + mid) <= row) lo = mid; else hi = mid;
        }
        b = lo;
        S = __ldg(a.start_pos + b) + (row - __ldg(a.cu_q + b)) + 1;
    } else {
        S = a.seq_lens[row];
    }
    const int t_begin = split * a.split_len;
    const int t_end = min(S, t_begin + a.split_len);

    constexpr int DK = kMla ? D + kMlaRopeWidth : D;     // key width
    __shared__ __align__(16) float q_s[HB][DK];
    __shared__ float m_s[4][HB];
    __shared__ float l_s[4][HB];
    __shared__ __align__(16) float o_s[4][HB][D];

    const TQ *qg = static_cast<const TQ *>(a.q) + ((size_t)row * a.Hq + h0) * D;
    for (int i = threadIdx.x; i < HB * D; i += 128) q_s[i / D][i % D] = to_f(qg[i]) * a.scale_log2;
    if constexpr (kMla) {
        constexpr int R = kMlaRopeWidth;
        const TQ *qr = static_cast<const TQ *>(a.q2) + ((size_t)row * a.Hq + h0) * R;
        for (int i = threadIdx.x; i < HB * R; i += 128) q_s[i / R][D + i % R] = to_f(qr[i]) * a.scale_log2;
    }
    __syncthreads();

    float m[HB], l[HB], o[HB][DPL];
#pragma unroll
    for (int h = 0; h < HB; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[h][i] = 0.f;
    }

    const size_t row_stride = (size_t)a.Hkv * D;
    const T *kb = static_cast<const T *>(a.k) + ((size_t)b * a.S_max * a.Hkv + j) * D;
    const T *vb = static_cast<const T *>(a.v) + ((size_t)b * a.S_max * a.Hkv + j) * D;

    for (int t0 = t_begin + warp * 32; t0 < t_end; t0 += 128) {
        const int t = t0 + lane;
        const bool valid = t < t_end;
        float s[HB];
#pragma unroll
        for (int h = 0; h < HB; ++h) s[h] = 0.f;
        float sv = 1.f;                         // the row's V scale (E4M3 cache)
        if (valid) {
            const T *kr = kb + (size_t)t * row_stride;
#pragma unroll 2
            for (int c = 0; c < D; c += 8) {
                float x[8];
                load8(kr + c, x);
#pragma unroll
                for (int h = 0; h < HB; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) s[h] = fmaf(q_s[h][c + e], x[e], s[h]);
            }
            if constexpr (kMla) {
                const T *kr2 = static_cast<const T *>(a.k2) + ((size_t)b * a.S_max + t) * kMlaRopeWidth;
#pragma unroll
                for (int c = 0; c < kMlaRopeWidth; c += 8) {
                    float x[8];
                    load8(kr2 + c, x);
#pragma unroll
                    for (int h = 0; h < HB; ++h)
#pragma unroll
                        for (int e = 0; e < 8; ++e) s[h] = fmaf(q_s[h][D + c + e], x[e], s[h]);
                }
            }
            if constexpr (kScaled) {
                const size_t srow = ((size_t)b * a.S_max + t) * a.Hkv + j;
                const float sk = __ldg(a.k_scale + srow);
                sv = __ldg(a.v_scale + srow);
#pragma unroll
                for (int h = 0; h < HB; ++h) s[h] *= sk;
            }
        }
        float p[HB];
#pragma unroll
        for (int h = 0; h < HB; ++h) {
            // lane 0 is always valid here (t0 < t_end), so the tile max is finite
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
            const T *vr = vb + (size_t)(t0 + tt) * row_stride;
            float vv[DPL];
#pragma unroll
            for (int i = 0; i < DPL; ++i) vv[i] = load1(vr + lane + 32 * i);
#pragma unroll
            for (int h = 0; h < HB; ++h) {
                const float pt = __shfl_sync(0xffffffffu, kScaled ? p[h] * sv : p[h], tt);
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
        for (int i = 0; i < DPL; ++i) o_s[warp][h][lane + 32 * i] = o[h][i];
    __syncthreads();

    for (int idx = threadIdx.x; idx < HB * D; idx += 128) {
        const int h = idx / D;
        const int d = idx % D;
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
        const size_t orow = (size_t)row * a.Hq + h0 + h;
        const float val = L > 0.f ? O / L : 0.f;
        if (a.n_split == 1) {
            a.out[orow * D + d] = val;
        } else {
            a.o_part[(orow * a.n_split + split) * D + d] = val;
            if (d == 0) a.lse_part[orow * a.n_split + split] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
}

template <typename TQ, typename T, int D, bool kChunk, bool kMla = false>
cudaError_t launch_d(const DecodeGqaArgs &a, cudaStream_t s) {
    const int G = a.Hq / a.Hkv;
    const int hb = (G % 8 == 0) ? 8 : (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
    const dim3 grid(a.n_split, a.Hkv * (G / hb), a.B);
    switch (hb) {
        case 8: decode_gqa_fma_kernel<TQ, T, D, 8, kChunk, kMla><<<grid, 128, 0, s>>>(a); break;
        case 4: decode_gqa_fma_kernel<TQ, T, D, 4, kChunk, kMla><<<grid, 128, 0, s>>>(a); break;
        case 2: decode_gqa_fma_kernel<TQ, T, D, 2, kChunk, kMla><<<grid, 128, 0, s>>>(a); break;
        default: decode_gqa_fma_kernel<TQ, T, D, 1, kChunk, kMla><<<grid, 128, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

template <typename TQ, typename T, bool kChunk>
cudaError_t launch_t(const DecodeGqaArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_d<TQ, T, 64, kChunk>(a, s);
        case 96: return launch_d<TQ, T, 96, kChunk>(a, s);
        case 128: return launch_d<TQ, T, 128, kChunk>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace mlakv
