// The two MLA projections on either side of the absorbed decode (qqstock article on DeepSeek
// MLA, section 2, "合并与吸收"): the key up-projection W_UK is absorbed into the query before
// the decode, and the value up-projection W_UV is applied once to the decode's latent output
// instead of once per cached token.
//   q_lat[b, h] = W_UK[h]ᵀ · q_nope[b, h]     W_UK [Hq, d_nope, r]   (rounded to bf16: the
//                                                                     decode's query operand)
//   out[b, h]   = W_UV[h]  · o_lat[b, h]      W_UV [Hq, d_v, r]      (fp32)
// Both are batched matrix-vector products per head: a few hundred KB of weights and
// activations per call, so the work is latency-bound, not bandwidth- or compute-bound. One
// block covers one head and 8 sequences. The block first moves the head's weights into shared
// memory with 16-byte cp.async copies (all in flight at once, one memory round trip), then
// splits the contraction index among up to 256 threads so that every SM sub-partition has
// several warps to issue from; the partial sums meet in shared memory. fp32 throughout, CUDA
// cores. Both kernels start as programmatic dependents of the previous launch in the stream:
// they prefetch the head's weights into L2 at once, wait for that launch before reading
// anything (their inputs may come from it), and let the next one start early.
#include "../../include/mlakv.h"
#include "common.cuh"
#include "ptx.cuh"

namespace mlakv {
namespace {

constexpr int BR = 8;                        // sequences per block
constexpr int kMaxThreads = 256;
constexpr int kChunkBytes = 32768;           // W_UK rows staged per pass

// W_UK: a thread owns two adjacent output columns; the d_nope rows are dealt round-robin to
// G groups of r/2 threads.
__host__ __device__ inline int absorb_groups(int r) { return kMaxThreads / (r / 2); }
__host__ __device__ inline int absorb_chunk_rows(int dn, int r) { return dn < kChunkBytes / (2 * r) ? dn : kChunkBytes / (2 * r); }
__host__ __device__ inline size_t absorb_smem(int dn, int r) {
    return (size_t)absorb_chunk_rows(dn, r) * r * 2 + (size_t)dn * BR * sizeof(float) +
           (size_t)absorb_groups(r) * BR * r * sizeof(float);
}
// W_UV: a thread owns one output column; the r/8 eight-wide slices of the latent index are
// dealt round-robin to G groups of d_v threads. Rows are padded by 16 bytes: the row stride
// is then 4 or 20 words modulo 32, so the eight threads of one 16-byte shared-memory access
// phase, reading consecutive rows, hit eight distinct groups of four banks.
__host__ __device__ inline int uv_groups(int r, int dv) {
    const int g = kMaxThreads / dv;
    return g < r / 8 ? g : r / 8;
}
__host__ __device__ inline int uv_row_stride(int r) { return r + 8; }
__host__ __device__ inline size_t uv_smem(int r, int dv) {
    return (size_t)dv * uv_row_stride(r) * 2 + (size_t)r * BR * sizeof(float) +
           (size_t)uv_groups(r, dv) * BR * dv * sizeof(float);
}

// q_lat[b, h, :] for b in [b0, b0 + BR). blockDim = G·r/2.
__global__ void __launch_bounds__(kMaxThreads) absorb_query_kernel(const __nv_bfloat16 *__restrict__ q_nope,
                                                                   const __nv_bfloat16 *__restrict__ w_uk,
                                                                   __nv_bfloat16 *__restrict__ q_lat, int B, int Hq,
                                                                   int dn, int r) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int ch = absorb_chunk_rows(dn, r), half = r / 2, T = blockDim.x, G = T / half;
    __nv_bfloat16 *ws = reinterpret_cast<__nv_bfloat16 *>(smem);              // [ch][r]
    float *qs = reinterpret_cast<float *>(smem + (size_t)ch * r * 2);         // [dn][BR]
    float *red = qs + (size_t)dn * BR;                                        // [G][BR][r]
    const int h = blockIdx.x, b0 = blockIdx.y * BR, cp = threadIdx.x % half, g = threadIdx.x / half;
    // warm L2 (and the address translation) with the head's weights while the previous
    // kernel finishes; a prefetch reads through the coherent L2, so it is safe before the wait
    for (size_t off = (size_t)threadIdx.x * 128; off < (size_t)dn * r * 2; off += (size_t)T * 128)
        prefetch_l2(reinterpret_cast<const unsigned char *>(w_uk + (size_t)h * dn * r) + off);
    griddep_wait();
    griddep_launch_dependents();
    float acc[BR][2];
#pragma unroll
    for (int bb = 0; bb < BR; ++bb) acc[bb][0] = acc[bb][1] = 0.f;
    for (int n0 = 0; n0 < dn; n0 += ch) {
        const int rows = dn - n0 < ch ? dn - n0 : ch;
        const __nv_bfloat16 *src = w_uk + ((size_t)h * dn + n0) * r;
        for (int v = threadIdx.x; v < rows * r / 8; v += T) cp_async16(ws + v * 8, src + v * 8);
        if (n0 == 0) {
            // the query rows, while the first weight copies are in flight: eight loads per
            // thread issued before any is stored, so they overlap
            const int nq = BR * dn;
            for (int i0 = threadIdx.x; i0 < nq; i0 += 8 * T) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * T, bb = i / dn, n = i - bb * dn;
                    x[u] = i < nq && b0 + bb < B ? __bfloat162float(q_nope[((size_t)(b0 + bb) * Hq + h) * dn + n]) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * T, bb = i / dn, n = i - bb * dn;
                    if (i < nq) qs[n * BR + bb] = x[u];
                }
            }
        }
        cp_async_wait_all();
        __syncthreads();
#pragma unroll 2
        for (int n = g; n < rows; n += G) {
            const uint32_t w2 = *reinterpret_cast<const uint32_t *>(ws + n * r + 2 * cp);
            const float w0 = bf16_lo(w2), w1 = bf16_hi(w2);
            const float4 qa = *reinterpret_cast<const float4 *>(qs + (n0 + n) * BR);
            const float4 qb = *reinterpret_cast<const float4 *>(qs + (n0 + n) * BR + 4);
            const float q[BR] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int bb = 0; bb < BR; ++bb) {
                acc[bb][0] = fmaf(q[bb], w0, acc[bb][0]);
                acc[bb][1] = fmaf(q[bb], w1, acc[bb][1]);
            }
        }
        __syncthreads();                       // the next pass overwrites ws
    }
#pragma unroll
    for (int bb = 0; bb < BR; ++bb)
        *reinterpret_cast<float2 *>(red + ((size_t)g * BR + bb) * r + 2 * cp) = make_float2(acc[bb][0], acc[bb][1]);
    __syncthreads();
    for (int i = threadIdx.x; i < BR * r; i += T) {
        const int bb = i / r, col = i - bb * r;
        float sum = 0.f;
        for (int gg = 0; gg < G; ++gg) sum += red[((size_t)gg * BR + bb) * r + col];
        if (b0 + bb < B) q_lat[((size_t)(b0 + bb) * Hq + h) * r + col] = __float2bfloat16_rn(sum);
    }
}

// out[b, h, :] for b in [b0, b0 + BR). blockDim = G·d_v.
__global__ void __launch_bounds__(kMaxThreads) apply_uv_kernel(const float *__restrict__ o_lat,
                                                               const __nv_bfloat16 *__restrict__ w_uv,
                                                               float *__restrict__ out, int B, int Hq, int r, int dv) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int rs = uv_row_stride(r), T = blockDim.x, G = T / dv, rv = r / 8;
    __nv_bfloat16 *wt = reinterpret_cast<__nv_bfloat16 *>(smem);              // [dv][rs]
    float *os = reinterpret_cast<float *>(smem + (size_t)dv * rs * 2);        // [r][BR]
    float *red = os + (size_t)r * BR;                                         // [G][BR][dv]
    const int h = blockIdx.x, b0 = blockIdx.y * BR, v = threadIdx.x % dv, g = threadIdx.x / dv;
    const __nv_bfloat16 *src = w_uv + (size_t)h * dv * r;
    for (size_t off = (size_t)threadIdx.x * 128; off < (size_t)dv * r * 2; off += (size_t)T * 128)
        prefetch_l2(reinterpret_cast<const unsigned char *>(src) + off);   // as in absorb_query_kernel
    griddep_wait();
    griddep_launch_dependents();
    for (int i = threadIdx.x; i < dv * rv; i += T) {
        const int row = i / rv, k = i - row * rv;
        cp_async16(wt + row * rs + k * 8, src + (size_t)row * r + k * 8);
    }
    const int no = BR * r;                     // latent rows: eight loads in flight per thread
    for (int i0 = threadIdx.x; i0 < no; i0 += 8 * T) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * T, bb = i / r, rr = i - bb * r;
            x[u] = i < no && b0 + bb < B ? o_lat[((size_t)(b0 + bb) * Hq + h) * r + rr] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * T, bb = i / r, rr = i - bb * r;
            if (i < no) os[rr * BR + bb] = x[u];
        }
    }
    cp_async_wait_all();
    __syncthreads();
    float acc[BR];
#pragma unroll
    for (int bb = 0; bb < BR; ++bb) acc[bb] = 0.f;
    for (int k = g; k < rv; k += G) {
        const uint4 w8 = *reinterpret_cast<const uint4 *>(wt + v * rs + k * 8);
        const uint32_t wp[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float w = (j & 1) ? bf16_hi(wp[j >> 1]) : bf16_lo(wp[j >> 1]);
            const float *o = os + (k * 8 + j) * BR;
            const float4 oa = *reinterpret_cast<const float4 *>(o);
            const float4 ob = *reinterpret_cast<const float4 *>(o + 4);
            acc[0] = fmaf(w, oa.x, acc[0]); acc[1] = fmaf(w, oa.y, acc[1]);
            acc[2] = fmaf(w, oa.z, acc[2]); acc[3] = fmaf(w, oa.w, acc[3]);
            acc[4] = fmaf(w, ob.x, acc[4]); acc[5] = fmaf(w, ob.y, acc[5]);
            acc[6] = fmaf(w, ob.z, acc[6]); acc[7] = fmaf(w, ob.w, acc[7]);
        }
    }
#pragma unroll
    for (int bb = 0; bb < BR; ++bb) red[((size_t)g * BR + bb) * dv + v] = acc[bb];
    __syncthreads();
    for (int i = threadIdx.x; i < BR * dv; i += T) {
        const int bb = i / dv, vv = i - bb * dv;
        float sum = 0.f;
        for (int gg = 0; gg < G; ++gg) sum += red[((size_t)gg * BR + bb) * dv + vv];
        if (b0 + bb < B) out[((size_t)(b0 + bb) * Hq + h) * dv + vv] = sum;
    }
}

}  // namespace
}  // namespace mlakv

using namespace mlakv;

extern "C" __attribute__((visibility("default"))) int attn_mla_absorb_query(const void *q_nope, const void *w_uk,
                                                                          void *q_lat, int B, int Hq, int d_nope,
                                                                          int r, mlakv_stream_t stream) {
    if (!q_nope || !w_uk || !q_lat)
        return report_error(ATTN_ERR_NULL, "attn_mla_absorb_query: q_nope, w_uk and q_lat must be non-NULL");
    if (B < 1 || Hq < 1 || d_nope < 1 || r < 1)
        return report_error(ATTN_ERR_SHAPE, "attn_mla_absorb_query: B, Hq, d_nope and r must be >= 1");
    if (r % 32 != 0 || r > 256 || d_nope > 512)
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_mla_absorb_query: r must be a multiple of 32 up to 256, "
                                                  "d_nope at most 512");
    if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_lat))
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_mla_absorb_query: every pointer must be 16-byte aligned");
    const size_t smem = absorb_smem(d_nope, r);
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(absorb_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = launch_pdl(absorb_query_kernel, dim3(Hq, (B + BR - 1) / BR), dim3(absorb_groups(r) * (r / 2)), smem,
                       reinterpret_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16 *>(q_nope),
                       static_cast<const __nv_bfloat16 *>(w_uk), static_cast<__nv_bfloat16 *>(q_lat), B, Hq, d_nope, r);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return report_cuda_error(e, "attn_mla_absorb_query: kernel launch");
    report_error(ATTN_OK, "");
    return ATTN_OK;
}

extern "C" __attribute__((visibility("default"))) int attn_mla_apply_uv(const float *o_lat, const void *w_uv,
                                                                      float *out, int B, int Hq, int r, int d_v,
                                                                      mlakv_stream_t stream) {
    if (!o_lat || !w_uv || !out)
        return report_error(ATTN_ERR_NULL, "attn_mla_apply_uv: o_lat, w_uv and out must be non-NULL");
    if (B < 1 || Hq < 1 || r < 1 || d_v < 1)
        return report_error(ATTN_ERR_SHAPE, "attn_mla_apply_uv: B, Hq, r and d_v must be >= 1");
    if (r % 32 != 0 || r > 256 || d_v > 256)
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_mla_apply_uv: r must be a multiple of 32 up to 256, "
                                                  "d_v at most 256");
    if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out))
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_mla_apply_uv: every pointer must be 16-byte aligned");
    const size_t smem = uv_smem(r, d_v);
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(apply_uv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = launch_pdl(apply_uv_kernel, dim3(Hq, (B + BR - 1) / BR), dim3(uv_groups(r, d_v) * d_v), smem,
                       reinterpret_cast<cudaStream_t>(stream), o_lat, static_cast<const __nv_bfloat16 *>(w_uv), out, B,
                       Hq, r, d_v);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return report_cuda_error(e, "attn_mla_apply_uv: kernel launch");
    report_error(ATTN_OK, "");
    return ATTN_OK;
}
