// The cache write of one decode step, fused with the rotary embedding ("模型架构｜MQA & GQA
// 调研", section "代码": Attention.forward rotates the new q and k with the cis table, writes
// k and v into the cache at start_pos, then reads the cache; qqstock MLA article, section 3:
// q_rope and the shared rope key are rotated, the latent c is cached as is).
//
// One block per sequence. The block's work is cut into 16-byte units of three kinds: the
// query heads (rotated into q_out), the new key heads (rotated into the cache row), and the
// unrotated part (copied into the other cache row). A head vector is rotated as consecutive
// pairs (x[2j], x[2j+1]) times the table entry (cos, sin) for the sequence's position, in
// fp32, rounded to nearest-even when the type is bf16. A position outside [0, S_max) appends
// nothing, writes q_out = 0 for that sequence and new length 0. The kernel starts as a
// programmatic dependent of the previous launch and lets the next one (the decode) launch
// early; the decode's own dependency wait orders its cache reads after these writes.
#include "../../include/mlakv.h"
#include "common.cuh"

#include <stdio.h>

namespace mlakv {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void to_f32(const uint4 &u, float *x) {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 from_f32(const float *x) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_f32(const uint4 &u, float *x) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
    }
    __device__ static uint4 from_f32(const float *x) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);   // .x = low half
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

struct AppendArgs {
    const void *q, *rot_new, *plain_new;    // [B, Hq, W], [B, Hr, W], [B, Hp, Wp]
    const int *positions;                   // [B]
    const float2 *cis;                      // [S_max, W/2] (cos, sin)
    void *q_out, *rot_cache, *plain_cache;  // [B, Hq, W], [B, S_max, Hr, W], [B, S_max, Hp, Wp]
    int *new_lens;                          // [B] or null
    int Hq, Hr, W, Hp, Wp, S_max;
};

template <typename T>
__global__ void __launch_bounds__(128) append_rope_kernel(AppendArgs a) {
    constexpr int V = Vec<T>::N;
    const int b = blockIdx.x;
    griddep_wait();
    griddep_launch_dependents();
    const int p = a.positions[b];
    const bool ok = p >= 0 && p < a.S_max;
    if (threadIdx.x == 0 && a.new_lens) a.new_lens[b] = ok ? p + 1 : 0;
    const int nq = a.Hq * a.W / V, nr = a.Hr * a.W / V, np = a.Hp * a.Wp / V;
    const size_t qrow = (size_t)b * a.Hq * a.W;
    const size_t crow = ((size_t)b * a.S_max + (ok ? p : 0));     // cache row index (used only if ok)
    for (int u = threadIdx.x; u < nq + nr + np; u += blockDim.x) {
        if (u < nq + nr) {
            const bool is_q = u < nq;
            const int e = (is_q ? u : u - nq) * V;                // element offset within the row
            if (!ok) {
                if (is_q) *reinterpret_cast<uint4 *>(static_cast<T *>(a.q_out) + qrow + e) = make_uint4(0, 0, 0, 0);
                continue;
            }
            const T *src = is_q ? static_cast<const T *>(a.q) + qrow + e
                                : static_cast<const T *>(a.rot_new) + (size_t)b * a.Hr * a.W + e;
            T *dst = is_q ? static_cast<T *>(a.q_out) + qrow + e
                          : static_cast<T *>(a.rot_cache) + crow * a.Hr * a.W + e;
            float x[V], y[V];
            Vec<T>::to_f32(*reinterpret_cast<const uint4 *>(src), x);
            const float2 *cs = a.cis + (size_t)p * (a.W / 2) + (e % a.W) / 2;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                const float2 c = cs[i];
                y[2 * i] = x[2 * i] * c.x - x[2 * i + 1] * c.y;
                y[2 * i + 1] = x[2 * i] * c.y + x[2 * i + 1] * c.x;
            }
            *reinterpret_cast<uint4 *>(dst) = Vec<T>::from_f32(y);
        } else if (ok) {
            const int e = (u - nq - nr) * V;
            *reinterpret_cast<uint4 *>(static_cast<T *>(a.plain_cache) + crow * a.Hp * a.Wp + e) =
                *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.plain_new) + (size_t)b * a.Hp * a.Wp + e);
        }
    }
}

int launch_append(const AppendArgs &a, int B, attn_dtype dtype, mlakv_stream_t stream, const char *who) {
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = dtype == ATTN_BF16 ? launch_pdl(append_rope_kernel<__nv_bfloat16>, dim3(B), dim3(128), 0, s, a)
                                       : launch_pdl(append_rope_kernel<float>, dim3(B), dim3(128), 0, s, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        char what[96];
        snprintf(what, sizeof(what), "%s: kernel launch", who);
        return report_cuda_error(e, what);
    }
    report_error(ATTN_OK, "");
    return ATTN_OK;
}

}  // namespace
}  // namespace mlakv

using namespace mlakv;

extern "C" __attribute__((visibility("default"))) int attn_kv_append_rope(
    const void *q, const void *k_new, const void *v_new, const int *positions, const float *freqs_cis, void *q_out,
    void *k_cache, void *v_cache, int *new_lens, int B, int Hq, int Hkv, int D, int S_max, attn_dtype dtype,
    mlakv_stream_t stream) {
    const char *who = "attn_kv_append_rope";
    if (!q || !k_new || !v_new || !positions || !freqs_cis || !q_out || !k_cache || !v_cache)
        return report_error(ATTN_ERR_NULL, "attn_kv_append_rope: every pointer except new_lens must be non-NULL");
    if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || S_max < 1)
        return report_error(ATTN_ERR_SHAPE, "attn_kv_append_rope: B, Hq, Hkv, D and S_max must be >= 1");
    if (Hq % Hkv != 0)
        return report_error(ATTN_ERR_SHAPE, "attn_kv_append_rope: Hq must be a multiple of Hkv");
    if (dtype != ATTN_BF16 && dtype != ATTN_F32)
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_kv_append_rope: dtype must be ATTN_F32 or ATTN_BF16");
    const int v = dtype == ATTN_BF16 ? 8 : 4;
    if (D % v != 0)
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_kv_append_rope: D must be a multiple of 8 (bf16) or 4 (fp32)");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(positions) || !aligned16(freqs_cis) ||
        !aligned16(q_out) || !aligned16(k_cache) || !aligned16(v_cache) || (new_lens && !aligned16(new_lens)))
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_kv_append_rope: every pointer must be 16-byte aligned");
    AppendArgs a{q, k_new, v_new, positions, reinterpret_cast<const float2 *>(freqs_cis), q_out, k_cache, v_cache,
                 new_lens, Hq, Hkv, D, Hkv, D, S_max};
    return launch_append(a, B, dtype, stream, who);
}

extern "C" __attribute__((visibility("default"))) int attn_mla_append_rope(
    const void *q_rope, const void *c_new, const void *kr_new, const int *positions, const float *freqs_cis,
    void *q_rope_out, void *c_cache, void *krope_cache, int *new_lens, int B, int Hq, int r, int dr, int S_max,
    mlakv_stream_t stream) {
    const char *who = "attn_mla_append_rope";
    if (!q_rope || !c_new || !kr_new || !positions || !freqs_cis || !q_rope_out || !c_cache || !krope_cache)
        return report_error(ATTN_ERR_NULL, "attn_mla_append_rope: every pointer except new_lens must be non-NULL");
    if (B < 1 || Hq < 1 || r < 1 || dr < 1 || S_max < 1)
        return report_error(ATTN_ERR_SHAPE, "attn_mla_append_rope: B, Hq, r, dr and S_max must be >= 1");
    if (r % 8 != 0 || dr % 8 != 0)
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_mla_append_rope: r and dr must be multiples of 8");
    if (!aligned16(q_rope) || !aligned16(c_new) || !aligned16(kr_new) || !aligned16(positions) ||
        !aligned16(freqs_cis) || !aligned16(q_rope_out) || !aligned16(c_cache) || !aligned16(krope_cache) ||
        (new_lens && !aligned16(new_lens)))
        return report_error(ATTN_ERR_UNSUPPORTED, "attn_mla_append_rope: every pointer must be 16-byte aligned");
    AppendArgs a{q_rope, kr_new, c_new, positions, reinterpret_cast<const float2 *>(freqs_cis), q_rope_out,
                 krope_cache, c_cache, new_lens, Hq, 1, dr, 1, r, S_max};
    return launch_append(a, B, ATTN_BF16, stream, who);
}
