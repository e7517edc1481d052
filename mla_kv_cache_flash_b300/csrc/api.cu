// The library's C ABI (declared in include/mlakv.h): host-side validation, the split-KV
// plan, workspace carving and kernel dispatch. Nothing here allocates device memory or
// synchronises, except attn_check_status, whose job is to synchronise.
#include "../../include/mlakv.h"
#include "common.cuh"

#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#define MLAKV_API extern "C" __attribute__((visibility("default")))

namespace mlakv {
namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return ATTN_OK;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}


// SM count of the current device. The split plan must be the same for the workspace query
// and the launch; both run on the caller's current device. Without a device (a host with
// no GPU) the plan is made for a 148-SM part.
int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 148;
    }
    return n;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SplitPlan {
    int n_split;
    int split_len;
};

// Cut [0, max_S) into n_split pieces of split_len tokens (a multiple of `tile`). With
// n_split = 0 the count is the largest that keeps the whole grid (blocks_per_split ·
// n_split blocks) within one wave of `resident` blocks per SM, without making a piece
// shorter than `min_tiles` tiles. A second, partial wave of equally long blocks would nearly
// double the time (measured on B300: MQA decode 62.8 µs with 256 blocks, 95.4 µs with 320).
SplitPlan plan_splits(int max_S, int tile, long blocks_per_split, int n_split_req, int min_tiles,
                      int resident = 2) {
    SplitPlan p{1, tile};
    const int max_tiles = max_S > 0 ? (max_S + tile - 1) / tile : 1;
    int n;
    if (n_split_req > 0) {
        n = n_split_req;
    } else {
        const long slots = (long)resident * device_sms();
        n = (int)(slots / blocks_per_split);
        const int cap = max_tiles / (min_tiles > 0 ? min_tiles : 1);
        if (n > cap) n = cap;
        if (n > 64) n = 64;
        if (n < 1) n = 1;
    }
    if (n > max_tiles) n = max_tiles;
    const int tiles_per = (max_tiles + n - 1) / n;
    p.split_len = tiles_per * tile;
    p.n_split = max_S > 0 ? (max_S + p.split_len - 1) / p.split_len : 1;
    if (n_split_req > 0 && p.n_split < n_split_req) {
        // an explicit request is honoured exactly; trailing pieces are then empty
        p.n_split = n_split_req;
    }
    return p;
}

// ---------------------------------------------------------------- GQA decode plan

constexpr int kFmaTile = 128;

bool gqa_use_fma(attn_dtype dtype) { return dtype == ATTN_F32 || dtype == ATTN_FP8_E4M3; }

// E4M3 caches with up to 16 query heads per KV head run on the tensor-core fp8 kernel (the
// balanced split over persistent blocks, merged in-kernel); others on the CUDA-core kernel.
bool fp8_on_mma(int B, int Hq, int Hkv, int D, attn_dtype dtype) {
    return dtype == ATTN_FP8_E4M3 && decode_fp8_mma_eligible(B, Hq, Hkv, D);
}

SplitPlan gqa_plan(int B, int Hq, int Hkv, int D, int max_S, attn_dtype dtype, int n_split) {
    const int G = Hq / Hkv;
    // the fp8 tensor-core kernel: n_split reports the persistent grid size
    if (fp8_on_mma(B, Hq, Hkv, D, dtype)) return SplitPlan{decode_fp8_blocks(B, Hq, Hkv, D, n_split), 0};
    if (gqa_use_fma(dtype)) {
        const int hb = (G % 8 == 0) ? 8 : (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
        // 128-thread blocks: up to 8 resident per SM for 1-2 stacked heads (≈40 registers a
        // thread), 4 for 4-8 heads (≈110 registers)
        return plan_splits(max_S, kFmaTile, (long)B * Hkv * (G / hb), n_split, 2, hb <= 2 ? 8 : 4);
    }
    // bf16: the balanced split; n_split reports the persistent grid size
    if (decode_tc_gqa_eligible(B, Hq, Hkv, D)) return SplitPlan{decode_tc_gqa_blocks(B, Hq, Hkv, n_split), 0};
    return SplitPlan{decode_gqa_stream_blocks(B, Hq, Hkv, D, n_split), 0};
}

// Partials of the CUDA-core decode (merged by a second launch): o_part then lse_part, after
// the workspace's counter region (which this path leaves alone, so that a workspace shared
// with the bf16 kernels keeps its counters zero).
size_t partials_bytes(int B, int Hq, int Dv, int n_split) {
    if (n_split <= 1) return 0;
    const size_t rows = (size_t)B * Hq;
    return kCounterRegionBytes + align_up(rows * n_split * Dv * sizeof(float), 256) +
           align_up(rows * n_split * sizeof(float), 256);
}

void carve_partials(void *workspace, int B, int Hq, int Dv, int n_split, float **o_part, float **lse_part) {
    const size_t rows = (size_t)B * Hq;
    char *w = static_cast<char *>(workspace) + kCounterRegionBytes;
    *o_part = reinterpret_cast<float *>(w);
    *lse_part = reinterpret_cast<float *>(w + align_up(rows * n_split * Dv * sizeof(float), 256));
}

int check_gqa_shapes(int B, int Hq, int Hkv, int D, int S_max, int max_S, attn_dtype dtype, int n_split) {
    if (B < 1 || Hq < 1 || Hkv < 1 || S_max < 1)
        return fail(ATTN_ERR_SHAPE, "B, Hq, Hkv and S_max must be >= 1 (got B=%d Hq=%d Hkv=%d S_max=%d)",
                    B, Hq, Hkv, S_max);
    if (Hq % Hkv != 0)
        return fail(ATTN_ERR_SHAPE, "Hkv=%d does not divide Hq=%d: every KV group needs the same whole "
                    "number of query heads", Hkv, Hq);
    if (max_S < 0 || max_S > S_max)
        return fail(ATTN_ERR_SHAPE, "max_S=%d must lie in [0, S_max=%d]", max_S, S_max);
    if (n_split < 0 || n_split > 256)
        return fail(ATTN_ERR_SHAPE, "n_split=%d must lie in [0, 256]", n_split);
    if (D != 64 && D != 96 && D != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "head width D=%d not built (64, 96, 128)", D);
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_FP8_E4M3)
        return fail(ATTN_ERR_UNSUPPORTED, "dtype %d not built (ATTN_F32, ATTN_BF16, ATTN_FP8_E4M3)", (int)dtype);
    if (Hq / Hkv > 128)
        return fail(ATTN_ERR_UNSUPPORTED, "group size Hq/Hkv=%d above 128", Hq / Hkv);
    return ATTN_OK;
}

// ---------------------------------------------------------------- MLA decode plan

constexpr int kMlaRank = 128;
constexpr int kMlaRope = 48;
constexpr int kMlaHeadsPerBlock = 16;

int check_mla_shapes(int B, int Hq, int r, int dr, int S_max, int max_S, int n_split) {
    if (B < 1 || Hq < 1 || S_max < 1)
        return fail(ATTN_ERR_SHAPE, "B, Hq and S_max must be >= 1 (got B=%d Hq=%d S_max=%d)", B, Hq, S_max);
    if (max_S < 0 || max_S > S_max)
        return fail(ATTN_ERR_SHAPE, "max_S=%d must lie in [0, S_max=%d]", max_S, S_max);
    if (n_split < 0 || n_split > 256)
        return fail(ATTN_ERR_SHAPE, "n_split=%d must lie in [0, 256]", n_split);
    if (r != kMlaRank || dr != kMlaRope)
        return fail(ATTN_ERR_UNSUPPORTED, "MLA rank r=%d, rope width dr=%d not built (r=128, dr=48)", r, dr);
    if (Hq % kMlaHeadsPerBlock != 0 || Hq > 128)
        return fail(ATTN_ERR_UNSUPPORTED, "MLA head count Hq=%d must be a multiple of 16 up to 128", Hq);
    if (!decode_tc_mla_fits(B, Hq))
        return fail(ATTN_ERR_UNSUPPORTED, "MLA batch B=%d too large for the kernel's shared-memory plan", B);
    return ATTN_OK;
}



}  // namespace

// Lets other translation units report through attn_last_error().
int report_error(int code, const char *message) { return fail(code, "%s", message); }
int report_cuda_error(cudaError_t e, const char *what) { return cuda_fail(e, what); }

}  // namespace mlakv

using namespace mlakv;

MLAKV_API const char *attn_last_error(void) { return g_err; }

MLAKV_API const char *attn_version(void) { return "mlakv 0.1.0 (sm_103a)"; }

MLAKV_API int attn_set_device_checks(int on) { return set_device_checks(on); }
MLAKV_API int attn_device_checks(void) { return device_checks_on() ? 1 : 0; }

// ======================================================================== GQA decode

namespace {

// The CUDA-core decode (fp32 or E4M3 cache): split plan, workspace check, decode, merge.
int decode_fma(DecodeGqaArgs a, int B, int Hq, int Hkv, int D, float scale, int S_max, int max_S,
               attn_dtype dtype, int n_split, void *workspace, size_t ws_bytes, cudaStream_t s, const char *who) {
    const SplitPlan p = gqa_plan(B, Hq, Hkv, D, max_S, dtype, n_split);
    const size_t need = partials_bytes(B, Hq, D, p.n_split);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace)))
        return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu at %p", who,
                    need, workspace ? ws_bytes : (size_t)0, workspace);
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D;
    a.scale_log2 = scale * kLog2e;
    a.S_max = S_max;
    a.n_split = p.n_split;
    a.split_len = p.split_len;
    if (p.n_split > 1) carve_partials(workspace, B, Hq, D, p.n_split, &a.o_part, &a.lse_part);
    char what[96];
    cudaError_t e = dtype == ATTN_FP8_E4M3 ? launch_decode_gqa_fp8(a, s) : launch_decode_gqa_f32(a, s);
    if (e != cudaSuccess) {
        snprintf(what, sizeof(what), "%s: decode kernel launch", who);
        return cuda_fail(e, what);
    }
    if (p.n_split > 1) {
        e = launch_merge(a.o_part, a.lse_part, a.out, B * Hq, p.n_split, D, s);
        if (e != cudaSuccess) {
            snprintf(what, sizeof(what), "%s: merge kernel launch", who);
            return cuda_fail(e, what);
        }
    }
    return ok();
}

}  // namespace

MLAKV_API int attn_decode_gqa_num_splits(int B, int Hq, int Hkv, int D, int max_S, attn_dtype dtype,
                                         int n_split) {
    const int rc = check_gqa_shapes(B, Hq, Hkv, D, max_S > 0 ? max_S : 1, max_S, dtype, n_split);
    if (rc != ATTN_OK) return rc;
    return gqa_plan(B, Hq, Hkv, D, max_S, dtype, n_split).n_split;
}

MLAKV_API size_t attn_decode_gqa_workspace_size(int B, int Hq, int Hkv, int D, int max_S, attn_dtype dtype,
                                                int n_split) {
    if (check_gqa_shapes(B, Hq, Hkv, D, max_S > 0 ? max_S : 1, max_S, dtype, n_split) != ATTN_OK) return 0;
    if (!gqa_use_fma(dtype))
        return decode_tc_gqa_eligible(B, Hq, Hkv, D) ? decode_tc_gqa_workspace(B, Hq, Hkv, n_split)
                                                     : decode_gqa_stream_workspace(B, Hq, Hkv, D, n_split);
    if (fp8_on_mma(B, Hq, Hkv, D, dtype)) return decode_fp8_workspace(B, Hq, Hkv, D, n_split);
    const SplitPlan p = gqa_plan(B, Hq, Hkv, D, max_S, dtype, n_split);
    return partials_bytes(B, Hq, D, p.n_split);
}

MLAKV_API int attn_decode_gqa(const void *q, const void *k_cache, const void *v_cache, const int *seq_lens,
                              float *out, int B, int Hq, int Hkv, int D, float scale, int S_max, int max_S,
                              attn_dtype dtype, int n_split, void *workspace, size_t ws_bytes,
                              mlakv_stream_t stream) {
    if (!q || !k_cache || !v_cache || !seq_lens || !out)
        return fail(ATTN_ERR_NULL, "attn_decode_gqa: q, k_cache, v_cache, seq_lens and out must be non-NULL");
    int rc = check_gqa_shapes(B, Hq, Hkv, D, S_max, max_S, dtype, n_split);
    if (rc != ATTN_OK) return rc;
    if (dtype == ATTN_FP8_E4M3)
        return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_gqa: an fp8 cache needs its scales; call attn_decode_gqa_fp8");
    if (!isfinite(scale)) return fail(ATTN_ERR_SHAPE, "scale must be finite");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(seq_lens))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_gqa: every pointer must be 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (device_checks_on() && (rc = check_lengths(seq_lens, B, max_S, s, "attn_decode_gqa")) != ATTN_OK) return rc;
    if (!gqa_use_fma(dtype)) {
        // bf16: persistent blocks over an even share of all cached tokens, merged in-kernel
        const bool tc = decode_tc_gqa_eligible(B, Hq, Hkv, D);
        const size_t need = tc ? decode_tc_gqa_workspace(B, Hq, Hkv, n_split)
                               : decode_gqa_stream_workspace(B, Hq, Hkv, D, n_split);
        if (!workspace || ws_bytes < need || !aligned16(workspace))
            return fail(ATTN_ERR_WORKSPACE, "attn_decode_gqa: workspace of %zu bytes (16-byte aligned) needed, "
                        "got %zu at %p", need, workspace ? ws_bytes : (size_t)0, workspace);
        if (tc) {
            const cudaError_t e = launch_decode_tc_gqa(q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, scale * kLog2e,
                                                       S_max, n_split, workspace, s);
            if (e != cudaSuccess) return cuda_fail(e, "attn_decode_gqa: kernel launch");
            return ok();
        }
        DecodeStreamArgs a{};
        a.q = q; a.k = k_cache; a.v = v_cache; a.seq_lens = seq_lens; a.out = out;
        a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D;
        a.scale_log2 = scale * kLog2e;
        a.S_max = S_max;
        a.n_blocks = decode_gqa_stream_blocks(B, Hq, Hkv, D, n_split);
        a.aligned = decode_gqa_stream_aligned(B, Hq, Hkv, n_split) ? 1 : 0;
        // the arrival counters first, then the partial outputs, then their log-sum-exps
        const size_t n_cnt = decode_gqa_stream_counters(B, Hq, Hkv);
        char *w = static_cast<char *>(workspace);
        a.counters = reinterpret_cast<int *>(w);
        a.o_part = reinterpret_cast<float *>(w + counter_region_bytes(n_cnt));
        a.lse_part = reinterpret_cast<float *>(w + counter_region_bytes(n_cnt) +
                                               decode_gqa_stream_o_bytes(B, Hq, Hkv, D, n_split));
        cudaError_t e = clear_overflow_counters(a.counters, n_cnt, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_decode_gqa: clearing the arrival counters");
        e = launch_decode_gqa_stream(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_decode_gqa: kernel launch");
        return ok();
    }
    DecodeGqaArgs a{};
    a.q = q; a.k = k_cache; a.v = v_cache; a.seq_lens = seq_lens; a.out = out;
    return decode_fma(a, B, Hq, Hkv, D, scale, S_max, max_S, dtype, n_split, workspace, ws_bytes, s,
                      "attn_decode_gqa");
}

MLAKV_API int attn_decode_gqa_fp8(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                                  const float *v_scale, const int *seq_lens, float *out, int B, int Hq, int Hkv,
                                  int D, float scale, int S_max, int max_S, int n_split, void *workspace,
                                  size_t ws_bytes, mlakv_stream_t stream) {
    if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !seq_lens || !out)
        return fail(ATTN_ERR_NULL, "attn_decode_gqa_fp8: q, k_cache, v_cache, k_scale, v_scale, seq_lens and out "
                    "must be non-NULL");
    int rc = check_gqa_shapes(B, Hq, Hkv, D, S_max, max_S, ATTN_FP8_E4M3, n_split);
    if (rc != ATTN_OK) return rc;
    if (!isfinite(scale)) return fail(ATTN_ERR_SHAPE, "scale must be finite");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) ||
        !aligned16(v_scale) || !aligned16(out) || !aligned16(seq_lens))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_gqa_fp8: every pointer must be 16-byte aligned");
    if (device_checks_on() &&
        (rc = check_lengths(seq_lens, B, max_S, reinterpret_cast<cudaStream_t>(stream), "attn_decode_gqa_fp8")) !=
            ATTN_OK)
        return rc;
    if (fp8_on_mma(B, Hq, Hkv, D, ATTN_FP8_E4M3)) {
        const size_t need = decode_fp8_workspace(B, Hq, Hkv, D, n_split);
        if (!workspace || ws_bytes < need || !aligned16(workspace))
            return fail(ATTN_ERR_WORKSPACE, "attn_decode_gqa_fp8: workspace of %zu bytes (16-byte aligned) needed, "
                        "got %zu at %p", need, workspace ? ws_bytes : (size_t)0, workspace);
        const cudaError_t e = launch_decode_fp8_mma(q, k_cache, v_cache, k_scale, v_scale, seq_lens, out, B, Hq, Hkv,
                                                    D, scale * kLog2e, S_max, n_split, workspace,
                                                    reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "attn_decode_gqa_fp8: kernel launch");
        return ok();
    }
    DecodeGqaArgs a{};
    a.q = q; a.k = k_cache; a.v = v_cache; a.seq_lens = seq_lens; a.out = out;
    a.k_scale = k_scale; a.v_scale = v_scale;
    return decode_fma(a, B, Hq, Hkv, D, scale, S_max, max_S, ATTN_FP8_E4M3, n_split, workspace, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream), "attn_decode_gqa_fp8");
}

// ======================================================================== chunked prefill

namespace {

constexpr int kMaxGridZ = 65535;

int check_chunked(int B, int T, int Hq, int Hkv, int D, int S_max, int max_kv, attn_dtype dtype, int n_split,
                  const char *who) {
    if (T < 0 || T > kMaxGridZ)
        return fail(ATTN_ERR_SHAPE, "%s: T=%d new tokens must lie in [0, %d]", who, T, kMaxGridZ);
    if (dtype != ATTN_F32 && dtype != ATTN_BF16)
        return fail(ATTN_ERR_UNSUPPORTED, "%s: dtype must be ATTN_F32 or ATTN_BF16", who);
    return check_gqa_shapes(B, Hq, Hkv, D, S_max, max_kv, dtype, n_split);
}

// Blocks per split: one per (query row, KV head, block of stacked heads), as for the
// CUDA-core decode with the packed rows in place of the sequences.
SplitPlan chunked_plan(int T, int Hq, int Hkv, int D, int max_kv, int n_split) {
    return gqa_plan(T > 0 ? T : 1, Hq, Hkv, D, max_kv, ATTN_F32, n_split);
}

// bf16 at D = 128 with chunks of at least 128 new tokens on average: the tcgen05 prefill kernel
// in its cache form, 128 new tokens × one head per MMA tile, so the decode kernels' re-reading
// of the cache once per few new tokens is gone
bool chunk_on_prefill(int B, int T, int D, attn_dtype dtype) {
    return dtype == ATTN_BF16 && D == 128 && B > 0 && (long long)T >= 128LL * B;
}
// Shorter chunks: bf16 caches whose query groups are a multiple of 16 heads at D = 128 (and
// every MLA cache with Hq a multiple of 16) run on the tcgen05 decode kernel, 4 new tokens × 16
// heads per block reading each cached row once; other bf16 shapes on the register-MMA decode
// kernel; the rest on the CUDA-core form, one new token per block.
bool chunk_on_tc_gqa(int B, int Hq, int Hkv, int D, attn_dtype dtype) {
    return dtype == ATTN_BF16 && decode_tc_gqa_chunk_eligible(B, Hq, Hkv, D);
}
// other bf16 caches with up to 16 query heads per KV head: the register-MMA decode kernel,
// 16 / G new tokens × G heads per MMA tile, when the batch's tables fit beside its ring
bool chunk_on_stream(int B, int T, int Hq, int Hkv, int D, attn_dtype dtype, int n_split) {
    return dtype == ATTN_BF16 && !chunk_on_tc_gqa(B, Hq, Hkv, D, dtype) && decode_gqa_stream_chunk_eligible(Hq, Hkv) &&
           decode_gqa_stream_chunk_fits(B, T, Hq, Hkv, D, n_split);
}
bool chunk_on_tc_mla(int B, int Hq) { return Hq % 16 == 0 && Hq <= 128 && decode_tc_mla_chunk_fits(B); }

}  // namespace

MLAKV_API size_t attn_prefill_gqa_chunked_workspace_size(int B, int T, int Hq, int Hkv, int D, int max_kv,
                                                         attn_dtype dtype, int n_split) {
    if (check_chunked(B, T, Hq, Hkv, D, max_kv > 0 ? max_kv : 1, max_kv, dtype, n_split,
                      "attn_prefill_gqa_chunked_workspace_size") != ATTN_OK || T == 0)
        return 0;
    if (chunk_on_prefill(B, T, D, dtype)) return 0;
    if (chunk_on_tc_gqa(B, Hq, Hkv, D, dtype)) return decode_tc_gqa_chunk_workspace(B, T, Hq, Hkv, n_split);
    if (chunk_on_stream(B, T, Hq, Hkv, D, dtype, n_split))
        return decode_gqa_stream_chunk_workspace(B, T, Hq, Hkv, D, n_split);
    return partials_bytes(T, Hq, D, chunked_plan(T, Hq, Hkv, D, max_kv, n_split).n_split);
}

MLAKV_API int attn_prefill_gqa_chunked(const void *q, const void *k_cache, const void *v_cache, const int *cu_q,
                                       const int *start_pos, float *out, int B, int T, int Hq, int Hkv, int D,
                                       float scale, int S_max, int max_kv, attn_dtype dtype, int n_split,
                                       void *workspace, size_t ws_bytes, mlakv_stream_t stream) {
    const char *who = "attn_prefill_gqa_chunked";
    if (!q || !k_cache || !v_cache || !cu_q || !start_pos || !out)
        return fail(ATTN_ERR_NULL, "%s: q, k_cache, v_cache, cu_q, start_pos and out must be non-NULL", who);
    const int rc = check_chunked(B, T, Hq, Hkv, D, S_max, max_kv, dtype, n_split, who);
    if (rc != ATTN_OK) return rc;
    if (!isfinite(scale)) return fail(ATTN_ERR_SHAPE, "scale must be finite");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(cu_q) || !aligned16(start_pos) ||
        !aligned16(out))
        return fail(ATTN_ERR_UNSUPPORTED, "%s: every pointer must be 16-byte aligned", who);
    if (T == 0 || max_kv == 0) return ok();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (device_checks_on()) {
        const int crc = check_chunks(cu_q, start_pos, B, T, max_kv, s, who);
        if (crc != ATTN_OK) return crc;
    }
    if (chunk_on_prefill(B, T, D, dtype)) {
        PrefillArgs a{};
        a.q = q; a.k = k_cache; a.v = v_cache; a.cu_seqlens = cu_q; a.out = out;
        a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.T = T;
        a.scale_log2 = scale * kLog2e;
        a.max_seqlen = T < max_kv ? T : max_kv;      // no chunk is longer than either
        a.out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
        a.start_pos = start_pos; a.S_max = S_max;
        const cudaError_t e = launch_prefill(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_gqa_chunked: kernel launch");
        return ok();
    }
    if (chunk_on_tc_gqa(B, Hq, Hkv, D, dtype)) {
        const size_t need = decode_tc_gqa_chunk_workspace(B, T, Hq, Hkv, n_split);
        if (!workspace || ws_bytes < need || !aligned16(workspace))
            return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu at %p",
                        who, need, workspace ? ws_bytes : (size_t)0, workspace);
        const cudaError_t e = launch_decode_tc_gqa_chunk(q, k_cache, v_cache, cu_q, start_pos, out, B, T, Hq, Hkv,
                                                         scale * kLog2e, S_max, n_split, workspace, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_gqa_chunked: kernel launch");
        return ok();
    }
    if (chunk_on_stream(B, T, Hq, Hkv, D, dtype, n_split)) {
        const size_t need = decode_gqa_stream_chunk_workspace(B, T, Hq, Hkv, D, n_split);
        if (!workspace || ws_bytes < need || !aligned16(workspace))
            return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu at %p",
                        who, need, workspace ? ws_bytes : (size_t)0, workspace);
        const cudaError_t e = launch_decode_gqa_stream_chunk(q, k_cache, v_cache, cu_q, start_pos, out, B, T, Hq,
                                                             Hkv, D, scale * kLog2e, S_max, n_split, workspace, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_gqa_chunked: kernel launch");
        return ok();
    }
    const SplitPlan p = chunked_plan(T, Hq, Hkv, D, max_kv, n_split);
    const size_t need = partials_bytes(T, Hq, D, p.n_split);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace)))
        return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu at %p", who,
                    need, workspace ? ws_bytes : (size_t)0, workspace);
    DecodeGqaArgs a{};
    a.q = q; a.k = k_cache; a.v = v_cache; a.out = out;
    a.cu_q = cu_q; a.start_pos = start_pos; a.n_seq = B;
    a.B = T; a.Hq = Hq; a.Hkv = Hkv; a.D = D;
    a.scale_log2 = scale * kLog2e;
    a.S_max = S_max;
    a.n_split = p.n_split;
    a.split_len = p.split_len;
    if (p.n_split > 1) carve_partials(workspace, T, Hq, D, p.n_split, &a.o_part, &a.lse_part);
    cudaError_t e = dtype == ATTN_BF16 ? launch_prefill_chunked_bf16(a, s) : launch_decode_gqa_f32(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_gqa_chunked: kernel launch");
    if (p.n_split > 1) {
        e = launch_merge(a.o_part, a.lse_part, out, T * Hq, p.n_split, D, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_gqa_chunked: merge kernel launch");
    }
    return ok();
}

MLAKV_API size_t attn_prefill_mla_chunked_workspace_size(int B, int T, int Hq, int max_kv, int n_split) {
    if (check_chunked(B, T, Hq, 1, 128, max_kv > 0 ? max_kv : 1, max_kv, ATTN_BF16, n_split,
                      "attn_prefill_mla_chunked_workspace_size") != ATTN_OK || T == 0)
        return 0;
    if (chunk_on_prefill(B, T, kMlaRank, ATTN_BF16)) return 0;
    if (chunk_on_tc_mla(B, Hq)) return decode_tc_mla_chunk_workspace(B, T, Hq, n_split);
    return partials_bytes(T, Hq, kMlaRank, chunked_plan(T, Hq, 1, kMlaRank, max_kv, n_split).n_split);
}

MLAKV_API int attn_prefill_mla_chunked(const void *q_lat, const void *q_rope, const void *c_cache,
                                       const void *krope_cache, const int *cu_q, const int *start_pos, float *out_lat,
                                       int B, int T, int Hq, int r, int dr, float scale, int S_max, int max_kv,
                                       int n_split, void *workspace, size_t ws_bytes, mlakv_stream_t stream) {
    const char *who = "attn_prefill_mla_chunked";
    if (!q_lat || !q_rope || !c_cache || !krope_cache || !cu_q || !start_pos || !out_lat)
        return fail(ATTN_ERR_NULL, "%s: q_lat, q_rope, c_cache, krope_cache, cu_q, start_pos and out_lat must be "
                    "non-NULL", who);
    const int rc = check_chunked(B, T, Hq, 1, 128, S_max, max_kv, ATTN_BF16, n_split, who);
    if (rc != ATTN_OK) return rc;
    if (r != kMlaRank || dr != kMlaRope)
        return fail(ATTN_ERR_UNSUPPORTED, "%s: MLA rank r=%d, rope width dr=%d not built (r=128, dr=48)", who, r, dr);
    if (!isfinite(scale)) return fail(ATTN_ERR_SHAPE, "scale must be finite");
    if (!aligned16(q_lat) || !aligned16(q_rope) || !aligned16(c_cache) || !aligned16(krope_cache) ||
        !aligned16(cu_q) || !aligned16(start_pos) || !aligned16(out_lat))
        return fail(ATTN_ERR_UNSUPPORTED, "%s: every pointer must be 16-byte aligned", who);
    if (T == 0 || max_kv == 0) return ok();
    if (device_checks_on()) {
        const int crc = check_chunks(cu_q, start_pos, B, T, max_kv, reinterpret_cast<cudaStream_t>(stream), who);
        if (crc != ATTN_OK) return crc;
    }
    if (chunk_on_prefill(B, T, kMlaRank, ATTN_BF16)) {
        // long chunks: the tcgen05 prefill kernel in its MLA form
        PrefillArgs a{};
        a.q = q_lat; a.q_rope = q_rope; a.k = c_cache; a.v = krope_cache; a.cu_seqlens = cu_q; a.out = out_lat;
        a.B = B; a.Hq = Hq; a.Hkv = 1; a.D = kMlaRank; a.T = T;
        a.scale_log2 = scale * kLog2e;
        a.max_seqlen = T < max_kv ? T : max_kv;
        a.out32 = (reinterpret_cast<uintptr_t>(out_lat) & 31u) == 0;
        a.start_pos = start_pos; a.S_max = S_max;
        const cudaError_t e = launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_mla_chunked: kernel launch");
        return ok();
    }
    if (chunk_on_tc_mla(B, Hq)) {
        const size_t need = decode_tc_mla_chunk_workspace(B, T, Hq, n_split);
        if (!workspace || ws_bytes < need || !aligned16(workspace))
            return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu at %p",
                        who, need, workspace ? ws_bytes : (size_t)0, workspace);
        const cudaError_t e = launch_decode_tc_mla_chunk(q_lat, q_rope, c_cache, krope_cache, cu_q, start_pos, out_lat,
                                                         B, T, Hq, scale * kLog2e, S_max, n_split, workspace,
                                                         reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_mla_chunked: kernel launch");
        return ok();
    }
    const SplitPlan p = chunked_plan(T, Hq, 1, kMlaRank, max_kv, n_split);
    const size_t need = partials_bytes(T, Hq, kMlaRank, p.n_split);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace)))
        return fail(ATTN_ERR_WORKSPACE, "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu at %p", who,
                    need, workspace ? ws_bytes : (size_t)0, workspace);
    DecodeGqaArgs a{};
    a.q = q_lat; a.q2 = q_rope; a.k = c_cache; a.v = c_cache; a.k2 = krope_cache; a.out = out_lat;
    a.cu_q = cu_q; a.start_pos = start_pos; a.n_seq = B;
    a.B = T; a.Hq = Hq; a.Hkv = 1; a.D = kMlaRank;
    a.scale_log2 = scale * kLog2e;
    a.S_max = S_max;
    a.n_split = p.n_split;
    a.split_len = p.split_len;
    if (p.n_split > 1) carve_partials(workspace, T, Hq, kMlaRank, p.n_split, &a.o_part, &a.lse_part);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_prefill_chunked_mla(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_mla_chunked: kernel launch");
    if (p.n_split > 1) {
        e = launch_merge(a.o_part, a.lse_part, out_lat, T * Hq, p.n_split, kMlaRank, s);
        if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_mla_chunked: merge kernel launch");
    }
    return ok();
}

// ======================================================================== MLA decode

MLAKV_API int attn_decode_mla_num_splits(int B, int Hq, int r, int dr, int max_S, int n_split) {
    const int rc = check_mla_shapes(B, Hq, r, dr, max_S > 0 ? max_S : 1, max_S, n_split);
    if (rc != ATTN_OK) return rc;
    return decode_tc_mla_blocks(B, Hq, n_split);
}

MLAKV_API size_t attn_decode_mla_workspace_size(int B, int Hq, int r, int dr, int max_S, int n_split) {
    if (check_mla_shapes(B, Hq, r, dr, max_S > 0 ? max_S : 1, max_S, n_split) != ATTN_OK) return 0;
    return decode_tc_mla_workspace(B, Hq, n_split);
}

MLAKV_API int attn_decode_mla_absorbed(const void *q_lat, const void *q_rope, const void *c_cache,
                                       const void *krope_cache, const int *seq_lens, float *out_lat, int B,
                                       int Hq, int r, int dr, float scale, int S_max, int max_S, int n_split,
                                       void *workspace, size_t ws_bytes, mlakv_stream_t stream) {
    if (!q_lat || !q_rope || !c_cache || !krope_cache || !seq_lens || !out_lat)
        return fail(ATTN_ERR_NULL, "attn_decode_mla_absorbed: every tensor pointer must be non-NULL");
    int rc = check_mla_shapes(B, Hq, r, dr, S_max, max_S, n_split);
    if (rc != ATTN_OK) return rc;
    if (!isfinite(scale)) return fail(ATTN_ERR_SHAPE, "scale must be finite");
    if (!aligned16(q_lat) || !aligned16(q_rope) || !aligned16(c_cache) || !aligned16(krope_cache) ||
        !aligned16(out_lat) || !aligned16(seq_lens))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_mla_absorbed: every pointer must be 16-byte aligned");
    if (device_checks_on() && (rc = check_lengths(seq_lens, B, max_S, reinterpret_cast<cudaStream_t>(stream),
                                                  "attn_decode_mla_absorbed")) != ATTN_OK)
        return rc;
    const size_t need = decode_tc_mla_workspace(B, Hq, n_split);
    if (!workspace || ws_bytes < need || !aligned16(workspace))
        return fail(ATTN_ERR_WORKSPACE, "attn_decode_mla_absorbed: workspace of %zu bytes (16-byte aligned) "
                    "needed, got %zu", need, workspace ? ws_bytes : (size_t)0);
    const cudaError_t e = launch_decode_tc_mla(q_lat, q_rope, c_cache, krope_cache, seq_lens, out_lat, B, Hq,
                                               scale * kLog2e, S_max, n_split, workspace,
                                               reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_mla_absorbed: kernel launch");
    return ok();
}

// ======================================================================== prefill

MLAKV_API int attn_prefill_gqa_causal(const void *q, const void *k, const void *v, const int *cu_seqlens,
                                      float *out, int B, int Hq, int Hkv, int D, float scale, int max_seqlen,
                                      int total_tokens, mlakv_stream_t stream) {
    if (B < 1 || Hq < 1 || Hkv < 1 || max_seqlen < 0 || total_tokens < 0)
        return fail(ATTN_ERR_SHAPE, "B, Hq, Hkv must be >= 1 and max_seqlen, total_tokens >= 0");
    if (!cu_seqlens || (total_tokens > 0 && (!q || !k || !v || !out)))
        return fail(ATTN_ERR_NULL, "attn_prefill_gqa_causal: q, k, v, cu_seqlens and out must be non-NULL");
    if (Hq % Hkv != 0)
        return fail(ATTN_ERR_SHAPE, "Hkv=%d does not divide Hq=%d", Hkv, Hq);
    if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "prefill head width D=%d not built (128)", D);
    if (!isfinite(scale)) return fail(ATTN_ERR_SHAPE, "scale must be finite");
    if (total_tokens == 0 || max_seqlen == 0) return ok();
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(cu_seqlens))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_prefill_gqa_causal: every pointer must be 16-byte aligned");
    if (device_checks_on()) {
        const int crc = check_offsets(cu_seqlens, B, total_tokens, max_seqlen, reinterpret_cast<cudaStream_t>(stream),
                                      "attn_prefill_gqa_causal");
        if (crc != ATTN_OK) return crc;
    }
    PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.cu_seqlens = cu_seqlens; a.out = out;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.T = total_tokens;
    a.scale_log2 = scale * kLog2e; a.max_seqlen = max_seqlen;
    a.out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    cudaError_t e = launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_prefill_gqa_causal: kernel launch");
    return ok();
}

// ======================================================================== merge, status

MLAKV_API int attn_merge_partials(const float *o_part, const float *lse_part, float *out, int rows, int n_split,
                                  int Dv, mlakv_stream_t stream) {
    if (!o_part || !lse_part || !out) return fail(ATTN_ERR_NULL, "attn_merge_partials: NULL pointer");
    if (rows < 0 || n_split < 1 || n_split > 256 || Dv < 4)
        return fail(ATTN_ERR_SHAPE, "attn_merge_partials: rows >= 0, 1 <= n_split <= 256, Dv >= 4");
    if (Dv % 4 != 0 || Dv > 512) return fail(ATTN_ERR_UNSUPPORTED, "Dv=%d must be a multiple of 4 up to 512", Dv);
    if (!aligned16(o_part) || !aligned16(out))
        return fail(ATTN_ERR_UNSUPPORTED, "attn_merge_partials: o_part and out must be 16-byte aligned");
    cudaError_t e = launch_merge(o_part, lse_part, out, rows, n_split, Dv, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_merge_partials: kernel launch");
    return ok();
}

MLAKV_API int attn_check_status(mlakv_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_check_status: stream");
    unsigned flag = 0, f = 0;
    int rc = decode_gqa_read_and_clear_status(s, &f);
    flag |= f;
    if (rc == 0) rc = decode_tc_read_and_clear_status(s, &f), flag |= f;
    if (rc == 0) rc = prefill_read_and_clear_status(s, &f), flag |= f;
    if (rc == 0) rc = selftest_read_and_clear_status(s, &f), flag |= f;
    if (rc == 0) rc = decode_fp8_read_and_clear_status(s, &f), flag |= f;
    if (rc != 0) return cuda_fail((cudaError_t)rc, "attn_check_status: reading the device flags");
    if (flag != 0) {
        // a decode that gave up may have left arrival counters set in the built-in scratch
        rc = noalloc_clear_counters(s);
        if (rc != 0) return cuda_fail((cudaError_t)rc, "attn_check_status: clearing the no-alloc counters");
        return fail(ATTN_ERR_TIMEOUT, "a kernel gave up a bounded wait (flags 0x%x); zero-fill any workspace "
                    "it used before reusing it", flag);
    }
    return ok();
}
