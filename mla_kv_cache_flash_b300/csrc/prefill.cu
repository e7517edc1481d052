// K4: causal GQA prefill on the 5th-generation tensor cores (tcgen05 MMA, tensor memory, TMA).
//
// The method ("模型架构｜MQA & GQA 调研", section "代码", Attention.forward over a whole prompt;
// the qqstock MLA code's scaled_dot_product_attention with is_causal=True): row i of a
// sequence attends keys 0 .. i of the same sequence through KV head h / G,
//   out[i, h] = Σ_{t ≤ i} softmax_t(scale · q[i,h]·k[t,j]) · v[t,j].
// It is the one dense contraction of the path, so both products run on tcgen05:
//
// One thread block = (sequence b, 128-row query tile qt, two query heads of one KV group).
// The two heads share the KV head, so every K/V tile that lands in shared memory feeds two
// 128×128 score tiles (GQA: each K/V byte is fetched once per pair of query heads, not per
// head). Query tiles with the most KV tiles are scheduled first. Warp roles:
//   warp 0     TMA producer: the two Q tiles once, then K and V tiles (128 keys × 128 columns,
//              128-byte swizzle) through a 2-stage ring.
//   warp 1     allocates 512 TMEM columns; lane 0 issues every MMA:
//                S_t = Q_t · K_nᵀ   (M=128, N=128, K=16 × 8; A, B K-major in shared memory)
//                O_t += P_t · V_n   (A = P from TMEM, B = V MN-major in shared memory)
//              and commits each group to an mbarrier.
//   warps 2-9  softmax, one warpgroup per query tile; thread = one query row (one TMEM
//              lane). It reads its 128 scores from TMEM, applies the causal mask on the
//              diagonal tile, keeps a running max m and sum l in the base-2 domain and writes
//              P = 2^(s·scale·log2 e − m) as bf16 back over its scores. The output is
//              rescaled only when the row max grows by more than 2^8 (the result is exact for
//              any reference value; this only bounds the range of P and l).
// At the end each softmax thread reads its O row from TMEM and writes O / l (fp32).
//
// TMEM: per query tile t, columns [256t, 256t+128) hold S (P aliases its first 64 columns,
// two bf16 per column) and [256t+128, 256t+256) hold O. An S tile is written only after the
// previous P·V of the same tile has completed, so P is never overwritten while in use.
//
// Precision: P is rounded to bf16 for the tensor cores, a relative error of up to 2^-8 per
// weight. Rows with many keys average it away, but rows near the start of a sequence see
// few keys (row 1 sees 2); in the first kSplitTiles query tiles P is therefore split into a
// bf16 head and a bf16 residual and both are multiplied with V, which leaves an error near
// 2^-16 there.
//
// Every wait is bounded (MLAKV_WAIT_TIMEOUT_NS): a wait that runs out sets a bit in
// g_prefill_status and the thread abandons its loop; every thread still reaches the final
// barrier, so tensor memory is always released.
#include "ptx.cuh"
#include "tcgen05.cuh"
#include "tensor_map.cuh"

#include <math.h>

namespace mlakv {

__device__ unsigned g_prefill_status;

namespace {

constexpr int HD = 128;                      // head width
constexpr int BM = 128;                      // query rows per tile
constexpr int BN = 128;                      // keys per KV tile
constexpr int NSTAGE = 2;                    // K/V ring depth
constexpr int TILE_BYTES = BM * HD * 2;      // one 128 × 128 bf16 tile: 32 KB
constexpr int BOX_BYTES = TILE_BYTES / 2;    // one TMA box: 128 rows × 64 columns (128 B)
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
constexpr int V_OFF = K_OFF + NSTAGE * TILE_BYTES;
constexpr int BAR_OFF = V_OFF + NSTAGE * TILE_BYTES;
constexpr int N_BARS = 16;
constexpr int SLOT_OFF = BAR_OFF + N_BARS * 8;
constexpr int SMEM = SLOT_OFF + 16 + 1024;   // + alignment slack
static_assert(SMEM <= 227 * 1024, "shared memory budget");

constexpr int kWarps = 10;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
// Query tiles 0 .. kSplitTiles-1 of a sequence (rows with at most 512 keys) multiply V with
// P as a bf16 head plus a bf16 residual; measured without it, bf16 P alone left errors up to
// 1.9e-3 in rows with 129-256 keys, and they shrink as rows see more keys.
constexpr int kSplitTiles = 4;

constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, false, false);   // Q K-major, K K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, HD, false, true);   // P from TMEM, V MN-major

// mbarrier slots (8 bytes each) inside the barrier block
enum : int {
    kQFull = 0,
    kKFull = 1,          // + stage
    kVFull = 3,          // + stage
    kKvEmpty = 5,        // + stage
    kSFull = 7,          // + query tile
    kPReady = 9,         // + query tile
    kODone = 11          // + query tile
};

// Row max of x = s·c (c = scale·log2 e) over one row of a score tile in TMEM (128 columns at
// s_addr). DIAG: the diagonal tile of a causal sequence, where key i is visible to `row` only
// if i <= row (key 0 always is, so the result is finite).
template <bool DIAG>
__device__ __forceinline__ float row_max(uint32_t s_addr, float c, int row) {
    float mx = -INFINITY;
#pragma unroll
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(s_addr + ch * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float x = __uint_as_float(r[i]) * c;
            mx = (!DIAG || ch * 32 + i <= row) ? fmaxf(mx, x) : mx;
        }
    }
    return mx;
}

// P = 2^(s·c − m) for the same row (0 for hidden keys), as bf16 pairs over TMEM columns
// [0, 64) of the row's S region; P columns of chunk k lie below the S columns still to be
// read, so each chunk is read before anything overwrites it. With SPLIT the bf16 residuals
// p − bf16(p) go to columns [64, 128) after the whole row has been read. Adds the unrounded
// weights to l.
template <bool DIAG, bool SPLIT>
__device__ __forceinline__ void write_p(uint32_t s_addr, float c, float m, int row, float &l) {
    uint32_t lo[SPLIT ? BN / 2 : 1];
#pragma unroll
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(s_addr + ch * 32, r);
        tmem_ld_wait(r);
        uint32_t hi[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k0 = ch * 32 + 2 * i;
            float p0 = fast_exp2(fmaf(__uint_as_float(r[2 * i]), c, -m));
            float p1 = fast_exp2(fmaf(__uint_as_float(r[2 * i + 1]), c, -m));
            if (DIAG) {
                p0 = k0 <= row ? p0 : 0.f;
                p1 = k0 + 1 <= row ? p1 : 0.f;
            }
            l += p0 + p1;
            hi[i] = pack_bf16x2(p0, p1);
            if constexpr (SPLIT) lo[ch * 16 + i] = pack_bf16x2(p0 - bf16_lo(hi[i]), p1 - bf16_hi(hi[i]));
        }
        tmem_st16(s_addr + ch * 16, hi);
    }
    if constexpr (SPLIT) {
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t part[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) part[i] = lo[ch * 16 + i];
            tmem_st16(s_addr + 64 + ch * 16, part);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const PrefillArgs a, int n_qt, int heads_per_cta) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + BAR_OFF + 8 * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + SLOT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // work item; the longest query tiles (most KV tiles) come first
    const int n_hgrp = a.Hq / heads_per_cta;
    const int per_qt = a.B * n_hgrp;
    const int qt = n_qt - 1 - (int)(blockIdx.x / per_qt);
    const int rem = (int)(blockIdx.x % per_qt);
    const int b = rem / n_hgrp;
    const int h0 = (rem % n_hgrp) * heads_per_cta;
    const int n_mt = heads_per_cta;                 // query tiles in this block (heads h0, h0+1)
    const int j = h0 / (a.Hq / a.Hkv);              // their KV head

    griddep_wait();
    const int seq0 = a.cu_seqlens[b];
    const int S = a.cu_seqlens[b + 1] - seq0;
    if (qt * BM >= S) return;                       // the whole block leaves before any setup
    const int n_kv = qt + 1;                        // KV tiles 0 .. qt (causal, equal lengths)
    const bool split_p = qt < kSplitTiles;          // short rows: P as bf16 head + residual

    if (threadIdx.x == 0) {
        mbar_init(bar(kQFull), 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(kKFull + s), 1);
            mbar_init(bar(kVFull + s), 1);
            mbar_init(bar(kKvEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(kSFull + t), 1);
            mbar_init(bar(kPReady + t), 128);
            mbar_init(bar(kODone + t), 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            const int q_tok = seq0 + qt * BM;
            mbar_arrive_expect_tx(bar(kQFull), n_mt * TILE_BYTES);
            for (int t = 0; t < n_mt; ++t)
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_3d(sb + Q_OFF + t * TILE_BYTES + bx * BOX_BYTES, &qmap, bx * 64, h0 + t, q_tok,
                                bar(kQFull), l2_evict_first_policy());
            int issued = 0;
            for (int n = 0; n < n_kv; ++n) {
                const int s = n % NSTAGE;
                if (!mbar_wait_bounded(bar(kKvEmpty + s), ((n / NSTAGE) & 1) ^ 1, &g_prefill_status, kStatusEmptyWait))
                    break;
                const int k_tok = seq0 + n * BN;
                mbar_arrive_expect_tx(bar(kKFull + s), TILE_BYTES);
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_3d_nohint(sb + K_OFF + s * TILE_BYTES + bx * BOX_BYTES, &kmap, bx * 64, j, k_tok,
                                       bar(kKFull + s));
                mbar_arrive_expect_tx(bar(kVFull + s), TILE_BYTES);
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_3d_nohint(sb + V_OFF + s * TILE_BYTES + bx * BOX_BYTES, &vmap, bx * 64, j, k_tok,
                                       bar(kVFull + s));
                issued = n + 1;
            }
            // no copy may still be in flight when the block exits
            mbar_wait_bounded(bar(kQFull), 0, &g_prefill_status, kStatusDrainWait);
            for (int n = issued > NSTAGE ? issued - NSTAGE : 0; n < issued; ++n) {
                mbar_wait_bounded(bar(kKFull + n % NSTAGE), (n / NSTAGE) & 1, &g_prefill_status, kStatusDrainWait);
                mbar_wait_bounded(bar(kVFull + n % NSTAGE), (n / NSTAGE) & 1, &g_prefill_status, kStatusDrainWait);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait_bounded(bar(kQFull), 0, &g_prefill_status, kStatusFullWait);
            for (int n = 0; n < n_kv && ok; ++n) {
                const int s = n % NSTAGE;
                const uint32_t ph = (n / NSTAGE) & 1;
                if (!mbar_wait_bounded(bar(kKFull + s), ph, &g_prefill_status, kStatusFullWait)) {
                    ok = false;
                    break;
                }
                for (int t = 0; t < n_mt && ok; ++t) {
                    // the previous P·V of this tile must be done before S overwrites P
                    if (n > 0 && !mbar_wait_bounded(bar(kODone + t), (n - 1) & 1, &g_prefill_status, kStatusMmaWait)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qa = sb + Q_OFF + t * TILE_BYTES;
                    const uint32_t ka = sb + K_OFF + s * TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
                        umma_ss(tmem + 256 * t, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                                kIdescS, kk > 0);
                    }
                    umma_commit(bar(kSFull + t));
                }
                if (!ok) break;
                if (!mbar_wait_bounded(bar(kVFull + s), ph, &g_prefill_status, kStatusFullWait)) {
                    ok = false;
                    break;
                }
                const uint32_t va = sb + V_OFF + s * TILE_BYTES;
                for (int t = 0; t < n_mt && ok; ++t) {
                    if (!mbar_wait_bounded(bar(kPReady + t), n & 1, &g_prefill_status, kStatusMmaWait)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t o = tmem + 256 * t + 128;
                    const uint32_t p = tmem + 256 * t;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_ts(o, p + kk * 8, sdesc_sw128(va + kk * 2048, BOX_BYTES, 1024), kIdescPV,
                                (n > 0 || kk > 0) ? 1u : 0u);
                    if (split_p) {
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            umma_ts(o, p + 64 + kk * 8, sdesc_sw128(va + kk * 2048, BOX_BYTES, 1024), kIdescPV, 1u);
                    }
                    umma_commit(bar(kODone + t));
                }
                // release the stage; the last one is never reused, so nothing arrives after exit
                if (ok && n + 1 < n_kv) umma_commit(bar(kKvEmpty + s));
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 2) >> 2;               // query tile of this warpgroup
        const int quarter = warp & 3;                // the TMEM lanes this warp may touch
        const int row = quarter * 32 + lane;         // query row within the tile
        if (t < n_mt) {
            const uint32_t s_addr = tmem + 256 * t + ((uint32_t)(quarter * 32) << 16);
            const uint32_t o_addr = s_addr + 128;
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            for (int n = 0; n < n_kv; ++n) {
                // the warp decides together: the TMEM accesses below are warp-collective
                const bool got = mbar_wait_bounded(bar(kSFull + t), n & 1, &g_prefill_status, kStatusFullWait);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool diag = n == qt;
                const float mt = diag ? row_max<true>(s_addr, a.scale_log2, row)
                                      : row_max<false>(s_addr, a.scale_log2, row);
                float alpha = 1.f;
                bool grow = false;
                if (n == 0) {
                    m_ref = mt;
                } else if (mt > m_ref + kRescaleLog2) {
                    alpha = fast_exp2(m_ref - mt);
                    m_ref = mt;
                    l *= alpha;
                    grow = true;
                }
                if (__any_sync(0xffffffffu, grow)) {
                    // O (complete up to tile n-1: S_n was issued after that P·V finished) *= alpha
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + c * 32, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(o_addr + c * 32, r);
                    }
                }
                if (split_p)
                    diag ? write_p<true, true>(s_addr, a.scale_log2, m_ref, row, l)
                         : write_p<false, true>(s_addr, a.scale_log2, m_ref, row, l);
                else if (diag)
                    write_p<true, false>(s_addr, a.scale_log2, m_ref, row, l);
                else
                    write_p<false, false>(s_addr, a.scale_log2, m_ref, row, l);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kPReady + t));
            }
            const bool done = ok && mbar_wait_bounded(bar(kODone + t), (n_kv - 1) & 1, &g_prefill_status, kStatusMmaWait);
            if (__all_sync(0xffffffffu, done)) {
                tc_fence_after();
                const int q_row = qt * BM + row;
                const float inv = 1.f / l;
                float4 *dst = reinterpret_cast<float4 *>(a.out + ((size_t)(seq0 + q_row) * a.Hq + h0 + t) * HD);
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + c * 32, r);
                    tmem_ld_wait(r);
                    if (q_row < S) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[c * 8 + i] = make_float4(
                                __uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t st) {
    if (a.D != HD) return cudaErrorInvalidValue;
    CUtensorMap qm, km, vm;
    const uint32_t box[3] = {64, 1, BM};
    {
        const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)a.Hq, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)a.Hq * HD * 2};
        cudaError_t e = encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box,
                                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)a.Hkv, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)a.Hkv * HD * 2};
        cudaError_t e = encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dims, strides, box,
                                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e == cudaSuccess)
            e = encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dims, strides, box,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e != cudaSuccess) return e;
    }
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int G = a.Hq / a.Hkv;
    const int heads_per_cta = (G % 2 == 0) ? 2 : 1;
    const int n_qt = (a.max_seqlen + BM - 1) / BM;
    const long blocks = (long)n_qt * a.B * (a.Hq / heads_per_cta);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
    const cudaError_t e = launch_pdl(prefill_kernel, dim3((unsigned)blocks), dim3(kThreads), SMEM, st, qm, km, vm, a,
                                     n_qt, heads_per_cta);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int prefill_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_prefill_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
