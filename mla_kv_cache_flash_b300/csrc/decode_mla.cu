// K3: MLA decode with W_UK absorbed into the query (qqstock article on DeepSeek MLA,
// sections 2, 3 and 6). Every head attends the same cached latent row [c_t ‖ kr_t]
// (r = 128, dr = 48: 352 bytes per token in bf16) and averages c_t itself, so this is MQA
// with key width 176 and value width 128 whose value is the first 128 columns of the key
// row: each latent byte is read from HBM once and serves every head, twice (as key and
// as value).
//
// One thread block = (sequence b, block of 16 heads, split). Warp 4 streams the split's
// c and kr rows through an NS-stage shared-memory ring with TMA (c: four 64-byte-swizzled
// boxes of 32 columns; kr: three 32-byte-swizzled boxes of 16 columns; 64-token stages).
// Warps 0-3 each own 16 tokens of a stage and run, with the 16 heads as the M rows:
//   S = [q_lat ‖ q_rope]·[c ‖ kr]ᵀ   11 k-steps of mma.sync m16n8k16 (bf16 → fp32);
//   online softmax in the base-2 domain (scores · scale·log2 e);
//   O += P·c                         P in registers as bf16, c fragments by ldmatrix.trans
//                                    from the same stage buffer the scores used.
// Tokens past the sequence end are masked and their c rows zeroed. The four warps' states
// are merged in shared memory; the block writes out_lat = O/l, or the normalised partial
// and lse = ln Σ e^s for the log-sum-exp merge kernel. Waits are bounded.
#include "ptx.cuh"
#include "tensor_map.cuh"

#include <math.h>

namespace mlakv {

__device__ unsigned g_decode_mla_status;

namespace {

constexpr int R = 128;               // kv_lora_rank
constexpr int DR = 48;               // rope width
constexpr int DK = R + DR;           // key width
constexpr int kT = 64;               // tokens per stage
constexpr int kHeads = 16;           // heads per block (one MMA M tile)
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int NS = 4;

constexpr int C_BOX = kT * 64;       // one c box: 64 rows × 64 B (32 columns)
constexpr int C_BYTES = 4 * C_BOX;   // 16 KB
constexpr int KR_BOX = kT * 32;      // one kr box: 64 rows × 32 B (16 columns)
constexpr int KR_BYTES = 3 * KR_BOX; // 6 KB
constexpr int STAGE = C_BYTES + KR_BYTES;
constexpr int QPITCH = DK * 2 + 16;  // padded q row (368 B): conflict-free ldmatrix
constexpr int Q_OFF = NS * STAGE;
constexpr int BAR_OFF = Q_OFF + kHeads * QPITCH;
constexpr int SMEM = BAR_OFF + 2 * NS * 8 + 1024;
constexpr int MERGE_BYTES = kConsumers * kHeads * (R + 2) * 4;
static_assert(MERGE_BYTES <= NS * STAGE, "merge scratch must fit in the stage buffers");
static_assert(STAGE % 1024 == 0, "stage buffers keep the swizzle alignment");

// c: 16-byte chunk `cidx` (0..15) of row `row`, 64-byte swizzle (chunk c at c ^ ((row>>1)&3))
__device__ __forceinline__ uint32_t c_off(int row, int cidx) {
    return (cidx >> 2) * C_BOX + row * 64 + (((cidx & 3) ^ ((row >> 1) & 3)) << 4);
}
// kr: 16-byte chunk `cidx` (0..5) of row `row`, 32-byte swizzle (chunk c at c ^ ((row>>2)&1))
__device__ __forceinline__ uint32_t kr_off(int row, int cidx) {
    return C_BYTES + (cidx >> 1) * KR_BOX + row * 32 + (((cidx & 1) ^ ((row >> 2) & 1)) << 4);
}
// key chunk `kc` (0..21) of a token row: c for kc < 16, kr after
__device__ __forceinline__ uint32_t key_off(int row, int kc) {
    return kc < 16 ? c_off(row, kc) : kr_off(row, kc - 16);
}

__global__ void __launch_bounds__(kThreads, 2)
decode_mla_kernel(const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap krmap,
                  const DecodeMlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + BAR_OFF;
    const uint32_t empty0 = full0 + NS * 8;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h0 = blockIdx.y * kHeads;
    const int b = blockIdx.z;
    const int split = blockIdx.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumers);
        }
        fence_mbar_init();
    }
    // everything above overlaps the previous kernel in the stream; the inputs are read below
    griddep_wait();
    griddep_launch_dependents();
    const int S = a.seq_lens[b];
    const int t_begin = split * a.split_len;
    const int t_end = min(S, t_begin + a.split_len);
    const int n_tiles = t_end > t_begin ? (t_end - t_begin + kT - 1) / kT : 0;

    // [q_lat ‖ q_rope] rows of this head block → padded shared rows
    {
        const uint4 *ql = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q_lat) +
                                                          ((size_t)b * a.Hq + h0) * R);
        const uint4 *qr = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q_rope) +
                                                          ((size_t)b * a.Hq + h0) * DR);
        for (int i = threadIdx.x; i < kHeads * (DK / 8); i += kThreads) {
            const int r = i / (DK / 8), c = i % (DK / 8);
            const uint4 v = c < R / 8 ? __ldg(ql + r * (R / 8) + c) : __ldg(qr + r * (DR / 8) + (c - R / 8));
            *reinterpret_cast<uint4 *>(smem + Q_OFF + r * QPITCH + c * 16) = v;
        }
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&cmap);
            prefetch_tensormap(&krmap);
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % NS;
                if (!mbar_wait_bounded(empty0 + 8 * s, ((i / NS) & 1) ^ 1, &g_decode_mla_status, kStatusEmptyWait))
                    break;
                const uint32_t dst = sbase + s * STAGE;
                mbar_arrive_expect_tx(full0 + 8 * s, STAGE);
                const int t = t_begin + i * kT;
#pragma unroll
                for (int bx = 0; bx < 4; ++bx) tma_load_3d(dst + bx * C_BOX, &cmap, bx * 32, t, b, full0 + 8 * s, pol);
#pragma unroll
                for (int bx = 0; bx < 3; ++bx)
                    tma_load_3d(dst + C_BYTES + bx * KR_BOX, &krmap, bx * 16, t, b, full0 + 8 * s, pol);
                issued = i + 1;
            }
            for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
                mbar_wait_bounded(full0 + 8 * (i % NS), (i / NS) & 1, &g_decode_mla_status, kStatusDrainWait);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, cq = lane & 3, mi = lane >> 3, ri = lane & 7;
    float o[R / 8][4];
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
    for (int nd = 0; nd < R / 8; ++nd)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;
    const uint32_t qbase = sbase + Q_OFF;
    bool ok = true;

    for (int i = 0; i < n_tiles; ++i) {
        const int s = i % NS;
        if (!mbar_wait_bounded(full0 + 8 * s, (i / NS) & 1, &g_decode_mla_status, kStatusFullWait)) {
            ok = false;
            break;
        }
        const uint32_t tb = sbase + s * STAGE;
        const int t0 = t_begin + i * kT + warp * 16;
        const int n_valid = min(16, t_end - t0);
        if (n_valid > 0) {
            if (n_valid < 16) {
                // zero the c rows past the sequence end so 0·(stale value) cannot make NaN
                uint8_t *cbuf = smem + s * STAGE;
                for (int idx = lane; idx < 16 * 16; idx += 32) {
                    const int r = idx >> 4;
                    if (r >= n_valid)
                        *reinterpret_cast<uint4 *>(cbuf + c_off(warp * 16 + r, idx & 15)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t b0, b1, b2, b3, a0, a1, a2, a3;
                const int row = warp * 16 + (mi >> 1) * 8 + ri;
                ldsm_x4(tb + key_off(row, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                ldsm_x4(qbase + ((mi & 1) * 8 + ri) * QPITCH + (2 * kk + (mi >> 1)) * 16, a0, a1, a2, a3);
                mma_bf16_16816(sc[0], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(sc[1], a0, a1, a2, a3, b2, b3);
            }
            uint32_t pa[4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float x[4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = nt * 8 + 2 * cq + e;
                        x[nt * 2 + e] = tok < n_valid ? sc[nt][2 * r + e] * a.scale_log2 : -INFINITY;
                    }
                float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(m[r], mx);                 // finite: token 0 of the slice is valid
                const float alpha = fast_exp2(m[r] - mn);
                m[r] = mn;
                const uint32_t lo = pack_bf16x2(fast_exp2(x[0] - mn), fast_exp2(x[1] - mn));
                const uint32_t hi = pack_bf16x2(fast_exp2(x[2] - mn), fast_exp2(x[3] - mn));
                pa[r] = lo;
                pa[2 + r] = hi;
                l[r] = l[r] * alpha + (bf16_lo(lo) + bf16_hi(lo) + bf16_lo(hi) + bf16_hi(hi));
#pragma unroll
                for (int nd = 0; nd < R / 8; ++nd) {
                    o[nd][2 * r] *= alpha;
                    o[nd][2 * r + 1] *= alpha;
                }
            }
#pragma unroll
            for (int pq = 0; pq < R / 16; ++pq) {
                uint32_t b0, b1, b2, b3;
                const int row = warp * 16 + (mi & 1) * 8 + ri;
                ldsm_x4_t(tb + c_off(row, 2 * pq + (mi >> 1)), b0, b1, b2, b3);
                mma_bf16_16816(o[2 * pq], pa[0], pa[1], pa[2], pa[3], b0, b1);
                mma_bf16_16816(o[2 * pq + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    if (!ok) return;

    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
    float *mrg = reinterpret_cast<float *>(smem);   // [warp][head][R+2]
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float lr = l[r];
        lr += __shfl_xor_sync(0xffffffffu, lr, 1);
        lr += __shfl_xor_sync(0xffffffffu, lr, 2);
        float *row = mrg + (warp * kHeads + r * 8 + g) * (R + 2);
#pragma unroll
        for (int nd = 0; nd < R / 8; ++nd) {
            row[nd * 8 + 2 * cq] = o[nd][2 * r];
            row[nd * 8 + 2 * cq + 1] = o[nd][2 * r + 1];
        }
        if (cq == 0) {
            row[R] = m[r];
            row[R + 1] = lr;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
    for (int idx = threadIdx.x; idx < kHeads * R; idx += kConsumers * 32) {
        const int h = idx / R, d = idx % R;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mrg[(w * kHeads + h) * (R + 2) + R]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float *row = mrg + (w * kHeads + h) * (R + 2);
                const float f = fast_exp2(row[R] - M);
                L = fmaf(row[R + 1], f, L);
                O = fmaf(row[d], f, O);
            }
        }
        const size_t orow = (size_t)b * a.Hq + h0 + h;
        const float val = L > 0.f ? O / L : 0.f;
        if (a.n_split == 1) {
            a.out[orow * R + d] = val;
        } else {
            a.o_part[(orow * a.n_split + split) * R + d] = val;
            if (d == 0) a.lse_part[orow * a.n_split + split] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
}

}  // namespace

int decode_mla_tile_tokens() { return kT; }

cudaError_t launch_decode_mla(const DecodeMlaArgs &a, cudaStream_t st) {
    CUtensorMap cm, km;
    {
        const uint64_t dims[3] = {(uint64_t)R, (uint64_t)a.S_max, (uint64_t)a.B};
        const uint64_t strides[2] = {(uint64_t)R * 2, (uint64_t)a.S_max * R * 2};
        const uint32_t box[3] = {32, kT, 1};
        cudaError_t e = encode_tensor_map(&cm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.c, dims, strides, box,
                                          CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {(uint64_t)DR, (uint64_t)a.S_max, (uint64_t)a.B};
        const uint64_t strides[2] = {(uint64_t)DR * 2, (uint64_t)a.S_max * DR * 2};
        const uint32_t box[3] = {16, kT, 1};
        cudaError_t e = encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.kr, dims, strides, box,
                                          CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e != cudaSuccess) return e;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const dim3 grid(a.n_split, a.Hq / kHeads, a.B);
    const cudaError_t e = launch_pdl(decode_mla_kernel, grid, dim3(kThreads), SMEM, st, cm, km, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int decode_mla_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_decode_mla_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_decode_mla_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
