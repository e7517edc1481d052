// K1 (tensor-core form): split-KV decode for GQA/MHA/MQA over a bf16 cache.
//
// The method ("模型架构｜MQA & GQA 调研", section "代码", Attention.forward with one new token):
// out[b,h] = softmax(scale · q[b,h]·K[b,:S_b,j]ᵀ) · V[b,:S_b,j] with j = h / G. The page
// expands K/V with repeat_kv, which reads every K/V byte once per query head; here the G
// query heads of KV head j are stacked as the M rows of one MMA tile, so each K/V byte
// leaves HBM once and feeds all G heads.
//
// One thread block = (sequence b, KV head j, block of up to 16·MT heads of j's group, split).
// Warp 4 is the producer: it streams the split's K and V rows through an NS-stage ring of
// shared-memory buffers with TMA tensor loads (64-token stages, 64-byte swizzled boxes of 32
// columns, L2 evict-first hint). Warps 0-3 are consumers; each owns 16 tokens of every stage:
//   S = Q·Kᵀ      mma.sync m16n8k16 (bf16 → fp32), heads on M, tokens on N, Q from smem;
//   softmax       per-head running max/sum in the base-2 domain (scores · scale·log2 e),
//                 quad shuffles for the row max, rescale factor 2^(m_old − m_new);
//   O += P·V      P rounded to bf16 in registers (the S accumulator layout is the A-operand
//                 layout), V fragments by ldmatrix.trans.
// Tokens past the sequence end are masked to −inf, and their V rows are zeroed in shared
// memory so stale cache contents never reach the output. At the end the four warps' states
// are merged in shared memory; the block writes out = O/l (one split) or the normalised
// partial and lse = ln Σ e^s for the log-sum-exp merge kernel.
//
// Every mbarrier wait is bounded (MLAKV_WAIT_TIMEOUT_CYCLES); a wait that runs out sets a bit in
// g_decode_gqa_status and the block returns, so a broken pipeline cannot hang the GPU.
#include "ptx.cuh"
#include "tensor_map.cuh"

#include <math.h>

namespace mlakv {

__device__ unsigned g_decode_gqa_status;

namespace {

constexpr int kT = 64;             // tokens per pipeline stage
constexpr int kConsumers = 4;      // consumer warps, 16 tokens of each stage apiece
constexpr int kThreads = (kConsumers + 1) * 32;

template <int D, int MT, int NS>
struct Cfg {
    static constexpr int NB = D / 32;               // 64-byte boxes per token row
    static constexpr int BOX = kT * 64;             // one box: kT rows of 64 bytes
    static constexpr int KV = NB * BOX;             // K (or V) bytes per stage
    static constexpr int STAGE = 2 * KV;
    static constexpr int HEADS = 16 * MT;
    static constexpr int QPITCH = D * 2 + 16;       // padded Q row: conflict-free ldmatrix
    static constexpr int Q_OFF = NS * STAGE;
    static constexpr int BAR_OFF = Q_OFF + HEADS * QPITCH;
    static constexpr int SMEM = BAR_OFF + 2 * NS * 8 + 1024;   // + alignment slack
    static constexpr int MERGE_BYTES = kConsumers * HEADS * (D + 2) * 4;
    static_assert(MERGE_BYTES <= NS * STAGE, "merge scratch must fit in the stage buffers");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Byte offset of 16-byte chunk `cidx` (along D) of token row `row` inside one K/V stage
// buffer laid out as NB boxes of [kT rows × 64 B] with the 64-byte TMA swizzle
// (address bits [4,5] ^= bits [7,8], i.e. chunk c of row r sits at c ^ ((r >> 1) & 3)).
__device__ __forceinline__ uint32_t kv_off(int row, int cidx) {
    const int box = cidx >> 2;
    const int c = (cidx & 3) ^ ((row >> 1) & 3);
    return box * (kT * 64) + row * 64 + c * 16;
}

template <int D, int MT, int NS>
__global__ void __launch_bounds__(kThreads, 2)
decode_gqa_bf16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const DecodeGqaArgs a) {
    using C = Cfg<D, MT, NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + C::BAR_OFF;
    const uint32_t empty0 = full0 + NS * 8;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.Hq / a.Hkv;
    const int n_hblk = (G + C::HEADS - 1) / C::HEADS;
    const int j = blockIdx.y / n_hblk;
    const int hb = blockIdx.y % n_hblk;
    const int heads = min(C::HEADS, G - hb * C::HEADS);
    const int h0 = j * G + hb * C::HEADS;
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

    // q rows of this head block → padded shared rows (zero rows beyond `heads`)
    {
        const uint4 *qg = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) +
                                                          ((size_t)b * a.Hq + h0) * D);
        for (int i = threadIdx.x; i < C::HEADS * (D / 8); i += kThreads) {
            const int r = i / (D / 8), c = i % (D / 8);
            const uint4 v = r < heads ? __ldg(qg + (size_t)r * (D / 8) + c) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(smem + C::Q_OFF + r * C::QPITCH + c * 16) = v;
        }
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % NS;
                if (!mbar_wait_bounded(empty0 + 8 * s, ((i / NS) & 1) ^ 1, &g_decode_gqa_status, kStatusEmptyWait))
                    break;
                const uint32_t dst = sbase + s * C::STAGE;
                mbar_arrive_expect_tx(full0 + 8 * s, C::STAGE);
                const int t = t_begin + i * kT;
#pragma unroll
                for (int bx = 0; bx < C::NB; ++bx) {
                    tma_load_4d(dst + bx * C::BOX, &kmap, bx * 32, j, t, b, full0 + 8 * s, pol);
                    tma_load_4d(dst + C::KV + bx * C::BOX, &vmap, bx * 32, j, t, b, full0 + 8 * s, pol);
                }
                issued = i + 1;
            }
            // no copy may still be in flight when the block exits
            for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
                mbar_wait_bounded(full0 + 8 * (i % NS), (i / NS) & 1, &g_decode_gqa_status, kStatusDrainWait);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2;      // row group inside an MMA fragment
    const int cq = lane & 3;      // column pair inside an MMA fragment
    const int mi = lane >> 3;     // ldmatrix: which 8x8 matrix this lane addresses
    const int ri = lane & 7;      // ldmatrix: which row of it
    float o[MT][D / 8][4];
    float m[MT][2], l[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            m[mt][r] = -INFINITY;
            l[mt][r] = 0.f;
        }
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nd][e] = 0.f;
    }
    const uint32_t qbase = sbase + C::Q_OFF;
    bool ok = true;

    for (int i = 0; i < n_tiles && ok; ++i) {
        const int s = i % NS;
        if (!mbar_wait_bounded(full0 + 8 * s, (i / NS) & 1, &g_decode_gqa_status, kStatusFullWait)) {
            ok = false;
            break;
        }
        const uint32_t kb = sbase + s * C::STAGE;
        const uint32_t vb = kb + C::KV;
        const int t0 = t_begin + i * kT + warp * 16;       // first token of this warp's slice
        const int n_valid = min(16, t_end - t0);
        if (n_valid > 0) {
            if (n_valid < 16) {
                // zero the V rows past the sequence end so 0·(stale value) cannot make NaN
                uint8_t *vrow = smem + s * C::STAGE + C::KV;
                for (int idx = lane; idx < 16 * C::NB * 4; idx += 32) {
                    const int r = idx / (C::NB * 4);
                    if (r >= n_valid) {
                        const int row = warp * 16 + r, cidx = idx % (C::NB * 4);
                        *reinterpret_cast<uint4 *>(vrow + kv_off(row, cidx)) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // S = Q·Kᵀ for the warp's 16 tokens
            float sc[MT][2][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b0, b1, b2, b3;
                {
                    const int row = warp * 16 + (mi >> 1) * 8 + ri;
                    ldsm_x4(kb + kv_off(row, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    const int hrow = mt * 16 + (mi & 1) * 8 + ri;
                    ldsm_x4(qbase + hrow * C::QPITCH + (2 * kk + (mi >> 1)) * 16, a0, a1, a2, a3);
                    mma_bf16_16816(sc[mt][0], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(sc[mt][1], a0, a1, a2, a3, b2, b3);
                }
            }
            // online softmax (base 2) and P in bf16 as the A operand of P·V
            uint32_t pa[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float x[4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = nt * 8 + 2 * cq + e;
                            x[nt * 2 + e] = tok < n_valid ? sc[mt][nt][2 * r + e] * a.scale_log2 : -INFINITY;
                        }
                    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float mn = fmaxf(m[mt][r], mx);            // finite: token 0 of the slice is valid
                    const float alpha = fast_exp2(m[mt][r] - mn);
                    m[mt][r] = mn;
                    float p[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) p[e] = fast_exp2(x[e] - mn);
                    const uint32_t lo = pack_bf16x2(p[0], p[1]);     // tokens 2cq, 2cq+1
                    const uint32_t hi = pack_bf16x2(p[2], p[3]);     // tokens 8+2cq, 9+2cq
                    pa[mt][r] = lo;
                    pa[mt][2 + r] = hi;
                    // the row sum uses the rounded weights, so Σ weights = 1 after normalising
                    const float ps = bf16_lo(lo) + bf16_hi(lo) + bf16_lo(hi) + bf16_hi(hi);
                    l[mt][r] = l[mt][r] * alpha + ps;
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd) {
                        o[mt][nd][2 * r] *= alpha;
                        o[mt][nd][2 * r + 1] *= alpha;
                    }
                }
            }
            // O += P·V
#pragma unroll
            for (int pq = 0; pq < D / 16; ++pq) {
                uint32_t b0, b1, b2, b3;
                const int row = warp * 16 + (mi & 1) * 8 + ri;
                ldsm_x4_t(vb + kv_off(row, 2 * pq + (mi >> 1)), b0, b1, b2, b3);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    mma_bf16_16816(o[mt][2 * pq], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
                    mma_bf16_16816(o[mt][2 * pq + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b2, b3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    if (!ok) return;

    // ---------------------------------------------------------------- merge the 4 warps
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");   // all stages consumed
    float *mrg = reinterpret_cast<float *>(smem);                          // [warp][head][D+2]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float lr = l[mt][r];
            lr += __shfl_xor_sync(0xffffffffu, lr, 1);
            lr += __shfl_xor_sync(0xffffffffu, lr, 2);
            const int h = mt * 16 + r * 8 + g;
            float *row = mrg + (warp * C::HEADS + h) * (D + 2);
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                row[nd * 8 + 2 * cq] = o[mt][nd][2 * r];
                row[nd * 8 + 2 * cq + 1] = o[mt][nd][2 * r + 1];
            }
            if (cq == 0) {
                row[D] = m[mt][r];
                row[D + 1] = lr;
            }
        }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
    for (int idx = threadIdx.x; idx < heads * D; idx += kConsumers * 32) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mrg[(w * C::HEADS + h) * (D + 2) + D]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float *row = mrg + (w * C::HEADS + h) * (D + 2);
                const float f = fast_exp2(row[D] - M);
                L = fmaf(row[D + 1], f, L);
                O = fmaf(row[d], f, O);
            }
        }
        const size_t orow = (size_t)b * a.Hq + h0 + h;
        const float val = L > 0.f ? O / L : 0.f;
        if (a.n_split == 1) {
            a.out[orow * D + d] = val;
        } else {
            a.o_part[(orow * a.n_split + split) * D + d] = val;
            if (d == 0) a.lse_part[orow * a.n_split + split] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
}

template <int D, int MT, int NS>
cudaError_t launch_cfg(const DecodeGqaArgs &a, cudaStream_t st) {
    using C = Cfg<D, MT, NS>;
    CUtensorMap km, vm;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)a.Hkv, (uint64_t)a.S_max, (uint64_t)a.B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)a.Hkv * D * 2, (uint64_t)a.S_max * a.Hkv * D * 2};
    const uint32_t box[4] = {32, 1, kT, 1};
    cudaError_t e = encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k, dims, strides, box,
                                      CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess)
        e = encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.v, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e != cudaSuccess) return e;
    auto kern = decode_gqa_bf16_kernel<D, MT, NS>;
    static bool attr_set = false;   // per process; the attribute is per function
    if (!attr_set) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int G = a.Hq / a.Hkv;
    const dim3 grid(a.n_split, a.Hkv * ((G + C::HEADS - 1) / C::HEADS), a.B);
    e = launch_pdl(kern, grid, dim3(kThreads), C::SMEM, st, km, vm, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeGqaArgs &a, cudaStream_t st) {
    constexpr int NS = D == 128 ? 3 : (D == 96 ? 4 : 6);
    const int G = a.Hq / a.Hkv;
    if (G <= 16) return launch_cfg<D, 1, NS>(a, st);
    return launch_cfg<D, 2, NS>(a, st);
}

}  // namespace

int decode_gqa_bf16_tile_tokens(int, int) { return kT; }

int decode_gqa_bf16_heads_per_block(int G) { return G <= 16 ? 16 : 32; }

cudaError_t launch_decode_gqa_bf16(const DecodeGqaArgs &a, cudaStream_t st) {
    switch (a.D) {
        case 64: return launch_d<64>(a, st);
        case 96: return launch_d<96>(a, st);
        case 128: return launch_d<128>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

int decode_gqa_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_decode_gqa_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_decode_gqa_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
