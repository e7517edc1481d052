// K1 over an 8-bit E4M3 cache on the tensor cores ("MHA, MQA và GQA" ebook: an fp8 cache
// halves every byte of the cache; "模型架构｜MQA & GQA 调研", section "代码", Attention.forward
// with one new token): out[b,h] = softmax(scale · q[b,h]·K[b,:S_b,j]ᵀ) · V[b,:S_b,j], j = h / G,
// where a cached row is e4m3(code) · its fp32 scale (one scale per row of K and of V).
//
// Work split (streamk.cuh): the segments (sequence b, KV head j) are cut into 64-token tiles
// laid end to end, and each persistent block takes an equal run of tiles, whatever the
// lengths (the producer warp finds the run's start once, lane-parallel, and every warp walks
// its pieces incrementally). A segment a block covers whole is written to `out`; one it
// shares with its neighbours becomes a partial (normalised output and ln Σ e^s) in one of the
// block's two slots. The producer warp publishes each such piece once the consumers have
// stored it (an acquire-release arrival on the segment's counter, in the workspace's counter
// region); the last block to arrive combines the segment's partials inside this launch: the
// producer warp for the block's first piece, the consumers (idle by then) for its last.
//
// Block = 4 consumer warps + 1 producer warp. The producer brings each tile's K and V codes
// into a 4-stage shared-memory ring with TMA tensor loads, the tile's K and V row scales on
// the same barrier (for up to 4 KV heads, when S_max·Hkv is a multiple of 4, those of all
// heads of the tile's 64 tokens as one contiguous bulk copy each, else the 128 the block needs
// by 4-byte asynchronous copies), and with a piece's first tile the piece's G bf16 query rows.
// Each consumer warp takes 16 tokens of a tile and builds its mma.sync m16n8k16 operands
// (fp16 in, fp32 accumulate) straight from the codes in the stage, widening them in
// registers (every E4M3 value is an fp16 value, so the widening is exact; one instruction per
// two codes). The query heads sit on the MMA's N side in blocks of 8 (one block for G <= 8,
// two up to 16):
//   S = K·Qᵀ  the slice's 16 tokens on M. A thread's K operand for two k-steps is 8
//             consecutive codes of one token row, so the feature order inside each 32-wide
//             block is permuted (the same way for Q: a dot product does not depend on the
//             order of its terms). Each token's products times its K scale, in the base-2
//             domain (scale · log2 e). The bf16 query is rounded to fp16 once per piece:
//             exact for |q| in [2^-14, 65504], off by at most 2^-25 below;
//   softmax   running max and sum per head (a column) across the 8 lanes that hold its rows;
//   Oᵀ += Vᵀ·Pᵀ  the weights times each token's V scale and 2^10 (the sum l takes the
//             unscaled weights; the 2^10 keeps small weights out of fp16's subnormal range and
//             is divided out at the end), split into an fp16 head and an fp16 residual (about
//             2^-22 of each weight left); the score fragment, transposed by movmatrix, is the
//             B operand, and each part is multiplied with the V codes. A thread's A operand is
//             a pair of tokens at one feature: it loads D/8 consecutive codes of each of its
//             four tokens and interleaves them with byte permutes, so output feature
//             d = (D/8)·g + 2mb (+1) sits at row g (+8) of the mb-th 16-row block.
// Codes of tokens past the segment are zeroed (the stage may hold anything there).
// At a piece's end the four warps' states are combined through a small shared buffer.
//
// Every mbarrier wait is bounded (MLAKV_WAIT_TIMEOUT_CYCLES); a wait that runs out sets a bit
// in g_decode_fp8_status and the warp skips its remaining work but still meets its partners
// at every barrier, so the block always reaches its end.
#include "ptx.cuh"
#include "streamk.cuh"
#include "tensor_map.cuh"

#include <cuda_fp8.h>
#include <math.h>

namespace mlakv {

__device__ unsigned g_decode_fp8_status;

namespace {

constexpr int TT = 64;            // tokens per tile
constexpr int NS = 4;             // ring stages
constexpr int kConsumers = 4;     // consumer warps, 16 tokens of each tile apiece
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kBulkHeads = 4;     // bulk scale copies: [64 tokens][Hkv] floats, Hkv up to this
constexpr float kWeightScale = 1024.f;    // 2^10: keeps the scaled weights out of fp16 subnormals

template <int D>
struct Cfg {
    static constexpr int CODES = TT * D;                       // one tile of K (or V) codes, bytes
    static constexpr int SCALES = TT * kBulkHeads * 4;         // one tile of K (or V) scales, bytes
    static constexpr int QROWS = 16 * D * 2;                   // the query rows of a piece starting here
    static constexpr int STAGE = 2 * CODES + 2 * SCALES + QROWS;
    static constexpr int STAGE_PAD = (STAGE + 127) / 128 * 128;
    static constexpr int RING = NS * STAGE_PAD;
    static constexpr int BAR_OFF = RING;
    // ring barriers, the publication and end barriers, padded to 16 bytes; then the "last to
    // arrive" flags of the block's (at most two) shared pieces, the walk's start (b, q, i0) and
    // its tile range [t, t_end)
    static constexpr int MISC_OFF = BAR_OFF + ((2 * NS + 2) * 8 + 15) / 16 * 16;
    // the piece's query rows in fp16, [16][QROW]: a row stride of 16 words mod 32 keeps the
    // 16-byte operand loads of two rows in different banks
    static constexpr int QROW = D % 64 == 0 ? D + 32 : D;
    static constexpr int QS_OFF = MISC_OFF + 48;
    static constexpr int CMB_OFF = QS_OFF + 16 * QROW * 2;     // piece-end rows [warp][G][D + 2] floats
    __host__ __device__ static size_t prefix_off(int G) { return CMB_OFF + (size_t)kConsumers * G * (D + 2) * 4; }
    // then the tile prefix [B+1] and the lengths [B+1]
    static size_t smem_bytes(int B, int G) { return prefix_off(G) + (size_t)2 * (B + 1) * 4 + 128; }
    static_assert(STAGE % 16 == 0 && CODES % 16 == 0 && SCALES % 16 == 0, "16-byte alignment of the stage parts");
    static_assert(BAR_OFF % 8 == 0 && QS_OFF % 16 == 0 && CMB_OFF % 16 == 0, "aligned barriers and rows");
    static_assert(D % 32 == 0, "whole 32-feature blocks");
};

// Four E4M3 codes (bytes 0..3 of w) → two fp16 pairs: lo = (byte 0, byte 1), hi = (byte 2,
// byte 3), the lower byte in the lower half. Exact.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Transpose of an 8×8 matrix of 16-bit values held one pair per lane (row lane / 4, columns
// 2·(lane % 4) and +1): afterwards each lane holds its row of the transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t r;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// Byte permute: result byte i = byte sel_i of the pair (a = bytes 0..3, b = bytes 4..7).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Two floats → fp16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float f16_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// D = A·B + D, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Contiguous global → shared bulk copy (16-byte aligned addresses, size a multiple of 16),
// completing `bytes` on `bar`.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t smem_dst, const void *gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_dst), "l"(gmem_src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed (the arrival is
// one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// How the balanced split cut segment (b, j): its first tile fs in the global tile order, its
// pieces (one per block that holds any of its tiles) and the partial slot each piece's block
// wrote (a block's first piece goes to its slot 0, its last to slot 1).
struct SegSplit {
    long long fs, T;
    int n, c0, n_pieces;
    bool sparse;              // fewer tiles than blocks: every block holds at most one tile
    __device__ SegSplit(const int *prefix, int seg_per_seq, int b, int j, int S, long long T_, int n_blocks)
        : T(T_), n(n_blocks) {
        const int nb = stream_tiles(S, TT);
        fs = (long long)seg_per_seq * prefix[b] + (long long)j * nb;
        sparse = T < n;
        c0 = stream_block_of(fs, T, n);
        n_pieces = sparse ? nb : stream_block_of(fs + nb - 1, T, n) - c0 + 1;
    }
    __device__ int slot(int ip) const {
        if (sparse) return 2 * stream_block_of(fs + ip, T, n);
        if (ip == 0) return stream_start(c0, T, n) < fs ? 2 * c0 + 1 : 2 * c0;
        return 2 * (c0 + ip);
    }
};

struct Fp8Args {
    const void *q;            // [B, Hq, D] bf16
    const float *k_scale;     // [B, S_max, Hkv]
    const float *v_scale;
    const int *seq_lens;      // [B]
    float *out;               // [B, Hq, D]
    float *o_part;            // [2·n_blocks, G, D]
    float *lse_part;          // [2·n_blocks, G]
    int *counters;            // [B·Hkv] at the workspace's start, zero between calls
    int B, Hq, Hkv, S_max, n_blocks;
    float scale_log2;
};

// out[b, jG .. jG+G-1] from the segment's partials (normalised rows and log-sum-exps), by
// threads tid = 0 .. nthr-1 of the caller's group: six pieces' rows loaded at a time (all in
// flight together), combined with a running maximum.
template <int D>
__device__ void merge_segment(const Fp8Args &a, const SegSplit &sp, int b, int j, int G, int tid, int nthr) {
    constexpr int PB = 6;
    for (int idx = tid; idx < G * (D / 4); idx += nthr) {
        const int h = idx / (D / 4), col = idx % (D / 4);
        float M = -INFINITY, W = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int ip0 = 0; ip0 < sp.n_pieces; ip0 += PB) {
            float lse[PB];
            float4 x[PB];
#pragma unroll
            for (int v = 0; v < PB; ++v) {
                lse[v] = -INFINITY;
                x[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ip0 + v < sp.n_pieces) {
                    const size_t pr = (size_t)sp.slot(ip0 + v) * G + h;
                    lse[v] = __ldcg(a.lse_part + pr);
                    x[v] = __ldcg(reinterpret_cast<const float4 *>(a.o_part + pr * D) + col);
                }
            }
            float Mb = M;
#pragma unroll
            for (int v = 0; v < PB; ++v) Mb = fmaxf(Mb, lse[v]);
            if (Mb == -INFINITY) continue;
            const float r = fast_exp2((M - Mb) * kLog2e);       // 0 while M = -inf
            W *= r;
            acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
#pragma unroll
            for (int v = 0; v < PB; ++v) {
                const float wv = lse[v] == -INFINITY ? 0.f : fast_exp2((lse[v] - Mb) * kLog2e);
                W += wv;
                acc.x = fmaf(wv, x[v].x, acc.x);
                acc.y = fmaf(wv, x[v].y, acc.y);
                acc.z = fmaf(wv, x[v].z, acc.z);
                acc.w = fmaf(wv, x[v].w, acc.w);
            }
            M = Mb;
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        reinterpret_cast<float4 *>(a.out + ((size_t)b * a.Hq + (size_t)j * G + h) * D)[col] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// Resident blocks per SM the register cap below is chosen for: 15 warps put four on some SM
// sub-partition, whose 16384 registers then give each thread at most 128 (10 warps: 168).
// HB = head blocks of 8 (G <= 8: one, G <= 16: two).
template <int D, int HB>
constexpr int kResident = D == 128 || HB == 2 ? 2 : 3;
template <int D, int HB>
constexpr int kMaxRegs = kResident<D, HB> == 3 ? 128 : 168;

template <int D, int HB>
__global__ void __launch_bounds__(kThreads) __maxnreg__((kMaxRegs<D, HB>))
decode_fp8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const Fp8Args a) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t sb = smem_u32(smem);
    const uint32_t full0 = sb + C::BAR_OFF, empty0 = full0 + 8 * NS, pub_bar = empty0 + 8 * NS, end_bar = pub_bar + 8;
    const int G = a.Hq / a.Hkv;
    int *last_flag = reinterpret_cast<int *>(smem + C::MISC_OFF);     // [2]
    int *walk_start = last_flag + 2;                                   // [3]: b, q, i0
    long long *walk_range = reinterpret_cast<long long *>(smem + C::MISC_OFF + 24);   // [2]: t, t_end
    float *cmb = reinterpret_cast<float *>(smem + C::CMB_OFF);          // [warp][G][D + 2]
    int *prefix = reinterpret_cast<int *>(smem + C::prefix_off(G));     // [B+1]
    int *lens = prefix + (a.B + 1);                                      // [B]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    // scales by bulk copy: a tile's [64 tokens][Hkv] block is contiguous, 16-byte aligned and a
    // multiple of 16 bytes long (up to the cache end) when S_max·Hkv is a multiple of 4
    const bool bulk = a.Hkv <= kBulkHeads && (a.S_max * a.Hkv) % 4 == 0;
    const int sst = bulk ? a.Hkv : 1;            // scale stride between tokens in the stage

    // The producer warp sets the block up (ring barriers, the tile prefix over the sequences)
    // and signals the consumers on named barrier kPrologueBar without waiting for them, so
    // its first copies go out as early as possible.
    constexpr int kPrologueBar = 2;
    uint64_t pol = 0;
    if (warp == kConsumers) {
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) {
                // the TMA arrival, and without bulk scale copies the 32 scale-copy lanes
                mbar_init(full0 + 8 * s, bulk ? 1 : 1 + 32);
                mbar_init(empty0 + 8 * s, kConsumers);
            }
            mbar_init(pub_bar, kConsumers);
            mbar_init(end_bar, 1);
            fence_mbar_init();
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
        pol = l2_evict_first_policy();
    }
    griddep_wait();
    griddep_launch_dependents();
    if (warp == kConsumers) {
        // tile prefix over the sequences (warp scan, 32 sequences at a time)
        int carry = 0;
        for (int base = 0; base < a.B; base += 32) {
            const int b = base + lane;
            const int len = b < a.B ? __ldg(a.seq_lens + b) : 0;
            if (b < a.B) lens[b] = len;
            const int v = stream_tiles(len, TT);
            int x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (b < a.B) prefix[b] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) prefix[a.B] = carry;
        __syncwarp();
        // this block's tile range and where it starts, for every warp's walker
        const long long T = (long long)a.Hkv * carry;
        const long long t0 = T > 0 ? stream_start(c, T, a.n_blocks) : 0;
        const long long t1 = T > 0 ? stream_start(c + 1, T, a.n_blocks) : 0;
        int b0 = 0, q0 = 0, i00 = 0;
        if (t0 < t1) seq_walk_start(prefix, a.B, a.Hkv, t0, lane, b0, q0, i00);
        if (lane == 0) {
            walk_start[0] = b0;
            walk_start[1] = q0;
            walk_start[2] = i00;
            walk_range[0] = t0;
            walk_range[1] = t1;
        }
        __syncwarp();
        bar_arrive_named(kPrologueBar, kThreads);
    } else {
        bar_sync_named(kPrologueBar, kThreads);
    }

    const int seg_per_seq = a.Hkv;
    const long long T = (long long)seg_per_seq * prefix[a.B];
    if (c == 0 && warp < kConsumers) {
        // sequences with an empty cache own no tile: their output is zero (a warp per sequence)
        for (int b = warp; b < a.B; b += kConsumers)
            if (lens[b] <= 0)
                for (int i = lane; i < a.Hq * D / 4; i += 32)
                    reinterpret_cast<float4 *>(a.out + (size_t)b * a.Hq * D)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    SeqWalker walk{prefix, lens, a.B, seg_per_seq, 1, 0, 0, 0, 0, 0, 0};
    walk.set(walk_start[0], walk_start[1], walk_start[2], walk_range[0], walk_range[1]);
    const SeqWalker walk0 = walk;

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        bool ok = true;
        int g = 0;
        Piece p;
        while (ok && walk.next(p)) {
            const int j = p.gi;
            const uint32_t qbytes = (uint32_t)(G * D * 2);
            const __nv_bfloat16 *qsrc = static_cast<const __nv_bfloat16 *>(a.q) + ((size_t)p.b * a.Hq + (size_t)j * G) * D;
            for (int i = 0; i < p.n_t; ++i, ++g) {
                const int s = g % NS;
                const uint32_t dst = sb + s * C::STAGE_PAD;
                const uint32_t fb = full0 + 8 * s;
                // every lane waits: each of them may write into the stage below
                if (!mbar_wait_bounded(empty0 + 8 * s, ((g / NS) & 1) ^ 1, &g_decode_fp8_status, kStatusEmptyWait))
                    ok = false;
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const int t0 = (p.i0 + i) * TT;
                const uint32_t qb = i == 0 ? qbytes : 0u;      // the piece's query rows with its first tile
                if (bulk) {
                    if (lane == 0) {
                        const uint32_t sbytes = (uint32_t)(min(TT, a.S_max - t0) * a.Hkv * 4);
                        const size_t soff = ((size_t)p.b * a.S_max + t0) * a.Hkv;
                        mbar_arrive_expect_tx(fb, 2 * C::CODES + 2 * sbytes + qb);
                        tma_load_4d(dst, &kmap, 0, j, t0, p.b, fb, pol);
                        tma_load_4d(dst + C::CODES, &vmap, 0, j, t0, p.b, fb, pol);
                        bulk_copy(dst + 2 * C::CODES, a.k_scale + soff, sbytes, fb, pol);
                        bulk_copy(dst + 2 * C::CODES + C::SCALES, a.v_scale + soff, sbytes, fb, pol);
                        if (qb) bulk_copy(dst + 2 * C::CODES + 2 * C::SCALES, qsrc, qb, fb, pol);
                    }
                } else {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(fb, 2 * C::CODES + qb);
                        tma_load_4d(dst, &kmap, 0, j, t0, p.b, fb, pol);
                        tma_load_4d(dst + C::CODES, &vmap, 0, j, t0, p.b, fb, pol);
                        if (qb) bulk_copy(dst + 2 * C::CODES + 2 * C::SCALES, qsrc, qb, fb, pol);
                    }
                    // the tile's K and V scales: lane L copies those of tokens t0 + L and t0 + 32 + L
                    // (rows past the cache end are left as they are; their weights are zero)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int t = t0 + 32 * u + lane;
                        if (t < a.S_max) {
                            const size_t srow = ((size_t)p.b * a.S_max + t) * a.Hkv + j;
                            cp_async4(dst + 2 * C::CODES + 4 * (32 * u + lane), a.k_scale + srow);
                            cp_async4(dst + 2 * C::CODES + C::SCALES + 4 * (32 * u + lane), a.v_scale + srow);
                        }
                    }
                    cp_async_arrive_noinc(fb);
                }
            }
        }
        // no copy may still be in flight when the block exits
        for (int i = g > NS ? g - NS : 0; i < g; ++i)
            mbar_wait_bounded(full0 + 8 * (i % NS), (i / NS) & 1, &g_decode_fp8_status, kStatusDrainWait);
        asm volatile("cp.async.wait_all;" ::: "memory");
        // Publish the block's shared pieces, in order, as the consumers finish them (they arrive
        // on pub_bar once their partial rows are stored): one arrival on the segment's counter,
        // whose acquire-release orders those rows before it and the other blocks' rows after
        // it. The last block to arrive merges the segment and resets the counter: this warp,
        // while the consumers go on, unless it is the block's last piece (then the consumers,
        // idle by then, merge it at the block's end). This keeps the round trips off the
        // consumers' path.
        SeqWalker w2 = walk0;
        int u = 0;
        while (w2.next(p)) {
            if (p.whole) continue;
            const bool final_piece = w2.t >= w2.t_end;
            const bool arrived = mbar_wait_bounded(pub_bar, u & 1, &g_decode_fp8_status, kStatusPublishWait);
            const SegSplit sp(prefix, seg_per_seq, p.b, p.gi, p.S, T, a.n_blocks);
            int last = 0;
            if (lane == 0 && arrived) {
                int *cnt = a.counters + (size_t)p.b * a.Hkv + p.gi;
                last = atomic_add_acq_rel_gpu(cnt, 1) == sp.n_pieces - 1;
                if (last) *cnt = 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last && !final_piece) {
                __syncwarp();
                merge_segment<D>(a, sp, p.b, p.gi, G, lane, 32);
            }
            if (lane == 0) last_flag[u] = last && final_piece;
            ++u;
        }
        // the flags are written: release the consumers' end of block
        __syncwarp();
        if (lane == 0) mbar_arrive(end_bar);
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Fragment coordinates of mma.sync m16n8k16: g8 = lane / 4 picks a row (A, C) or a column
    // (B), cq = lane % 4 a pair of k indices (A, B) or of columns (C).
    const int g8 = lane >> 2, cq = lane & 3;
    constexpr int NW = D / 32;                    // 32-feature blocks: two k-steps of S each
    constexpr int NM = D / 16;                    // 16-feature row blocks of Oᵀ
    constexpr int kBar = 1, kNum = kConsumers * 32;
    const int r0 = 16 * warp;                     // this warp's first token of every tile
    __half *qs = reinterpret_cast<__half *>(smem + C::QS_OFF);
    bool ok = true;
    int g = 0, k = 0, n_pub = 0;
    // the block's shared pieces (at most its first and its last): (sequence, KV head, length)
    int pb0 = 0, pj0 = 0, ps0 = 0, pb1 = 0, pj1 = 0, ps1 = 0;
    Piece p;
    while (walk.next(p)) {
        const int j = p.gi;
        // Oᵀ accumulators: o[hb][mb] holds features f(mb, g8) (e = 0, 1) and f(mb, g8 + 8)
        // (e = 2, 3) of heads 8hb + 2cq (e even) and 8hb + 2cq + 1 (e odd), where
        // f(mb, g8) = (D/8)·g8 + 2mb and f(mb, g8 + 8) = (D/8)·g8 + 2mb + 1.
        float o[HB][NM][4], m[HB][2], l[HB][2];
#pragma unroll
        for (int hb = 0; hb < HB; ++hb) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                m[hb][e] = -INFINITY;
                l[hb][e] = 0.f;
            }
#pragma unroll
            for (int mb = 0; mb < NM; ++mb)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[hb][mb][e] = 0.f;
        }
        uint32_t qb[HB][NW][4];       // Qᵀ B operands, k-steps 2w (0, 1) and 2w + 1 (2, 3)

        const int t_end = min(p.S, (p.i0 + p.n_t) * TT);
        for (int i = 0; i < p.n_t; ++i, ++g) {
            const int s = g % NS;
            if (ok && !mbar_wait_bounded(full0 + 8 * s, (g / NS) & 1, &g_decode_fp8_status, kStatusFullWait)) ok = false;
            const uint8_t *stage = smem + s * C::STAGE_PAD;
            if (i == 0) {
                // the piece's query rows, rounded to fp16 (rows past G zero); the barrier also
                // orders this piece's use of the combine buffer after the previous piece's
                const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(stage + 2 * C::CODES + 2 * C::SCALES);
                for (int idx = threadIdx.x; idx < 8 * HB * (D / 8); idx += kNum) {
                    const int r = idx / (D / 8), c8 = idx % (D / 8);
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (ok && r < G) v = *reinterpret_cast<const uint4 *>(qg + r * D + 8 * c8);
                    *reinterpret_cast<uint4 *>(qs + r * C::QROW + 8 * c8) =
                        make_uint4(pack_f16x2(bf16_lo(v.x), bf16_hi(v.x)), pack_f16x2(bf16_lo(v.y), bf16_hi(v.y)),
                                   pack_f16x2(bf16_lo(v.z), bf16_hi(v.z)), pack_f16x2(bf16_lo(v.w), bf16_hi(v.w)));
                }
                bar_sync_named(kBar, kNum);
                // B operand of S for head 8hb + g8 in the permuted feature order: k-step 2w + h
                // takes features 32w + 8cq + 4h + {0,1} (b0) and + {2,3} (b1)
#pragma unroll
                for (int hb = 0; hb < HB; ++hb)
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(qs + (8 * hb + g8) * C::QROW + 32 * w + 8 * cq);
                        qb[hb][w][0] = v.x;
                        qb[hb][w][1] = v.y;
                        qb[hb][w][2] = v.z;
                        qb[hb][w][3] = v.w;
                    }
            }
            const int n_valid = min(16, t_end - ((p.i0 + i) * TT + r0));
            if (ok && n_valid > 0) {
                const uint8_t *kc = stage + r0 * D, *vc = stage + C::CODES + r0 * D;
                // the scales of this thread's S rows, tokens g8 and g8 + 8 of the slice
                const float *ksc = reinterpret_cast<const float *>(stage + 2 * C::CODES) + r0 * sst + (bulk ? j : 0);
                const float *vsc = ksc + C::SCALES / 4;
                const bool live0 = g8 < n_valid, live1 = g8 + 8 < n_valid;
                const float ks0 = live0 ? ksc[g8 * sst] * a.scale_log2 : 0.f;
                const float ks1 = live1 ? ksc[(g8 + 8) * sst] * a.scale_log2 : 0.f;
                const float vs0 = live0 ? vsc[g8 * sst] * kWeightScale : 0.f;
                const float vs1 = live1 ? vsc[(g8 + 8) * sst] * kWeightScale : 0.f;
                // S = K·Qᵀ over the slice's 16 tokens (rows) and the head blocks (columns): A is
                // eight consecutive codes of K rows g8 and g8 + 8 per 32-feature block
                float sc[HB][4];
#pragma unroll
                for (int hb = 0; hb < HB; ++hb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[hb][e] = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const uint2 c0 = *reinterpret_cast<const uint2 *>(kc + g8 * D + 32 * w + 8 * cq);
                    const uint2 c1 = *reinterpret_cast<const uint2 *>(kc + (g8 + 8) * D + 32 * w + 8 * cq);
                    uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
                    widen4(c0.x, a0, a2);
                    widen4(c1.x, a1, a3);
                    widen4(c0.y, a4, a6);
                    widen4(c1.y, a5, a7);
#pragma unroll
                    for (int hb = 0; hb < HB; ++hb) {
                        mma_f16_16816(sc[hb], a0, a1, a2, a3, qb[hb][w][0], qb[hb][w][1]);
                        mma_f16_16816(sc[hb], a4, a5, a6, a7, qb[hb][w][2], qb[hb][w][3]);
                    }
                }
                // V codes of tokens 2cq, 2cq+1, 8+2cq, 9+2cq, features (D/8)·g8 .. + D/8 - 1
                // (zero past the segment: the stage may hold anything there)
                uint32_t vw[4][NW];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = (e >> 1) * 8 + 2 * cq + (e & 1);
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(vc + tok * D + (D / 8) * g8);
#pragma unroll
                    for (int w = 0; w < NW; ++w) vw[e][w] = tok < n_valid ? src[w] : 0u;
                }
                // online softmax (base 2) per head (column) over the tokens (rows, across g8);
                // the weights times scale_v · 2^10 split into fp16 head and residual, then
                // transposed into the B operand of Oᵀ += Vᵀ·Pᵀ (tokens 2cq, 2cq+1 | 8+2cq, 9+2cq
                // of head 8hb + g8)
                uint32_t pb[HB][4];
#pragma unroll
                for (int hb = 0; hb < HB; ++hb) {
                    float x[4];
                    x[0] = live0 ? sc[hb][0] * ks0 : -INFINITY;
                    x[1] = live0 ? sc[hb][1] * ks0 : -INFINITY;
                    x[2] = live1 ? sc[hb][2] * ks1 : -INFINITY;
                    x[3] = live1 ? sc[hb][3] * ks1 : -INFINITY;
                    float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
#pragma unroll
                        for (int off = 4; off < 32; off <<= 1) mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], off));
                    }
                    float alpha[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float mn = fmaxf(m[hb][e], mx[e]);          // finite: token 0 is valid
                        alpha[e] = fast_exp2(m[hb][e] - mn);
                        m[hb][e] = mn;
                    }
                    float pw[4], wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pw[e] = fast_exp2(x[e] - m[hb][e & 1]);
                        wv[e] = pw[e] * (e < 2 ? vs0 : vs1);
                    }
                    l[hb][0] = l[hb][0] * alpha[0] + (pw[0] + pw[2]);
                    l[hb][1] = l[hb][1] * alpha[1] + (pw[1] + pw[3]);
                    const uint32_t h0 = pack_f16x2(wv[0], wv[1]), h1 = pack_f16x2(wv[2], wv[3]);
                    const uint32_t e0 = pack_f16x2(wv[0] - f16_lo(h0), wv[1] - f16_hi(h0));
                    const uint32_t e1 = pack_f16x2(wv[2] - f16_lo(h1), wv[3] - f16_hi(h1));
                    pb[hb][0] = movmatrix_trans(h0);
                    pb[hb][1] = movmatrix_trans(h1);
                    pb[hb][2] = movmatrix_trans(e0);
                    pb[hb][3] = movmatrix_trans(e1);
#pragma unroll
                    for (int mb = 0; mb < NM; ++mb) {
                        o[hb][mb][0] *= alpha[0];
                        o[hb][mb][1] *= alpha[1];
                        o[hb][mb][2] *= alpha[0];
                        o[hb][mb][3] *= alpha[1];
                    }
                }
                // Oᵀ += Vᵀ·Pᵀ for the two parts; A rows g8 / g8 + 8 of row block mb are features
                // f(mb, g8) / f(mb, g8 + 8): byte pairs (token, token + 1) of one feature
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    uint32_t lo[4], hi[4];   // row blocks 2w (lo) and 2w + 1 (hi): a0, a1, a2, a3
                    widen4(prmt(vw[0][w], vw[1][w], 0x5140u), lo[0], lo[1]);
                    widen4(prmt(vw[0][w], vw[1][w], 0x7362u), hi[0], hi[1]);
                    widen4(prmt(vw[2][w], vw[3][w], 0x5140u), lo[2], lo[3]);
                    widen4(prmt(vw[2][w], vw[3][w], 0x7362u), hi[2], hi[3]);
#pragma unroll
                    for (int hb = 0; hb < HB; ++hb) {
                        mma_f16_16816(o[hb][2 * w], lo[0], lo[1], lo[2], lo[3], pb[hb][0], pb[hb][1]);
                        mma_f16_16816(o[hb][2 * w], lo[0], lo[1], lo[2], lo[3], pb[hb][2], pb[hb][3]);
                        mma_f16_16816(o[hb][2 * w + 1], hi[0], hi[1], hi[2], hi[3], pb[hb][0], pb[hb][1]);
                        mma_f16_16816(o[hb][2 * w + 1], hi[0], hi[1], hi[2], hi[3], pb[hb][2], pb[hb][3]);
                    }
                }
            }
            __syncwarp();                 // the stage is read
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }

        // -------------------------------------------------------------- end of the piece
        // each warp's (Oᵀ, m, l) of the G heads through the combine buffer, then combined
        float *mine = cmb + (size_t)warp * G * (D + 2);
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float lr = l[hb][e];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) lr += __shfl_xor_sync(0xffffffffu, lr, off);
                const int h = 8 * hb + 2 * cq + e;
                if (h < G) {
                    float *row = mine + h * (D + 2);
#pragma unroll
                    for (int mb = 0; mb < NM; ++mb) {
                        row[(D / 8) * g8 + 2 * mb] = o[hb][mb][e];
                        row[(D / 8) * g8 + 2 * mb + 1] = o[hb][mb][2 + e];
                    }
                    if (g8 == 0) {
                        row[D] = ok ? m[hb][e] : -INFINITY;
                        row[D + 1] = ok ? lr : 0.f;
                    }
                }
            }
        bar_sync_named(kBar, kNum);
        const int slot = 2 * c + (k == 0 ? 0 : 1);
        for (int idx = threadIdx.x; idx < G * D; idx += kNum) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, cmb[((size_t)w * G + h) * (D + 2) + D]);
            float Lsum = 0.f, val = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float *row = cmb + ((size_t)w * G + h) * (D + 2);
                const float f = M == -INFINITY ? 0.f : fast_exp2(row[D] - M);
                Lsum = fmaf(row[D + 1], f, Lsum);
                val = fmaf(row[d], f, val);
            }
            const float inv = Lsum > 0.f ? 1.f / (Lsum * kWeightScale) : 0.f;
            if (p.whole) {
                a.out[((size_t)p.b * a.Hq + (size_t)j * G + h) * D + d] = val * inv;
            } else {
                const size_t pr = (size_t)slot * G + h;
                a.o_part[pr * D + d] = val * inv;
                if (d == 0) a.lse_part[pr] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
            }
        }
        if (!p.whole) {
            // the rows are stored: hand the piece to the producer warp for publication
            __syncwarp();
            if (lane == 0) mbar_arrive(pub_bar);
            if (n_pub == 0) {
                pb0 = p.b; pj0 = j; ps0 = p.S;
            } else {
                pb1 = p.b; pj1 = j; ps1 = p.S;
            }
            ++n_pub;
        }
        ++k;
    }

    // ------------------------------------------------------------ merge the segment of the
    // block's last piece if the block arrived last on it
    if (n_pub > 0 && !mbar_wait_bounded(end_bar, 0, &g_decode_fp8_status, kStatusPublishWait)) n_pub = 0;
    for (int u = 0; u < n_pub; ++u) {
        if (!last_flag[u]) continue;
        const int b = u ? pb1 : pb0, j = u ? pj1 : pj0;
        const SegSplit sp(prefix, seg_per_seq, b, j, u ? ps1 : ps0, T, a.n_blocks);
        merge_segment<D>(a, sp, b, j, G, threadIdx.x, kNum);
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return 148;
    }
    return n;
}

size_t smem_for(int D, int B, int G) {
    return D == 64 ? Cfg<64>::smem_bytes(B, G) : D == 96 ? Cfg<96>::smem_bytes(B, G) : Cfg<128>::smem_bytes(B, G);
}

// Persistent blocks: as many as reside on every SM (the register cap's count, fewer when the
// shared memory, 228 KiB per SM with 1 KiB reserved per block, holds fewer); n_split > 0 caps
// them at n_split per (sequence, KV head).
int fp8_blocks(int B, int Hq, int Hkv, int D, int n_split) {
    const int by_regs = Hq / Hkv > 8 ? kResident<64, 2> : D == 128 ? kResident<128, 1> : kResident<64, 1>;
    const int by_smem = (int)((228 * 1024) / (smem_for(D, B, Hq / Hkv) + 1024));
    const int per_sm = max(1, min(by_regs, by_smem));
    long long n = (long long)per_sm * sm_count();
    const long long per_seg = n_split > 0 ? n_split : kMaxPieces;
    if (per_seg * B * Hkv < n) n = per_seg * B * Hkv;
    return (int)(n < 1 ? 1 : n);
}

template <int D, int HB>
cudaError_t launch_d(const CUtensorMap &km, const CUtensorMap &vm, const Fp8Args &a, cudaStream_t st) {
    const size_t smem = Cfg<D>::smem_bytes(a.B, a.Hq / a.Hkv);
    auto kern = decode_fp8_kernel<D, HB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(a.n_blocks), dim3(kThreads), smem, st, km, vm, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool decode_fp8_mma_eligible(int B, int Hq, int Hkv, int D) {
    return Hq / Hkv <= 16 && (D == 64 || D == 96 || D == 128) && smem_for(D, B, Hq / Hkv) <= 227 * 1024;
}

int decode_fp8_blocks(int B, int Hq, int Hkv, int D, int n_split) { return fp8_blocks(B, Hq, Hkv, D, n_split); }

// Workspace: one arrival counter per (sequence, KV head) in the counter region, then two
// partial slots of G rows × D floats per block and their log-sum-exps.
size_t decode_fp8_workspace(int B, int Hq, int Hkv, int D, int n_split) {
    const size_t rows = 2 * (size_t)fp8_blocks(B, Hq, Hkv, D, n_split) * (Hq / Hkv);
    return counter_region_bytes((size_t)B * Hkv) + (rows * D * 4 + 255) / 256 * 256 + (rows * 4 + 255) / 256 * 256;
}

cudaError_t launch_decode_fp8_mma(const void *q, const void *k, const void *v, const float *k_scale,
                                  const float *v_scale, const int *seq_lens, float *out, int B, int Hq, int Hkv,
                                  int D, float scale_log2, int S_max, int n_split, void *ws, cudaStream_t st) {
    Fp8Args a{};
    a.q = q; a.k_scale = k_scale; a.v_scale = v_scale; a.seq_lens = seq_lens; a.out = out;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.S_max = S_max; a.scale_log2 = scale_log2;
    a.n_blocks = fp8_blocks(B, Hq, Hkv, D, n_split);
    const size_t rows = 2 * (size_t)a.n_blocks * (Hq / Hkv);
    char *w = static_cast<char *>(ws);
    a.counters = reinterpret_cast<int *>(w);
    w += counter_region_bytes((size_t)B * Hkv);
    a.o_part = reinterpret_cast<float *>(w);
    a.lse_part = reinterpret_cast<float *>(w + (rows * D * 4 + 255) / 256 * 256);
    CUtensorMap km, vm;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)Hkv, (uint64_t)S_max, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)D, (uint64_t)Hkv * D, (uint64_t)S_max * Hkv * D};
    const uint32_t box[4] = {(uint32_t)D, 1, (uint32_t)TT, 1};
    cudaError_t e = encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, k, dims, strides, box,
                                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess)
        e = encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, v, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess) e = clear_overflow_counters(a.counters, (size_t)B * Hkv, st);
    if (e != cudaSuccess) return e;
    switch (D) {
        case 64: return Hq / Hkv > 8 ? launch_d<64, 2>(km, vm, a, st) : launch_d<64, 1>(km, vm, a, st);
        case 96: return Hq / Hkv > 8 ? launch_d<96, 2>(km, vm, a, st) : launch_d<96, 1>(km, vm, a, st);
        case 128: return Hq / Hkv > 8 ? launch_d<128, 2>(km, vm, a, st) : launch_d<128, 1>(km, vm, a, st);
        default: return cudaErrorInvalidValue;
    }
}

int decode_fp8_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_decode_fp8_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_decode_fp8_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
