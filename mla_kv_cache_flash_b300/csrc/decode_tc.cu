// K1 for wide query groups and K3 (MLA) on the 5th-generation tensor cores: decode over a
// bf16 cache when 16 or more query heads share each cached row.
//
// The method: out[b,h] = softmax(scale · q[b,h]·K[b,:S_b,j]ᵀ) · V[b,:S_b,j], j = h / G
// ("模型架构｜MQA & GQA 调研", section "代码", Attention.forward with one new token). MLA's
// absorbed form is the same with K = [c ‖ kr] (176 columns) and V = c (qqstock article on
// DeepSeek MLA, sections 2, 3 and 6): every head reads the one latent row.
// With G heads per row the work is about 2·G flops per cached byte (16 at G = 16 over the
// 176-wide MLA key and 128-wide value, 32 for MQA with 32 heads), which is past what
// register-fragment tensor cores sustain at HBM speed on one SM. So here both products run as
// tcgen05 MMAs with the accumulators in tensor memory, and the cached tokens - not the
// heads - form the 128-row M side:
//   Sᵀ = K·Qᵀ        M = 128 tokens of a tile, N = the block's N query heads (16 or 32),
//                    K = key width; A (the cache tile) and B (the query rows) K-major in
//                    shared memory, 128-byte swizzle (32-byte for MLA's 48-wide rope part).
//   softmax          one thread per token row reads its N scores from TMEM: base-2 scores,
//                    a per-head reference maximum m, weights p = 2^(s − m) as a bf16 head
//                    plus a bf16 residual (p − head), per-thread partial sums l. The reference is raised (and O and l scaled
//                    down) only when a score exceeds it by more than 2^8, which a block-wide
//                    vote detects; the result does not depend on the reference, it only
//                    bounds the range of p.
//   Oᵀ += Vᵀ·Pᵀ     M = 128 value columns, N heads, K = 128 tokens: Vᵀ is the cache tile read
//                    MN-major from the same shared memory that TMA filled, Pᵀ is the
//                    softmax threads' bf16 rows (one token's N weights each) in shared memory,
//                    multiplied once for the heads and once for the residuals.
// Precision: a bf16 weight alone is off by up to 2^-9 of itself, which a sequence of a few
// tokens does not average away (measured: 3.1e-3 on 5-token rows); with the residual the
// weights carry about 16 significant bits, and the sums l use the same two-part values.
//
// The work is split like the register-MMA decode kernel (streamk.cuh): segments = (sequence,
// KV head, block of N query heads), cut into 128-token tiles laid end to end; each persistent
// block (one per SM) takes an equal run of tiles. A segment a block covers whole is written
// to `out`; a shared one leaves a normalised partial and ln Σ e^s in the block's slot, and the
// last block to finish the segment (acquire-release arrival counter) combines them.
//
// Warp roles (192 threads, one block per SM; two for 16-head MLA):
//   warp 0     TMA producer: per piece the query rows into a slot (two slots where shared
//              memory allows), per tile the cache rows into an NS-stage ring (L2 evict-first).
//   warp 1     allocates 128 TMEM columns (S double buffer at 0 and 32; O at 64: N columns
//              for the weights' heads, N for their residuals, summed at the end); lane 0
//              issues the MMAs: S(g) as soon as tile g lands, P·V(g−1) after it.
//   warps 2-5  softmax, one thread per token row / TMEM lane; at a piece end the same
//              threads read Oᵀ (lane = value column) and write the output or the partial.
// Tokens past a sequence's end get weight 0 and their value rows are zeroed in shared memory
// before P·V, so stale cache contents never reach the output.
//
// Every mbarrier wait is bounded (MLAKV_WAIT_TIMEOUT_CYCLES); a wait that runs out sets a bit
// in g_decode_tc_status and the thread skips later waits, while still meeting its partners at
// every named barrier, so the block always reaches its end and frees its tensor memory.
#include "ptx.cuh"
#include "streamk.cuh"
#include "tcgen05.cuh"
#include "tensor_map.cuh"

#include <math.h>

namespace mlakv {

__device__ unsigned g_decode_tc_status;

namespace {

constexpr int kGqa = 0, kMla = 1;
constexpr int TILE = 128;                 // tokens per tile (TMEM lanes)
constexpr int DV = 128;                   // value width: D of GQA, r of MLA
constexpr int BOX = TILE * 128;           // one 128-byte-swizzled box: 128 rows × 64 columns
constexpr int ROPE_BOX = TILE * 32;       // one 32-byte-swizzled box: 128 rows × 16 columns
constexpr int kSoftmax = 128;             // threads of one softmax warpgroup
constexpr int kPlist = 256;               // partial slots a merge can list in shared memory
constexpr float kRescaleLog2 = 8.0f;
constexpr int kChunkTokens = 4;           // chunked prefill: new tokens per segment (N = 64)

// CH: chunked prefill. A block's N columns are then kChunkTokens new tokens × 16 query heads
// (column i·16 + h), and each column has its own key limit (bottom-right causal).
template <int KIND, int N, bool CH = false>
struct Cfg {
    static_assert(CH ? N == 16 * kChunkTokens : (N == 16 || N == 32), "16 or 32 query heads per block, "
                  "or a chunk of kChunkTokens tokens × 16 heads");
    static constexpr int NT = CH ? kChunkTokens : 1;            // new tokens per block
    static constexpr int HB = CH ? 16 : N;                      // query heads per block
    // softmax warpgroups (4 warps each) and the columns each owns: one warpgroup for up to 32
    // columns; a 64-column chunk block splits its columns between two, so that each thread
    // forms 32 weights per token row and two softmax warps share each SM sub-partition
    static constexpr int NWG = N > 32 ? 2 : 1;
    static constexpr int NC = N / NWG;
    static constexpr int NSM = kSoftmax * NWG;                  // softmax threads
    static constexpr int THREADS = 64 + NSM;                    // + the TMA and MMA warps
    // ring stage: the key tile (2 boxes of K or c), then V (2 boxes) or kr (3 boxes)
    static constexpr int STAGE = 2 * BOX + (KIND == kGqa ? 2 * BOX : 3 * ROPE_BOX);
    // blocks per SM: two for 16-head MLA (two independent tile chains share the SM's tensor
    // pipe and TMA engine, each filling the other's gaps), one otherwise
    static constexpr int CPS = KIND == kMla && N == 16 ? 2 : 1;
    static constexpr int NS = CH ? (KIND == kGqa ? 2 : 3) : KIND == kGqa ? 3 : CPS == 2 ? 2 : 4;
    static constexpr int V_OFF = KIND == kGqa ? 2 * BOX : 0;     // value tile inside a stage
    static constexpr int Q_BOX = N * 128;                       // N query rows × 64 columns
    static constexpr int QR_BOX = N * 32;                       // N rows × 16 rope columns
    static constexpr int Q_BYTES = 2 * Q_BOX + (KIND == kMla ? 3 * QR_BOX : 0);
    static constexpr int Q_SLOT = (Q_BYTES + 1023) / 1024 * 1024;
    // query slots: two (the next piece's rows load early) where shared memory allows
    static constexpr int QS = (KIND == kGqa && N == 32) || CPS == 2 || CH ? 1 : 2;
    // one token's weights as 2N bf16: the N heads, then the N residuals; the P·V product
    // takes both as one N = 2N operand (one MMA chain instead of two). Stored as rows of
    // PROW bytes (the swizzle width) in blocks of TILE rows along the 2N columns.
    static constexpr int PROW = N == 16 ? 64 : 128;
    static constexpr int P_ROW = 2 * N * 2;
    static constexpr int P_BYTES = TILE * P_ROW;
    static constexpr uint32_t P_LAYOUT = N == 16 ? kSw64 : kSw128;
    static constexpr int Q_OFF = NS * STAGE;
    // weight buffers: two (the softmax of tile g + 1 need not wait for P·V(g)) where shared
    // memory allows
    static constexpr int PB = (N == 16 && CPS == 1) || CH ? 2 : 1;
    // tensor memory: two S buffers of N columns (32 apart at least), then O (2N columns)
    static constexpr uint32_t S_COLS = N < 32 ? 32 : N;
    static constexpr uint32_t O_COL = 2 * S_COLS;
    static constexpr uint32_t TMEM_COLS = O_COL + 2 * N <= 128 ? 128 : 256;
    static constexpr int P_OFF = Q_OFF + QS * Q_SLOT;
    static constexpr int BAR_OFF = P_OFF + PB * P_BYTES;
    static constexpr int N_BARS = 2 * NS + 12;
    static constexpr int SCR_OFF = BAR_OFF + 256;
    static constexpr int MAXRED_OFF = SCR_OFF;                  // [4][N] per-warp tile maxima
    static constexpr int LRED_OFF = MAXRED_OFF + 4 * N * 4;     // [4][N] per-warp sums
    static constexpr int STAT_OFF = LRED_OFF + 4 * N * 4;       // [N] 1/L, [N] lse
    static constexpr int MISC_OFF = STAT_OFF + 2 * N * 4;       // TMEM base, merge flag
    static constexpr int SHREC_OFF = MISC_OFF + 16;             // [2] shared-segment records
    static constexpr int PLIST_OFF = SHREC_OFF + 2 * 64;
    static constexpr int PREFIX_OFF = PLIST_OFF + kPlist * 4;
    static_assert(STAGE % 1024 == 0 && Q_SLOT % 1024 == 0 && P_BYTES % 1024 == 0, "swizzle alignment");
    static_assert(N_BARS * 8 <= 256, "barrier area");
    // after the tile prefix [B+1]: the keys per sequence [B] (decode: seq_lens), then for
    // chunked prefill the first new-token row [B+1] and the segment prefix [B+1]
    // the prefix arrays, then the walk's start (b, q, i0)
    static size_t smem_bytes(int B) { return PREFIX_OFF + (size_t)(B + 1) * 4 * (CH ? 4 : 2) + 16 + 1024; }
};

// Barrier indices.
template <int NS>
struct Bars {
    static constexpr int FULL = 0, EMPTY = NS, QFULL = 2 * NS, QEMPTY = 2 * NS + 2, SFULL = 2 * NS + 4,
                         SFREE = 2 * NS + 6, PREADY = 2 * NS + 8, PVDONE = 2 * NS + 10;   // PREADY, PVDONE: one per weight buffer
};

struct TcArgs {
    const int *seq_lens;    // [B] (chunked prefill: unused)
    const int *cu_q;        // chunked prefill: [B+1] first new-token row of each sequence
    const int *start_pos;   // chunked prefill: [B] keys cached before each chunk
    float *out;             // [B, Hq, 128]
    float *o_part;          // [2·n_blocks, N, 128]
    float *lse_part;        // [2·n_blocks, N]
    int *counters;          // [segments] at the workspace's start, zero between calls
    int B, Hq, G;           // G: query heads per KV head (MLA: all Hq)
    int seg_per_seq;        // segments per sequence (chunked prefill: per query block): KV heads × head blocks
    int n_hblk;             // head blocks of N per KV head
    float scale_log2;
    int n_blocks;
    int aligned;
};

// Reduce N per-thread values over the 32 lanes of a warp, one head per lane group: after the
// call, lane L holds the reduction for head L >> (5 − log2 N). Halving exchange: at each step
// a lane keeps half of its heads and receives its partner's values for them.
template <int N, bool MAX>
__device__ __forceinline__ float xpose_reduce(float (&v)[N], int lane) {
#pragma unroll
    for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
            const float send = up ? v[j] : v[j + n / 2];
            const float keep = up ? v[j + n / 2] : v[j];
            const float r = __shfl_xor_sync(0xffffffffu, send, o);
            v[j] = MAX ? fmaxf(keep, r) : keep + r;
        }
    }
    float x = v[0];
#pragma unroll
    for (int o = N == 32 ? 0 : 1; o > 0; o >>= 1) {
        const float r = __shfl_xor_sync(0xffffffffu, x, o);
        x = MAX ? fmaxf(x, r) : x + r;
    }
    return x;
}

template <int N>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 64) tmem_ld64_sync(taddr, r);
    else if constexpr (N == 32) tmem_ld32_sync(taddr, r);
    else tmem_ld16_sync(taddr, r);
}

// Per-column reductions over a warp for N columns (see xpose_reduce): calls put(head, value)
// on the lanes that hold a head's result. N = 64 reduces its two halves of 32 in turn.
template <int N, bool MAX, typename Put>
__device__ __forceinline__ void reduce_cols(const float (&x)[N], int lane, Put put) {
    constexpr int H = N < 32 ? N : 32;
    constexpr int SHIFT = H == 32 ? 0 : 1;
#pragma unroll
    for (int half = 0; half < N / H; ++half) {
        float v[H];
#pragma unroll
        for (int h = 0; h < H; ++h) v[h] = x[half * H + h];
        const float r = xpose_reduce<H, MAX>(v, lane);
        if ((lane & ((1 << SHIFT) - 1)) == 0) put(half * H + (lane >> SHIFT), r);
    }
}

// Where a segment's rows live. Decode: one query row per head, out row (b, h0 + column).
// Chunked prefill: column n is new token n / 16 of the block and head h0 + n % 16; the token
// sits at packed row row0 + n / 16 and sees keys [0, kbase + n / 16 + 1).
struct SegInfo {
    int gi, hb, q;          // KV head, head block, segment index within the sequence
    int row0, nvalid;       // first output row, valid new tokens (decode: b, 1)
    int h0;                 // first query head
    int kbase;              // chunked prefill: keys before the block's first token
    int seg;                // global segment index (arrival counter)
};

template <int N>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&r)[N]) {
    if constexpr (N == 32) tmem_st32(taddr, r); else tmem_st16(taddr, r);
}

template <int KIND, int N, bool CH>
__global__ void __launch_bounds__(Cfg<KIND, N, CH>::THREADS, Cfg<KIND, N, CH>::CPS)
decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,    // K (GQA) or c (MLA)
                 const __grid_constant__ CUtensorMap vmap,    // V (GQA) or kr (MLA)
                 const __grid_constant__ CUtensorMap qmap,    // q (GQA) or q_lat (MLA)
                 const __grid_constant__ CUtensorMap qrmap,   // q_rope (MLA)
                 const TcArgs a) {
    using C = Cfg<KIND, N, CH>;
    using BI = Bars<C::NS>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + C::BAR_OFF + 8 * i; };
    float *maxred = reinterpret_cast<float *>(smem + C::MAXRED_OFF);
    float *lred = reinterpret_cast<float *>(smem + C::LRED_OFF);
    float *stat = reinterpret_cast<float *>(smem + C::STAT_OFF);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    int *plist = reinterpret_cast<int *>(smem + C::PLIST_OFF);
    int *prefix = reinterpret_cast<int *>(smem + C::PREFIX_OFF);
    int *klen = prefix + (a.B + 1);       // keys per sequence (decode: a copy of seq_lens)
    int *cu = klen + (a.B + 1);           //   first new-token row per sequence, [B+1]
    int *segpre = cu + (a.B + 1);         //   segments before each sequence, [B+1]
    int *wstart = prefix + (CH ? 4 : 2) * (a.B + 1);   // decode: the walk's start b, q, i0

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(BI::FULL + s), 1);
            mbar_init(bar(BI::EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(BI::QFULL + i), 1);
            mbar_init(bar(BI::QEMPTY + i), 1);
            mbar_init(bar(BI::SFULL + i), 1);
            mbar_init(bar(BI::SFREE + i), 4 * C::NWG);
        }
        for (int i = 0; i < C::PB; ++i) {
            mbar_init(bar(BI::PREADY + i), 4 * C::NWG);
            mbar_init(bar(BI::PVDONE + i), 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sb + C::MISC_OFF, C::TMEM_COLS);
        tmem_relinquish();
    }
    uint64_t pol = 0;                         // producer: L2 evict-first for the streamed rows
    if (threadIdx.x == 0) {
        // the descriptors are kernel parameters, which no earlier kernel writes
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        prefetch_tensormap(&qmap);
        if (KIND == kMla) prefetch_tensormap(&qrmap);
        pol = l2_evict_first_policy();
    }
    // everything above overlaps the previous kernel in the stream; the inputs are read below
    griddep_wait();
    griddep_launch_dependents();
    if (CH && warp == 0) {
        // per sequence: n new tokens at rows cu_q[b] .., seeing keys up to start_pos[b] + n;
        // ceil(n / NT) query blocks of seg_per_seq segments each, every one over those keys
        int carry = 0, scarry = 0;
        for (int base = 0; base < a.B; base += 32) {
            const int b = base + lane;
            int n = 0, st = 0, c0 = 0;
            if (b < a.B) {
                c0 = __ldg(a.cu_q + b);
                n = __ldg(a.cu_q + b + 1) - c0;
                st = __ldg(a.start_pos + b);
            }
            const int keys = n > 0 ? st + n : 0;
            const int nseg = (n + C::NT - 1) / C::NT * a.seg_per_seq;
            const int v = nseg * stream_tiles(keys, TILE);
            int x = v, y = nseg;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int xu = __shfl_up_sync(0xffffffffu, x, o);
                const int yu = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) x += xu, y += yu;
            }
            if (b < a.B) {
                prefix[b] = carry + x - v;
                segpre[b] = scarry + y - nseg;
                klen[b] = keys;
                cu[b] = c0;
            }
            carry += __shfl_sync(0xffffffffu, x, 31);
            scarry += __shfl_sync(0xffffffffu, y, 31);
        }
        if (lane == 0) {
            prefix[a.B] = carry;
            segpre[a.B] = scarry;
            cu[a.B] = __ldg(a.cu_q + a.B);
        }
    } else if (warp == 0) {
        // tile prefix over the sequences (warp scan, 32 sequences at a time; the lengths of
        // up to 128 sequences are loaded in one round trip)
        int carry = 0;
        for (int base = 0; base < a.B; base += 128) {
            int len[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int b = base + 32 * j + lane;
                len[j] = b < a.B ? __ldg(a.seq_lens + b) : 0;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (base + 32 * j >= a.B) break;
                const int b = base + 32 * j + lane;
                if (b < a.B) klen[b] = len[j];
                const int v = stream_tiles(len[j], TILE);
                int x = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (b < a.B) prefix[b] = carry + x - v;
                carry += __shfl_sync(0xffffffffu, x, 31);
            }
        }
        if (lane == 0) prefix[a.B] = carry;
        __syncwarp();
        // where this block's tile range starts (streamed split): found once, lane-parallel
        const long long T0 = (long long)a.seg_per_seq * carry;
        int b0 = 0, q0 = 0, i00 = 0;
        if (!a.aligned && T0 > 0) {
            const long long t0 = stream_start(blockIdx.x, T0, a.n_blocks);
            if (t0 < stream_start(blockIdx.x + 1, T0, a.n_blocks))
                seq_walk_start(prefix, a.B, a.seg_per_seq, t0, lane, b0, q0, i00);
        }
        if (lane == 0) {
            wstart[0] = b0;
            wstart[1] = q0;
            wstart[2] = i00;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    // tiles of all segments, laid end to end
    const long long T = CH ? (long long)prefix[a.B] : (long long)a.seg_per_seq * prefix[a.B];
    const int c = blockIdx.x;
    SeqWalker walk{prefix, klen, a.B, a.seg_per_seq / a.n_hblk, a.n_hblk, 0, 0, 0, 0, 0, 0};
    if (!CH && a.aligned) {
        // block c streams segment c whole
        const int b = c / a.seg_per_seq, q = c % a.seg_per_seq;
        const int nb = stream_tiles(klen[b], TILE);
        const long long t = (long long)a.seg_per_seq * prefix[b] + (long long)q * nb;
        walk.set(b, q, 0, t, t + nb);
    } else if (T > 0) {
        if constexpr (CH) {
            walk.t = stream_start(c, T, a.n_blocks);
            walk.t_end = stream_start(c + 1, T, a.n_blocks);
        } else {
            walk.set(wstart[0], wstart[1], wstart[2], stream_start(c, T, a.n_blocks), stream_start(c + 1, T, a.n_blocks));
        }
    }
    ChunkPieceWalker cwalk{prefix, klen, a.B, TILE, walk.t, walk.t_end};
    auto next_piece = [&](Piece &p) {
        if constexpr (CH) return cwalk.next(p);
        else return walk.next(p);
    };
    // the rows, heads and counter of a piece's segment
    auto seg_info = [&](const Piece &p) {
        SegInfo r;
        if constexpr (CH) {
            r.q = p.gi;
            const int qb = r.q / a.seg_per_seq, rem = r.q % a.seg_per_seq;
            r.gi = rem / a.n_hblk;
            r.hb = rem % a.n_hblk;
            const int n = cu[p.b + 1] - cu[p.b];
            r.row0 = cu[p.b] + qb * C::NT;
            r.nvalid = min(C::NT, n - qb * C::NT);
            r.kbase = klen[p.b] - n + qb * C::NT;
            r.h0 = r.gi * a.G + r.hb * C::HB;
            r.seg = segpre[p.b] + r.q;
        } else {
            r.gi = p.gi;
            r.hb = p.hb;
            r.q = p.gi * a.n_hblk + p.hb;
            r.row0 = p.b;
            r.nvalid = 1;
            r.kbase = 0;
            r.h0 = p.gi * a.G + p.hb * N;
            r.seg = p.b * a.seg_per_seq + r.q;
        }
        return r;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && walk.t < walk.t_end) {
            int g = 0, k = 0;
            bool ok = true;
            Piece p;
            // A piece's query rows go to slot k % QS once the piece that used the slot before
            // has issued its last score MMA. With one slot, the piece's first tile is requested
            // before that wait, so the cache stream does not pause at the piece boundary.
            // the query rows: decode, heads h0 .. h0+N-1 of sequence b (box N heads × 1);
            // chunked prefill, heads h0 .. h0+15 of packed rows row0 .. row0+NT-1 (box 16 × NT)
            auto load_q = [&](const Piece &pc, int kq) {
                const int qs = kq % C::QS;
                if (kq >= C::QS && !mbar_wait_bounded(bar(BI::QEMPTY + qs), ((kq / C::QS) - 1) & 1,
                                                      &g_decode_tc_status, kStatusEmptyWait))
                    return false;
                const SegInfo si = seg_info(pc);
                const uint32_t qd = sb + C::Q_OFF + qs * C::Q_SLOT;
                const uint32_t qb = bar(BI::QFULL + qs);
                mbar_arrive_expect_tx(qb, C::Q_BYTES);
                tma_load_3d(qd, &qmap, 0, si.h0, si.row0, qb, pol);
                tma_load_3d(qd + C::Q_BOX, &qmap, 64, si.h0, si.row0, qb, pol);
                if constexpr (KIND == kMla) {
#pragma unroll
                    for (int i = 0; i < 3; ++i)
                        tma_load_3d(qd + 2 * C::Q_BOX + i * C::QR_BOX, &qrmap, 16 * i, si.h0, si.row0, qb, pol);
                }
                return true;
            };
            while (ok && next_piece(p)) {
                // the query rows go after the piece's first tile: for the first piece, so the
                // cache stream starts at once; with one query slot, so it does not pause at the
                // piece boundary
                const bool q_late = C::QS == 1 || k == 0;
                if (!q_late && !load_q(p, k)) {
                    ok = false;
                    break;
                }
                for (int i = 0; i < p.n_t; ++i, ++g) {
                    const int s = g % NS;
                    if (!mbar_wait_bounded(bar(BI::EMPTY + s), ((g / NS) & 1) ^ 1, &g_decode_tc_status,
                                           kStatusEmptyWait)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sb + s * C::STAGE;
                    const uint32_t fb = bar(BI::FULL + s);
                    mbar_arrive_expect_tx(fb, C::STAGE);
                    const int t = (p.i0 + i) * TILE;
                    if constexpr (KIND == kGqa) {
                        const int j = CH ? seg_info(p).gi : p.gi;
                        tma_load_4d(dst, &kmap, 0, j, t, p.b, fb, pol);
                        tma_load_4d(dst + BOX, &kmap, 64, j, t, p.b, fb, pol);
                        tma_load_4d(dst + 2 * BOX, &vmap, 0, j, t, p.b, fb, pol);
                        tma_load_4d(dst + 3 * BOX, &vmap, 64, j, t, p.b, fb, pol);
                    } else {
                        tma_load_3d(dst, &kmap, 0, t, p.b, fb, pol);
                        tma_load_3d(dst + BOX, &kmap, 64, t, p.b, fb, pol);
#pragma unroll
                        for (int r = 0; r < 3; ++r) tma_load_3d(dst + 2 * BOX + r * ROPE_BOX, &vmap, 16 * r, t, p.b, fb, pol);
                    }
                    if (q_late && i == 0 && !load_q(p, k)) {
                        ok = false;
                        ++g;
                        break;
                    }
                }
                ++k;
            }
            // no copy may still be in flight when the block exits
            for (int i = g > NS ? g - NS : 0; i < g; ++i)
                mbar_wait_bounded(bar(BI::FULL + i % NS), (i / NS) & 1, &g_decode_tc_status, kStatusDrainWait);
            for (int i = k > C::QS ? k - C::QS : 0; i < k; ++i)
                mbar_wait_bounded(bar(BI::QFULL + i % C::QS), (i / C::QS) & 1, &g_decode_tc_status, kStatusDrainWait);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 issues every MMA. Two products are due at any time: S(g), into S buffer
        // g & 1, once tile g has landed (and the softmax has read S(g − 2)); and P·V(g − 1),
        // once the softmax has written that tile's weights. Lane 0 polls both and issues
        // whichever is ready first: P·V(g − 1) releases tile g − 1's ring stage, so it must
        // not wait for tile g to land, and S(g) must not wait for the softmax of tile g − 1.
        // A piece's last P·V is issued before the next piece's first S, so the piece's
        // epilogue never waits for the next piece's data.
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(TILE, N, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(DV, 2 * N, true, true);
            const uint32_t t_o = tmem + C::O_COL;
            bool ok = true;
            auto issue_s = [&](int gg, int s, uint32_t qd) {
                const uint32_t kt = sb + s * C::STAGE;
                const uint32_t d = tmem + C::S_COLS * (gg & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * BOX + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * C::Q_BOX + (kk & 3) * 32;
                    umma_ss(d, sdesc(kt + off, 16, 1024, kSw128), sdesc(qd + qoff, 16, 1024, kSw128), idesc_s,
                            kk > 0 ? 1u : 0u);
                }
                if constexpr (KIND == kMla) {
#pragma unroll
                    for (int kk = 0; kk < 3; ++kk)
                        umma_ss(d, sdesc(kt + 2 * BOX + kk * ROPE_BOX, 16, 256, kSw32),
                                sdesc(qd + 2 * C::Q_BOX + kk * C::QR_BOX, 16, 256, kSw32), idesc_s, 1u);
                }
                umma_commit(bar(BI::SFULL + (gg & 1)));
            };
            auto issue_pv = [&](int gg, int s, bool first) {
                const uint32_t v = sb + s * C::STAGE + C::V_OFF;
                const uint32_t pb = sb + C::P_OFF + (gg % C::PB) * C::P_BYTES;
                // 16 tokens per MMA; columns [0, N) of O take the weights' heads, [N, 2N) their residuals
#pragma unroll
                for (int kk = 0; kk < TILE / 16; ++kk)
                    umma_ss(t_o, sdesc(v + kk * 2048, BOX, 1024, kSw128),
                            sdesc(pb + kk * 16 * C::PROW, TILE * C::PROW, 8 * C::PROW, C::P_LAYOUT), idesc_o,
                            (!first || kk > 0) ? 1u : 0u);
                umma_commit(bar(BI::PVDONE + gg % C::PB));
                umma_commit(bar(BI::EMPTY + s));
            };
            auto ready_pv = [&](int gg) { return mbar_test_wait(bar(BI::PREADY + gg % C::PB), (gg / C::PB) & 1); };
            int g = 0, k = 0;
            bool pend = false, pend_first = false;   // P·V of tile pend_g not yet issued
            int pend_g = 0, pend_s = 0;
            Piece p;
            while (ok && next_piece(p)) {
                const int qs = k % C::QS;
                const uint32_t qd = sb + C::Q_OFF + qs * C::Q_SLOT;
                for (int i = 0; ok && i < p.n_t; ++i, ++g) {
                    const int s = g % NS;
                    bool s_done = false;
                    const long long t0 = clock64();
                    while (!s_done || pend) {
                        if (pend && ready_pv(pend_g)) {
                            tc_fence_after();
                            issue_pv(pend_g, pend_s, pend_first);
                            pend = false;
                            continue;
                        }
                        if (!s_done && mbar_test_wait(bar(BI::FULL + s), (g / NS) & 1) &&
                            (g < 2 || mbar_test_wait(bar(BI::SFREE + (g & 1)), ((g >> 1) - 1) & 1)) &&
                            (i > 0 || mbar_test_wait(bar(BI::QFULL + qs), (k / C::QS) & 1))) {
                            tc_fence_after();
                            issue_s(g, s, qd);
                            if (i == p.n_t - 1) umma_commit(bar(BI::QEMPTY + qs));
                            s_done = true;
                            continue;
                        }
                        if (clock64() - t0 > MLAKV_WAIT_TIMEOUT_CYCLES) {
                            atomicOr(&g_decode_tc_status, kStatusMmaWait);
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    pend = true;
                    pend_g = g;
                    pend_s = s;
                    pend_first = i == 0;
                    if (i == p.n_t - 1) {
                        if (!mbar_wait_bounded(bar(BI::PREADY + g % C::PB), (g / C::PB) & 1, &g_decode_tc_status,
                                               kStatusMmaWait)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(g, s, i == 0);
                        pend = false;
                    }
                }
                ++k;
            }
            // the last products finish before the block frees tensor memory
            if (ok && g > 0)
                mbar_wait_bounded(bar(BI::PVDONE + (g - 1) % C::PB), ((g - 1) / C::PB) & 1, &g_decode_tc_status,
                                  kStatusMmaWait);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        // NWG warpgroups of four warps; warpgroup wg owns columns [wg·NC, wg·NC + NC) of the
        // block's N, with its own running maxima, rescale votes and named barrier (1 + wg);
        // barrier 3 spans all softmax warps. A thread owns one token row / TMEM lane.
        constexpr int NC = C::NC, NSM = C::NSM;
        const int row = 32 * (warp & 3) + lane;           // token row, TMEM lane, value column
        const int tid = threadIdx.x - 64;                 // 0 .. NSM - 1
        const int wg = tid / kSoftmax;
        const int sw = (tid % kSoftmax) >> 5;             // warp within the warpgroup
        const int tw = tid % kSoftmax;                    // thread within the warpgroup
        const int col0 = wg * NC;                         // first column of this warpgroup
        const int gbar = 1 + wg;
        const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t t_o = tmem + lane_addr + C::O_COL;
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t parity, unsigned code) {
            if (ok && !mbar_wait_bounded(b, parity, &g_decode_tc_status, code)) ok = false;
        };
        if (!CH && c == 0) {
            // sequences with an empty cache own no tile: their output is zero
            for (int b = 0; b < a.B; ++b)
                if (prefix[b + 1] == prefix[b])
                    for (int i = tid; i < a.Hq * DV / 4; i += NSM)
                        reinterpret_cast<float4 *>(a.out + (size_t)b * a.Hq * DV)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // The output row of column n of a segment: (row0 + n / HB) of the [rows, Hq, DV] output,
        // head h0 + n % HB; chunked prefill writes only the block's valid new tokens.
        auto out_row = [&](int row0, int h0, int n) {
            return ((size_t)(row0 + n / C::HB) * a.Hq + h0 + n % C::HB) * DV;
        };
        // Shared segments this block left a partial of (its first and last piece at most): their
        // records in shared memory, the arrival count thread 0 saw in a register, read only at
        // the end, so the counter's round trip never stalls the stream; the last arrival merges.
        struct Shared {
            long long fs;                     // the segment's first tile in the stream
            int row0, nvalid, h0, seg, nb;    // output rows, first query head, segment, its tiles
            int c0, c1, first_odd;            // its first and last owner blocks (filled at the end)
        };
        Shared *shrec = reinterpret_cast<Shared *>(smem + C::SHREC_OFF);
        int seen0 = 0, seen1 = 0, n_shared = 0;
        int g = 0, k = 0;
        Piece p;
        while (next_piece(p)) {
            const SegInfo si = seg_info(p);
            // chunked prefill: key limit of each new token among this warpgroup's columns
            // (column h is token col0 / HB + h / HB; 0: no such token)
            constexpr int NTW = (NC + C::HB - 1) / C::HB;
            int lim[NTW];
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const int tok = col0 / C::HB + j;
                lim[j] = tok < si.nvalid ? si.kbase + tok + 1 : 0;
            }
            // the reference maximum of each column (the same in every thread of the warpgroup)
            // and this thread's share of each column's weight sum. Chunked prefill starts the
            // reference at −1e30 rather than −∞: a column may see no visible key for a while
            // (its token's limit lies before the piece), and 2^(−∞ − (−1e30)) = 0 is then its
            // weight, where 2^(−∞ − (−∞)) would be NaN; the first visible score raises it.
            constexpr float kMInit = CH ? -1e30f : -INFINITY;
            float m[NC], l[NC];
#pragma unroll
            for (int h = 0; h < NC; ++h) {
                m[h] = kMInit;
                l[h] = 0.f;
            }
            for (int i = 0; i < p.n_t; ++i, ++g) {
                const int s = g % NS;
                wait(bar(BI::SFULL + (g & 1)), (g >> 1) & 1, kStatusMmaWait);
                tc_fence_after();
                uint32_t sr[NC];
                tmem_ld_row<NC>(tmem + lane_addr + C::S_COLS * (g & 1) + col0, sr);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BI::SFREE + (g & 1)));

                const int key = (p.i0 + i) * TILE + row;
                const bool valid = key < p.S;
                float x[NC];
#pragma unroll
                for (int h = 0; h < NC; ++h) {
                    const bool vis = CH ? key < lim[h / C::HB] : valid;
                    x[h] = vis ? __uint_as_float(sr[h]) * a.scale_log2 : -INFINITY;
                }
                bool need = i == 0;
                if (!need) {
                    bool ex = false;
#pragma unroll
                    for (int h = 0; h < NC; ++h) ex |= x[h] - m[h] > kRescaleLog2;
                    need = bar_any(gbar, kSoftmax, ex);
                }
                if (need) {
                    // new reference: the running maximum per column over all rows so far
                    reduce_cols<NC, true>(x, lane, [&](int h, float v) { maxred[sw * N + col0 + h] = v; });
                    bar_sync_named(gbar, kSoftmax);
                    // the factor old → new reference of column h, recomputed where needed rather
                    // than held, the rescale being rare
                    auto factor = [&](int h, float &mn) {
                        const int gc = col0 + h;
                        const float tm = fmaxf(fmaxf(maxred[gc], maxred[N + gc]), fmaxf(maxred[2 * N + gc], maxred[3 * N + gc]));
                        mn = fmaxf(m[h], tm);
                        return fast_exp2(m[h] - mn);
                    };
                    if (i > 0) {
                        // O holds the tiles before this one: scale this warpgroup's columns of
                        // both halves to the new reference
                        wait(bar(BI::PVDONE + (g - 1) % C::PB), ((g - 1) / C::PB) & 1, kStatusMmaWait);
                        tc_fence_after();
#pragma unroll
                        for (int ch = 0; ch < 2 * NC / 16; ++ch) {     // 16 columns at a time
                            const int hc = (ch * 16) % NC;            // first column of the chunk
                            const uint32_t ta = t_o + (ch * 16 < NC ? 0 : N) + col0 + hc;
                            uint32_t o[16];
                            tmem_ld16_sync(ta, o);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                float mn;
                                o[j] = __float_as_uint(__uint_as_float(o[j]) * factor(hc + j, mn));
                            }
                            tmem_st16(ta, o);
                        }
                        tmem_st_wait();
                    }
#pragma unroll
                    for (int h = 0; h < NC; ++h) {
                        float mn;
                        l[h] *= factor(h, mn);
                        m[h] = mn;
                    }
                }
                // weights as bf16 head + bf16 residual; the sums take the two-part values (chunked
                // prefill: the fp32 weights, which differ from them by under 2^-16 of themselves).
                // The token's 2N weights [heads | residuals] go to the weight buffer as 16-byte
                // chunks: chunk cc of a PROW-byte row of block cc / CPR, swizzled (128-byte rows:
                // chunk at cc ^ (row & 7); 64-byte rows: cc ^ ((row >> 1) & 3)); this thread's are
                // chunks col0 / 8 .. of each half.
                constexpr int CPR = C::PROW / 16;
                const int swz = C::PROW == 128 ? row & 7 : (row >> 1) & 3;
                auto weights8 = [&](int h0, uint4 &wk, uint4 &wr) {     // columns h0 .. h0 + 7
                    uint32_t k4[4], r4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int h = h0 + 2 * u;
                        const float p0 = fast_exp2(x[h] - m[h]), p1 = fast_exp2(x[h + 1] - m[h + 1]);
                        const uint32_t w = pack_bf16x2(p0, p1);
                        const uint32_t r = pack_bf16x2(p0 - bf16_lo(w), p1 - bf16_hi(w));
                        k4[u] = w;
                        r4[u] = r;
                        if (CH) {
                            l[h] += p0;
                            l[h + 1] += p1;
                        } else {
                            l[h] += bf16_lo(w) + bf16_lo(r);
                            l[h + 1] += bf16_hi(w) + bf16_hi(r);
                        }
                    }
                    wk = make_uint4(k4[0], k4[1], k4[2], k4[3]);
                    wr = make_uint4(r4[0], r4[1], r4[2], r4[3]);
                };
                uint8_t *pbuf = smem + C::P_OFF + (g % C::PB) * C::P_BYTES + row * C::PROW;
                auto chunk_at = [&](int cc) {
                    return reinterpret_cast<uint4 *>(pbuf + (cc / CPR) * TILE * C::PROW + (((cc % CPR) ^ swz) << 4));
                };
                if constexpr (CH) {
                    // the weight buffer is free once P·V(g − PB) has completed; each 8 columns'
                    // weights are stored as soon as they are formed
                    if (g >= C::PB) wait(bar(BI::PVDONE + g % C::PB), ((g / C::PB) - 1) & 1, kStatusMmaWait);
#pragma unroll
                    for (int c8 = 0; c8 < NC / 8; ++c8) {
                        uint4 wk, wr;
                        weights8(8 * c8, wk, wr);
                        *chunk_at(col0 / 8 + c8) = wk;
                        *chunk_at(N / 8 + col0 / 8 + c8) = wr;
                    }
                } else {
                    uint4 wk[NC / 8], wr[NC / 8];
#pragma unroll
                    for (int c8 = 0; c8 < NC / 8; ++c8) weights8(8 * c8, wk[c8], wr[c8]);
                    // the weight buffer is free once P·V(g − PB) has completed
                    if (g >= C::PB) wait(bar(BI::PVDONE + g % C::PB), ((g / C::PB) - 1) & 1, kStatusMmaWait);
#pragma unroll
                    for (int c8 = 0; c8 < NC / 8; ++c8) {
                        *chunk_at(col0 / 8 + c8) = wk[c8];
                        *chunk_at(N / 8 + col0 / 8 + c8) = wr[c8];
                    }
                }
                if (!valid && wg == 0) {
                    // a row past the sequence end: zero its value row (weight 0 · stale data)
                    uint8_t *vr = smem + s * C::STAGE + C::V_OFF + row * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        *reinterpret_cast<uint4 *>(vr + ch * 16) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(vr + BOX + ch * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BI::PREADY + g % C::PB));
            }

            // ---------------------------------------------------------- end of the piece
            reduce_cols<NC, false>(l, lane, [&](int h, float v) { lred[sw * N + col0 + h] = v; });
            bar_sync_named(gbar, kSoftmax);
            if (tw < NC) {
                const int gc = col0 + tw;
                const float L = lred[gc] + lred[N + gc] + lred[2 * N + gc] + lred[3 * N + gc];
                float mh = m[0];
#pragma unroll
                for (int h = 1; h < NC; ++h) mh = tw == h ? m[h] : mh;
                stat[gc] = ok && L > 0.f ? 1.f / L : 0.f;
                stat[N + gc] = ok && L > 0.f ? (mh + log2f(L)) * kLn2 : -INFINITY;
            }
            wait(bar(BI::PVDONE + (g - 1) % C::PB), ((g - 1) / C::PB) & 1, kStatusMmaWait);
            tc_fence_after();
            uint32_t o[NC], o2[NC];
            tmem_ld_row<NC>(t_o + col0, o);
            tmem_ld_row<NC>(t_o + N + col0, o2);
            tc_fence_before();
            bar_sync_named(gbar, kSoftmax);                // stat written
            const int slot = 2 * c + (k == 0 ? 0 : 1);
#pragma unroll
            for (int h = 0; h < NC; ++h) {
                const int gc = col0 + h;
                const float val = (__uint_as_float(o[h]) + __uint_as_float(o2[h])) * stat[gc];
                if (!p.whole) a.o_part[((size_t)slot * N + gc) * DV + row] = val;
                else if (!CH || gc / C::HB < si.nvalid) a.out[out_row(si.row0, si.h0, gc) + row] = val;
            }
            if (!p.whole) {
                if (tw < NC) a.lse_part[(size_t)slot * N + col0 + tw] = stat[N + col0 + tw];
                // publish: the partial's stores, ordered before thread 0's release by the
                // barrier, are visible to whichever block later acquires the counter. Thread 0
                // keeps the count it saw in a register of its own, read only at the end.
                bar_sync_named(3, NSM);
                if (tid == 0) {
                    if (n_shared == 0) seen0 = atomic_add_acq_rel_gpu(a.counters + si.seg, 1);
                    else seen1 = atomic_add_acq_rel_gpu(a.counters + si.seg, 1);
                    Shared &r = shrec[n_shared];
                    if constexpr (CH) {
                        r.nb = stream_tiles(klen[p.b], TILE);
                        r.fs = (long long)prefix[p.b] + (long long)si.q * r.nb;
                    } else {
                        r.nb = prefix[p.b + 1] - prefix[p.b];
                        r.fs = (long long)a.seg_per_seq * prefix[p.b] + (long long)si.q * r.nb;
                    }
                    r.row0 = si.row0;
                    r.nvalid = si.nvalid;
                    r.h0 = si.h0;
                    r.seg = si.seg;
                }
                ++n_shared;
            }
            ++k;
        }

        // ---------------------------------------------------------- merge the shared segments
        // this block arrived last at
        const bool sparse = T < a.n_blocks;
        const int w8 = tid >> 5;                          // softmax warp 0 .. NSM/32 - 1
        for (int j = 0; j < n_shared; ++j) {
            bar_sync_named(3, NSM);               // misc[1] and plist are free; records written
            // the blocks holding tiles of this segment: c0 .. c1 (three divisions, one per warp);
            // first_odd: block c0 started before the segment, so it holds it in its second slot
            Shared &rs = shrec[j];
            if (lane == 0 && w8 == 0) rs.c0 = stream_block_of(rs.fs, T, a.n_blocks);
            if (lane == 0 && w8 == 1) rs.c1 = stream_block_of(rs.fs + rs.nb - 1, T, a.n_blocks);
            if (lane == 0 && w8 == 2) rs.first_odd = rs.fs > 0 && stream_block_of(rs.fs - 1, T, a.n_blocks) ==
                                                                    stream_block_of(rs.fs, T, a.n_blocks);
            bar_sync_named(3, NSM);
            const Shared q = rs;
            // with fewer tiles than blocks each block owns at most one tile: one partial per tile
            const int n_pieces = sparse ? q.nb : q.c1 - q.c0 + 1;
            if (tid == 0) {
                const bool last = (j == 0 ? seen0 : seen1) == n_pieces - 1;
                misc[1] = last;
                if (last) a.counters[q.seg] = 0;
            }
            bar_sync_named(3, NSM);
            if (!misc[1]) continue;
            // thread 0's acquire, then the barrier, order the loads below after every
            // other block's release of its partial
            // the partners' slots: consecutive blocks from c0 (their first slot; c0's second
            // when it started before the segment), or, with more blocks than tiles, the owner
            // of each tile, listed once in shared memory
            const bool listed = sparse && n_pieces <= kPlist;
            auto slot_of = [&](int i) {
                if (sparse) return 2 * stream_block_of(q.fs + i, T, a.n_blocks);
                if (i == 0) return 2 * q.c0 + q.first_odd;
                return 2 * (q.c0 + i);
            };
            if (listed) {
                for (int i = tid; i < n_pieces; i += NSM) plist[i] = slot_of(i);
                bar_sync_named(3, NSM);
            }
            auto slot_at = [&](int i) { return listed ? plist[i] : slot_of(i); };
            // Softmax warp w8 combines rows w8, w8 + NW, ..., lane = float4 column block. The
            // partials come PC at a time with their log-sum-exps, all rows' loads in flight
            // together (one L2 round trip per PC partials), folded in with a running maximum.
            constexpr int NW = NSM / 32, RPW = N / NW, PC = NW > 4 ? 2 : 4;
            float M[RPW], W[RPW];
            float4 acc[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                M[r] = -INFINITY;
                W[r] = 0.f;
                acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int i0 = 0; i0 < n_pieces; i0 += PC) {
                float lv[PC][RPW];
                float4 xv[PC][RPW];
#pragma unroll
                for (int u = 0; u < PC; ++u) {
                    const bool in = i0 + u < n_pieces;
                    const size_t base = in ? (size_t)slot_at(i0 + u) * N : 0;
#pragma unroll
                    for (int r = 0; r < RPW; ++r) {
                        const int rr = w8 + NW * r;
                        lv[u][r] = in ? __ldcg(a.lse_part + base + rr) : -INFINITY;
                        if (in) xv[u][r] = __ldcg(reinterpret_cast<const float4 *>(a.o_part + (base + rr) * DV) + lane);
                    }
                }
#pragma unroll
                for (int u = 0; u < PC; ++u)
#pragma unroll
                    for (int r = 0; r < RPW; ++r) {
                        if (lv[u][r] == -INFINITY) continue;
                        const float mn = fmaxf(M[r], lv[u][r]);
                        const float f = fast_exp2((M[r] - mn) * kLog2e);     // 0 while M = -inf
                        const float w = fast_exp2((lv[u][r] - mn) * kLog2e);
                        M[r] = mn;
                        W[r] = W[r] * f + w;
                        acc[r].x = fmaf(w, xv[u][r].x, acc[r].x * f);
                        acc[r].y = fmaf(w, xv[u][r].y, acc[r].y * f);
                        acc[r].z = fmaf(w, xv[u][r].z, acc[r].z * f);
                        acc[r].w = fmaf(w, xv[u][r].w, acc[r].w * f);
                    }
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int n = w8 + NW * r;
                if (CH && n / C::HB >= q.nvalid) continue;
                const float inv = W[r] > 0.f ? 1.f / W[r] : 0.f;
                reinterpret_cast<float4 *>(a.out + out_row(q.row0, q.h0, n))[lane] =
                    make_float4(acc[r].x * inv, acc[r].y * inv, acc[r].z * inv, acc[r].w * inv);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
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

int heads_per_block(int G) { return G % 32 == 0 ? 32 : 16; }

template <int KIND>
size_t smem_for(int N, int B) {
    return N == 32 ? Cfg<KIND, 32>::smem_bytes(B) : Cfg<KIND, 16>::smem_bytes(B);
}

// Segments (sequence, KV head, head block) and the grid over them. Aligned mode: when the
// segments number between half the resident blocks and all of them, each gets a block.
struct Plan {
    long long segs;
    int n_blocks;
    bool aligned;
};

Plan plan(long long segs, int n_split, int cps, bool whole_blocks = true) {
    Plan p{segs, 1, false};
    const int sms = cps * sm_count();          // resident blocks
    if (n_split == 0 && segs <= sms && 2 * segs >= sms) {
        p.aligned = true;
        p.n_blocks = (int)segs;
        return p;
    }
    // MLA (whole_blocks): a whole number k of blocks per segment when that fills at least 85 %
    // of the resident slots: with segments of equal length every block then holds one piece
    // of one segment (no block ends on a second, shared segment), which costs less than the
    // last 15 % of slots gain (16-head MLA, 64 equal segments on B300: 256 blocks 25.4 us,
    // 296 blocks 27.8 us, 259 blocks 28.6 us). The GQA/MQA kernel, one block per SM, keeps
    // every SM streaming instead (MQA, 64 segments: 148 blocks 52.8 us, 128 blocks 54.0 us).
    // Ragged lengths stay balanced either way. A merge over more than kPlist partials lists
    // them on the fly.
    long long n = sms;
    const long long k = segs > 0 ? sms / segs : 0;
    if (whole_blocks && k >= 1 && 100 * k * segs >= 85LL * sms) n = k * segs;
    const long long per_seg = n_split > 0 ? n_split : kMaxPieces;
    if (per_seg * segs < n) n = per_seg * segs;
    p.n_blocks = (int)(n < 1 ? 1 : n);
    return p;
}

// Workspace: one arrival counter per segment at the start (the library's counter region),
// then two partial slots of N rows × DV floats per block, then their log-sum-exps.
size_t ws_bytes(const Plan &p, int N) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    return counter_region_bytes((size_t)p.segs) + up((size_t)2 * p.n_blocks * N * DV * 4) +
           up((size_t)2 * p.n_blocks * N * 4);
}

TcArgs carve(const Plan &pl, int N, void *ws) {
    TcArgs a{};
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    char *w = static_cast<char *>(ws);
    a.counters = reinterpret_cast<int *>(w);
    w += counter_region_bytes((size_t)pl.segs);
    a.o_part = reinterpret_cast<float *>(w);
    a.lse_part = reinterpret_cast<float *>(w + up((size_t)2 * pl.n_blocks * N * DV * 4));
    a.n_blocks = pl.n_blocks;
    a.aligned = pl.aligned ? 1 : 0;
    return a;
}

template <int KIND, int N, bool CH>
cudaError_t launch(const CUtensorMap &km, const CUtensorMap &vm, const CUtensorMap &qm, const CUtensorMap &qrm,
                   const TcArgs &a, cudaStream_t st) {
    const size_t smem = Cfg<KIND, N, CH>::smem_bytes(a.B);
    auto kern = decode_tc_kernel<KIND, N, CH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(a.n_blocks), dim3(Cfg<KIND, N, CH>::THREADS), smem, st, km, vm, qm, qrm, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Tensor maps of a GQA cache pair [B, S_max, Hkv, 128] (boxes of 64 columns × 128 tokens of one
// KV head) and of its queries [rows, Hq, 128] (boxes of 64 columns × qh heads × qt rows).
cudaError_t gqa_maps(const void *q, const void *k, const void *v, int B, int Hkv, int S_max, int rows, int Hq,
                     int qh, int qt, CUtensorMap *km, CUtensorMap *vm, CUtensorMap *qm) {
    const uint64_t dims[4] = {128, (uint64_t)Hkv, (uint64_t)S_max, (uint64_t)B};
    const uint64_t strides[3] = {256, (uint64_t)Hkv * 256, (uint64_t)S_max * Hkv * 256};
    const uint32_t box[4] = {64, 1, TILE, 1};
    cudaError_t e = encode_tensor_map(km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dims, strides, box,
                                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess)
        e = encode_tensor_map(vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess) {
        const uint64_t qdims[3] = {128, (uint64_t)Hq, (uint64_t)rows};
        const uint64_t qstrides[2] = {256, (uint64_t)Hq * 256};
        const uint32_t qbox[3] = {64, (uint32_t)qh, (uint32_t)qt};
        e = encode_tensor_map(qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, qdims, qstrides, qbox,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    return e;
}

// Tensor maps of the MLA latent cache c [B, S_max, 128] (two 64-column boxes a tile), the rope
// keys kr [B, S_max, 48] (three 16-column boxes), and of the queries q_lat [rows, Hq, 128] and
// q_rope [rows, Hq, 48] (boxes of qh heads × qt rows).
cudaError_t mla_maps(const void *q_lat, const void *q_rope, const void *c_cache, const void *kr_cache, int B,
                     int S_max, int rows, int Hq, int qh, int qt, CUtensorMap *cm, CUtensorMap *krm, CUtensorMap *qm,
                     CUtensorMap *qrm) {
    const uint64_t cdims[3] = {128, (uint64_t)S_max, (uint64_t)B};
    const uint64_t cstrides[2] = {256, (uint64_t)S_max * 256};
    const uint32_t cbox[3] = {64, TILE, 1};
    cudaError_t e = encode_tensor_map(cm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c_cache, cdims, cstrides, cbox,
                                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess) {
        const uint64_t dims[3] = {48, (uint64_t)S_max, (uint64_t)B};
        const uint64_t strides[2] = {96, (uint64_t)S_max * 96};
        const uint32_t box[3] = {16, TILE, 1};
        e = encode_tensor_map(krm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kr_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    if (e == cudaSuccess) {
        const uint64_t dims[3] = {128, (uint64_t)Hq, (uint64_t)rows};
        const uint64_t strides[2] = {256, (uint64_t)Hq * 256};
        const uint32_t box[3] = {64, (uint32_t)qh, (uint32_t)qt};
        e = encode_tensor_map(qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_lat, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    if (e == cudaSuccess) {
        const uint64_t dims[3] = {48, (uint64_t)Hq, (uint64_t)rows};
        const uint64_t strides[2] = {96, (uint64_t)Hq * 96};
        const uint32_t box[3] = {16, (uint32_t)qh, (uint32_t)qt};
        e = encode_tensor_map(qrm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_rope, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    return e;
}

// Chunked prefill: the grid is one block per SM over the balanced split (the number of
// segments depends on the device-side chunk lengths); n_split > 0 caps it at n_split blocks
// per segment of the host-side bound. Segments: at most ceil((T + B·(NT−1)) / NT) query blocks
// × seg_per_qb.
constexpr int kChunkN = 16 * kChunkTokens;

long long chunk_segs_bound(int B, int T, int seg_per_qb) {
    return (long long)((T + (long long)B * (kChunkTokens - 1)) / kChunkTokens) * seg_per_qb;
}

Plan chunk_plan(int B, int T, int seg_per_qb, int n_split) {
    Plan p{chunk_segs_bound(B, T, seg_per_qb), sm_count(), false};
    if (n_split > 0 && (long long)n_split * p.segs < p.n_blocks) p.n_blocks = (int)(n_split * p.segs);
    if (p.n_blocks < 1) p.n_blocks = 1;
    return p;
}

}  // namespace

// ------------------------------------------------------------------ GQA (D = 128, G % 16 == 0)

bool decode_tc_gqa_eligible(int B, int Hq, int Hkv, int D) {
    const int G = Hq / Hkv;
    return D == 128 && G % 16 == 0 && smem_for<kGqa>(heads_per_block(G), B) <= 227 * 1024;
}

static Plan gqa_plan_tc(int B, int Hq, int Hkv, int n_split) {
    const int G = Hq / Hkv;
    return plan((long long)B * Hkv * (G / heads_per_block(G)), n_split,
                heads_per_block(G) == 32 ? Cfg<kGqa, 32>::CPS : Cfg<kGqa, 16>::CPS, false);
}

int decode_tc_gqa_blocks(int B, int Hq, int Hkv, int n_split) { return gqa_plan_tc(B, Hq, Hkv, n_split).n_blocks; }

size_t decode_tc_gqa_workspace(int B, int Hq, int Hkv, int n_split) {
    return ws_bytes(gqa_plan_tc(B, Hq, Hkv, n_split), heads_per_block(Hq / Hkv));
}

cudaError_t launch_decode_tc_gqa(const void *q, const void *k, const void *v, const int *seq_lens, float *out, int B,
                                 int Hq, int Hkv, float scale_log2, int S_max, int n_split, void *ws, cudaStream_t st) {
    const int G = Hq / Hkv;
    const int N = heads_per_block(G);
    const Plan pl = gqa_plan_tc(B, Hq, Hkv, n_split);
    TcArgs a = carve(pl, N, ws);
    a.seq_lens = seq_lens;
    a.out = out;
    a.B = B;
    a.Hq = Hq;
    a.G = G;
    a.n_hblk = G / N;
    a.seg_per_seq = Hkv * a.n_hblk;
    a.scale_log2 = scale_log2;
    CUtensorMap km, vm, qm;
    cudaError_t e = gqa_maps(q, k, v, B, Hkv, S_max, B, Hq, N, 1, &km, &vm, &qm);
    if (e == cudaSuccess) e = clear_overflow_counters(a.counters, (size_t)pl.segs, st);
    if (e != cudaSuccess) return e;
    return N == 32 ? launch<kGqa, 32, false>(km, vm, qm, qm, a, st) : launch<kGqa, 16, false>(km, vm, qm, qm, a, st);
}

// Chunked prefill over a GQA cache with 16 or more query heads per KV head (G % 16 == 0).
bool decode_tc_gqa_chunk_eligible(int B, int Hq, int Hkv, int D) {
    return D == 128 && (Hq / Hkv) % 16 == 0 && Cfg<kGqa, kChunkN, true>::smem_bytes(B) <= 227 * 1024;
}

size_t decode_tc_gqa_chunk_workspace(int B, int T, int Hq, int Hkv, int n_split) {
    return ws_bytes(chunk_plan(B, T, Hq / 16, n_split), kChunkN);
}

int decode_tc_gqa_chunk_blocks(int B, int T, int Hq, int Hkv, int n_split) {
    (void)Hkv;
    return chunk_plan(B, T, Hq / 16, n_split).n_blocks;
}

cudaError_t launch_decode_tc_gqa_chunk(const void *q, const void *k, const void *v, const int *cu_q,
                                       const int *start_pos, float *out, int B, int T, int Hq, int Hkv,
                                       float scale_log2, int S_max, int n_split, void *ws, cudaStream_t st) {
    const int G = Hq / Hkv;
    const Plan pl = chunk_plan(B, T, Hq / 16, n_split);
    TcArgs a = carve(pl, kChunkN, ws);
    a.cu_q = cu_q;
    a.start_pos = start_pos;
    a.out = out;
    a.B = B;
    a.Hq = Hq;
    a.G = G;
    a.n_hblk = G / 16;
    a.seg_per_seq = Hkv * a.n_hblk;
    a.scale_log2 = scale_log2;
    CUtensorMap km, vm, qm;
    cudaError_t e = gqa_maps(q, k, v, B, Hkv, S_max, T, Hq, 16, kChunkTokens, &km, &vm, &qm);
    if (e == cudaSuccess) e = clear_overflow_counters(a.counters, (size_t)pl.segs, st);
    if (e != cudaSuccess) return e;
    return launch<kGqa, kChunkN, true>(km, vm, qm, qm, a, st);
}

// ------------------------------------------------------------------ MLA (r = 128, dr = 48, Hq % 16 == 0)

bool decode_tc_mla_fits(int B, int Hq) { return smem_for<kMla>(heads_per_block(Hq), B) <= 227 * 1024; }

static Plan mla_plan_tc(int B, int Hq, int n_split) {
    return plan((long long)B * (Hq / heads_per_block(Hq)), n_split,
                heads_per_block(Hq) == 32 ? Cfg<kMla, 32>::CPS : Cfg<kMla, 16>::CPS);
}

int decode_tc_mla_blocks(int B, int Hq, int n_split) { return mla_plan_tc(B, Hq, n_split).n_blocks; }

size_t decode_tc_mla_workspace(int B, int Hq, int n_split) {
    return ws_bytes(mla_plan_tc(B, Hq, n_split), heads_per_block(Hq));
}

cudaError_t launch_decode_tc_mla(const void *q_lat, const void *q_rope, const void *c_cache, const void *kr_cache,
                                 const int *seq_lens, float *out, int B, int Hq, float scale_log2, int S_max,
                                 int n_split, void *ws, cudaStream_t st) {
    const int N = heads_per_block(Hq);
    const Plan pl = mla_plan_tc(B, Hq, n_split);
    TcArgs a = carve(pl, N, ws);
    a.seq_lens = seq_lens;
    a.out = out;
    a.B = B;
    a.Hq = Hq;
    a.G = Hq;
    a.n_hblk = Hq / N;
    a.seg_per_seq = a.n_hblk;
    a.scale_log2 = scale_log2;
    CUtensorMap cm, krm, qm, qrm;
    cudaError_t e = mla_maps(q_lat, q_rope, c_cache, kr_cache, B, S_max, B, Hq, N, 1, &cm, &krm, &qm, &qrm);
    if (e == cudaSuccess) e = clear_overflow_counters(a.counters, (size_t)pl.segs, st);
    if (e != cudaSuccess) return e;
    return N == 32 ? launch<kMla, 32, false>(cm, krm, qm, qrm, a, st) : launch<kMla, 16, false>(cm, krm, qm, qrm, a, st);
}

// MLA chunked prefill: kChunkTokens new tokens × 16 heads per block.
bool decode_tc_mla_chunk_fits(int B) { return Cfg<kMla, kChunkN, true>::smem_bytes(B) <= 227 * 1024; }

size_t decode_tc_mla_chunk_workspace(int B, int T, int Hq, int n_split) {
    return ws_bytes(chunk_plan(B, T, Hq / 16, n_split), kChunkN);
}

int decode_tc_mla_chunk_blocks(int B, int T, int Hq, int n_split) { return chunk_plan(B, T, Hq / 16, n_split).n_blocks; }

cudaError_t launch_decode_tc_mla_chunk(const void *q_lat, const void *q_rope, const void *c_cache,
                                       const void *kr_cache, const int *cu_q, const int *start_pos, float *out,
                                       int B, int T, int Hq, float scale_log2, int S_max, int n_split, void *ws,
                                       cudaStream_t st) {
    const Plan pl = chunk_plan(B, T, Hq / 16, n_split);
    TcArgs a = carve(pl, kChunkN, ws);
    a.cu_q = cu_q;
    a.start_pos = start_pos;
    a.out = out;
    a.B = B;
    a.Hq = Hq;
    a.G = Hq;
    a.n_hblk = Hq / 16;
    a.seg_per_seq = a.n_hblk;
    a.scale_log2 = scale_log2;
    CUtensorMap cm, krm, qm, qrm;
    cudaError_t e = mla_maps(q_lat, q_rope, c_cache, kr_cache, B, S_max, T, Hq, 16, kChunkTokens, &cm, &krm, &qm, &qrm);
    if (e == cudaSuccess) e = clear_overflow_counters(a.counters, (size_t)pl.segs, st);
    if (e != cudaSuccess) return e;
    return launch<kMla, kChunkN, true>(cm, krm, qm, qrm, a, st);
}

int decode_tc_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_decode_tc_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_decode_tc_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
