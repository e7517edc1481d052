// K1 (tensor-core form): decode for GQA/MHA/MQA over a bf16 cache, split evenly over the GPU.
//
// The method ("模型架构｜MQA & GQA 调研", section "代码", Attention.forward with one new token):
// out[b,h] = softmax(scale · q[b,h]·K[b,:S_b,j]ᵀ) · V[b,:S_b,j] with j = h / G. The page
// expands K/V with repeat_kv, which reads every K/V byte once per query head; here the G
// query heads of KV head j are stacked as the M rows of one MMA tile, so each K/V byte
// leaves HBM once and feeds all G heads.
//
// Work split (streamk.cuh): the cache is walked in tiles of TT tokens × HG KV heads (the
// heads of one token range are read together: in the [B, S_max, Hkv, D] cache their rows
// are neighbours, which HBM serves far faster than the same rows fetched at different
// times), and each persistent block takes an equal share of all tiles, whatever the sequence
// lengths. A block streams its share without pausing at segment boundaries: a segment it
// covers whole is written to `out`, one it shares with a neighbour becomes a partial
// (normalised output and ln Σ e^s) that the stream-K merge kernel combines.
//
// Block = 4 consumer warps + 1 producer warp, one block per SM. The producer streams each
// tile's K and V rows through an NS-stage shared-memory ring with TMA tensor loads (one
// 64-byte swizzled box of 32 columns × TT tokens per head, L2 evict-first hint) and, one
// segment ahead, the segment's query rows into one of two query buffers. Consumer warp w
// owns KV head w / WPH of the group and TS = TT / WPH tokens of each tile (WPH = 4 / HG warps
// per head), in slices of 16:
//   S = Q·Kᵀ      mma.sync m16n8k16 (bf16 → fp32), query heads on M, tokens on N;
//   softmax       per-head running max/sum in the base-2 domain (scores · scale·log2 e),
//                 quad shuffles for the row max, rescale factor 2^(m_old − m_new);
//   O += P·V      P rounded to bf16 in registers (the S accumulator layout is the A-operand
//                 layout), V fragments by ldmatrix.trans.
// Tokens past the sequence end are masked to −inf, and their V rows are zeroed in shared
// memory so stale cache contents never reach the output. At a segment's end a warp that
// owns its head alone (HG = 4) writes its rows directly; otherwise the warps sharing a head
// combine their states in shared memory.
//
// Every mbarrier wait is bounded (MLAKV_WAIT_TIMEOUT_CYCLES); a wait that runs out sets a bit
// in g_decode_gqa_status, after which the warp skips all further work but still meets its
// partners at every barrier, so a broken pipeline cannot hang the GPU.
#include "ptx.cuh"
#include "streamk.cuh"
#include "tensor_map.cuh"

#include <math.h>

namespace mlakv {

__device__ unsigned g_decode_gqa_status;

namespace {

constexpr int kLseCache = 512;     // per warp: cached partial log-sum-exps of a merge

// NC consumer warps (4 or 8) + 1 producer warp.
template <int D, int MT, int HG, int NS, int NC>
struct Cfg {
    static constexpr int kThreads = (NC + 1) * 32;
    static constexpr int TT = HG == 4 ? 32 : 16 * NC;   // tokens per tile
    static constexpr int WPH = NC / HG;             // warps per KV head
    static constexpr int TS = TT / WPH;             // tokens per warp per tile
    static constexpr int SLICES = TS / 16;
    static constexpr int NB = D / 32;               // 64-byte column boxes per token row
    static constexpr int BOX = TT * 64;             // one box: TT rows of 64 bytes (one head)
    static constexpr int KV = NB * HG * BOX;        // K (or V) bytes per stage
    static constexpr int STAGE = 2 * KV;
    static constexpr int HEADS = 16 * MT;           // MMA rows per KV head
    static constexpr int Q_OFF = NS * STAGE;
    static_assert(BOX % 512 == 0 && STAGE % 1024 == 0, "swizzle alignment");
    static_assert(TT % WPH == 0 && TS % 16 == 0, "whole 16-token slices per warp");
    static_assert(SLICES >= 1, "at least one 16-token slice per warp");
};

// Shared-memory layout after the ring: two query buffers of NB boxes of q_rows rows, the
// barriers, the combine scratch (warps sharing a head) and the tile prefix.
struct Layout {
    int q_box, q_buf, bar, scr, fac, stats, plist, prefix, total;
};

template <int D, int MT, int HG, int NS, int NC>
Layout layout(int q_rows, int heads, int B, int n_blocks, bool chunked) {
    using C = Cfg<D, MT, HG, NS, NC>;
    constexpr int kConsumers = NC;
    Layout L;
    L.q_box = q_rows * 64;
    L.q_buf = C::NB * L.q_box;
    L.bar = C::Q_OFF + 2 * L.q_buf;
    L.scr = L.bar + 256;
    const int scr_floats = C::WPH > 1 ? kConsumers * heads * (D + 2) : 0;
    L.fac = L.scr + scr_floats * 4;
    L.stats = L.fac + (C::WPH > 1 ? HG * heads * (C::WPH + 1) * 4 : 0);
    L.plist = L.stats + 2 * HG * heads * 4 + 16;
    L.prefix = L.plist + kConsumers * (n_blocks + kLseCache) * 4;
    // tile prefix [B+1], keys per sequence [B]; chunked prefill also the first new-token rows
    // [B+1] and the segment prefix [B+1]; then the walk's start (b, q, i0)
    L.total = L.prefix + (chunked ? 4 : 2) * (B + 1) * 4 + 16 + 1024;
    return L;
}

// Byte offset of 16-byte chunk `cidx` (along D) of row `row` in a buffer of 64-byte-wide
// boxes whose `row` 0 sits at a 512-byte boundary, written by TMA with the 64-byte swizzle
// (address bits [4,5] ^= bits [7,8]: chunk c of row r sits at c ^ ((r >> 1) & 3)).
__device__ __forceinline__ uint32_t sw64(int row, int cidx) {
    return row * 64 + ((((cidx & 3) ^ ((row >> 1) & 3))) << 4);
}

// CH: chunked prefill. The M rows of a KV head's MMA tile are then NT = a.nt new tokens × G
// query heads (row i·G + g), each token with its own key limit (bottom-right causal); the
// query rows of a KV-head group arrive as one box of NT tokens × HG·G heads.
template <int D, int MT, int HG, int NS, int NC, bool CH>
__global__ void __launch_bounds__((NC + 1) * 32, 1)
decode_gqa_bf16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const __grid_constant__ CUtensorMap qmap, const DecodeStreamArgs a, const Layout L,
                       int q_rows_loaded) {
    using C = Cfg<D, MT, HG, NS, NC>;
    constexpr int TT = C::TT, WPH = C::WPH, TS = C::TS;
    constexpr int kConsumers = NC, kThreads = C::kThreads;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + L.bar;             // NS barriers
    const uint32_t empty0 = full0 + NS * 8;           // NS barriers
    const uint32_t qfull0 = empty0 + NS * 8;          // 2 barriers
    const uint32_t qempty0 = qfull0 + 16;             // 2 barriers
    const int heads = a.heads;
    float *scr = reinterpret_cast<float *>(smem + L.scr);     // [warp][head][D+2]   (WPH > 1)
    float *fac = reinterpret_cast<float *>(smem + L.fac);     // [hg·head][WPH + 1]  (WPH > 1)
    float *stats = reinterpret_cast<float *>(smem + L.stats); // [2][hg·head] merge max, 1/sum
    int *flag = reinterpret_cast<int *>(stats + 2 * HG * a.heads);   // "this block merges"
    int *plist = reinterpret_cast<int *>(smem + L.plist);     // per warp: partial rows of a merge,
                                                              // then kLseCache cached lse values
    int *prefix = reinterpret_cast<int *>(smem + L.prefix);   // [B+1]
    int *lens = prefix + (a.B + 1);                            // [B] keys per sequence
    int *cu = lens + (a.B + 1);                                // chunked: [B+1] first new-token row
    int *segpre = cu + (a.B + 1);                              // chunked: [B+1] segments before b
    int *wstart = prefix + (CH ? 4 : 2) * (a.B + 1);           // decode: the walk's start b, q, i0

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.Hq / a.Hkv;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumers);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull0 + 8 * i, 1);
            mbar_init(qempty0 + 8 * i, kConsumers);
        }
        fence_mbar_init();
    }
    // query rows past those loaded are only ever read as padding rows: keep them zero
    for (int i = threadIdx.x; i < 2 * L.q_buf / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + C::Q_OFF)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    uint64_t pol = 0;                         // producer: L2 evict-first for the streamed rows
    if (warp == kConsumers && lane == 0) {
        // the descriptors are kernel parameters, which no earlier kernel writes
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        prefetch_tensormap(&qmap);
        pol = l2_evict_first_policy();
    }

    // everything above overlaps the previous kernel in the stream; the inputs are read below
    griddep_wait();
    griddep_launch_dependents();
    const int ntok = CH ? a.nt : 1;                // new tokens per segment
    if (CH && warp == 0) {
        // per sequence: n new tokens at rows cu_q[b] .., seeing keys up to start_pos[b] + n;
        // ceil(n / nt) query blocks of Hkv / HG segments each, every one over those keys
        const int per_qb = a.Hkv / HG;
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
            const int nseg = (n + ntok - 1) / ntok * per_qb;
            const int v = nseg * stream_tiles(keys, TT);
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
                lens[b] = keys;
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
        // where this block's tile range starts (streamed split): found once, lane-parallel
        const int spp = (a.Hkv / HG) * a.n_hblk;
        const long long T0 = (long long)spp * carry;
        int b0 = 0, q0 = 0, i00 = 0;
        if (!a.aligned && T0 > 0) {
            const long long t0 = stream_start(blockIdx.x, T0, a.n_blocks);
            if (t0 < stream_start(blockIdx.x + 1, T0, a.n_blocks)) seq_walk_start(prefix, a.B, spp, t0, lane, b0, q0, i00);
        }
        if (lane == 0) {
            wstart[0] = b0;
            wstart[1] = q0;
            wstart[2] = i00;
        }
    }
    __syncthreads();

    const int seg_per_seq = (a.Hkv / HG) * a.n_hblk;      // chunked: per query block
    const long long T = CH ? (long long)prefix[a.B] : (long long)seg_per_seq * prefix[a.B];
    const int c = blockIdx.x;
    if (!CH && c == 0 && warp < kConsumers) {
        // sequences with an empty cache own no tile: their output is zero (a warp per sequence)
        for (int b = warp; b < a.B; b += kConsumers)
            if (prefix[b + 1] == prefix[b])
                for (int i = lane; i < a.Hq * D / 4; i += 32)
                    reinterpret_cast<float4 *>(a.out + (size_t)b * a.Hq * D)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    SeqWalker walk{prefix, lens, a.B, a.Hkv / HG, a.n_hblk, 0, 0, 0, 0, 0, 0};
    if (!CH && a.aligned) {
        // block c streams segment c whole
        const int b = c / seg_per_seq, q = c % seg_per_seq;
        const int nb = stream_tiles(lens[b], TT);
        const long long t = (long long)seg_per_seq * prefix[b] + (long long)q * nb;
        walk.set(b, q, 0, t, t + nb);
    } else if (T > 0) {
        if constexpr (CH) {
            walk.t = stream_start(c, T, a.n_blocks);
            walk.t_end = stream_start(c + 1, T, a.n_blocks);
        } else {
            walk.set(wstart[0], wstart[1], wstart[2], stream_start(c, T, a.n_blocks), stream_start(c + 1, T, a.n_blocks));
        }
    }
    ChunkPieceWalker cwalk{prefix, lens, a.B, TT, walk.t, walk.t_end};
    AlignedChunkWalker awalk{0, 0, a.Hkv / HG, 0, 0, TT, 0};
    if (CH && a.aligned) {
        // block c: sequence c / Hkv, KV head c % Hkv (HG = 1), all of its query blocks
        awalk.b = c / a.Hkv;
        awalk.j = c % a.Hkv;
        if (awalk.b < a.B) {
            const int n = cu[awalk.b + 1] - cu[awalk.b];
            awalk.nqb = (n + ntok - 1) / ntok;
            awalk.S = lens[awalk.b];
        }
    }
    auto next_piece = [&](Piece &p) {
        if constexpr (CH) return a.aligned ? awalk.next(p) : cwalk.next(p);
        else return walk.next(p);
    };
    // A piece's segment: KV-head group gi, head block hb, index q within the sequence (and the
    // arrival counter seg); decode rows are heads of sequence b, chunked-prefill rows are the
    // query block's new tokens at packed rows row0 .., nvalid of them, seeing keys < kbase + i + 1.
    struct SegG {
        int gi, hb, q, seg, row0, nvalid, kbase;
    };
    auto seg_info = [&](const Piece &p) {
        SegG r;
        if constexpr (CH) {
            r.q = p.gi;
            const int qb = r.q / seg_per_seq;
            r.gi = r.q % seg_per_seq;
            r.hb = 0;
            const int n = cu[p.b + 1] - cu[p.b];
            r.row0 = cu[p.b] + qb * ntok;
            r.nvalid = min(ntok, n - qb * ntok);
            r.kbase = lens[p.b] - n + qb * ntok;
            r.seg = segpre[p.b] + r.q;
        } else {
            r.gi = p.gi;
            r.hb = p.hb;
            r.q = p.gi * a.n_hblk + p.hb;
            r.seg = p.b * seg_per_seq + r.q;
            r.row0 = p.b;
            r.nvalid = 1;
            r.kbase = 0;
        }
        return r;
    };
    // Output row of query row h (0 .. heads-1) of KV head jj: decode, head jj·G + hb·HEADS + h of
    // sequence b; chunked prefill, head jj·G + h % G of packed row row0 + h / G
    auto out_row = [&](const SegG &si, int jj, int h) {
        if constexpr (CH) return (size_t)(si.row0 + h / G) * a.Hq + jj * G + h % G;
        else return (size_t)si.row0 * a.Hq + jj * G + si.hb * C::HEADS + h;
    };
    auto row_valid = [&](const SegG &si, int h) { return !CH || h / G < si.nvalid; };

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && (walk.t < walk.t_end || (CH && a.aligned && awalk.nqb > 0))) {
            int g = 0, k = 0;
            bool ok = true;
            Piece p;
            while (ok && next_piece(p)) {
                const int qb = k & 1;
                if (k >= 2 && !mbar_wait_bounded(qempty0 + 8 * qb, ((k >> 1) - 1) & 1, &g_decode_gqa_status,
                                                 kStatusEmptyWait)) {
                    ok = false;
                    break;
                }
                const SegG si = seg_info(p);
                const int j0 = si.gi * HG;
                const int h0 = j0 * G + si.hb * C::HEADS;
                mbar_arrive_expect_tx(qfull0 + 8 * qb, C::NB * q_rows_loaded * 64);
#pragma unroll
                for (int bx = 0; bx < C::NB; ++bx)
                    tma_load_3d(sbase + C::Q_OFF + qb * L.q_buf + bx * L.q_box, &qmap, bx * 32, h0, si.row0,
                                qfull0 + 8 * qb, pol);
                for (int i = 0; i < p.n_t; ++i, ++g) {
                    const int s = g % NS;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ((g / NS) & 1) ^ 1, &g_decode_gqa_status, kStatusEmptyWait)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sbase + s * C::STAGE;
                    mbar_arrive_expect_tx(full0 + 8 * s, C::STAGE);
                    const int t = (p.i0 + i) * TT;
                    // the HG heads of each column box back to back: neighbouring rows in HBM
#pragma unroll
                    for (int bx = 0; bx < C::NB; ++bx)
#pragma unroll
                        for (int hh = 0; hh < HG; ++hh)
                            tma_load_4d(dst + (bx * HG + hh) * C::BOX, &kmap, bx * 32, j0 + hh, t, p.b, full0 + 8 * s, pol);
#pragma unroll
                    for (int bx = 0; bx < C::NB; ++bx)
#pragma unroll
                        for (int hh = 0; hh < HG; ++hh)
                            tma_load_4d(dst + C::KV + (bx * HG + hh) * C::BOX, &vmap, bx * 32, j0 + hh, t, p.b,
                                        full0 + 8 * s, pol);
                }
                ++k;
            }
            // no copy may still be in flight when the block exits
            for (int i = g > NS ? g - NS : 0; i < g; ++i)
                mbar_wait_bounded(full0 + 8 * (i % NS), (i / NS) & 1, &g_decode_gqa_status, kStatusDrainWait);
            for (int i = k > 2 ? k - 2 : 0; i < k; ++i)
                mbar_wait_bounded(qfull0 + 8 * (i & 1), (i >> 1) & 1, &g_decode_gqa_status, kStatusDrainWait);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int hw = warp / WPH;    // KV head of the group this warp serves
    const int sub = warp % WPH;   // its share of each tile's tokens
    const int g8 = lane >> 2;     // row group inside an MMA fragment
    const int cq = lane & 3;      // column pair inside an MMA fragment
    const int mi = lane >> 3;     // ldmatrix: which 8x8 matrix this lane addresses
    const int ri = lane & 7;      // ldmatrix: which row of it
    // the query-buffer row of this lane's ldmatrix row (m = (mi & 1)·8 + ri of each 16-row MMA
    // tile): decode, the head's rows from qrow0; chunked prefill, token m / G of the box's
    // [token][HG·G heads] rows, or a zero padding row past the block's tokens
    const int qrow0 = a.n_hblk == 1 ? hw * G : 0;
    const int qm = (mi & 1) * 8 + ri;
    const int my_qrow = !CH ? qrow0 + qm
                      : qm < ntok * G ? (qm / G) * (HG * G) + hw * G + qm % G : ntok * HG * G;
    bool ok = true;               // false once a wait has given up: the warp then only keeps
                                  // step with its partners at the named barriers
    int g = 0, k = 0;
    Piece p;
    while (next_piece(p)) {
        const SegG si = seg_info(p);
        const int qb = k & 1;
        const uint32_t qbase = sbase + C::Q_OFF + qb * L.q_buf;
        if (ok && !mbar_wait_bounded(qfull0 + 8 * qb, (k >> 1) & 1, &g_decode_gqa_status, kStatusFullWait)) ok = false;
        float o[MT][D / 8][4];
        float m[MT][2], l[MT][2];
        // chunked prefill: the key limit of this thread's two rows (g8 and g8 + 8: tokens
        // (g8) / G and (g8 + 8) / G of the block; 0 for rows past its new tokens). Their running
        // maxima start at −1e30 rather than −∞: a row may see no visible key in a slice or a
        // whole piece, and 2^(−∞ − (−1e30)) = 0 is then its weight, where −∞ − (−∞) is NaN.
        int lim[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int tok = (r * 8 + g8) / G;
            lim[r] = CH && r * 8 + g8 < ntok * G && tok < si.nvalid ? si.kbase + tok + 1 : 0;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                m[mt][r] = CH ? -1e30f : -INFINITY;
                l[mt][r] = 0.f;
            }
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][nd][e] = 0.f;
        }
        const int t_end = min(p.S, (p.i0 + p.n_t) * TT);
        for (int i = 0; i < p.n_t; ++i, ++g) {
            const int s = g % NS;
            if (ok && !mbar_wait_bounded(full0 + 8 * s, (g / NS) & 1, &g_decode_gqa_status, kStatusFullWait))
                ok = false;
            if (ok) {
                const uint32_t kb = sbase + s * C::STAGE + hw * C::BOX;    // this head's K rows
                const uint32_t vb = kb + C::KV;
#pragma unroll
                for (int sl = 0; sl < C::SLICES; ++sl) {
                    const int r0 = sub * TS + sl * 16;                      // first row of the slice
                    const int n_valid = min(16, t_end - ((p.i0 + i) * TT + r0));
                    if (n_valid <= 0) continue;
                    if (n_valid < 16) {
                        // zero the V rows past the sequence end so 0·(stale value) cannot make NaN
                        uint8_t *vrow = smem + s * C::STAGE + C::KV + hw * C::BOX;
                        for (int idx = lane; idx < 16 * C::NB * 4; idx += 32) {
                            const int r = idx / (C::NB * 4), cidx = idx % (C::NB * 4);
                            if (r >= n_valid)
                                *reinterpret_cast<uint4 *>(vrow + (cidx >> 2) * HG * C::BOX + sw64(r0 + r, cidx)) =
                                    make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    // S = Q·Kᵀ for the slice's 16 tokens
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
                        const int cb = 2 * kk + (mi & 1);
                        ldsm_x4(kb + (cb >> 2) * HG * C::BOX + sw64(r0 + (mi >> 1) * 8 + ri, cb), b0, b1, b2, b3);
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            uint32_t a0, a1, a2, a3;
                            const int ca = 2 * kk + (mi >> 1);
                            ldsm_x4(qbase + (ca >> 2) * L.q_box + sw64(my_qrow + mt * 16, ca), a0, a1, a2, a3);
                            mma_bf16_16816(sc[mt][0], a0, a1, a2, a3, b0, b1);
                            mma_bf16_16816(sc[mt][1], a0, a1, a2, a3, b2, b3);
                        }
                    }
                    // online softmax (base 2) and P in bf16 as the A operand of P·V
                    // chunked prefill also keeps each weight's bf16 residual (p − bf16(p)) and
                    // multiplies it with V as well: rows of a chunk near a sequence's start see
                    // only a few keys, where a 2^-9 rounding of each weight does not average away
                    uint32_t pa[MT][4], pres[MT][4];
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
                                    const bool vis = tok < n_valid &&
                                                     (!CH || (p.i0 + i) * TT + r0 + tok < lim[r]);
                                    x[nt * 2 + e] = vis ? sc[mt][nt][2 * r + e] * a.scale_log2 : -INFINITY;
                                }
                            float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                            const float mn = fmaxf(m[mt][r], mx);    // finite: token 0 of the slice is valid
                            const float alpha = fast_exp2(m[mt][r] - mn);
                            m[mt][r] = mn;
                            float pr[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) pr[e] = fast_exp2(x[e] - mn);
                            const uint32_t lo = pack_bf16x2(pr[0], pr[1]);   // tokens 2cq, 2cq+1
                            const uint32_t hi = pack_bf16x2(pr[2], pr[3]);   // tokens 8+2cq, 9+2cq
                            pa[mt][r] = lo;
                            pa[mt][2 + r] = hi;
                            // the row sum uses the rounded weights, so Σ weights = 1 after normalising
                            float ps = bf16_lo(lo) + bf16_hi(lo) + bf16_lo(hi) + bf16_hi(hi);
                            if constexpr (CH) {
                                const uint32_t lo2 = pack_bf16x2(pr[0] - bf16_lo(lo), pr[1] - bf16_hi(lo));
                                const uint32_t hi2 = pack_bf16x2(pr[2] - bf16_lo(hi), pr[3] - bf16_hi(hi));
                                pres[mt][r] = lo2;
                                pres[mt][2 + r] = hi2;
                                ps += bf16_lo(lo2) + bf16_hi(lo2) + bf16_lo(hi2) + bf16_hi(hi2);
                            }
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
                        const int cv = 2 * pq + (mi >> 1);
                        ldsm_x4_t(vb + (cv >> 2) * HG * C::BOX + sw64(r0 + (mi & 1) * 8 + ri, cv), b0, b1, b2, b3);
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            mma_bf16_16816(o[mt][2 * pq], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
                            mma_bf16_16816(o[mt][2 * pq + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b2, b3);
                            if constexpr (CH) {
                                mma_bf16_16816(o[mt][2 * pq], pres[mt][0], pres[mt][1], pres[mt][2], pres[mt][3], b0, b1);
                                mma_bf16_16816(o[mt][2 * pq + 1], pres[mt][0], pres[mt][1], pres[mt][2], pres[mt][3], b2,
                                               b3);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // the query rows of this piece are no longer read
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty0 + 8 * qb);

        const int j = si.gi * HG + hw;                         // this warp's KV head
        // its query rows in this block: heads (decode) or new tokens × heads (chunked prefill)
        const int n_rows = CH ? heads : min(heads, G - si.hb * C::HEADS);
        const int slot = 2 * c + (k == 0 ? 0 : 1);
        const size_t part_row0 = (size_t)slot * HG * heads + hw * heads;
        if constexpr (WPH == 1) {
            // ---------------------------------------------------------- direct write
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float lr = l[mt][r];
                    lr += __shfl_xor_sync(0xffffffffu, lr, 1);
                    lr += __shfl_xor_sync(0xffffffffu, lr, 2);
                    const int h = mt * 16 + r * 8 + g8;
                    if (h >= n_rows || (p.whole && !row_valid(si, h))) continue;
                    const float inv = ok && lr > 0.f ? 1.f / lr : 0.f;
                    float *dst = p.whole ? a.out + out_row(si, j, h) * D : a.o_part + (part_row0 + h) * D;
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd)
                        *reinterpret_cast<float2 *>(dst + nd * 8 + 2 * cq) =
                            make_float2(o[mt][nd][2 * r] * inv, o[mt][nd][2 * r + 1] * inv);
                    if (!p.whole && cq == 0)
                        a.lse_part[part_row0 + h] = ok && lr > 0.f ? (m[mt][r] + log2f(lr)) * kLn2 : -INFINITY;
                }
        } else {
            // ---------------------------------------------------------- combine the WPH warps of each head
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");   // scratch free
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float lr = l[mt][r];
                    lr += __shfl_xor_sync(0xffffffffu, lr, 1);
                    lr += __shfl_xor_sync(0xffffffffu, lr, 2);
                    const int h = mt * 16 + r * 8 + g8;
                    if (h < heads) {
                        float *row = scr + (warp * heads + h) * (D + 2);
#pragma unroll
                        for (int nd = 0; nd < D / 8; ++nd) {
                            row[nd * 8 + 2 * cq] = o[mt][nd][2 * r];
                            row[nd * 8 + 2 * cq + 1] = o[mt][nd][2 * r + 1];
                        }
                        if (cq == 0) {
                            row[D] = ok ? m[mt][r] : -INFINITY;
                            row[D + 1] = lr;
                        }
                    }
                }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
            // per (head of the group, query row): the warps' weights 2^(m_w − M) / L and ln Σ e^s
            for (int idx = threadIdx.x; idx < HG * heads; idx += kConsumers * 32) {
                const int hh = idx / heads, h = idx % heads;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < WPH; ++w) M = fmaxf(M, scr[((hh * WPH + w) * heads + h) * (D + 2) + D]);
                float f[WPH], Lsum = 0.f;
#pragma unroll
                for (int w = 0; w < WPH; ++w) {
                    const float *row = scr + ((hh * WPH + w) * heads + h) * (D + 2);
                    f[w] = M == -INFINITY ? 0.f : fast_exp2(row[D] - M);
                    Lsum = fmaf(row[D + 1], f[w], Lsum);
                }
                const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
                for (int w = 0; w < WPH; ++w) fac[idx * (WPH + 1) + w] = f[w] * inv;
                fac[idx * (WPH + 1) + WPH] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
            for (int idx = threadIdx.x; idx < HG * n_rows * D; idx += kConsumers * 32) {
                const int hh = idx / (n_rows * D), h = (idx / D) % n_rows, d = idx % D;
                const int fi = hh * heads + h;
                float val = 0.f;
#pragma unroll
                for (int w = 0; w < WPH; ++w)
                    val = fmaf(scr[((hh * WPH + w) * heads + h) * (D + 2) + d], fac[fi * (WPH + 1) + w], val);
                const int jj = si.gi * HG + hh;
                if (p.whole) {
                    if (row_valid(si, h)) a.out[out_row(si, jj, h) * D + d] = val;
                } else {
                    const size_t pr = (size_t)slot * HG * heads + hh * heads + h;
                    a.o_part[pr * D + d] = val;
                    if (d == 0) a.lse_part[pr] = fac[fi * (WPH + 1) + WPH];
                }
            }
        }
        // ---------------------------------------------------------- finish a shared segment
        // Publish this block's partial; the last of the segment's blocks to arrive combines all
        // of them and resets the arrival counter for the next call. A block's first piece is
        // finished while its stream goes on with the next one. With one warp per KV head
        // (WPH = 1) each warp does this for its own head alone, with no block-wide barrier;
        // otherwise the consumer warps do it together.
        if (!p.whole) {
            const Piece &q = p;
            const int nb = stream_tiles(q.S, TT);
            // the segment's first tile in the stream
            const long long fs = (CH ? (long long)prefix[q.b] : (long long)seg_per_seq * prefix[q.b]) +
                                 (long long)si.q * nb;
            // the partial slots of all blocks holding tiles of this segment: blocks c0 .. c1, or,
            // with fewer tiles than blocks (each block then owns at most one tile), the owners of
            // the segment's nb tiles
            const bool sparse = T < a.n_blocks;
            const int c0 = stream_block_of(fs, T, a.n_blocks);
            const int n_pieces = sparse ? nb : stream_block_of(fs + nb - 1, T, a.n_blocks) - c0 + 1;
            auto slot_of = [&](int i) {
                if (sparse) return 2 * stream_block_of(fs + i, T, a.n_blocks);
                if (i == 0) return stream_start(c0, T, a.n_blocks) < fs ? 2 * c0 + 1 : 2 * c0;
                return 2 * (c0 + i);
            };
            const int seg = si.seg;
            // rows of heads hh0 .. hh0+n_hh-1 of the group, merged by n_thr threads from t0:
            // partial row bases cached in wl, their lse values in wc
            auto merge_rows = [&](int hh0, int n_hh, int t0, int n_thr, int *wl, float *wc) {
                for (int i = t0; i < n_pieces; i += n_thr) wl[i] = slot_of(i) * HG * heads;
                if (WPH == 1) __syncwarp(); else asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
                const int rows = n_hh * n_rows;
                const bool cached = rows * n_pieces <= kLseCache;
                if (cached)
                    for (int e = t0; e < rows * n_pieces; e += n_thr) {
                        const int r = e / n_pieces, i = e % n_pieces;
                        wc[e] = __ldcg(a.lse_part + wl[i] + (hh0 + r / n_rows) * heads + r % n_rows);
                    }
                if (WPH == 1) __syncwarp(); else asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
                for (int idx = t0; idx < rows * (D / 4); idx += n_thr) {
                    const int r = idx / (D / 4), col = idx % (D / 4);
                    const int off = (hh0 + r / n_rows) * heads + r % n_rows;
                    auto lse_at = [&](int i) { return cached ? wc[r * n_pieces + i] : __ldcg(a.lse_part + wl[i] + off); };
                    float M = -INFINITY;
                    for (int i = 0; i < n_pieces; ++i) M = fmaxf(M, lse_at(i));
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    float W = 0.f;
                    // eight partial rows in flight at a time
                    for (int i0 = 0; i0 < n_pieces; i0 += 8) {
                        float4 x[8];
    #pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (i0 + u < n_pieces)
                                x[u] = __ldcg(reinterpret_cast<const float4 *>(a.o_part + ((size_t)wl[i0 + u] + off) * D) + col);
    #pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (i0 + u < n_pieces) {
                                const float w = M == -INFINITY ? 0.f : fast_exp2((lse_at(i0 + u) - M) * kLog2e);
                                W += w;
                                acc.x = fmaf(w, x[u].x, acc.x);
                                acc.y = fmaf(w, x[u].y, acc.y);
                                acc.z = fmaf(w, x[u].z, acc.z);
                                acc.w = fmaf(w, x[u].w, acc.w);
                            }
                    }
                    const float inv = W > 0.f ? 1.f / W : 0.f;
                    const int jj = si.gi * HG + hh0 + r / n_rows;
                    if (row_valid(si, r % n_rows)) {
                        float4 *dst = reinterpret_cast<float4 *>(a.out + out_row(si, jj, r % n_rows) * D);
                        dst[col] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                    }
                }
            };
            if constexpr (WPH == 1) {
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    int *cnt = a.counters + (size_t)seg * HG + hw;
                    const int prev = atomic_add_acq_rel_gpu(cnt, 1);
                    last = prev == n_pieces - 1;
                    if (last) *cnt = 0;
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    int *wl = plist + warp * (a.n_blocks + kLseCache);
                    merge_rows(hw, 1, lane, 32, wl, reinterpret_cast<float *>(wl + a.n_blocks));
                }
            } else {
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
                if (threadIdx.x == 0) {
                    int *cnt = a.counters + (size_t)seg * HG;
                    const int prev = atomic_add_acq_rel_gpu(cnt, 1);
                    *flag = prev == n_pieces - 1;
                    if (prev == n_pieces - 1) *cnt = 0;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
                if (*flag) {
                    __threadfence();
                    merge_rows(0, HG, threadIdx.x, kConsumers * 32, plist, reinterpret_cast<float *>(plist + a.n_blocks));
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");   // flag, lists reused
            }
        }
        ++k;
    }

}

// Ring depth per configuration: about 192 KB of K/V in flight per SM, less where the
// combine scratch of warps sharing a head needs room, or (chunked prefill) the query buffers
// hold several new tokens of every head of the group.
template <int D, int MT, int HG, int NC, bool CH>
constexpr int ring_depth() {
    constexpr int stage = 2 * (D / 32) * HG * (HG == 4 ? 32 : 16 * NC) * 64;
    constexpr int budget = (HG == 4 ? 192 * 1024 : MT == 2 ? 128 * 1024 : 176 * 1024) - (CH ? 40 * 1024 : 0);
    constexpr int n = budget / stage;
    return n < 2 ? 2 : n;
}

int mt_for(int G) { return G <= 16 ? 1 : 2; }

// KV heads per tile: 4 when they divide Hkv and a head's query rows fit one MMA tile,
// else 2, else 1.
int hg_for(int Hkv, int G) {
    if (G > 16) return 1;
    if (Hkv % 4 == 0) return 4;
    if (Hkv % 2 == 0) return 2;
    return 1;
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

// query rows: the group's HG·G rows (one head block when n_hblk > 1), plus the padding
// the last head's 16·MT-row MMA tile reaches past them; chunked prefill, nt tokens × HG·G
// heads, plus one zero row that stands for the rows past the block's tokens
template <int HG, int MT, bool CH>
void query_rows(const DecodeStreamArgs &a, int &q_loaded, int &q_rows) {
    const int G = a.Hq / a.Hkv;
    q_loaded = CH ? a.nt * HG * G : a.n_hblk == 1 ? HG * G : a.heads;
    q_rows = CH ? (q_loaded + 1 + 7) / 8 * 8 : ((a.n_hblk == 1 ? (HG - 1) * G : 0) + 16 * MT + 7) / 8 * 8;
}

template <int D, int MT, int HG, int NS, int NC, bool CH>
int layout_total(const DecodeStreamArgs &a) {
    int q_loaded, q_rows;
    query_rows<HG, MT, CH>(a, q_loaded, q_rows);
    return layout<D, MT, HG, NS, NC>(q_rows, a.heads, a.B, a.n_blocks, CH).total;
}

template <int D, int MT, int HG, int NS, int NC, bool CH>
cudaError_t launch_ns(const DecodeStreamArgs &a, cudaStream_t st) {
    using C = Cfg<D, MT, HG, NS, NC>;
    const int G = a.Hq / a.Hkv;
    int q_loaded, q_rows;
    query_rows<HG, MT, CH>(a, q_loaded, q_rows);
    const Layout L = layout<D, MT, HG, NS, NC>(q_rows, a.heads, a.B, a.n_blocks, CH);
    if (L.total > 227 * 1024) return cudaErrorInvalidValue;
    CUtensorMap km, vm, qm;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)a.Hkv, (uint64_t)a.S_max, (uint64_t)a.B};
    const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)a.Hkv * D * 2, (uint64_t)a.S_max * a.Hkv * D * 2};
    const uint32_t box[4] = {32, 1, (uint32_t)C::TT, 1};
    cudaError_t e = encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k, dims, strides, box,
                                      CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess)
        e = encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.v, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (e == cudaSuccess) {
        // decode: [B, Hq, D], a box of q_loaded heads of one sequence; chunked prefill:
        // [T, Hq, D], a box of HG·G heads × nt packed rows
        const uint64_t qdims[3] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)(CH ? a.T : a.B)};
        const uint64_t qstrides[2] = {(uint64_t)D * 2, (uint64_t)a.Hq * D * 2};
        const uint32_t qbox[3] = {32, (uint32_t)(CH ? HG * G : q_loaded), (uint32_t)(CH ? a.nt : 1)};
        e = encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, qdims, qstrides, qbox,
                              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    if (e != cudaSuccess) return e;
    auto kern = decode_gqa_bf16_kernel<D, MT, HG, NS, NC, CH>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(a.n_blocks), dim3(C::kThreads), L.total, st, km, vm, qm, a, L, q_loaded);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The ring as deep as ring_depth gives, or two stages where the per-sequence tables of a large
// batch (8 bytes a sequence, beside the ring) would not fit in shared memory beside it.
template <int D, int MT, int HG, int NC, bool CH>
cudaError_t launch_cfg(const DecodeStreamArgs &a, cudaStream_t st) {
    constexpr int NS = ring_depth<D, MT, HG, NC, CH>();
    if (NS == 2 || layout_total<D, MT, HG, NS, NC, CH>(a) <= 227 * 1024) return launch_ns<D, MT, HG, NS, NC, CH>(a, st);
    return launch_ns<D, MT, HG, 2, NC, CH>(a, st);
}

// One KV head per tile with a single MMA row tile per head: 7 consumer warps over 112-token
// tiles, for nearly twice the latency hiding per SM (8 warps in all keep 255 registers per
// thread available; the combine scratch of 32-row heads would not fit beside them).
template <int D, int MT, bool CH>
cudaError_t launch_mt(const DecodeStreamArgs &a, cudaStream_t st) {
    switch (a.hg) {
        case 4: return launch_cfg<D, MT, 4, 4, CH>(a, st);
        case 2: return launch_cfg<D, MT, 2, 4, CH>(a, st);
        default: return MT == 1 ? launch_cfg<D, MT, 1, 7, CH>(a, st) : launch_cfg<D, MT, 1, 4, CH>(a, st);
    }
}

template <int D>
cudaError_t launch_d(const DecodeStreamArgs &a, cudaStream_t st) {
    return mt_for(a.Hq / a.Hkv) == 1 ? launch_mt<D, 1, false>(a, st) : launch_mt<D, 2, false>(a, st);
}

// Chunked prefill: one 16-row MMA tile per KV head (MT = 1) holds 16 / G new tokens.
template <int D>
cudaError_t launch_d_chunk(const DecodeStreamArgs &a, cudaStream_t st) {
    return launch_mt<D, 1, true>(a, st);
}

}  // namespace

// Aligned mode: when the (sequence, KV head, head block) segments number between half the
// SMs and all of them, each gets a block of its own and nothing is shared or merged (the
// merge of a segment split between blocks can only start after its last piece, which
// lengthens the tail of a short call more than the uneven segment lengths do).
bool decode_gqa_stream_aligned(int B, int Hq, int Hkv, int n_split) {
    const int G = Hq / Hkv;
    const int MT = mt_for(G);
    const long long segs = (long long)B * Hkv * ((G + 16 * MT - 1) / (16 * MT));
    const int sms = sm_count();
    return n_split == 0 && segs <= sms && 2 * segs >= sms;
}

int decode_gqa_stream_blocks(int B, int Hq, int Hkv, int D, int n_split) {
    (void)D;
    const int G = Hq / Hkv;
    const int MT = mt_for(G);
    const int n_hblk = (G + 16 * MT - 1) / (16 * MT);
    if (decode_gqa_stream_aligned(B, Hq, Hkv, n_split)) return B * Hkv * n_hblk;
    long long n = sm_count();
    const long long segs = (long long)B * (Hkv / hg_for(Hkv, G)) * n_hblk;
    const long long cap = (long long)(n_split > 0 ? n_split : kMaxPieces) * segs;
    if (cap < n) n = cap;
    return (int)(n < 1 ? 1 : n);
}

// Partial rows: two slots per block, hg·heads query rows per slot.
static size_t stream_part_rows(int B, int Hq, int Hkv, int D, int n_split) {
    const int G = Hq / Hkv;
    const int heads = G < 16 * mt_for(G) ? G : 16 * mt_for(G);
    return 2 * (size_t)decode_gqa_stream_blocks(B, Hq, Hkv, D, n_split) * hg_for(Hkv, G) * heads;
}

size_t decode_gqa_stream_o_bytes(int B, int Hq, int Hkv, int D, int n_split) {
    return (stream_part_rows(B, Hq, Hkv, D, n_split) * D * sizeof(float) + 255) / 256 * 256;
}

size_t decode_gqa_stream_lse_bytes(int B, int Hq, int Hkv, int D, int n_split) {
    return (stream_part_rows(B, Hq, Hkv, D, n_split) * sizeof(float) + 255) / 256 * 256;
}

// One arrival counter per (sequence, KV head, head block), at the workspace's start.
size_t decode_gqa_stream_counters(int B, int Hq, int Hkv) {
    const int G = Hq / Hkv;
    const int MT = mt_for(G);
    return (size_t)B * Hkv * ((G + 16 * MT - 1) / (16 * MT));
}

size_t decode_gqa_stream_workspace(int B, int Hq, int Hkv, int D, int n_split) {
    return counter_region_bytes(decode_gqa_stream_counters(B, Hq, Hkv)) +
           decode_gqa_stream_o_bytes(B, Hq, Hkv, D, n_split) + decode_gqa_stream_lse_bytes(B, Hq, Hkv, D, n_split);
}

cudaError_t launch_decode_gqa_stream(const DecodeStreamArgs &a0, cudaStream_t st) {
    DecodeStreamArgs a = a0;
    const int G = a.Hq / a.Hkv;
    const int MT = mt_for(G);
    a.heads = G < 16 * MT ? G : 16 * MT;
    a.n_hblk = (G + 16 * MT - 1) / (16 * MT);
    a.hg = a.aligned ? 1 : hg_for(a.Hkv, G);
    a.tile_tokens = a.hg == 4 ? 32 : (a.hg == 1 && MT == 1) ? 112 : 64;
    cudaError_t e;
    switch (a.D) {
        case 64: e = launch_d<64>(a, st); break;
        case 96: e = launch_d<96>(a, st); break;
        case 128: e = launch_d<128>(a, st); break;
        default: return cudaErrorInvalidValue;
    }
    return e;
}

// ------------------------------------------------------------------ chunked prefill
// Query groups of up to 16 heads: 16 / G new tokens × G heads fill one 16-row MMA tile per KV
// head, and every cached row a block reads feeds all of them. The grid is one block per SM
// over the balanced split (the segments depend on the device-side chunk lengths); at most
// ceil((T + B·(nt − 1)) / nt) query blocks of Hkv / HG segments each.
static int chunk_tokens(int G) { return 16 / G; }

bool decode_gqa_stream_chunk_eligible(int Hq, int Hkv) { return Hq / Hkv <= 16; }

static long long stream_chunk_segs(int B, int T, int Hq, int Hkv) {
    const int G = Hq / Hkv, nt = chunk_tokens(G);
    return (T + (long long)B * (nt - 1)) / nt * (Hkv / hg_for(Hkv, G));
}

// Aligned chunk plan: when the (sequence, KV head) pairs number between half the SMs and all
// of them, each gets a block that walks its query blocks itself (one pass over the cache for a
// chunk of up to 16 / G tokens) and nothing is shared or merged, as for the decode.
static bool stream_chunk_aligned(int B, int Hkv, int n_split) {
    const long long pairs = (long long)B * Hkv;
    const int sms = sm_count();
    return n_split == 0 && pairs <= sms && 2 * pairs >= sms;
}

int decode_gqa_stream_chunk_blocks(int B, int T, int Hq, int Hkv, int n_split) {
    if (stream_chunk_aligned(B, Hkv, n_split)) return B * Hkv;
    long long n = sm_count();
    if (n_split > 0) {
        const long long cap = (long long)n_split * stream_chunk_segs(B, T, Hq, Hkv);
        if (cap < n) n = cap;
    }
    return (int)(n < 1 ? 1 : n);
}

// Workspace: one arrival counter per (segment, KV head of its group) in the counter region,
// then two partial slots of HG·(nt·G) rows per block and their log-sum-exps.
size_t decode_gqa_stream_chunk_workspace(int B, int T, int Hq, int Hkv, int D, int n_split) {
    const int G = Hq / Hkv, hg = hg_for(Hkv, G);        // (the aligned plan needs no more)
    const size_t rows = 2 * (size_t)decode_gqa_stream_chunk_blocks(B, T, Hq, Hkv, n_split) * hg * chunk_tokens(G) * G;
    const size_t n_cnt = (size_t)stream_chunk_segs(B, T, Hq, Hkv) * hg;
    return counter_region_bytes(n_cnt) + (rows * D * sizeof(float) + 255) / 256 * 256 +
           (rows * sizeof(float) + 255) / 256 * 256;
}

// The chunk mode's plan (everything but the pointers), shared by the launch and the fit check.
static DecodeStreamArgs chunk_plan_args(int B, int T, int Hq, int Hkv, int D, int n_split) {
    DecodeStreamArgs a{};
    const int G = Hq / Hkv;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.T = T;
    a.nt = chunk_tokens(G);
    a.heads = a.nt * G;
    a.n_hblk = 1;
    a.aligned = stream_chunk_aligned(B, Hkv, n_split) ? 1 : 0;
    a.hg = a.aligned ? 1 : hg_for(Hkv, G);
    a.tile_tokens = a.hg == 4 ? 32 : a.hg == 1 ? 112 : 64;
    a.n_blocks = decode_gqa_stream_chunk_blocks(B, T, Hq, Hkv, n_split);
    return a;
}

// Does the chunk mode's shared memory (its per-sequence tables beside a ring of at least two
// stages) fit for this batch? The launch takes the configuration launch_mt<D, 1, true> picks.
template <int D>
static bool chunk_fits_d(const DecodeStreamArgs &a) {
    constexpr int kMax = 227 * 1024;
    switch (a.hg) {
        case 4: return layout_total<D, 1, 4, 2, 4, true>(a) <= kMax;
        case 2: return layout_total<D, 1, 2, 2, 4, true>(a) <= kMax;
        default: return layout_total<D, 1, 1, 2, 7, true>(a) <= kMax;
    }
}

bool decode_gqa_stream_chunk_fits(int B, int T, int Hq, int Hkv, int D, int n_split) {
    const DecodeStreamArgs a = chunk_plan_args(B, T, Hq, Hkv, D, n_split);
    return D == 64 ? chunk_fits_d<64>(a) : D == 96 ? chunk_fits_d<96>(a) : D == 128 ? chunk_fits_d<128>(a) : false;
}

cudaError_t launch_decode_gqa_stream_chunk(const void *q, const void *k, const void *v, const int *cu_q,
                                           const int *start_pos, float *out, int B, int T, int Hq, int Hkv, int D,
                                           float scale_log2, int S_max, int n_split, void *ws, cudaStream_t st) {
    DecodeStreamArgs a = chunk_plan_args(B, T, Hq, Hkv, D, n_split);
    a.q = q; a.k = k; a.v = v; a.out = out; a.cu_q = cu_q; a.start_pos = start_pos;
    a.scale_log2 = scale_log2;
    a.S_max = S_max;
    const size_t rows = 2 * (size_t)a.n_blocks * a.hg * a.heads;
    const size_t n_cnt = (size_t)stream_chunk_segs(B, T, Hq, Hkv) * a.hg;
    char *w = static_cast<char *>(ws);
    a.counters = reinterpret_cast<int *>(w);
    a.o_part = reinterpret_cast<float *>(w + counter_region_bytes(n_cnt));
    a.lse_part = reinterpret_cast<float *>(w + counter_region_bytes(n_cnt) + (rows * D * sizeof(float) + 255) / 256 * 256);
    cudaError_t e = clear_overflow_counters(a.counters, n_cnt, st);
    if (e != cudaSuccess) return e;
    switch (D) {
        case 64: return launch_d_chunk<64>(a, st);
        case 96: return launch_d_chunk<96>(a, st);
        case 128: return launch_d_chunk<128>(a, st);
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
