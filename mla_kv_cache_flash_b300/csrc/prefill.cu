// K4: causal GQA prefill on the 5th-generation tensor cores (tcgen05 MMA, tensor memory, TMA).
//
// The method ("模型架构｜MQA & GQA 调研", section "代码", Attention.forward over a whole prompt;
// the qqstock MLA code's scaled_dot_product_attention with is_causal=True): row i of a
// sequence attends keys 0 .. i of the same sequence through KV head h / G,
//   out[i, h] = Σ_{t ≤ i} softmax_t(scale · q[i,h]·k[t,j]) · v[t,j].
// It is the one dense contraction of the path, so both products run on tcgen05.
//
// Work item = (sequence b, 128-row query tile qt, two query heads of one KV group; one head
// when the group size is odd). The two heads share the KV head, so every K/V tile that lands
// in shared memory feeds two 128×128 score tiles. The kernel is persistent: one block per
// SM walks a fixed list of items, longest (most KV tiles) first, dealt to the blocks in
// alternating order so their totals stay even. One item's output stores and the next item's
// Q load overlap the MMAs. Warp roles:
//   warp 0     TMA producer: each item's two Q tiles, then its K and V tiles (128 keys × 128
//              columns, 128-byte swizzle) through a 2-stage ring that runs across items.
//   warp 1     allocates 512 TMEM columns once; the warp runs the MMA loop and lane 0
//              issues every MMA:
//                S_t = Q_t · K_nᵀ   (M=128, N=128, K=16 × 8; A, B K-major in shared memory)
//                O_t += P_t · V_n   (A = P from TMEM, B = V MN-major in shared memory)
//              and commits each group to an mbarrier.
//   warps 2-9  softmax, one warpgroup per query tile; thread = one query row (one TMEM
//              lane). It reads its 128 scores from TMEM in 32-column quarters (the next
//              quarter's load in flight while one is processed), masks the diagonal tile,
//              keeps a running max m and sum l in the base-2 domain and writes
//              P = 2^(s·scale·log2 e − m) as bf16 over its scores. The output is rescaled
//              only when the row max grows by more than 2^8 (the result is exact for any
//              reference value; this only bounds the range of P and l). At the end of an
//              item it reads its O row from TMEM and writes O / l (fp32): a full tile through
//              a shared staging buffer and TMA stores, a sequence's partial last tile from
//              registers.
// The softmax uses Blackwell's paired fp32 FMA/add (two lanes of work per instruction) and
// the three-input max, which halve its instruction count.
//
// TMEM: per query tile t, columns [256t, 256t+128) hold S and [256t+128, 256t+256) hold O.
// P (two bf16 per column) overwrites S in place: keys 32q .. 32q+31 use the first 16 of
// columns [32q, 32q+32), and the residual of the first kSplitTiles tiles the other 16. The
// next S of a tile is issued after that tile's P·V, and one thread's MMAs run in issue order,
// so P is read before it is overwritten.
//
// Precision: P is rounded to bf16 for the tensor cores, a relative error of up to 2^-8 per
// weight. Rows with many keys average it away, but rows near the start of a sequence see
// few keys (row 1 sees 2); in the first kSplitTiles query tiles P is therefore split into a
// bf16 head and a bf16 residual and both are multiplied with V, which leaves an error near
// 2^-16 there.
//
// Cache form (chunked prefill over an existing cache: "模型架构｜MQA & GQA 调研", section
// "代码", the new tokens written at start_pos before attending): K and V come from the caches
// [B, S_max, Hkv, D] through 4D tensor maps, and row i of sequence b's chunk sees cache rows
// 0 .. start_pos[b] + i. An
// item then covers KV tiles 0 .. (start_pos + last row) / 128, and the mask starts at the tile
// holding key start_pos + first row: with an unaligned start_pos two tiles are masked, each
// row by its own limit. V rows past the chunk's end (the cache may hold anything there, NaN
// included) are zeroed in shared memory by the MMA warp before P·V reads them; their weights
// are 0, but 0 · NaN is not. The item list spans the longest chunk, found by every warp at
// block start from cu_seqlens.
//
// MLA form (the qqstock DeepSeek MLA article, sections 2 and 6: with W_UK absorbed, MLA is
// MQA whose key is the latent row c with its decoupled RoPE part kr, and whose value is c):
// the cache form over c [B, S_max, 128] and kr [B, S_max, 48]. Each latent tile in shared
// memory is both the K operand of the score (with the rope part: three more K = 16 steps over
// 32-byte swizzled boxes of q_rope and kr) and the V operand of P·V; c and kr arrive on one
// barrier, and a stage is free once both P·V MMAs reading it are done.
//
// Every wait is bounded (MLAKV_WAIT_TIMEOUT_CYCLES): a wait that runs out sets a bit in
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
constexpr int BM = 128;                      // query rows per tile (TMEM lanes)
constexpr int BN = 128;                      // keys per KV tile
constexpr int NSTAGE = 2;                    // K/V ring depth
constexpr int TILE_BYTES = BM * HD * 2;      // one 128 × 128 bf16 tile: 32 KB
constexpr int BOX_BYTES = TILE_BYTES / 2;    // one TMA box: 128 rows × 64 columns (128 B)
constexpr int Q_SLOTS = 2;                   // Q tiles rotate through two slots
constexpr int OST_BYTES = BM * 32 * 4;       // output staging: 128 rows × 32 fp32 columns, per query tile
constexpr int RT_BYTES = 3 * BM * 32;        // MLA rope part of a tile: three 16-column boxes (32-byte swizzle)
constexpr int RBOX_BYTES = BM * 32;
constexpr int N_BARS = 24;

// The kernel's three forms: packed K/V (causal prefill), K/V caches (chunked prefill), and
// the MLA latent caches (chunked MLA prefill, W_UK absorbed).
enum Form : int { kPacked = 0, kCache = 1, kMla = 2 };

// Shared memory: Q slots, (MLA) q_rope slots, the K stages (MLA: the latent rows c, which
// are also V), the V stages (MLA: the rope keys kr), two output staging buffers, barriers.
template <int FORM>
struct Lay {
    static constexpr bool MLA = FORM == kMla;
    static constexpr int Q_OFF = 0;
    static constexpr int QR_OFF = Q_OFF + Q_SLOTS * TILE_BYTES;
    static constexpr int K_OFF = QR_OFF + (MLA ? Q_SLOTS * RT_BYTES : 0);
    static constexpr int V_OFF = K_OFF + NSTAGE * TILE_BYTES;
    static constexpr int OST_OFF = V_OFF + NSTAGE * (MLA ? RT_BYTES : TILE_BYTES);
    static constexpr int BAR_OFF = OST_OFF + 2 * OST_BYTES;
    static constexpr int SLOT_OFF = BAR_OFF + N_BARS * 8;
    static constexpr int SMEM = SLOT_OFF + 16 + 1024;   // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(K_OFF % 1024 == 0 && OST_OFF % 1024 == 0 && QR_OFF % 256 == 0 && V_OFF % 256 == 0,
                  "128-byte swizzled tiles on 1024 bytes, 32-byte swizzled boxes on 256");
};

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
    kQFull = 0,          // + Q slot
    kQEmpty = 3,         // + Q slot: the last S MMA reading the slot is done
    kKFull = 6,          // + stage
    kVFull = 8,          // + stage
    kKEmpty = 10,        // + stage: both S MMAs reading the K tile are done
    kVEmpty = 12,        // + stage: both P·V MMAs reading the V tile are done
    kSFull = 14,         // + query tile
    kPReady = 16,        // + query tile
    kODone = 18          // + query tile
};

// ------------------------------------------------------------------ paired fp32 arithmetic
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// The largest (NEG: smallest) visible raw score of one row of the S tile in TMEM, so that the
// row max of x = s·c is c times it (c = scale·log2 e; NEG when c < 0). DIAG: a masked tile,
// where key i is visible only if i <= row (key 0 of an item's first tile always is, so the
// result there is finite). The row is read in 32-column quarters, the next quarter's load in
// flight while the current one is reduced; eight independent partial extrema keep the
// dependency chains short.
template <bool DIAG, bool NEG>
__device__ __forceinline__ float row_extreme(uint32_t s_addr, int row) {
    constexpr float kNone = NEG ? INFINITY : -INFINITY;
    float e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = kNone;
    uint32_t ra[32], rb[32];
    tmem_ld32(s_addr, ra);
    tmem_ld_wait(ra);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t(&cur)[32] = (q & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (q & 1) ? ra : rb;
        if (q < 3) tmem_ld32(s_addr + 32 * (q + 1), nxt);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            float v0 = __uint_as_float(cur[i]), v1 = __uint_as_float(cur[i + 1]);
            if (DIAG) {
                v0 = 32 * q + i <= row ? v0 : kNone;
                v1 = 32 * q + i + 1 <= row ? v1 : kNone;
            }
            const int k = (i >> 1) & 7;
            e[k] = NEG ? fmin3(e[k], v0, v1) : fmax3(e[k], v0, v1);
        }
        if (q < 3) tmem_ld_wait(nxt);
    }
    return NEG ? fminf(fmin3(e[0], e[1], e[2]), fmin3(fmin3(e[3], e[4], e[5]), e[6], e[7]))
               : fmaxf(fmax3(e[0], e[1], e[2]), fmax3(fmax3(e[3], e[4], e[5]), e[6], e[7]));
}

// P = 2^(s·c − m) for the same row (0 for hidden keys), as bf16 pairs. Keys 32q .. 32q+31
// (quarter q) own TMEM columns [32q, 32q+32) of the row's S region: P goes to the first 16 of
// them and, with SPLIT, the bf16 residual p − bf16(p) to the last 16. A quarter's columns are
// written only after that quarter of S has been read, while the next quarter's load is in
// flight (it reads other columns). Adds the unrounded weights to l.
template <bool DIAG, bool SPLIT>
__device__ __forceinline__ void write_p(uint32_t s_addr, float c, float m, int row, float &l) {
    const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-m, -m);
    uint64_t acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = 0;
    uint32_t ra[32], rb[32];
    tmem_ld32(s_addr, ra);
    tmem_ld_wait(ra);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t(&cur)[32] = (q & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (q & 1) ? ra : rb;
        if (q < 3) tmem_ld32(s_addr + 32 * (q + 1), nxt);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k0 = 32 * q + 2 * i;           // key index within the tile
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), c2, nm2), x0, x1);
            float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            if (DIAG) {
                p0 = k0 <= row ? p0 : 0.f;
                p1 = k0 + 1 <= row ? p1 : 0.f;
            }
            acc[i & 3] = fadd2(acc[i & 3], f2pack(p0, p1));
            hi[i] = pack_bf16x2(p0, p1);
            if constexpr (SPLIT) lo[i] = pack_bf16x2(p0 - bf16_lo(hi[i]), p1 - bf16_hi(hi[i]));
        }
        tmem_st16(s_addr + 32 * q, hi);
        if constexpr (SPLIT) tmem_st16(s_addr + 32 * q + 16, lo);
        if (q < 3) tmem_ld_wait(nxt);
    }
    float a0, a1;
    f2unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), a0, a1);
    l += a0 + a1;
}

// Shared → global tensor store of one box (completion tracked by the bulk async-group).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's bulk stores have read their shared-memory source (it may be rewritten).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 32-byte store of eight floats (the address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float *p, float a0, float a1, float a2, float a3, float a4, float a5,
                                             float a6, float a7) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(a0), "f"(a1), "f"(a2),
                 "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7)
                 : "memory");
}

// The k-th item of block `blk` (of `nblk`) in the dealt order: item positions are taken in
// rounds of nblk, alternating direction, over the list sorted longest first.
struct Item {
    int qt, b, h0;
};
__device__ __forceinline__ bool item_at(int k, int blk, int nblk, int n_items, int per_qt, int n_hgrp,
                                        int heads_per_cta, int n_qt, Item &it) {
    const int pos = k * nblk + ((k & 1) ? (nblk - 1 - blk) : blk);
    if (pos >= n_items) return false;
    it.qt = n_qt - 1 - pos / per_qt;
    const int rem = pos % per_qt;
    it.b = rem / n_hgrp;
    it.h0 = (rem % n_hgrp) * heads_per_cta;
    return true;
}

// One item's extent. kv0: the position of the item's sequence's row 0 among its keys
// (start_pos in the cache form, else 0); nkv: KV tiles the item reads; mask_from: the first
// of them holding a key hidden from some row.
struct Span {
    int seq0, S, kv0, nkv, mask_from;
};
template <bool CACHE>
__device__ __forceinline__ bool item_span(const PrefillArgs &a, const Item &it, Span &sp) {
    sp.seq0 = a.cu_seqlens[it.b];
    sp.S = a.cu_seqlens[it.b + 1] - sp.seq0;
    if (it.qt * BM >= sp.S) return false;
    if (CACHE) {
        sp.kv0 = a.start_pos[it.b];
        const int last = min((it.qt + 1) * BM, sp.S) - 1;          // the item's last row
        sp.nkv = (sp.kv0 + last) / BN + 1;
        sp.mask_from = (sp.kv0 + it.qt * BM) / BN;
    } else {
        sp.kv0 = 0;
        sp.nkv = it.qt + 1;
        sp.mask_from = it.qt;
    }
    return true;
}

// Query tiles of the longest sequence, at most n_qt (warp-collective).
__device__ __forceinline__ int longest_tiles(const int *cu, int B, int n_qt, int lane) {
    int mx = 0;
    for (int b = lane; b < B; b += 32) mx = max(mx, cu[b + 1] - cu[b]);
    mx = __reduce_max_sync(0xffffffffu, mx);
    return min(n_qt, (mx + BM - 1) / BM);
}

// Zero rows z0 .. 127 of a V tile in shared memory (both 64-column boxes; a row's 128 bytes
// in a box are its own whatever the swizzle), then make the writes visible to the tensor core.
__device__ __forceinline__ void zero_v_rows(uint8_t *tile, int z0, int lane) {
    for (int i = lane; i < (BN - z0) * 16; i += 32) {
        const int r = z0 + (i >> 4), c = i & 15;
        *reinterpret_cast<uint4 *>(tile + (c >> 3) * BOX_BYTES + r * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// qmap: Q (MLA: q_lat); qrmap: MLA q_rope (the other forms do not read it); kmap: K (MLA: the
// latent cache c); vmap: V (MLA: the rope cache kr); omap: the fp32 output.
template <int FORM>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap qrmap,
               const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap omap, const PrefillArgs a, int n_qt, int heads_per_cta) {
    constexpr bool CACHE = FORM != kPacked;
    constexpr bool MLA = FORM == kMla;
    using L = Lay<FORM>;
    constexpr int Q_OFF = L::Q_OFF, QR_OFF = L::QR_OFF, K_OFF = L::K_OFF, V_OFF = L::V_OFF, OST_OFF = L::OST_OFF;
    constexpr int BAR_OFF = L::BAR_OFF, SLOT_OFF = L::SLOT_OFF;
    // bytes one Q slot and one K/V stage receive
    constexpr uint32_t Q_TX = TILE_BYTES + (MLA ? RT_BYTES : 0);
    constexpr uint32_t KV_TX = TILE_BYTES + (MLA ? RT_BYTES : 0);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + BAR_OFF + 8 * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + SLOT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_hgrp = a.Hq / heads_per_cta;
    const int per_qt = a.B * n_hgrp;
    const int n_mt = heads_per_cta;                 // query tiles per item (heads h0, h0+1)
    const int G = a.Hq / a.Hkv;
    const int blk = blockIdx.x, nblk = gridDim.x;

    if (threadIdx.x == 0) {
        for (int q = 0; q < Q_SLOTS; ++q) {
            mbar_init(bar(kQFull + q), 1);
            mbar_init(bar(kQEmpty + q), 1);
        }
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(kKFull + s), 1);
            mbar_init(bar(kVFull + s), 1);
            mbar_init(bar(kKEmpty + s), 1);
            mbar_init(bar(kVEmpty + s), 1);
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
    griddep_wait();                                 // cu_seqlens and the inputs are read below
    if (CACHE) n_qt = longest_tiles(a.cu_seqlens, a.B, n_qt, lane);
    const int n_items = n_qt * per_qt;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            const uint64_t pol_q = l2_evict_first_policy();
            int g_kv = 0, qc = 0;                    // K/V tiles and Q tiles loaded so far
            bool ok = true;
            Item it;
            Span sp;
            for (int k = 0; ok && item_at(k, blk, nblk, n_items, per_qt, n_hgrp, heads_per_cta, n_qt, it); ++k) {
                if (!item_span<CACHE>(a, it, sp)) continue;
                const int j = it.h0 / G;
                // Q tile t of this item goes to slot qc % 3; the slot's previous tile must be
                // done with (its last S MMA complete)
                for (int t = 0; t < n_mt && ok; ++t, ++qc) {
                    const int q = qc % Q_SLOTS, u = qc / Q_SLOTS;
                    if (u > 0 && !mbar_wait_bounded(bar(kQEmpty + q), (u - 1) & 1, &g_prefill_status, kStatusEmptyWait)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(kQFull + q), Q_TX);
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_3d(sb + Q_OFF + q * TILE_BYTES + bx * BOX_BYTES, &qmap, bx * 64, it.h0 + t,
                                    sp.seq0 + it.qt * BM, bar(kQFull + q), pol_q);
                    if (MLA)
                        for (int bx = 0; bx < 3; ++bx)
                            tma_load_3d(sb + QR_OFF + q * RT_BYTES + bx * RBOX_BYTES, &qrmap, bx * 16, it.h0 + t,
                                        sp.seq0 + it.qt * BM, bar(kQFull + q), pol_q);
                }
                for (int n = 0; ok && n < sp.nkv; ++n, ++g_kv) {
                    const int s = g_kv % NSTAGE;
                    const uint32_t free_ph = ((g_kv / NSTAGE) & 1) ^ 1;
                    // the tile's first key: a row of the packed K/V, or a position in the cache
                    const int k_tok = CACHE ? n * BN : sp.seq0 + n * BN;
                    if (MLA) {
                        // c (K and V) and kr share one barrier; the stage is free once both
                        // P·V MMAs reading it (issued after its S MMAs) are done
                        if (!mbar_wait_bounded(bar(kVEmpty + s), free_ph, &g_prefill_status, kStatusEmptyWait)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(kKFull + s), KV_TX);
                        for (int bx = 0; bx < 2; ++bx)
                            tma_load_3d_nohint(sb + K_OFF + s * TILE_BYTES + bx * BOX_BYTES, &kmap, bx * 64, k_tok, it.b,
                                               bar(kKFull + s));
                        for (int bx = 0; bx < 3; ++bx)
                            tma_load_3d_nohint(sb + V_OFF + s * RT_BYTES + bx * RBOX_BYTES, &vmap, bx * 16, k_tok, it.b,
                                               bar(kKFull + s));
                        continue;
                    }
                    if (!mbar_wait_bounded(bar(kKEmpty + s), free_ph, &g_prefill_status, kStatusEmptyWait)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(kKFull + s), TILE_BYTES);
                    for (int bx = 0; bx < 2; ++bx) {
                        if (CACHE)
                            tma_load_4d_nohint(sb + K_OFF + s * TILE_BYTES + bx * BOX_BYTES, &kmap, bx * 64, j, k_tok,
                                               it.b, bar(kKFull + s));
                        else
                            tma_load_3d_nohint(sb + K_OFF + s * TILE_BYTES + bx * BOX_BYTES, &kmap, bx * 64, j, k_tok,
                                               bar(kKFull + s));
                    }
                    if (!mbar_wait_bounded(bar(kVEmpty + s), free_ph, &g_prefill_status, kStatusEmptyWait)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(kVFull + s), TILE_BYTES);
                    for (int bx = 0; bx < 2; ++bx) {
                        if (CACHE)
                            tma_load_4d_nohint(sb + V_OFF + s * TILE_BYTES + bx * BOX_BYTES, &vmap, bx * 64, j, k_tok,
                                               it.b, bar(kVFull + s));
                        else
                            tma_load_3d_nohint(sb + V_OFF + s * TILE_BYTES + bx * BOX_BYTES, &vmap, bx * 64, j, k_tok,
                                               bar(kVFull + s));
                    }
                }
            }
            // no copy may still be in flight when the block exits
            for (int i = qc > Q_SLOTS ? qc - Q_SLOTS : 0; i < qc; ++i)
                mbar_wait_bounded(bar(kQFull + i % Q_SLOTS), (i / Q_SLOTS) & 1, &g_prefill_status, kStatusDrainWait);
            for (int g = g_kv > NSTAGE ? g_kv - NSTAGE : 0; g < g_kv; ++g) {
                mbar_wait_bounded(bar(kKFull + g % NSTAGE), (g / NSTAGE) & 1, &g_prefill_status, kStatusDrainWait);
                if (!MLA)
                    mbar_wait_bounded(bar(kVFull + g % NSTAGE), (g / NSTAGE) & 1, &g_prefill_status, kStatusDrainWait);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop, so the descriptors stay warp-uniform; lane 0 alone
        // issues the MMAs and the commits that track them. Descriptors are built once: a
        // byte offset inside shared memory (< 256 KB) adds to the 14-bit start-address field
        // in 16-byte units without carrying out of it.
        //
        // Issue order for iteration g (KV tile g of this block): S_0(g), P·V_1(g−1), S_1(g),
        // P·V_0(g). Each tile's chain S → softmax → P·V → next S is offset by half a period
        // from the other's, so one tile's softmax runs while the tensor core works for the
        // other. S_t(g) overwrites P_t, which P·V_t(g−1) reads; it is issued after that P·V
        // without waiting for it to finish: MMAs issued by one thread execute in issue order,
        // so the earlier one has read its operands before the later one writes (waiting for
        // the completion cost an mbarrier round trip, 550-800 cycles, twice per iteration,
        // with the tensor pipe idle). The commit after S_t(g) still tracks every earlier MMA,
        // so "S_t(g) full" also means P·V_t(g−1) is done when the softmax rescales O_t.
        //
        // MLA: S adds q_rope · krᵀ (three K = 16 steps over the 32-byte swizzled boxes) to
        // q_lat · cᵀ, and P·V reads its B operand from the c stage.
        const uint64_t q_desc = sdesc_sw128(sb + Q_OFF, 16, 1024);
        const uint64_t k_desc = sdesc_sw128(sb + K_OFF, 16, 1024);
        const uint64_t v_desc = sdesc_sw128(sb + (MLA ? K_OFF : V_OFF), BOX_BYTES, 1024);
        const uint64_t qr_desc = sdesc(sb + QR_OFF, 16, 256, kSw32);
        const uint64_t kr_desc = sdesc(sb + V_OFF, 16, 256, kSw32);
        auto wait_all = [&](int idx, uint32_t parity, unsigned code) {
            const bool got = mbar_wait_bounded(bar(idx), parity, &g_prefill_status, code);
            return __all_sync(0xffffffffu, got);
        };
        auto issue_s = [&](int t, int qslot, int s) {     // S_t = Q(slot) · K(stage s)ᵀ
            if (lane == 0) {
                const uint64_t kd = k_desc + (uint64_t)((s * TILE_BYTES) >> 4);
                const uint64_t qd = q_desc + (uint64_t)((qslot * TILE_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
                    umma_ss(tmem + 256 * t, qd + off, kd + off, kIdescS, kk > 0);
                }
                if (MLA) {
                    const uint64_t qrd = qr_desc + (uint64_t)((qslot * RT_BYTES) >> 4);
                    const uint64_t krd = kr_desc + (uint64_t)((s * RT_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 3; ++kk)
                        umma_ss(tmem + 256 * t, qrd + ((kk * RBOX_BYTES) >> 4), krd + ((kk * RBOX_BYTES) >> 4), kIdescS,
                                1u);
                }
                umma_commit(bar(kSFull + t));
            }
            __syncwarp();
        };
        auto issue_pv = [&](int t, int s, bool first, bool split) {   // O_t (+)= P_t · V(stage s)
            if (lane == 0) {
                const uint32_t p = tmem + 256 * t;
                const uint64_t vd = v_desc + (uint64_t)((s * TILE_BYTES) >> 4);
                // keys 16kk .. 16kk+15: P in columns 32·(kk/2) + 8·(kk%2) .. +8, residual 16 further
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_ts(p + 128, p + 32 * (kk >> 1) + 8 * (kk & 1), vd + ((kk * 2048) >> 4), kIdescPV,
                            (!first || kk > 0) ? 1u : 0u);
                if (split) {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_ts(p + 128, p + 32 * (kk >> 1) + 16 + 8 * (kk & 1), vd + ((kk * 2048) >> 4), kIdescPV,
                                1u);
                }
                umma_commit(bar(kODone + t));
            }
            __syncwarp();
        };
        auto commit = [&](int idx) {
            if (lane == 0) umma_commit(bar(idx));
            __syncwarp();
        };
        int g = 0, qc = 0;                           // iterations and Q tiles of this block so far
        bool ok = true;
        // the deferred P·V_1 of the previous iteration
        bool pend = false, pend_first = false, pend_split = false;
        int pend_s = 0;
        auto flush_pv1 = [&]() {
            if (!pend) return true;
            if (!wait_all(kPReady + 1, (g - 1) & 1, kStatusMmaWait)) return false;
            tc_fence_after();
            issue_pv(1, pend_s, pend_first, pend_split);
            commit(kVEmpty + pend_s);                // both P·V of that stage are issued
            pend = false;
            return true;
        };
        Item it;
        Span sp;
        for (int k = 0; ok && item_at(k, blk, nblk, n_items, per_qt, n_hgrp, heads_per_cta, n_qt, it); ++k) {
            if (!item_span<CACHE>(a, it, sp)) continue;
            const bool split_p = sp.kv0 + it.qt * BM < kSplitTiles * BM;
            const int q0 = qc % Q_SLOTS, u0 = qc / Q_SLOTS;
            const int q1 = (qc + 1) % Q_SLOTS, u1 = (qc + 1) / Q_SLOTS;
            qc += n_mt;
            for (int n = 0; n < sp.nkv; ++n, ++g) {
                const int s = g % NSTAGE;
                const uint32_t ph = (g / NSTAGE) & 1;
                // at an item boundary the previous item's last P·V_1 goes first: S_0 may wait
                // for the new Q tiles
                if (n == 0 && !(ok = flush_pv1())) break;
                if (!(ok = wait_all(kKFull + s, ph, kStatusFullWait))) break;
                if (n == 0 && !(ok = wait_all(kQFull + q0, u0 & 1, kStatusFullWait))) break;
                if (MLA && n == sp.nkv - 1) {
                    // latent rows past the chunk's end (first at z0 >= 1 of this tile) hold
                    // anything; as values their weights are 0, so they must be finite
                    const int z0 = sp.kv0 + sp.S - n * BN;
                    if (z0 < BN) zero_v_rows(smem + K_OFF + s * TILE_BYTES, z0, lane);
                }
                tc_fence_after();
                issue_s(0, q0, s);
                if (n == sp.nkv - 1) commit(kQEmpty + q0);
                if (n_mt == 1 && !MLA) commit(kKEmpty + s);
                if (n_mt == 2) {
                    if (!(ok = flush_pv1())) break;
                    if (n == 0 && !(ok = wait_all(kQFull + q1, u1 & 1, kStatusFullWait))) break;
                    tc_fence_after();
                    issue_s(1, q1, s);
                    if (n == sp.nkv - 1) commit(kQEmpty + q1);
                    if (!MLA) commit(kKEmpty + s);       // both S MMAs of this K tile are issued
                }
                if (!(ok = (MLA || wait_all(kVFull + s, ph, kStatusFullWait)) &&
                           wait_all(kPReady + 0, g & 1, kStatusMmaWait)))
                    break;
                if (CACHE && !MLA && n == sp.nkv - 1) {
                    // cache rows past the chunk's end (first at z0 >= 1 of this tile) hold
                    // anything; their weights are 0, so their values must be finite
                    const int z0 = sp.kv0 + sp.S - n * BN;
                    if (z0 < BN) zero_v_rows(smem + V_OFF + s * TILE_BYTES, z0, lane);
                }
                tc_fence_after();
                issue_pv(0, s, n == 0, split_p);
                if (n_mt == 2) {
                    pend = true;
                    pend_s = s;
                    pend_first = n == 0;
                    pend_split = split_p;
                } else {
                    commit(kVEmpty + s);
                }
            }
        }
        if (ok) ok = flush_pv1();                   // the last iteration's P·V_1 (iteration g-1)
        // the last commits must have arrived before the block exits
        for (int i = g > NSTAGE ? g - NSTAGE : 0; i < g; ++i) {
            if (!MLA)
                mbar_wait_bounded(bar(kKEmpty + i % NSTAGE), (i / NSTAGE) & 1, &g_prefill_status, kStatusDrainWait);
            mbar_wait_bounded(bar(kVEmpty + i % NSTAGE), (i / NSTAGE) & 1, &g_prefill_status, kStatusDrainWait);
        }
        for (int i = qc > Q_SLOTS ? qc - Q_SLOTS : 0; i < qc; ++i)
            mbar_wait_bounded(bar(kQEmpty + i % Q_SLOTS), (i / Q_SLOTS) & 1, &g_prefill_status, kStatusDrainWait);
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 2) >> 2;               // query tile of this warpgroup
        const int quarter = warp & 3;                // the TMEM lanes this warp may touch
        const int row = quarter * 32 + lane;         // query row within the tile
        const uint32_t s_addr = tmem + 256 * t + ((uint32_t)(quarter * 32) << 16);
        const uint32_t o_addr = s_addr + 128;
        const bool neg = a.scale_log2 < 0.f;         // the row max of s·c is then c·min(s)
        int g = 0;
        bool ok = t < n_mt;
        Item it;
        Span sp;
        for (int k = 0; ok && item_at(k, blk, nblk, n_items, per_qt, n_hgrp, heads_per_cta, n_qt, it); ++k) {
            if (!item_span<CACHE>(a, it, sp)) continue;
            const int seq0 = sp.seq0, S = sp.S;
            const bool split_p = sp.kv0 + it.qt * BM < kSplitTiles * BM;
            float m_ref = -INFINITY, l = 0.f;
            for (int n = 0; n < sp.nkv; ++n, ++g) {
                // the warp decides together: the TMEM accesses below are warp-collective
                const bool got = mbar_wait_bounded(bar(kSFull + t), g & 1, &g_prefill_status, kStatusFullWait);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // a masked tile: key k of the tile is visible to this row iff k <= lim
                const bool diag = n >= sp.mask_from;
                const int lim = row + sp.kv0 + it.qt * BM - n * BN;
                const float ext = neg ? (diag ? row_extreme<true, true>(s_addr, lim) : row_extreme<false, true>(s_addr, lim))
                                      : (diag ? row_extreme<true, false>(s_addr, lim) : row_extreme<false, false>(s_addr, lim));
                const float mt = ext * a.scale_log2;
                float alpha = 1.f;
                bool grow = false;
                if (n == 0) {
                    m_ref = mt;                      // key 0 of the first tile is always visible
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
                        uint32_t o[32];
                        tmem_ld32(o_addr + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(o_addr + c * 32, o);
                    }
                }
                if (split_p)
                    diag ? write_p<true, true>(s_addr, a.scale_log2, m_ref, lim, l)
                         : write_p<false, true>(s_addr, a.scale_log2, m_ref, lim, l);
                else if (diag)
                    write_p<true, false>(s_addr, a.scale_log2, m_ref, lim, l);
                else
                    write_p<false, false>(s_addr, a.scale_log2, m_ref, lim, l);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(kPReady + t));
            }
            if (!ok) break;
            // epilogue: the item's last P·V of this tile is iteration g-1
            const bool done = mbar_wait_bounded(bar(kODone + t), (g - 1) & 1, &g_prefill_status, kStatusMmaWait);
            if (!__all_sync(0xffffffffu, done)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int q_row = it.qt * BM + row;
            const float inv = 1.f / l;
            if ((it.qt + 1) * BM <= S) {
                // a full tile: four 32-column chunks through this tile's shared staging buffer
                // (128-byte swizzle: chunk j of row r at (j ^ r % 8)·16 in the row's 128 bytes),
                // each written to global memory by one TMA store, which coalesces what one row
                // per thread would scatter over 32 rows per store instruction
                const uint32_t ost = sb + OST_OFF + t * OST_BYTES;
                const int bar_id = 1 + t;
                const bool issuer = quarter == 0 && lane == 0;     // one thread of the warpgroup
#pragma unroll 1
                for (int c2 = 0; c2 < HD / 64; ++c2) {
                    // two chunks' columns from TMEM with one wait
                    uint32_t o[2][32];
                    tmem_ld32(o_addr + c2 * 64, o[0]);
                    tmem_ld32(o_addr + c2 * 64 + 32, o[1]);
                    tmem_ld_wait(o[0]);
                    tmem_ld_wait(o[1]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (issuer) bulk_wait_read();              // the previous store has read the buffer
                        bar_sync_named(bar_id, 128);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t dsts = ost + row * 128 + ((j ^ (row & 7)) << 4);
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dsts),
                                         "f"(__uint_as_float(o[h][4 * j]) * inv),
                                         "f"(__uint_as_float(o[h][4 * j + 1]) * inv),
                                         "f"(__uint_as_float(o[h][4 * j + 2]) * inv),
                                         "f"(__uint_as_float(o[h][4 * j + 3]) * inv)
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        bar_sync_named(bar_id, 128);
                        if (issuer) {
                            tma_store_3d(&omap, ost, (2 * c2 + h) * 32, it.h0 + t, seq0 + it.qt * BM);
                            bulk_commit();
                        }
                    }
                }
            } else {
            float *dst = a.out + ((size_t)(seq0 + q_row) * a.Hq + it.h0 + t) * HD;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_addr + c * 32, o);
                tmem_ld_wait(o);
                if (q_row < S && !a.out32) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        reinterpret_cast<float4 *>(dst)[c * 8 + i] = make_float4(
                            __uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                            __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
                } else if (q_row < S) {
                    // 32-byte stores: a thread writes its own row, so every store of a warp
                    // touches 32 rows; the wider store halves their number
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_global_v8(dst + c * 32 + 8 * i, __uint_as_float(o[8 * i]) * inv,
                                     __uint_as_float(o[8 * i + 1]) * inv, __uint_as_float(o[8 * i + 2]) * inv,
                                     __uint_as_float(o[8 * i + 3]) * inv, __uint_as_float(o[8 * i + 4]) * inv,
                                     __uint_as_float(o[8 * i + 5]) * inv, __uint_as_float(o[8 * i + 6]) * inv,
                                     __uint_as_float(o[8 * i + 7]) * inv);
                }
            }
            }
            // the next item's first P·V overwrites O; it waits for this warpgroup's next
            // "P ready", which comes after these loads
            tc_fence_before();
        }
    }

    if (warp >= 2) bulk_wait_all();            // every output store has landed
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

template <int FORM>
cudaError_t launch_form(const PrefillArgs &a, cudaStream_t st, const CUtensorMap &qm, const CUtensorMap &qrm,
                        const CUtensorMap &km, const CUtensorMap &vm, const CUtensorMap &om) {
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(prefill_kernel<FORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<FORM>::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int G = a.Hq / a.Hkv;
    const int heads_per_cta = (G % 2 == 0) ? 2 : 1;
    const int n_qt = (a.max_seqlen + BM - 1) / BM;
    const long n_items = (long)n_qt * a.B * (a.Hq / heads_per_cta);
    if (n_items <= 0) return cudaSuccess;
    if (n_items > 0x7fffffffL) return cudaErrorInvalidValue;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int grid = (int)(n_items < sms ? n_items : sms);
    const cudaError_t e = launch_pdl(prefill_kernel<FORM>, dim3(grid), dim3(kThreads), Lay<FORM>::SMEM, st, qm, qrm, km,
                                     vm, om, a, n_qt, heads_per_cta);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t st) {
    if (a.D != HD) return cudaErrorInvalidValue;
    const bool mla = a.q_rope != nullptr, cache = a.start_pos != nullptr;
    if (mla && (!cache || a.Hkv != 1)) return cudaErrorInvalidValue;
    constexpr auto SW128 = CU_TENSOR_MAP_SWIZZLE_128B, SW32 = CU_TENSOR_MAP_SWIZZLE_32B;
    constexpr auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    constexpr auto L2_256 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    CUtensorMap qm, qrm, km, vm, om;
    const uint32_t box128[3] = {64, 1, BM};              // 64 columns of one head, 128 rows
    cudaError_t e;
    {
        const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)a.Hq, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)a.Hq * HD * 2};
        e = encode_tensor_map(&qm, BF16, 3, a.q, dims, strides, box128, SW128, L2_256);
        if (e != cudaSuccess) return e;
    }
    if (mla) {
        // q_rope [T, Hq, 48] and kr [B, S_max, 48] in 16-column boxes (32-byte swizzle); the
        // latent cache c [B, S_max, 128] in 64-column boxes: coordinates (column, position, sequence)
        const uint64_t qr_dims[3] = {48, (uint64_t)a.Hq, (uint64_t)a.T};
        const uint64_t qr_strides[2] = {96, (uint64_t)a.Hq * 96};
        const uint32_t qr_box[3] = {16, 1, BM};
        e = encode_tensor_map(&qrm, BF16, 3, a.q_rope, qr_dims, qr_strides, qr_box, SW32, L2_256);
        if (e != cudaSuccess) return e;
        const uint64_t c_dims[3] = {(uint64_t)HD, (uint64_t)a.S_max, (uint64_t)a.B};
        const uint64_t c_strides[2] = {(uint64_t)HD * 2, (uint64_t)a.S_max * HD * 2};
        const uint32_t c_box[3] = {64, BN, 1};
        e = encode_tensor_map(&km, BF16, 3, a.k, c_dims, c_strides, c_box, SW128, L2_256);
        if (e != cudaSuccess) return e;
        const uint64_t r_dims[3] = {48, (uint64_t)a.S_max, (uint64_t)a.B};
        const uint64_t r_strides[2] = {96, (uint64_t)a.S_max * 96};
        const uint32_t r_box[3] = {16, BN, 1};
        e = encode_tensor_map(&vm, BF16, 3, a.v, r_dims, r_strides, r_box, SW32, L2_256);
        if (e != cudaSuccess) return e;
    } else if (cache) {
        // the caches [B, S_max, Hkv, D]: coordinates (column, KV head, position, sequence)
        const uint64_t dims[4] = {(uint64_t)HD, (uint64_t)a.Hkv, (uint64_t)a.S_max, (uint64_t)a.B};
        const uint64_t strides[3] = {(uint64_t)HD * 2, (uint64_t)a.Hkv * HD * 2, (uint64_t)a.S_max * a.Hkv * HD * 2};
        const uint32_t box4[4] = {64, 1, BN, 1};
        e = encode_tensor_map(&km, BF16, 4, a.k, dims, strides, box4, SW128, L2_256);
        if (e == cudaSuccess) e = encode_tensor_map(&vm, BF16, 4, a.v, dims, strides, box4, SW128, L2_256);
        if (e != cudaSuccess) return e;
    } else {
        const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)a.Hkv, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)HD * 2, (uint64_t)a.Hkv * HD * 2};
        e = encode_tensor_map(&km, BF16, 3, a.k, dims, strides, box128, SW128, L2_256);
        if (e == cudaSuccess) e = encode_tensor_map(&vm, BF16, 3, a.v, dims, strides, box128, SW128, L2_256);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)a.Hq, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)HD * 4, (uint64_t)a.Hq * HD * 4};
        const uint32_t obox[3] = {32, 1, BM};
        e = encode_tensor_map(&om, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.out, dims, strides, obox, SW128,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE);
        if (e != cudaSuccess) return e;
    }
    if (mla) return launch_form<kMla>(a, st, qm, qrm, km, vm, om);
    if (cache) return launch_form<kCache>(a, st, qm, qm, km, vm, om);
    return launch_form<kPacked>(a, st, qm, qm, km, vm, om);
}

int prefill_read_and_clear_status(cudaStream_t s, unsigned *flag) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_prefill_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return (int)e;
}

}  // namespace mlakv
