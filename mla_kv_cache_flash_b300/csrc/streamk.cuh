// The balanced work split of the bf16 decode kernels ("stream-K"), shared by the decode
// kernel that streams the work and the merge kernel that combines what it left split.
//
// Each (sequence b, group of hg KV heads, block hb of their query heads) is one segment: the
// sequence's seq_lens[b] cached tokens of those KV heads, cut into tiles of `tile` tokens
// (the hg heads of one token range stay together, so the rows the block reads lie close in
// memory). Segments are laid end to end, sequence-major, into one list of T tiles, and block
// c of the n persistent blocks takes tiles [start(c), start(c+1)) with start(c) =
// floor(c·T / n). A block walks its range segment by segment ("pieces"); a piece that covers
// its whole segment is final, any other is a partial result (normalised output +
// log-sum-exp) in one of the block's two slots: 2c for its first piece, 2c+1 for its last.
#pragma once

#include <stdint.h>

namespace mlakv {

__host__ __device__ __forceinline__ int stream_tiles(int len, int tile) { return (len + tile - 1) / tile; }

__host__ __device__ __forceinline__ long long stream_start(int c, long long T, int n) {
    if (T * n < (1LL << 32)) return (long long)((unsigned)c * (unsigned)T / (unsigned)n);
    return (long long)c * T / n;
}

// The block whose range holds tile t (0 <= t < T): the largest c with start(c) <= t.
// In 32-bit arithmetic when T·n fits (the usual case: a 64-bit division is a long software
// sequence on the GPU).
__host__ __device__ __forceinline__ int stream_block_of(long long t, long long T, int n) {
    if (T * n < (1LL << 32)) return (int)(((unsigned)(t + 1) * (unsigned)n - 1u) / (unsigned)T);
    return (int)(((t + 1) * n - 1) / T);
}

// off = q·nb + i0 with 0 <= i0 < nb: in 32 bits when off fits (a 64-bit division is a long
// software sequence on the GPU, and the walkers run it at every piece start).
__host__ __device__ __forceinline__ void split_offset(long long off, int nb, int &q, int &i0) {
    if (off < (1LL << 31)) {
        const unsigned u = (unsigned)off;
        q = (int)(u / (unsigned)nb);
        i0 = (int)(u - (unsigned)q * (unsigned)nb);
    } else {
        q = (int)(off / nb);
        i0 = (int)(off - (long long)q * nb);
    }
}

// One piece of a block's range: tiles [i0, i0 + n_t) of segment (b, gi, hb).
struct Piece {
    int b, gi, hb, S, i0, n_t;
    bool whole;                 // the piece is the whole segment
};

// Walks the pieces of a block's tile range [t, t_end) using the tile prefix over sequences.
struct PieceWalker {
    const int *prefix;          // prefix[b] = Σ_{b' < b} tiles(S_b'), b = 0 .. B
    const int *seq_lens;
    int B, seg_per_seq, n_hblk, tile;
    long long t, t_end;
    __device__ bool next(Piece &p) {
        if (t >= t_end) return false;
        // the last b with seg_per_seq · prefix[b] <= t (sequences with no tiles are skipped)
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)seg_per_seq * prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        p.b = lo;
        p.S = seq_lens[lo];
        const int nb = prefix[lo + 1] - prefix[lo];     // = stream_tiles(p.S, tile)
        const long long fb = (long long)seg_per_seq * prefix[lo];
        int q, i0;
        split_offset(t - fb, nb, q, i0);
        p.gi = q / n_hblk;
        p.hb = q % n_hblk;
        p.i0 = i0;
        const long long seg_end = fb + (long long)(q + 1) * nb;
        const long long end = seg_end < t_end ? seg_end : t_end;
        p.n_t = (int)(end - t);
        p.whole = p.i0 == 0 && end == seg_end;
        t = end;
        return true;
    }
};

// The same walk, incremental: the start position (sequence b, segment q of it, tile i0 of
// that) is found once, lane-parallel, by seq_walk_start; each further piece then follows from
// the previous one without a search or a division (a search and two divisions cost a single
// thread about a thousand cycles, paid at every piece start on the critical path).
struct SeqWalker {
    const int *prefix;          // prefix[b] = Σ_{b' < b} tiles(S_b'), b = 0 .. B
    const int *seq_lens;
    int B, n_groups, n_hblk;    // a sequence's segments: n_groups KV-head groups × n_hblk head blocks
    int b, gi, hb, i0;          // the next piece's segment (b, gi, hb) and first tile
    long long t, t_end;
    // position from seq_walk_start's (b, q, i0), q = gi·n_hblk + hb
    __device__ void set(int b_, int q, int i0_, long long t_, long long t_end_) {
        b = b_;
        gi = n_hblk == 1 ? q : q / n_hblk;
        hb = n_hblk == 1 ? 0 : q - gi * n_hblk;
        i0 = i0_;
        t = t_;
        t_end = t_end_;
    }
    __device__ bool next(Piece &p) {
        if (t >= t_end) return false;
        const int nb = prefix[b + 1] - prefix[b];
        const long long left = t_end - t;
        const int n_t = left < nb - i0 ? (int)left : nb - i0;
        p.b = b;
        p.S = seq_lens[b];
        p.gi = gi;
        p.hb = hb;
        p.i0 = i0;
        p.n_t = n_t;
        p.whole = i0 == 0 && n_t == nb;
        t += n_t;
        i0 += n_t;
        if (i0 == nb) {
            i0 = 0;
            if (++hb == n_hblk) {
                hb = 0;
                if (++gi == n_groups) {
                    gi = 0;
                    do {
                        ++b;
                    } while (b < B && prefix[b + 1] == prefix[b]);
                }
            }
        }
        return true;
    }
};

// Start position of tile t0 < T for a SeqWalker, by all 32 lanes of a warp: the sequence whose
// tiles hold t0 by a ballot over 32 sequences at a time, then one division. Every lane
// returns the same (b, q, i0).
__device__ __forceinline__ void seq_walk_start(const int *prefix, int B, int seg_per_seq, long long t0, int lane,
                                               int &b, int &q, int &i0) {
    b = 0;
    for (int base = 0; base < B; base += 32) {
        const int bb = base + lane;
        const bool hit = bb < B && (long long)seg_per_seq * prefix[bb] <= t0 &&
                         t0 < (long long)seg_per_seq * prefix[bb + 1];
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (m) {
            b = base + __ffs(m) - 1;
            break;
        }
    }
    split_offset(t0 - (long long)seg_per_seq * prefix[b], prefix[b + 1] - prefix[b], q, i0);
}

// Chunked prefill: sequence b owns nseg_b segments (its query blocks × KV heads × head
// blocks), each over the same lens[b] keys (the keys its last new token sees); prefix[b]
// counts the tiles of the sequences before b with that multiplicity. A piece's `gi` is its
// segment's index within the sequence (hb = 0); the kernel splits it.
struct ChunkPieceWalker {
    const int *prefix;          // [B+1] Σ_{b' < b} nseg_b' · tiles(lens[b'])
    const int *lens;            // [B]
    int B, tile;
    long long t, t_end;
    __device__ bool next(Piece &p) {
        if (t >= t_end) return false;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        p.b = lo;
        p.S = lens[lo];
        const int nb = stream_tiles(p.S, tile);
        const long long fb = prefix[lo];
        int q, i0;
        split_offset(t - fb, nb, q, i0);
        p.gi = q;
        p.hb = 0;
        p.i0 = i0;
        const long long seg_end = fb + (long long)(q + 1) * nb;
        const long long end = seg_end < t_end ? seg_end : t_end;
        p.n_t = (int)(end - t);
        p.whole = p.i0 == 0 && end == seg_end;
        t = end;
        return true;
    }
};

// Chunked prefill with one block per (sequence b, KV head j): the block's pieces are the
// segments of its query blocks, q = qb·per_qb + j for qb = 0 .. nqb − 1, each whole.
struct AlignedChunkWalker {
    int b, j, per_qb, nqb, S, tile, qb;
    __device__ bool next(Piece &p) {
        if (qb >= nqb) return false;
        p.b = b;
        p.gi = qb * per_qb + j;
        p.hb = 0;
        p.S = S;
        p.i0 = 0;
        p.n_t = stream_tiles(S, tile);
        p.whole = true;
        ++qb;
        return true;
    }
};

}  // namespace mlakv
