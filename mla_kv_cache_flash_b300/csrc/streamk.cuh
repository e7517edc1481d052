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
    return (long long)c * T / n;
}

// The block whose range holds tile t (0 <= t < T): the largest c with start(c) <= t.
__host__ __device__ __forceinline__ int stream_block_of(long long t, long long T, int n) {
    return (int)(((t + 1) * n - 1) / T);
}

}  // namespace mlakv
