// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define MLAKV_HIDDEN __attribute__((visibility("hidden")))

namespace mlakv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ argument bundles

struct DecodeGqaArgs {
    const void *q;          // [B, Hq, D]
    const void *k;          // [B, S_max, Hkv, D]
    const void *v;          // [B, S_max, Hkv, D]
    const int *seq_lens;    // [B]
    float *out;             // [B, Hq, D]
    float *o_part;          // [B, Hq, n_split, D]   (n_split > 1)
    float *lse_part;        // [B, Hq, n_split]      (n_split > 1)
    int B, Hq, Hkv, D;
    float scale_log2;       // scale · log2(e)
    int S_max;
    int n_split;
    int split_len;          // tokens per split (multiple of the kernel's tile)
    const float *k_scale;   // [B, S_max, Hkv] per-row scales of an E4M3 cache, else unused
    const float *v_scale;
    // chunked prefill (cu_q non-null): B counts the packed query rows, n_seq the sequences;
    // row r of sequence b sees the cache up to start_pos[b] + (r - cu_q[b]) inclusive
    const int *cu_q;        // [n_seq + 1]
    const int *start_pos;   // [n_seq]
    int n_seq;
    // MLA chunked prefill: q = q_lat [rows, Hq, 128], q2 = q_rope [rows, Hq, 48],
    // k = v = c [n_seq, S_max, 128], k2 = kr [n_seq, S_max, 48], Hkv = 1, D = 128
    const void *q2;
    const void *k2;
};

// GQA decode over a bf16 cache with the balanced ("stream-K") split of streamk.cuh.
struct DecodeStreamArgs {
    const void *q;          // [B, Hq, D]
    const void *k;          // [B, S_max, Hkv, D]
    const void *v;          // [B, S_max, Hkv, D]
    const int *seq_lens;    // [B]
    float *out;             // [B, Hq, D]
    float *o_part;          // [2·n_blocks, hg·heads, D]   partial outputs, two slots per block
    float *lse_part;        // [2·n_blocks, hg·heads]
    int B, Hq, Hkv, D;
    float scale_log2;       // scale · log2(e)
    int S_max;
    int n_blocks;           // persistent blocks (grid size)
    int heads;              // query-head rows per KV head and head block: min(G, 16·MT)
    int n_hblk;             // head blocks per KV head: ceil(G / (16·MT))
    int hg;                 // KV heads streamed together in one tile (1, 2 or 4)
    int tile_tokens;        // tokens per tile
    int *counters;          // [B · Hkv · n_hblk] at the workspace's start, zero between calls
    int aligned;            // 1: block c streams exactly segment c (no segment is shared)
    // chunked prefill: q is [T, Hq, D] packed by sequence; sequence b's cu_q[b+1] − cu_q[b]
    // new tokens see keys up to start_pos[b] + i; nt new tokens per segment
    const int *cu_q;        // [B+1]
    const int *start_pos;   // [B]
    int nt, T;
};

struct PrefillArgs {
    const void *q;          // [T, Hq, D]
    const void *k;          // [T, Hkv, D]
    const void *v;          // [T, Hkv, D]
    const int *cu_seqlens;  // [B+1]
    float *out;             // [T, Hq, D]
    int B, Hq, Hkv, D, T;
    float scale_log2;
    int max_seqlen;
    int out32;              // out is 32-byte aligned (the epilogue then stores 32 bytes at a time)
    // Cache form (chunked prefill): k and v are caches [B, S_max, Hkv, D] already holding the
    // chunks, and row i of sequence b's chunk sits at position start_pos[b] + i, seeing cache
    // rows 0 .. start_pos[b] + i. nullptr: k and v are packed like q, positions from 0.
    const int *start_pos;
    int S_max;
    // MLA form (with start_pos; Hkv = 1, D = r = 128): q is q_lat [T, Hq, 128], q_rope
    // [T, Hq, 48], k the latent cache c [B, S_max, 128] (keys and values), v the rope keys
    // kr [B, S_max, 48]; s = q_lat·c + q_rope·kr. nullptr: the GQA forms.
    const void *q_rope;
};

// ------------------------------------------------------------------ launchers (one per TU)

// K1: split-KV GQA decode. Writes out directly when n_split == 1, else the partials.
MLAKV_HIDDEN cudaError_t launch_decode_gqa_f32(const DecodeGqaArgs &a, cudaStream_t s);
// K1 over an E4M3 cache with per-row K and V scales (bf16 query), same grid and partials.
MLAKV_HIDDEN cudaError_t launch_decode_gqa_fp8(const DecodeGqaArgs &a, cudaStream_t s);
// Chunked prefill (cu_q set) on the same kernel over a bf16 cache; an fp32 cache goes through
// launch_decode_gqa_f32, which also takes cu_q.
MLAKV_HIDDEN cudaError_t launch_prefill_chunked_bf16(const DecodeGqaArgs &a, cudaStream_t s);
// Chunked prefill over the MLA latent cache (key [c ‖ kr], value c), bf16.
MLAKV_HIDDEN cudaError_t launch_prefill_chunked_mla(const DecodeGqaArgs &a, cudaStream_t s);
// K1 (bf16, balanced): the persistent grid size and the workspace it needs; the decode kernel
// also combines the segments it splits between blocks.
MLAKV_HIDDEN int decode_gqa_stream_blocks(int B, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN bool decode_gqa_stream_aligned(int B, int Hq, int Hkv, int n_split);
MLAKV_HIDDEN size_t decode_gqa_stream_workspace(int B, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN size_t decode_gqa_stream_o_bytes(int B, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN size_t decode_gqa_stream_lse_bytes(int B, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN size_t decode_gqa_stream_counters(int B, int Hq, int Hkv);
MLAKV_HIDDEN cudaError_t launch_decode_gqa_stream(const DecodeStreamArgs &a, cudaStream_t s);
// Chunked prefill on the same kernel for query groups of up to 16 heads: 16 / G new tokens ×
// G heads per MMA tile, each token with its own key limit.
MLAKV_HIDDEN bool decode_gqa_stream_chunk_eligible(int Hq, int Hkv);
// Whether a batch's per-sequence tables fit beside the chunk mode's ring (else the CUDA-core form).
MLAKV_HIDDEN bool decode_gqa_stream_chunk_fits(int B, int T, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN int decode_gqa_stream_chunk_blocks(int B, int T, int Hq, int Hkv, int n_split);
MLAKV_HIDDEN size_t decode_gqa_stream_chunk_workspace(int B, int T, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN cudaError_t launch_decode_gqa_stream_chunk(const void *q, const void *k, const void *v,
                                                        const int *cu_q, const int *start_pos, float *out, int B,
                                                        int T, int Hq, int Hkv, int D, float scale_log2, int S_max,
                                                        int n_split, void *ws, cudaStream_t st);
// K1 over an E4M3 cache on the tensor cores (mma.sync, up to 16 query heads per KV head): TMA
// code tiles widened to fp16 in shared memory, the balanced split over persistent blocks, shared
// segments merged in-kernel (arrival counters in the workspace's counter region).
MLAKV_HIDDEN bool decode_fp8_mma_eligible(int B, int Hq, int Hkv, int D);
MLAKV_HIDDEN int decode_fp8_blocks(int B, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN size_t decode_fp8_workspace(int B, int Hq, int Hkv, int D, int n_split);
MLAKV_HIDDEN cudaError_t launch_decode_fp8_mma(const void *q, const void *k, const void *v, const float *k_scale,
                                               const float *v_scale, const int *seq_lens, float *out, int B, int Hq,
                                               int Hkv, int D, float scale_log2, int S_max, int n_split, void *ws,
                                               cudaStream_t st);
// K2: log-sum-exp merge of the split partials.
MLAKV_HIDDEN cudaError_t launch_merge(const float *o_part, const float *lse_part, float *out,
                                      int rows, int n_split, int Dv, cudaStream_t s);
// K1 for Hq/Hkv a multiple of 16 at D = 128, and K3 (MLA absorbed decode, r = 128, dr = 48),
// on the tcgen05 tensor cores with the same balanced split; the workspace holds two partial
// slots per block and one zero-initialised arrival counter per segment.
MLAKV_HIDDEN bool decode_tc_gqa_eligible(int B, int Hq, int Hkv, int D);
MLAKV_HIDDEN int decode_tc_gqa_blocks(int B, int Hq, int Hkv, int n_split);
MLAKV_HIDDEN size_t decode_tc_gqa_workspace(int B, int Hq, int Hkv, int n_split);
MLAKV_HIDDEN cudaError_t launch_decode_tc_gqa(const void *q, const void *k, const void *v, const int *seq_lens,
                                              float *out, int B, int Hq, int Hkv, float scale_log2, int S_max,
                                              int n_split, void *ws, cudaStream_t st);
MLAKV_HIDDEN bool decode_tc_mla_fits(int B, int Hq);
MLAKV_HIDDEN int decode_tc_mla_blocks(int B, int Hq, int n_split);
MLAKV_HIDDEN size_t decode_tc_mla_workspace(int B, int Hq, int n_split);
MLAKV_HIDDEN cudaError_t launch_decode_tc_mla(const void *q_lat, const void *q_rope, const void *c_cache,
                                              const void *kr_cache, const int *seq_lens, float *out, int B, int Hq,
                                              float scale_log2, int S_max, int n_split, void *ws, cudaStream_t st);
// Chunked prefill on the same tcgen05 kernel: 4 new tokens × 16 query heads per block, each
// token with its own key limit (bottom-right causal); the workspace as for the decode.
MLAKV_HIDDEN bool decode_tc_gqa_chunk_eligible(int B, int Hq, int Hkv, int D);
MLAKV_HIDDEN size_t decode_tc_gqa_chunk_workspace(int B, int T, int Hq, int Hkv, int n_split);
MLAKV_HIDDEN int decode_tc_gqa_chunk_blocks(int B, int T, int Hq, int Hkv, int n_split);
MLAKV_HIDDEN cudaError_t launch_decode_tc_gqa_chunk(const void *q, const void *k, const void *v, const int *cu_q,
                                                    const int *start_pos, float *out, int B, int T, int Hq, int Hkv,
                                                    float scale_log2, int S_max, int n_split, void *ws,
                                                    cudaStream_t st);
MLAKV_HIDDEN bool decode_tc_mla_chunk_fits(int B);
MLAKV_HIDDEN size_t decode_tc_mla_chunk_workspace(int B, int T, int Hq, int n_split);
MLAKV_HIDDEN int decode_tc_mla_chunk_blocks(int B, int T, int Hq, int n_split);
MLAKV_HIDDEN cudaError_t launch_decode_tc_mla_chunk(const void *q_lat, const void *q_rope, const void *c_cache,
                                                    const void *kr_cache, const int *cu_q, const int *start_pos,
                                                    float *out, int B, int T, int Hq, float scale_log2, int S_max,
                                                    int n_split, void *ws, cudaStream_t st);
// K4: causal GQA prefill (D = 128).
MLAKV_HIDDEN cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s);
// Device error flags of the TUs that have bounded waits: read-and-clear (synchronous).
MLAKV_HIDDEN int decode_gqa_read_and_clear_status(cudaStream_t s, unsigned *flag);
MLAKV_HIDDEN int decode_tc_read_and_clear_status(cudaStream_t s, unsigned *flag);
MLAKV_HIDDEN int prefill_read_and_clear_status(cudaStream_t s, unsigned *flag);
MLAKV_HIDDEN int selftest_read_and_clear_status(cudaStream_t s, unsigned *flag);
MLAKV_HIDDEN int decode_fp8_read_and_clear_status(cudaStream_t s, unsigned *flag);
// Zeroes the counter region of the built-in no-alloc scratch on the current device (after a
// timeout); synchronous.
MLAKV_HIDDEN int noalloc_clear_counters(cudaStream_t s);

// Launch `kern` on `s` with programmatic stream serialisation allowed: the kernel may start
// before the previous kernel in the stream has finished, and must call griddep_wait() before
// it touches memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ------------------------------------------------------------------ workspace layout
//
// Every workspace any entry point takes starts with one fixed region that only arrival
// counters ever occupy; split partials always come after it. The kernels that merge split
// segments in-kernel find their counters at the workspace's start, and a call that completes
// leaves them zero. Because no partial is ever written into the region, one zero-filled
// workspace serves any sequence of calls, whatever their shapes. A call with more counters
// than the region holds extends it past the region and zeroes its counters itself (one
// memset on its stream) before its launch, since partials of other shapes may lie there.
constexpr size_t kCounterRegionBytes = size_t(64) << 10;
// The library's own split choice cuts a segment into at most this many pieces: the block that
// finishes a shared segment last reads every piece's partial row, a few at a time, so its
// merge grows with the piece count (B=1, 8192 tokens, 4 KV heads: 148 pieces 58 us, 37 pieces
// 28 us). An explicit n_split is taken as given.
constexpr int kMaxPieces = 32;   // 16384 int32 counters

inline size_t counter_region_bytes(size_t n_counters) {
    const size_t c = (n_counters * sizeof(int) + 255) / 256 * 256;
    return c > kCounterRegionBytes ? c : kCounterRegionBytes;
}

// The counters of a call that overflow the fixed region are zeroed by the call itself.
inline cudaError_t clear_overflow_counters(int *counters, size_t n_counters, cudaStream_t s) {
    if (n_counters * sizeof(int) <= kCounterRegionBytes) return cudaSuccess;
    return cudaMemsetAsync(counters, 0, n_counters * sizeof(int), s);
}

// Sets the thread's attn_last_error() message and returns `code`.
MLAKV_HIDDEN int report_error(int code, const char *message);
// Sets the message to "<what>: <CUDA error name> (<description>)" and returns ATTN_ERR_CUDA.
MLAKV_HIDDEN int report_cuda_error(cudaError_t e, const char *what);

// Device-side checks of the length arrays (input_checks.cu): off unless MLAKV_DEVICE_CHECKS=1 or
// attn_set_device_checks(1). Each runs on the stream, synchronises it and returns ATTN_OK or
// ATTN_ERR_INPUT (with attn_last_error set) before the caller launches anything.
MLAKV_HIDDEN bool device_checks_on();
MLAKV_HIDDEN int set_device_checks(int on);
// lens[i] in [0, bound], i < n
MLAKV_HIDDEN int check_lengths(const int *lens, int n, int bound, cudaStream_t s, const char *who);
// offsets[0] == 0, non-decreasing, offsets[n] <= T, every difference <= max_len
MLAKV_HIDDEN int check_offsets(const int *offsets, int n, int T, int max_len, cudaStream_t s, const char *who);
// the offsets rule without max_len, and 0 <= start[i], start[i] + cu[i+1] - cu[i] <= max_kv
MLAKV_HIDDEN int check_chunks(const int *cu, const int *start, int n, int T, int max_kv, cudaStream_t s,
                              const char *who);

// Every pointer the C ABI takes must sit on a 16-byte boundary.
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// bf16 → fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Programmatic dependent launch. griddep_wait() returns once every grid this one depends on
// has completed and its memory is visible (at once for a kernel launched without the
// attribute); griddep_launch_dependents() lets the next kernel in the stream launch now, so
// its blocks can be resident and set up while this grid finishes.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

}  // namespace mlakv
