/*
 * mlakv.h — C ABI of the KV-cache attention library (libmlakv.so), sm_103a.
 *
 * The library computes softmax(q·Kᵀ·scale)·V for new query tokens over a KV cache whose
 * KV heads are each shared by a group of query heads (GQA; MHA and MQA are its two ends),
 * causal GQA prefill over packed sequences, and MLA decode over a low-rank latent cache
 * with a decoupled RoPE key, with W_UK absorbed into the query.
 *
 * Sources, by page title and section:
 *   [MQA&GQA]  "模型架构｜MQA & GQA 调研" (lichtung612 blog): section "Grouped-query attention"
 *              (GQA-G, GQA-1 = MQA, GQA-H = MHA) and section "代码" (repeat_kv, and
 *              Attention.forward: cache layout (max_batch, max_seq, n_kv_heads, head_dim),
 *              cache write before read, scores/√d + mask, fp32 softmax, ·V).
 *   [EBOOK]    "MHA, MQA và GQA" (coregenaihub ebook): the KV-group count must divide the
 *              Q-head count; the sim rejects other counts rather than rounding.
 *   [MLA]      qqstock article on DeepSeek MLA: sections 1-3 (latent c, weight absorption,
 *              decoupled RoPE key shared by all heads), section 6 (MLA computes like MQA,
 *              V shares c with the un-RoPE'd K) and its MultiHeadLatentAttention code.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE memory owned by the caller, dense (C-contiguous) in
 *     the layout stated, 16-byte aligned. The library never allocates, frees or
 *     synchronises inside a compute call: it validates the host-side arguments, enqueues
 *     its kernels on `stream` and returns. Results are ready when the stream reaches them.
 *   - Query head h uses KV head h / (Hq/Hkv) (contiguous groups, the order repeat_kv's
 *     expand-then-reshape produces) [MQA&GQA, 代码].
 *   - Outputs and accumulators are fp32. bf16 inputs are widened exactly.
 *   - Errors found on the host return a negative status before anything is launched;
 *     the message is available from attn_last_error() on the same thread. Device-side data
 *     (seq_lens, cu_seqlens) are trusted to lie within the bounds stated.
 *   - Calls are reentrant. A workspace must not be shared by two calls that can run at
 *     the same time (different streams); calls on one stream are ordered by the stream.
 *   - Workspaces. Every workspace starts with a fixed 64 KiB region that holds only the
 *     arrival counters of the kernels that merge split segments themselves (bf16 GQA
 *     decode, MLA decode); split partials always lie after it. Zero-fill a workspace once
 *     before its first use: every call that completes leaves its counters zero again, so
 *     one buffer then serves any sequence of calls of any entry point, shape and dtype, as
 *     long as it is large enough for each. A call with more than 16384 counters zeroes its
 *     own (one memset on `stream`) before its launch. After attn_check_status reports
 *     ATTN_ERR_TIMEOUT, zero-fill any workspace the failed calls used before reusing it.
 */
#ifndef MLAKV_H
#define MLAKV_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *mlakv_stream_t;

/* Status codes. 0 = success; negative = error, nothing was launched (except ATTN_ERR_CUDA
 * when the launch itself failed, and ATTN_ERR_TIMEOUT, reported after the fact). */
enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,        /* a required pointer is NULL */
    ATTN_ERR_SHAPE = -2,       /* a size < 1 (or < 0 where 0 is allowed), or Hq % Hkv != 0 [EBOOK] */
    ATTN_ERR_UNSUPPORTED = -3, /* head width / rank / dtype / alignment not built in */
    ATTN_ERR_WORKSPACE = -4,   /* workspace NULL or smaller than the *_workspace_size query */
    ATTN_ERR_CUDA = -5,        /* a CUDA call or kernel launch failed (see attn_last_error) */
    ATTN_ERR_TIMEOUT = -6,     /* a kernel's bounded wait gave up (from attn_check_status) */
    ATTN_ERR_INPUT = -7        /* a device-side length, offset or start position out of its
                                  stated bounds (only with the device checks on, see
                                  attn_set_device_checks) */
};

/* Element type of q and of the cache for attn_decode_gqa (ATTN_F32, ATTN_BF16) and of the
 * cache for attn_decode_gqa_fp8 (ATTN_FP8_E4M3, whose query is bf16; attn_decode_gqa
 * refuses it). The workspace and split queries take all three. */
typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1, ATTN_FP8_E4M3 = 2 } attn_dtype;

/* ---------------------------------------------------------------------------------------
 * GQA / MHA / MQA decode: one new query token per sequence over its cache.
 * [MQA&GQA] Attention.forward with seqlen = 1 and no mask: the new token's K/V are already
 * in the cache, so sequence b attends cache positions 0 .. seq_lens[b]-1.
 *
 *   q        [B, Hq, D]            dtype
 *   k_cache  [B, S_max, Hkv, D]    dtype  (the page's cache_k layout)
 *   v_cache  [B, S_max, Hkv, D]    dtype
 *   seq_lens [B] int32, 0 <= seq_lens[b] <= max_S <= S_max. seq_lens[b] = 0 gives out = 0.
 *   out      [B, Hq, D] fp32, fully written.
 *   scale    multiplies q·k before the softmax (1/sqrt(D) for the page's forward).
 *   S_max    cache capacity (the row stride of the cache, in tokens).
 *   max_S    host-known upper bound on seq_lens; sizes the split-KV plan. Passing S_max is
 *            always valid.
 *   n_split  fp32 (and E4M3) cache: number of pieces each sequence's cache is cut into (each piece is
 *            processed by its own thread block and the pieces are merged by log-sum-exp);
 *            0 lets the library choose from B, Hkv, max_S and the device's SM count.
 *            bf16 cache: the work is always balanced over one persistent thread block per SM
 *            (all sequences' cached tokens are cut into equal shares, whatever their
 *            lengths); n_split > 0 caps the number of blocks at n_split per segment. A
 *            segment is one sequence's tokens for a group of up to 4 KV heads, or, when
 *            D = 128 and 16 or more query heads share each KV head (Hq/Hkv a multiple of
 *            16: those shapes run on the tcgen05 tensor cores), for one KV head and a block
 *            of 16 or 32 of its query heads.
 *   D        64, 96 or 128. Any Hq/Hkv with Hq % Hkv == 0 and Hq/Hkv <= 128.
 *   B        bf16 cache: the kernels keep 8 bytes of per-sequence tables in shared memory
 *            beside their K/V ring and take a shallower ring for a batch that would not fit
 *            beside the deepest one; at least 4800 sequences fit for every shape (at the
 *            Llama-3-8B shape, over 9000). A larger batch returns ATTN_ERR_CUDA.
 *   workspace, ws_bytes: scratch for the split partials, at least
 *            attn_decode_gqa_workspace_size(...) bytes with the same arguments; may be
 *            NULL when that size is 0. For a bf16 cache the workspace also holds one arrival
 *            counter per segment in its counter region (see "Workspaces" above): it must be
 *            zero-filled before its first use, and every call that completes leaves the
 *            counters zero again.
 * Returns ATTN_OK or an error code.
 * ------------------------------------------------------------------------------------- */
size_t attn_decode_gqa_workspace_size(int B, int Hq, int Hkv, int D, int max_S,
                                      attn_dtype dtype, int n_split);

/* The split count attn_decode_gqa uses for these arguments (n_split = 0 resolved). */
int attn_decode_gqa_num_splits(int B, int Hq, int Hkv, int D, int max_S, attn_dtype dtype,
                               int n_split);

int attn_decode_gqa(const void *q, const void *k_cache, const void *v_cache,
                    const int *seq_lens, float *out,
                    int B, int Hq, int Hkv, int D, float scale,
                    int S_max, int max_S, attn_dtype dtype, int n_split,
                    void *workspace, size_t ws_bytes, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * attn_decode_gqa for callers that may not allocate device memory. No source page has a
 * counterpart to this entry point; it exists for the library's users.
 *
 * attn_decode_gqa takes its split scratch from the caller. A caller that cannot allocate —
 * a plugin inside a host program that owns all device memory, a serving loop that must not
 * call cudaMalloc because it can synchronise the device and stall other streams, code that
 * runs where the allocator cannot be entered — calls this instead. It takes the same
 * arguments minus the workspace, and keeps the split partials in a fixed array built into
 * the library (attn_decode_gqa_noalloc_max_scratch() bytes, 16 MiB, held by every GPU that
 * loads the library until the process exits). It allocates and frees nothing.
 *   - Sizes whose partials need more than that return ATTN_ERR_WORKSPACE (ask for fewer
 *     splits, or use attn_decode_gqa).
 *   - The first call on a device looks up the array's device address on that device (the
 *     device must be current); make that first call before any stream capture. The address
 *     is kept until the process exits, so the device's primary context must live as long
 *     (no cudaDeviceReset in between).
 *   - Every call uses the same array, laid out like any workspace of this library (see
 *     "Workspaces" above). It starts zero-filled when the library loads, and a call that
 *     completes leaves its counters at zero again, so any sequence of shapes and dtypes
 *     is served correctly. When attn_check_status reports ATTN_ERR_TIMEOUT it also zeroes
 *     the array's counters on the current device. Calls whose kernels can overlap on the
 *     GPU — other streams, other host threads — race on it; order them.
 * Results are identical to attn_decode_gqa with the same arguments.
 * ------------------------------------------------------------------------------------- */
size_t attn_decode_gqa_noalloc_max_scratch(void);

int attn_decode_gqa_noalloc(const void *q, const void *k_cache, const void *v_cache,
                            const int *seq_lens, float *out,
                            int B, int Hq, int Hkv, int D, float scale,
                            int S_max, int max_S, attn_dtype dtype, int n_split,
                            mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * GQA decode over an 8-bit floating-point cache [EBOOK: fp8 halves every cache byte]:
 * attn_decode_gqa with the cached values e4m3(code)·scale, one fp32 scale per cached row
 * (sequence, token, KV head) for K and for V. E4M3: 1 sign, 4 exponent (bias 7) and
 * 3 mantissa bits, no infinities, largest finite 448; codes widen to fp32 exactly.
 *
 *   q          [B, Hq, D]           bf16
 *   k_cache, v_cache [B, S_max, Hkv, D] uint8 E4M3 codes
 *   k_scale, v_scale [B, S_max, Hkv]    fp32
 *   seq_lens, out, scale, S_max, max_S, n_split, workspace: as attn_decode_gqa with
 *   dtype = ATTN_FP8_E4M3 (use that dtype for the workspace and split queries). D in
 *   {64, 96, 128}. attn_decode_gqa itself refuses ATTN_FP8_E4M3 (it has no scales).
 * Up to 16 query heads per KV head: one launch on the tensor cores (mma.sync, codes widened
 * exactly to fp16 in registers, the weights times each row's V scale split into two fp16
 * parts so the products keep fp32 accuracy), the work balanced over persistent thread
 * blocks as for bf16 caches (n_split > 0 caps the blocks at n_split per (sequence, KV
 * head)); the workspace then holds one arrival counter per (sequence, KV head) in its
 * counter region, under the bf16 rules (zero-filled before first use, left zero by every
 * completed call). More query heads per KV head: the CUDA-core kernel, split partials
 * merged by a second launch (as for fp32 caches).
 * ------------------------------------------------------------------------------------- */
int attn_decode_gqa_fp8(const void *q, const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale, const int *seq_lens,
                        float *out, int B, int Hq, int Hkv, int D, float scale,
                        int S_max, int max_S, int n_split,
                        void *workspace, size_t ws_bytes, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * MLA decode with W_UK absorbed [MLA sections 2, 3, 6]: every head attends the same cached
 * latent row [c_t ‖ kr_t] and averages c_t itself:
 *   s_t = scale·(q_lat[b,h]·c_t + q_rope[b,h]·kr_t),  out_lat[b,h] = Σ_t softmax(s)_t c_t.
 * The caller forms q_lat[b,h] = W_UK[h]ᵀ q_nope[b,h] before the call and applies W_UV[h]
 * to out_lat after it (attn_mla_absorb_query and attn_mla_apply_uv below).
 *
 *   q_lat       [B, Hq, r]      bf16
 *   q_rope      [B, Hq, dr]     bf16 (RoPE already applied)
 *   c_cache     [B, S_max, r]   bf16
 *   krope_cache [B, S_max, dr]  bf16 (RoPE already applied; one head shared by all)
 *   seq_lens    [B] int32, 0 <= seq_lens[b] <= max_S <= S_max; 0 gives out_lat = 0.
 *   out_lat     [B, Hq, r] fp32, fully written.
 *   scale       1/sqrt(d_nope + dr) for the article's recombined query.
 *   r = 128, dr = 48 are built in; Hq a multiple of 16 up to 128.
 *   n_split, max_S, workspace: as for attn_decode_gqa with a bf16 cache (one persistent
 *            block per SM; a segment is one sequence and a block of 16 or 32 heads; the
 *            workspace holds arrival counters and must be zero-filled before its first use).
 * ------------------------------------------------------------------------------------- */
size_t attn_decode_mla_workspace_size(int B, int Hq, int r, int dr, int max_S, int n_split);
int attn_decode_mla_num_splits(int B, int Hq, int r, int dr, int max_S, int n_split);

int attn_decode_mla_absorbed(const void *q_lat, const void *q_rope, const void *c_cache,
                             const void *krope_cache, const int *seq_lens, float *out_lat,
                             int B, int Hq, int r, int dr, float scale,
                             int S_max, int max_S, int n_split,
                             void *workspace, size_t ws_bytes, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * The two projections around the absorbed MLA decode [MLA section 2]: W_UK is folded into
 * the query before the decode, W_UV is applied once to its latent output after it.
 *
 * attn_mla_absorb_query:  q_lat[b,h,:] = W_UK[h]ᵀ · q_nope[b,h,:], fp32 sums rounded to
 *                         nearest-even bf16 (the decode's query operand).
 *   q_nope  [B, Hq, d_nope]   bf16 (the non-RoPE part of the per-head query)
 *   w_uk    [Hq, d_nope, r]   bf16 (key up-projection, latent index last)
 *   q_lat   [B, Hq, r]        bf16, fully written.
 *   r a multiple of 32 up to 256; d_nope 1 .. 512.
 *
 * attn_mla_apply_uv:      out[b,h,:] = W_UV[h] · o_lat[b,h,:], fp32.
 *   o_lat   [B, Hq, r]        fp32 (attn_decode_mla_absorbed's out_lat)
 *   w_uv    [Hq, d_v, r]      bf16 (value up-projection, latent index last)
 *   out     [B, Hq, d_v]      fp32, fully written.
 *   r a multiple of 32 up to 256; d_v 1 .. 256.
 *
 * Both: B, Hq >= 1; pointers 16-byte aligned; ATTN_ERR_NULL / _SHAPE / _UNSUPPORTED before
 * any launch, ATTN_ERR_CUDA if the launch fails. Each may start before the previous kernel
 * on the stream has finished and waits for it before reading its inputs.
 * ------------------------------------------------------------------------------------- */
int attn_mla_absorb_query(const void *q_nope, const void *w_uk, void *q_lat,
                          int B, int Hq, int d_nope, int r, mlakv_stream_t stream);

int attn_mla_apply_uv(const float *o_lat, const void *w_uv, float *out,
                      int B, int Hq, int r, int d_v, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * The cache write of one decode step, fused with the rotary embedding [MQA&GQA "代码":
 * forward rotates the new q and k with the cis table, writes k and v at start_pos, then
 * reads the cache; MLA section 3: q_rope and the shared rope key are rotated, c is not].
 * A head vector of width W is rotated as W/2 consecutive pairs:
 *   (x[2j] + i·x[2j+1]) · (cos + i·sin),  (cos, sin) = freqs_cis[pos, j],
 * in fp32, the result rounded to nearest-even when the type is bf16.
 *
 * attn_kv_append_rope (GQA, decode: one new token per sequence)
 *   q          [B, Hq, D]           dtype (the new token's query, before RoPE)
 *   k_new      [B, Hkv, D]          dtype (before RoPE)
 *   v_new      [B, Hkv, D]          dtype
 *   positions  [B] int32 on the device: the row each sequence's token goes to (start_pos)
 *   freqs_cis  [S_max, D/2, 2] fp32 (cos, sin) per position and pair
 *   q_out      [B, Hq, D]           dtype, the rotated query (may be the same buffer as q)
 *   k_cache, v_cache [B, S_max, Hkv, D] dtype: row positions[b] of sequence b is written,
 *              nothing else is touched.
 *   new_lens   [B] int32 or NULL: positions[b] + 1, the decode's seq_lens.
 *   D a multiple of 8 (bf16) or 4 (fp32); Hq % Hkv == 0.
 *
 * attn_mla_append_rope (MLA, decode)
 *   q_rope [B, Hq, dr], c_new [B, r], kr_new [B, dr] bf16; freqs_cis [S_max, dr/2, 2] fp32;
 *   q_rope_out [B, Hq, dr] (may be q_rope); c_cache [B, S_max, r] gets c_new unrotated,
 *   krope_cache [B, S_max, dr] the rotated kr_new; new_lens as above. r, dr multiples of 8.
 *
 * Both: a position outside [0, S_max) appends nothing for that sequence, writes its q_out
 * rows as 0 and its new length as 0. Pointers 16-byte aligned. ATTN_ERR_NULL / _SHAPE /
 * _UNSUPPORTED before any launch, ATTN_ERR_CUDA if the launch fails. The kernel may start
 * before the previous kernel on the stream has finished and waits for it before reading.
 * ------------------------------------------------------------------------------------- */
int attn_kv_append_rope(const void *q, const void *k_new, const void *v_new, const int *positions,
                        const float *freqs_cis, void *q_out, void *k_cache, void *v_cache,
                        int *new_lens, int B, int Hq, int Hkv, int D, int S_max, attn_dtype dtype,
                        mlakv_stream_t stream);

int attn_mla_append_rope(const void *q_rope, const void *c_new, const void *kr_new,
                         const int *positions, const float *freqs_cis, void *q_rope_out,
                         void *c_cache, void *krope_cache, int *new_lens,
                         int B, int Hq, int r, int dr, int S_max, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Causal GQA prefill over packed variable-length sequences [MQA&GQA, Attention.forward
 * with the causal mask; MLA code's is_causal=True]: row i of sequence b attends keys
 * 0 .. i of the same sequence.
 *
 *   q          [T, Hq, D]  bf16, T = cu_seqlens[B]
 *   k, v       [T, Hkv, D] bf16 (each sequence's own keys/values)
 *   cu_seqlens [B+1] int32 on the device: 0, then running sums of the lengths.
 *   out        [T, Hq, D] fp32, every row written.
 *   max_seqlen   host-known upper bound on the lengths (sizes the grid), >= 0.
 *   total_tokens T, the row count of q/k/v/out (bounds the tensor maps), >= 0.
 *   D = 128. Hq % Hkv == 0. max_seqlen = 0 or T = 0 launches nothing.
 * ------------------------------------------------------------------------------------- */
int attn_prefill_gqa_causal(const void *q, const void *k, const void *v,
                            const int *cu_seqlens, float *out,
                            int B, int Hq, int Hkv, int D, float scale, int max_seqlen,
                            int total_tokens, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Chunked prefill over an existing cache [MQA&GQA "代码": seqlen new tokens at start_pos,
 * written into the cache first, see cached positions 0 .. start_pos + i]: new token i of
 * sequence b attends rows 0 .. start_pos[b] + i of its cache (bottom-right causal).
 *
 *   q          [T, Hq, D]            dtype, the new tokens packed by sequence
 *   k_cache, v_cache [B, S_max, Hkv, D] dtype, already holding the chunks
 *   cu_q       [B+1] int32 on the device: 0, then running sums of the chunk lengths (= T)
 *   start_pos  [B] int32 on the device: tokens cached before each chunk;
 *              start_pos[b] + n_b <= S_max
 *   out        [T, Hq, D] fp32, every row written.
 *   max_kv     host-known bound on start_pos[b] + n_b (sizes the split), 0 .. S_max
 *   dtype      ATTN_F32 or ATTN_BF16; D in {64, 96, 128}; 0 <= T <= 65535; T = 0 or
 *              max_kv = 0 launches nothing.
 *   n_split, workspace: size from attn_prefill_gqa_chunked_workspace_size with the same
 *              dtype; zero-filled before its first use (see "Workspaces").
 * Kernels, chosen from the host arguments alone:
 *   - bf16 at D = 128 with T >= 128·B (chunks of 128 new tokens or more on average): the
 *     tcgen05 prefill kernel of attn_prefill_gqa_causal reading K and V from the caches,
 *     128 new tokens × one query head per MMA tile; no split, no workspace (the size is 0
 *     and n_split is ignored). Cache rows past start_pos[b] + n_b may hold anything (NaN
 *     included): they never reach an output.
 *   - other bf16 caches with Hq/Hkv a multiple of 16 at D = 128: the tcgen05 decode kernel,
 *     4 new tokens × 16 query heads per thread block, so each cached row a block reads feeds
 *     all of them (n_split > 0 caps the blocks at n_split per segment);
 *   - other bf16 caches with at most 16 query heads per KV head: the register-MMA decode
 *     kernel, 16/G new tokens × G heads per MMA tile (n_split as for the tcgen05 form);
 *   - the rest (fp32 caches included): the CUDA-core kernel, each new token a decode over its
 *     visible cache (n_split as for an fp32 cache), then the K2 merge.
 * With n_b = 1 and start_pos = seq_lens − 1 this is one decode step.
 * ------------------------------------------------------------------------------------- */
size_t attn_prefill_gqa_chunked_workspace_size(int B, int T, int Hq, int Hkv, int D, int max_kv,
                                               attn_dtype dtype, int n_split);

int attn_prefill_gqa_chunked(const void *q, const void *k_cache, const void *v_cache,
                             const int *cu_q, const int *start_pos, float *out,
                             int B, int T, int Hq, int Hkv, int D, float scale,
                             int S_max, int max_kv, attn_dtype dtype, int n_split,
                             void *workspace, size_t ws_bytes, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * MLA chunked prefill with W_UK absorbed [MLA sections 2, 3 and 6, with the chunk mask of
 * MQA&GQA "代码"]: new token i of sequence b attends latent rows 0 .. start_pos[b] + i:
 *   s_t = scale·(q_lat·c_t + q_rope·kr_t),  out_lat = Σ_t softmax(s)_t c_t.
 *
 *   q_lat       [T, Hq, r]       bf16 (W_UK absorbed, e.g. by attn_mla_absorb_query)
 *   q_rope      [T, Hq, dr]      bf16 (RoPE applied)
 *   c_cache     [B, S_max, r]    bf16, krope_cache [B, S_max, dr] bf16, holding the chunks
 *   cu_q, start_pos, max_kv, n_split, workspace: as attn_prefill_gqa_chunked (workspace
 *               size from attn_prefill_mla_chunked_workspace_size).
 *   out_lat     [T, Hq, r] fp32, every row written (apply W_UV with attn_mla_apply_uv).
 *   r = 128, dr = 48; 1 <= Hq <= 128; 0 <= T <= 65535.
 * Kernels, chosen from the host arguments alone: T >= 128·B (chunks of 128 new tokens or more
 * on average, a whole prompt with start_pos = 0 included) runs on the tcgen05 prefill kernel
 * of attn_prefill_gqa_causal in its MLA form (128 new tokens × one head per MMA tile, each
 * latent tile both keys, with its rope part, and values; no split, no workspace, n_split
 * ignored; latent and rope rows past start_pos[b] + n_b may hold anything). Otherwise Hq a
 * multiple of 16 runs on the tcgen05 MLA decode kernel, 4 new tokens × 16 heads per thread
 * block reading each latent row once (n_split > 0 caps the blocks at n_split per segment);
 * other head counts on the CUDA-core kernel (each new token a decode over its visible latent
 * rows), then the K2 merge.
 * ------------------------------------------------------------------------------------- */
size_t attn_prefill_mla_chunked_workspace_size(int B, int T, int Hq, int max_kv, int n_split);

int attn_prefill_mla_chunked(const void *q_lat, const void *q_rope, const void *c_cache,
                             const void *krope_cache, const int *cu_q, const int *start_pos,
                             float *out_lat, int B, int T, int Hq, int r, int dr, float scale,
                             int S_max, int max_kv, int n_split,
                             void *workspace, size_t ws_bytes, mlakv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Log-sum-exp merge of split partials (the combine step of split-KV decode):
 *   out[row] = Σ_i e^{lse[row,i] − M} o[row,i,:] / Σ_i e^{lse[row,i] − M},  M = max_i lse[row,i]
 * where o[row,i,:] is piece i's normalised output and lse[row,i] = ln Σ_t e^{s_t} over the
 * piece (−inf for an empty piece). A row whose pieces are all empty gives 0.
 *
 *   o_part   [rows, n_split, Dv] fp32
 *   lse_part [rows, n_split] fp32
 *   out      [rows, Dv] fp32
 *   1 <= n_split <= 256, Dv a multiple of 4 up to 512.
 * ------------------------------------------------------------------------------------- */
int attn_merge_partials(const float *o_part, const float *lse_part, float *out,
                        int rows, int n_split, int Dv, mlakv_stream_t stream);

/* Message for the last non-zero status returned on this thread ("" if none). */
const char *attn_last_error(void);

/* Synchronises `stream`, then reads and clears the library's device-side error flags on
 * the current device. Returns ATTN_OK, ATTN_ERR_TIMEOUT if a kernel gave up a bounded
 * wait since the last check, or ATTN_ERR_CUDA if the stream reported an error. */
int attn_check_status(mlakv_stream_t stream);

/* Device-side checks of the length arrays (a debugging aid; off by default). The host checks
 * only the sizes it is given; seq_lens, cu_seqlens, cu_q and start_pos live on the device and
 * are trusted within their stated bounds (a length above the cache capacity would make a
 * kernel read past the cache). With the checks on, every entry point that takes such an array
 * first checks it on its stream with a small kernel, synchronises the stream, and returns
 * ATTN_ERR_INPUT (attn_last_error names the rule and the first offending index) before
 * launching anything else:
 *   attn_decode_gqa, attn_decode_gqa_fp8, attn_decode_mla_absorbed, attn_decode_gqa_noalloc:
 *       0 <= seq_lens[b] <= max_S;
 *   attn_prefill_gqa_causal: cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] <= total_tokens,
 *       each length <= max_seqlen;
 *   attn_prefill_gqa_chunked, attn_prefill_mla_chunked: cu_q as cu_seqlens with T, and
 *       0 <= start_pos[b], start_pos[b] + n_b <= max_kv.
 * The checks cost a launch and a synchronisation per call and cannot run under stream
 * capture. Turned on by MLAKV_DEVICE_CHECKS=1 in the environment when first consulted, or by
 * this call; process-wide, not thread-safe against concurrent calls. Returns the previous
 * setting (0 or 1). */
int attn_set_device_checks(int on);
int attn_device_checks(void);

/* Failure-path self-test (no source page has a counterpart; it exists to test the library).
 * Launches one thread that waits, bounded by `timeout_cycles` SM clock cycles (1e3 .. 1e9),
 * on an mbarrier that nothing arrives on. The wait runs out, the kernel records it in its
 * device status word and returns; the next attn_check_status on `stream` returns
 * ATTN_ERR_TIMEOUT and clears it, and the context stays usable. Returns ATTN_OK once the
 * kernel is launched, ATTN_ERR_SHAPE for a timeout outside the range, ATTN_ERR_CUDA if the
 * launch fails. */
int attn_selftest_bounded_wait(long long timeout_cycles, mlakv_stream_t stream);

/* Library version string. */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLAKV_H */
