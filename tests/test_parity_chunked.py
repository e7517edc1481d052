"""Chunked prefill over an existing cache (attn_prefill_gqa_chunked) against the fp64 CPU
oracle: new token i of a chunk at start_pos sees cache rows 0 .. start_pos + i.

fp32 caches: max |Δ| ≤ 1e-5; bf16 caches: ≤ 3e-3 (bf16 inputs, fp32 arithmetic).
"""

import numpy as np
import pytest
import torch

import mla_kv_cache_flash_b300 as mk
import oracle
import workloads as W
from workloads import to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(chunks, hq, hkv, d, s_max, dtype, seed):
    """chunks: (start_pos, n_new) per sequence; the cache already holds every chunk."""
    w = W.DecodeWorkload("chunked", 6, len(chunks), hq, hkv, d, s_max, dtype, lengths=(1,) * len(chunks), sub=seed)
    base = W.decode_inputs(w, DEV)                   # its caches serve as the sequences' caches
    n = np.array([c for _, c in chunks])
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    start = np.array([s for s, _ in chunks], dtype=np.int32)
    g = torch.Generator(device=DEV).manual_seed(7000 + seed)
    q = torch.randn((int(cu[-1]), hq, d), generator=g, device=DEV)
    q = q.to(torch.bfloat16) if dtype == "bf16" else q
    return q, base["k_cache"], base["v_cache"], cu, start, w.scale


def _check(chunks, hq, hkv, d, s_max, dtype, seed, tol, n_splits=(0, 1, 3)):
    q, k, v, cu, start, scale = _case(chunks, hq, hkv, d, s_max, dtype, seed)
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, start, scale)
    max_kv = int((start + np.diff(cu)).max())
    for n_split in n_splits:
        out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(start).to(DEV), max_kv,
                                     scale=scale, n_split=n_split)
        torch.cuda.synchronize()
        assert float(np.abs(to_f64(out) - ref).max()) <= tol, n_split


@pytest.mark.parametrize("hq,hkv,d", [(8, 4, 96), (8, 8, 64), (8, 1, 128), (32, 8, 128)])
def test_chunked_fp32(hq, hkv, d):
    # a chunk after a cached prefix, a chunk from the start, one token (a decode step), an
    # empty chunk, and a chunk that ends at the cache's last row
    _check(((300, 17), (0, 40), (999, 1), (5, 0), (200, 300)), hq, hkv, d, 1000, "fp32", hq + d, 1e-5)


# (32, 2, 128), (32, 1, 128) and (64, 2, 128): 16 or 32 query heads per KV head at D = 128,
# the tcgen05 form (4 new tokens × 16 heads per block); the others, up to 16 heads per KV
# head, the register-MMA form (16 / G new tokens × G heads per 16-row MMA tile: 8 × 2, 4 × 4,
# 1 × 16, 5 × 3 with a spare row, 2 × 8, and KV-head groups of 4, 2 and 1)
@pytest.mark.parametrize("hq,hkv,d", [(8, 4, 96), (32, 8, 128), (16, 1, 64), (32, 2, 128), (32, 1, 128),
                                      (64, 2, 128), (12, 4, 64), (6, 3, 96), (64, 8, 128), (16, 2, 96)])
def test_chunked_bf16(hq, hkv, d):
    _check(((1000, 64), (0, 129), (2047, 1), (127, 128)), hq, hkv, d, 2048, "bf16", hq + 2 * d, 3e-3)


@pytest.mark.parametrize("hq,hkv,d", [(32, 1, 128), (8, 4, 96)])
def test_chunked_bf16_ragged_small_chunks(hq, hkv, d):
    # chunk lengths that are not multiples of 4 (the tcgen05 form's token block), a chunk at
    # the cache's start, empty chunks between others, and a last chunk ending at S_max
    _check(((0, 1), (3, 2), (10, 3), (0, 0), (77, 5), (250, 6), (4, 7), (999, 9), (1015, 9)), hq, hkv, d, 1024,
           "bf16", 50 + hq, 3e-3, n_splits=(0, 1, 2, 7))


@pytest.mark.parametrize("hq,hkv", [(32, 1), (8, 4)])
def test_chunked_bf16_long_chunk(hq, hkv):
    # 512-token chunks, from the start and after a cached prefix
    _check(((0, 512), (700, 512), (3000, 48)), hq, hkv, 128 if hkv == 1 else 96, 4096, "bf16", 60 + hq, 3e-3,
           n_splits=(0, 3))


# bf16 at D = 128 with chunks averaging at least 128 tokens: the tcgen05 prefill kernel reading
# K and V from the caches. Start positions on and off the 128-key tile grid (0, 1, 127, 128,
# 700, 2000), chunks of 1, 128, 129, 200, 256, 300 and 512 tokens and an empty one; 32, 4, 3
# (one head per item) and 1 query heads per KV head.
_LONG = ((0, 300), (1, 128), (127, 129), (128, 256), (700, 512), (3000, 1), (0, 0), (2000, 200))


def _poison_past_chunks(cache, start, cu):
    """Fill every cache row at or past start_pos + n_b with NaN (the kernel must not let them
    reach a visible output through a zero weight)."""
    c = cache.clone()
    for b in range(c.shape[0]):
        c[b, int(start[b]) + int(cu[b + 1] - cu[b]):] = float("nan")
    return c


@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 1), (12, 4), (16, 16)])
def test_chunked_long_chunks_on_the_prefill_kernel(hq, hkv):
    q, k, v, cu, start, scale = _case(_LONG, hq, hkv, 128, 4096, "bf16", 90 + hq + hkv)
    k, v = _poison_past_chunks(k, start, cu), _poison_past_chunks(v, start, cu)
    T, B = int(cu[-1]), len(_LONG)
    assert T >= 128 * B
    assert mk.lib().attn_prefill_gqa_chunked_workspace_size(B, T, hq, hkv, 128, 3200, mk.ATTN_BF16, 0) == 0
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, start, scale)
    out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(start).to(DEV), 3200,
                                 scale=scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert bool(torch.isfinite(out).all())
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3


def test_chunked_long_chunks_negative_scale_and_loose_bound():
    """A negative scale (the row maximum is then the smallest raw score) and a max_kv far
    above every chunk end (the item list is cut to the longest chunk inside the kernel)."""
    chunks = ((5, 640), (0, 129), (4000, 96), (1300, 130))
    q, k, v, cu, start, _ = _case(chunks, 16, 2, 128, 4096, "bf16", 77)
    k = _poison_past_chunks(k, start, cu)
    v = _poison_past_chunks(v, start, cu)
    scale = -0.07
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, start, scale)
    out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(start).to(DEV), 4096,
                                 scale=scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3


def test_chunked_single_tokens_are_decode_steps():
    """Chunks of one token at start_pos = length − 1 give the decode of that length."""
    w = W.MINIMIND_GQA
    inp = W.decode_inputs(w, DEV)
    lens = inp["seq_lens"]
    B = w.batch
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    out = mk.prefill_gqa_chunked(inp["q"], inp["k_cache"], inp["v_cache"], cu, (lens - 1).contiguous(),
                                 int(lens.max()), scale=w.scale)
    dec = mk.decode_gqa(inp["q"], inp["k_cache"], inp["v_cache"], lens, scale=w.scale)
    torch.cuda.synchronize()
    ref = oracle.decode_gqa(to_f64(inp["q"]), to_f64(inp["k_cache"]), to_f64(inp["v_cache"]), lens.cpu().numpy(),
                            w.scale)
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3
    assert float((out - dec).abs().max()) <= 3e-3


def test_chunked_empty_batch_is_a_no_op():
    q = torch.zeros((0, 8, 96), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((2, 16, 4, 96), dtype=torch.bfloat16, device=DEV)
    cu = torch.zeros(3, dtype=torch.int32, device=DEV)
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    out = mk.prefill_gqa_chunked(q, k, k, cu, st, 0)
    torch.cuda.synchronize()
    assert out.shape == (0, 8, 96)


def test_chunked_minimind_four_new_tokens():
    """The bench's chunked line: the MiniMind caches with each sequence's last 4 rows as its
    chunk, every output against the oracle."""
    w = W.MINIMIND_GQA
    inp = W.decode_inputs(w, DEV)
    lens = inp["seq_lens"]
    B, n = w.batch, 4
    g = torch.Generator(device=DEV).manual_seed(w.seed + 700)
    q = torch.randn((B * n, w.n_q_heads, w.head_dim), generator=g, device=DEV).to(torch.bfloat16)
    cu = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=DEV)
    start = (lens - n).contiguous()
    out = mk.prefill_gqa_chunked(q, inp["k_cache"], inp["v_cache"], cu, start, int(lens.max()), scale=w.scale)
    torch.cuda.synchronize()
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(inp["k_cache"]), to_f64(inp["v_cache"]), cu.cpu().numpy(),
                                     start.cpu().numpy(), w.scale)
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3



# --------------------------------------------------------------------------------- MLA

def _mla_case(chunks, hq, s_max, seed):
    w = W.MlaWorkload("mla_chunked", 6, len(chunks), hq, 96, 128, 48, 96, s_max, lengths=(1,) * len(chunks),
                      sub=seed)
    inp = W.mla_inputs(w, DEV)                       # its latent caches serve as the sequences' caches
    n = np.array([c for _, c in chunks])
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    start = np.array([s for s, _ in chunks], dtype=np.int32)
    g = torch.Generator(device=DEV).manual_seed(8000 + seed)
    T = int(cu[-1])
    q_lat = torch.randn((T, hq, 128), generator=g, device=DEV).to(torch.bfloat16)
    q_rope = torch.randn((T, hq, 48), generator=g, device=DEV).to(torch.bfloat16)
    return q_lat, q_rope, inp["c_cache"], inp["kr_cache"], cu, start, w.scale


@pytest.mark.parametrize("hq", [16, 8, 32, 3])
def test_mla_chunked(hq):
    chunks = ((300, 17), (0, 40), (999, 1), (5, 0), (200, 300))
    q_lat, q_rope, c, kr, cu, start, scale = _mla_case(chunks, hq, 1000, hq)
    ref = oracle.mla_prefill_absorbed(to_f64(q_lat), to_f64(q_rope), to_f64(c), to_f64(kr), cu, start, scale)
    max_kv = int((start + np.diff(cu)).max())
    for n_split in (0, 1, 3):
        out = mk.prefill_mla_chunked(q_lat, q_rope, c, kr, torch.from_numpy(cu).to(DEV),
                                     torch.from_numpy(start).to(DEV), max_kv, scale, n_split=n_split)
        torch.cuda.synchronize()
        assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3, n_split


def test_mla_chunked_single_tokens_are_decode_steps():
    """One-token chunks at start_pos = length − 1 give the absorbed MLA decode."""
    lens = (1, 129, 700, 2000)
    w = W.MlaWorkload("mla_chunk1", 6, len(lens), 16, 96, 128, 48, 96, 2000, lengths=lens, sub=40)
    inp = W.mla_inputs(w, DEV)
    q_lat = mk.mla_absorb_query(inp["q_nope"], inp["w_uk"])
    B = len(lens)
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    out = mk.prefill_mla_chunked(q_lat, inp["q_rope"], inp["c_cache"], inp["kr_cache"], cu,
                                 (inp["seq_lens"] - 1).contiguous(), max(lens), w.scale)
    dec = mk.decode_mla_absorbed(q_lat, inp["q_rope"], inp["c_cache"], inp["kr_cache"], inp["seq_lens"], w.scale)
    torch.cuda.synchronize()
    ref = oracle.mla_decode_absorbed(to_f64(q_lat), to_f64(inp["q_rope"]), to_f64(inp["c_cache"]),
                                     to_f64(inp["kr_cache"]), inp["seq_lens"].cpu().numpy(), w.scale)
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3
    assert float((out - dec).abs().max()) <= 3e-3


def test_mla_chunked_ragged_and_long():
    # the tcgen05 decode form's edge cases: chunks of 1 .. 9 tokens (not multiples of 4), empty
    # chunks, a 512-token chunk and one ending at S_max, with the split plan forced several
    # ways (nine sequences keep the average chunk under 128 tokens, off the prefill kernel)
    chunks = ((0, 1), (3, 2), (10, 3), (0, 0), (77, 5), (1200, 9), (0, 512), (1528, 512), (0, 0))
    q_lat, q_rope, c, kr, cu, start, scale = _mla_case(chunks, 16, 2040, 41)
    ref = oracle.mla_prefill_absorbed(to_f64(q_lat), to_f64(q_rope), to_f64(c), to_f64(kr), cu, start, scale)
    max_kv = int((start + np.diff(cu)).max())
    for n_split in (0, 1, 2, 5):
        out = mk.prefill_mla_chunked(q_lat, q_rope, c, kr, torch.from_numpy(cu).to(DEV),
                                     torch.from_numpy(start).to(DEV), max_kv, scale, n_split=n_split)
        torch.cuda.synchronize()
        assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3, n_split


@pytest.mark.parametrize("hq", [16, 8, 3, 32])
def test_mla_chunked_long_chunks_on_the_prefill_kernel(hq):
    # chunks averaging 128 tokens or more: the tcgen05 prefill kernel's MLA form, each latent
    # tile serving as keys (with its rope part) and as values; every latent and rope row past
    # a chunk is NaN. 3 heads: one head per item.
    q_lat, q_rope, c, kr, cu, start, scale = _mla_case(_LONG, hq, 4096, 120 + hq)
    c, kr = _poison_past_chunks(c, start, cu), _poison_past_chunks(kr, start, cu)
    T, B = int(cu[-1]), len(_LONG)
    assert mk.lib().attn_prefill_mla_chunked_workspace_size(B, T, hq, 3200, 0) == 0
    ref = oracle.mla_prefill_absorbed(to_f64(q_lat), to_f64(q_rope), to_f64(c), to_f64(kr), cu, start, scale)
    out = mk.prefill_mla_chunked(q_lat, q_rope, c, kr, torch.from_numpy(cu).to(DEV), torch.from_numpy(start).to(DEV),
                                 3200, scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert bool(torch.isfinite(out).all())
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3


def test_mla_prefill_from_an_empty_cache():
    """MLA prefill of whole prompts (start_pos = 0): row i sees latent rows 0 .. i."""
    chunks = ((0, 1000), (0, 129), (0, 384), (0, 1))
    q_lat, q_rope, c, kr, cu, start, scale = _mla_case(chunks, 16, 1024, 55)
    ref = oracle.mla_prefill_absorbed(to_f64(q_lat), to_f64(q_rope), to_f64(c), to_f64(kr), cu, start, scale)
    out = mk.prefill_mla_chunked(q_lat, q_rope, c, kr, torch.from_numpy(cu).to(DEV), torch.from_numpy(start).to(DEV),
                                 1000, scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3


def test_mla_chunked_four_new_tokens_bench_size():
    """The bench's MLA chunked line: the MiniMind MLA caches (B = 64, 4096 rows) with each
    sequence's last 4 rows as its chunk, every output against the oracle."""
    w = W.MINIMIND_MLA
    inp = W.mla_inputs(w, DEV)
    B, n = w.batch, 4
    g = torch.Generator(device=DEV).manual_seed(w.seed + 800)
    q_lat = torch.randn((B * n, w.n_q_heads, w.kv_lora_rank), generator=g, device=DEV).to(torch.bfloat16)
    q_rope = torch.randn((B * n, w.n_q_heads, w.rope_dim), generator=g, device=DEV).to(torch.bfloat16)
    cu = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=DEV)
    start = (inp["seq_lens"] - n).contiguous()
    out = mk.prefill_mla_chunked(q_lat, q_rope, inp["c_cache"], inp["kr_cache"], cu, start,
                                 int(inp["seq_lens"].max()), w.scale)
    torch.cuda.synchronize()
    ref = oracle.mla_prefill_absorbed(to_f64(q_lat), to_f64(q_rope), to_f64(inp["c_cache"]),
                                      to_f64(inp["kr_cache"]), cu.cpu().numpy(), start.cpu().numpy(), w.scale)
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3


# ------------------------------------------------------------- the 512-token chunk lines

def _sampled_chunk_check(out, q_rows, refs):
    """refs: {b: (lo, hi, oracle rows)}; compares every row and head of the sampled sequences."""
    for b, (lo, hi, ref) in refs.items():
        err = float(np.abs(to_f64(out[lo:hi]) - ref).max())
        assert err <= 3e-3, (b, err)


def test_chunked_prefill_512_at_the_bench_size():
    """The bench's GQA long-chunk line (Llama-3-8B layer, 16 caches of 4096 rows, the last 512
    of each the new tokens) in the one launch bench.py times; sequences 0, 7 and 15 against the
    oracle, every row and head."""
    w = W.LLAMA3_8B_CHUNK512
    inp = W.decode_inputs(w, DEV)
    B, n = w.batch, 512
    g = torch.Generator(device=DEV).manual_seed(w.seed + 700)
    q = torch.randn((B * n, w.n_q_heads, w.head_dim), generator=g, device=DEV).to(torch.bfloat16)
    cu = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=DEV)
    start = (inp["seq_lens"] - n).contiguous()
    assert mk.lib().attn_prefill_gqa_chunked_workspace_size(B, B * n, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                            w.s_max, mk.ATTN_BF16, 0) == 0
    out = mk.prefill_gqa_chunked(q, inp["k_cache"], inp["v_cache"], cu, start, w.s_max, scale=w.scale)
    torch.cuda.synchronize()
    mk.check_status()
    refs = {}
    st = start.cpu().numpy()
    for b in (0, 7, 15):
        lo, hi = b * n, (b + 1) * n
        refs[b] = (lo, hi, oracle.prefill_gqa_chunked(to_f64(q[lo:hi]), to_f64(inp["k_cache"][b:b + 1]),
                                                      to_f64(inp["v_cache"][b:b + 1]), np.array([0, n]),
                                                      st[b:b + 1], w.scale))
    _sampled_chunk_check(out, q, refs)


def test_mla_chunked_prefill_512_at_the_bench_size():
    """The bench's MLA long-chunk line (MiniMind MLA, 32 latent caches of 4096 rows, the last 512
    of each the new tokens) in the one launch bench.py times; sequences 0, 13 and 31 against the
    oracle, every row and head."""
    w = W.MINIMIND_MLA_CHUNK512
    inp = W.mla_inputs(w, DEV)
    B, n = w.batch, 512
    g = torch.Generator(device=DEV).manual_seed(w.seed + 800)
    q_lat = torch.randn((B * n, w.n_q_heads, w.kv_lora_rank), generator=g, device=DEV).to(torch.bfloat16)
    q_rope = torch.randn((B * n, w.n_q_heads, w.rope_dim), generator=g, device=DEV).to(torch.bfloat16)
    cu = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=DEV)
    start = (inp["seq_lens"] - n).contiguous()
    out = mk.prefill_mla_chunked(q_lat, q_rope, inp["c_cache"], inp["kr_cache"], cu, start, w.s_max, w.scale)
    torch.cuda.synchronize()
    mk.check_status()
    refs = {}
    st = start.cpu().numpy()
    for b in (0, 13, 31):
        lo, hi = b * n, (b + 1) * n
        refs[b] = (lo, hi, oracle.mla_prefill_absorbed(to_f64(q_lat[lo:hi]), to_f64(q_rope[lo:hi]),
                                                       to_f64(inp["c_cache"][b:b + 1]), to_f64(inp["kr_cache"][b:b + 1]),
                                                       np.array([0, n]), st[b:b + 1], w.scale))
    _sampled_chunk_check(out, q_lat, refs)


@pytest.mark.parametrize("case", range(6))
def test_long_chunks_random_shapes(case):
    """Seeded random batches on the prefill kernel's cache and MLA forms: chunk lengths 1-700,
    start positions anywhere that fits, 2-6 sequences (the average kept at 128 or more so the
    prefill kernel runs), group sizes 1-16, every cache row past a chunk NaN."""
    rng = np.random.default_rng(5000 + case)
    B = int(rng.integers(2, 7))
    s_max = int(rng.choice([768, 1024, 1536]))
    n = rng.integers(1, 701, size=B)
    n[0] = max(int(n[0]), 128 * B - int(n[1:].sum()), 1)          # average >= 128 tokens
    n = np.minimum(n, s_max)
    while int(n.sum()) < 128 * B:
        n[int(np.argmin(n))] = min(s_max, int(n.min()) + 128)
    start = np.array([int(rng.integers(0, s_max - int(x) + 1)) for x in n])
    chunks = tuple((int(s), int(x)) for s, x in zip(start, n))
    hq, hkv = [(8, 8), (16, 4), (12, 4), (32, 2), (6, 3), (16, 1)][case]
    q, k, v, cu, st, scale = _case(chunks, hq, hkv, 128, s_max, "bf16", 300 + case)
    k, v = _poison_past_chunks(k, st, cu), _poison_past_chunks(v, st, cu)
    T = int(cu[-1])
    assert mk.lib().attn_prefill_gqa_chunked_workspace_size(B, T, hq, hkv, 128, s_max, mk.ATTN_BF16, 0) == 0
    max_kv = int((st + np.diff(cu)).max())
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, st, scale)
    out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(st).to(DEV), max_kv,
                                 scale=scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3, chunks
    # the same chunks through the MLA form (16 heads, or 8 on odd cases)
    mq = 16 if case % 2 == 0 else 8
    ql, qr, c, kr, cu2, st2, mscale = _mla_case(chunks, mq, s_max, 400 + case)
    c, kr = _poison_past_chunks(c, st2, cu2), _poison_past_chunks(kr, st2, cu2)
    mref = oracle.mla_prefill_absorbed(to_f64(ql), to_f64(qr), to_f64(c), to_f64(kr), cu2, st2, mscale)
    mout = mk.prefill_mla_chunked(ql, qr, c, kr, torch.from_numpy(cu2).to(DEV), torch.from_numpy(st2).to(DEV),
                                  max_kv, mscale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(mout) - mref).max()) <= 3e-3, chunks


def test_long_chunks_cache_capacity_off_the_tile_grid():
    """S_max = 1000 (not a multiple of 128): the last K/V tile of a chunk ending at S_max reaches
    past the cache (zeros from the tensor map), one ending 3 rows short has NaN rows to zero
    inside it; both forms."""
    chunks = ((700, 300), (0, 997), (500, 130))
    q, k, v, cu, st, scale = _case(chunks, 16, 4, 128, 1000, "bf16", 333)
    k, v = _poison_past_chunks(k, st, cu), _poison_past_chunks(v, st, cu)
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, st, scale)
    out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(st).to(DEV), 1000,
                                 scale=scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3
    ql, qr, c, kr, cu2, st2, mscale = _mla_case(chunks, 16, 1000, 334)
    c, kr = _poison_past_chunks(c, st2, cu2), _poison_past_chunks(kr, st2, cu2)
    mref = oracle.mla_prefill_absorbed(to_f64(ql), to_f64(qr), to_f64(c), to_f64(kr), cu2, st2, mscale)
    mout = mk.prefill_mla_chunked(ql, qr, c, kr, torch.from_numpy(cu2).to(DEV), torch.from_numpy(st2).to(DEV), 1000,
                                  mscale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(mout) - mref).max()) <= 3e-3


@pytest.mark.parametrize("hq,hkv,d", [(8, 4, 96), (32, 2, 128), (12, 4, 64)])
def test_short_chunks_large_batches(hq, hkv, d):
    """2500 sequences with chunks of 0-3 new tokens (far below 128 on average: the decode
    kernels' chunk modes) over caches of at most 64 rows: the per-sequence tables then take a
    shallower ring, or the next kernel form. Every output within the derived bf16-weight bound
    of the chunk modes, which carry each weight's bf16 residual (about 2^-16 relative)."""
    rng = np.random.default_rng(2500 + hq)
    B = 2500
    n = rng.integers(0, 4, size=B)
    start = np.array([int(rng.integers(0, 64 - int(x) + 1)) for x in n])
    chunks = tuple((int(s), int(x)) for s, x in zip(start, n))
    q, k, v, cu, st, scale = _case(chunks, hq, hkv, d, 64, "bf16", 500 + hq)
    max_kv = int((st + np.diff(cu)).max())
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, st, scale)
    out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(st).to(DEV), max_kv,
                                 scale=scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3


def test_long_chunks_after_a_long_context():
    """512- and 300-token chunks after 130000 and 99000 cached rows (items of about a thousand
    KV tiles) on the prefill kernel's cache and MLA forms, NaN past every chunk."""
    chunks = ((130000, 512), (99000, 300))
    q, k, v, cu, st, scale = _case(chunks, 16, 2, 128, 131072, "bf16", 777)
    k, v = _poison_past_chunks(k, st, cu), _poison_past_chunks(v, st, cu)
    ref = oracle.prefill_gqa_chunked(to_f64(q), to_f64(k), to_f64(v), cu, st, scale)
    out = mk.prefill_gqa_chunked(q, k, v, torch.from_numpy(cu).to(DEV), torch.from_numpy(st).to(DEV), 130512,
                                 scale=scale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(out) - ref).max()) <= 3e-3
    ql, qr, c, kr, cu2, st2, mscale = _mla_case(chunks, 16, 131072, 778)
    c, kr = _poison_past_chunks(c, st2, cu2), _poison_past_chunks(kr, st2, cu2)
    mref = oracle.mla_prefill_absorbed(to_f64(ql), to_f64(qr), to_f64(c), to_f64(kr), cu2, st2, mscale)
    mout = mk.prefill_mla_chunked(ql, qr, c, kr, torch.from_numpy(cu2).to(DEV), torch.from_numpy(st2).to(DEV),
                                  130512, mscale)
    torch.cuda.synchronize()
    mk.check_status()
    assert float(np.abs(to_f64(mout) - mref).max()) <= 3e-3
