"""Seeded synthetic inputs for the KV-cache attention workloads.

This module only draws random numbers and lays them out; it holds none of the attention
arithmetic. Both sides use it: the tests and ``bench.py`` hand the very same tensors to
the CUDA library and (copied to the host, widened to float64) to the CPU oracle.

Recipe (every workload):
  * values: ``torch.randn`` in float32 from a ``torch.Generator`` seeded per workload on
    the device that will hold the tensor, then rounded to bfloat16 with
    round-to-nearest-even (``.to(torch.bfloat16)``) for the bf16 workloads; the fp32
    workload keeps the float32 draws;
  * lengths: drawn on the host with ``numpy.random.default_rng(seed)``, integers
    uniform over the inclusive range, stored as int32;
  * seeds: ``1000 + workload index``; a sub-case k of a workload adds ``10 * k``;
  * an fp8 cache (``fp8_decode_inputs``): fp32 draws stored as E4M3 codes with one fp32
    scale per cached row, the row's largest magnitude over 448;
  * a decode step's new token (``append_inputs``): q, k_new, v_new drawn as above, and a
    rotation table of (cos, sin) of angles uniform in [-π, π), one per position and pair.

The shapes are those of the model layers the pages account for: the MiniMind hidden-768
attention (8 Q heads, 4 KV heads of width 96; MLA rank 128 + RoPE 48), and the
Llama-3-8B layer (32 Q heads, 8 KV groups, head width 128).
"""

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    index: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    s_max: int
    dtype: str                       # "fp32" or "bf16"
    lengths: tuple = None            # fixed per-sequence lengths, or None
    length_range: tuple = None       # (lo, hi) inclusive uniform draw, or None
    sub: int = 0

    @property
    def seed(self):
        return 1000 + self.index + 10 * self.sub

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)


@dataclass(frozen=True)
class MlaWorkload:
    name: str
    index: int
    batch: int
    n_q_heads: int
    nope_dim: int
    kv_lora_rank: int
    rope_dim: int
    v_head_dim: int
    s_max: int
    lengths: tuple = None
    length_range: tuple = None
    weight_std: float = 1.0 / math.sqrt(128.0)
    sub: int = 0

    @property
    def seed(self):
        return 1000 + self.index + 10 * self.sub

    @property
    def scale(self):
        # softmax scale of the recombined [nope ‖ rope] query: 1/sqrt(96 + 48) = 1/12
        return 1.0 / math.sqrt(self.nope_dim + self.rope_dim)


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    index: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    lengths: tuple = None
    length_range: tuple = None
    sub: int = 0

    @property
    def seed(self):
        return 1000 + self.index + 10 * self.sub

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)


TINY_FP32 = {
    hkv: DecodeWorkload(f"tiny_gqa_decode_fp32_hkv{hkv}", 0, 2, 8, hkv, 64, 128, "fp32",
                        lengths=(37, 128), sub=sub)
    for sub, hkv in enumerate((2, 8, 1))
}
MINIMIND_GQA = DecodeWorkload("minimind_gqa_decode_b32_hq8_hkv4_d96", 1, 32, 8, 4, 96, 2048,
                              "bf16", length_range=(512, 2048))
LLAMA3_8B = {
    hkv: DecodeWorkload(f"llama3_8b_decode_b64_s8192_hq32_hkv{hkv}", 2, 64, 32, hkv, 128, 8192,
                        "bf16", lengths=(8192,) * 64, sub=sub)
    for sub, hkv in enumerate((32, 8, 1))
}
MINIMIND_MLA = MlaWorkload("minimind_mla_decode_b64_s4096_hq16_r128_dr48", 3, 64, 16, 96, 128,
                           48, 96, 4096, lengths=(4096,) * 64)
PREFILL_UNIFORM = PrefillWorkload("causal_prefill_b8_s2048_hq32_hkv8_d128", 4, 8, 32, 8, 128,
                                  lengths=(2048,) * 8)
PREFILL_RAGGED = PrefillWorkload("causal_prefill_ragged_b8_s256to4096_hq32_hkv8_d128", 4, 8, 32, 8,
                                 128, length_range=(256, 4096), sub=1)
# chunked prefill of long chunks: the Llama-3-8B layer over 16 caches of 4096 rows whose last
# 512 rows are the new tokens (start_pos = 3584)
LLAMA3_8B_CHUNK512 = DecodeWorkload("llama3_8b_chunked_prefill_b16_s4096_chunk512_hq32_hkv8_d128", 7, 16, 32, 8,
                                    128, 4096, "bf16", lengths=(4096,) * 16)
# and the MiniMind MLA layer (W_UK absorbed) over 32 latent caches of 4096 rows, the last 512 new
MINIMIND_MLA_CHUNK512 = MlaWorkload("minimind_mla_chunked_prefill_b32_s4096_chunk512_hq16_r128_dr48", 8, 32, 16,
                                    96, 128, 48, 96, 4096, lengths=(4096,) * 32)


def draw_lengths(n, lengths, length_range, seed):
    """Per-sequence lengths: the fixed tuple, or integers uniform over the inclusive
    ``length_range`` drawn with ``numpy.random.default_rng(seed)``."""
    if lengths is not None:
        out = np.asarray(lengths, dtype=np.int32)
        if out.shape != (n,):
            raise ValueError("lengths must have one entry per sequence")
        return out
    lo, hi = length_range
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n).astype(np.int32)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, device, dtype, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16) if dtype == "bf16" else x


def decode_inputs(w, device="cpu", seed=None):
    """q [B,Hq,D], k_cache/v_cache [B,S_max,Hkv,D] (bf16 or fp32), seq_lens [B] int32."""
    seed = w.seed if seed is None else seed
    gen = _gen(device, seed)
    q = _randn((w.batch, w.n_q_heads, w.head_dim), gen, device, w.dtype)
    k = _randn((w.batch, w.s_max, w.n_kv_heads, w.head_dim), gen, device, w.dtype)
    v = _randn((w.batch, w.s_max, w.n_kv_heads, w.head_dim), gen, device, w.dtype)
    lens = torch.from_numpy(draw_lengths(w.batch, w.lengths, w.length_range, seed)).to(device)
    return {"q": q, "k_cache": k, "v_cache": v, "seq_lens": lens}


def mla_inputs(w, device="cpu", seed=None):
    """q_nope [B,Hq,d_nope], q_rope [B,Hq,dr], c_cache [B,S_max,r], kr_cache [B,S_max,dr],
    W_UK [Hq,d_nope,r], W_UV [Hq,d_v,r] (std ``weight_std``), all bf16; seq_lens int32."""
    seed = w.seed if seed is None else seed
    gen = _gen(device, seed)
    b, h = w.batch, w.n_q_heads
    q_nope = _randn((b, h, w.nope_dim), gen, device, "bf16")
    q_rope = _randn((b, h, w.rope_dim), gen, device, "bf16")
    c_cache = _randn((b, w.s_max, w.kv_lora_rank), gen, device, "bf16")
    kr_cache = _randn((b, w.s_max, w.rope_dim), gen, device, "bf16")
    w_uk = _randn((h, w.nope_dim, w.kv_lora_rank), gen, device, "bf16", std=w.weight_std)
    w_uv = _randn((h, w.v_head_dim, w.kv_lora_rank), gen, device, "bf16", std=w.weight_std)
    lens = torch.from_numpy(draw_lengths(b, w.lengths, w.length_range, seed)).to(device)
    return {"q_nope": q_nope, "q_rope": q_rope, "c_cache": c_cache, "kr_cache": kr_cache,
            "w_uk": w_uk, "w_uv": w_uv, "seq_lens": lens}


def prefill_inputs(w, device="cpu", seed=None):
    """Packed q [T,Hq,D], k/v [T,Hkv,D] bf16 and cu_seqlens [B+1] int32 (T = Σ S_b)."""
    seed = w.seed if seed is None else seed
    lens = draw_lengths(w.batch, w.lengths, w.length_range, seed)
    cu = np.zeros(w.batch + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    total = int(cu[-1])
    gen = _gen(device, seed)
    q = _randn((total, w.n_q_heads, w.head_dim), gen, device, "bf16")
    k = _randn((total, w.n_kv_heads, w.head_dim), gen, device, "bf16")
    v = _randn((total, w.n_kv_heads, w.head_dim), gen, device, "bf16")
    return {"q": q, "k": k, "v": v, "cu_seqlens": torch.from_numpy(cu).to(device),
            "lengths": lens, "max_seqlen": int(lens.max()) if len(lens) else 0}


def append_inputs(batch, n_q_heads, n_kv_heads, head_dim, s_max, device="cpu", seed=0, dtype="bf16",
                  rot_dim=None):
    """The new token of one decode step: q [B,Hq,D], k_new/v_new [B,Hkv,D] (``dtype``), and a
    rotation table freqs_cis [S_max, rot_dim/2, 2] fp32 of (cos, sin) of angles drawn
    uniformly in [-π, π) (the table is an input of the method; its angles are arbitrary
    here). ``rot_dim`` defaults to ``head_dim``."""
    gen = _gen(device, seed)
    rot_dim = head_dim if rot_dim is None else rot_dim
    q = _randn((batch, n_q_heads, head_dim), gen, device, dtype)
    k_new = _randn((batch, n_kv_heads, head_dim), gen, device, dtype)
    v_new = _randn((batch, n_kv_heads, head_dim), gen, device, dtype)
    ang = (torch.rand((s_max, rot_dim // 2), generator=gen, device=device, dtype=torch.float32) * 2 - 1) * math.pi
    cis = torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).contiguous()
    return {"q": q, "k_new": k_new, "v_new": v_new, "freqs_cis": cis}


def fp8_decode_inputs(w, device="cpu", seed=None):
    """A decode workload with an E4M3 cache: q [B,Hq,D] bf16; the K and V rows are fp32
    N(0,1) draws stored as E4M3 codes [B,S_max,Hkv,D] uint8 with one fp32 scale per row
    [B,S_max,Hkv] (the row's largest magnitude over 448, so the codes span the format's
    range; the conversion is torch's ``float8_e4m3fn`` cast); seq_lens as ``decode_inputs``."""
    seed = w.seed if seed is None else seed
    gen = _gen(device, seed)
    q = _randn((w.batch, w.n_q_heads, w.head_dim), gen, device, "bf16")
    out = {"q": q}
    for name in ("k", "v"):
        x = _randn((w.batch, w.s_max, w.n_kv_heads, w.head_dim), gen, device, "fp32")
        sc = (x.abs().amax(dim=-1) / 448.0).clamp_min(1e-12)
        out[name + "_cache"] = (x / sc[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
        out[name + "_scale"] = sc.contiguous()
    out["seq_lens"] = torch.from_numpy(draw_lengths(w.batch, w.lengths, w.length_range, seed)).to(device)
    return out


def to_f64(t):
    """Host float64 copy of a tensor's exact values (bf16 and fp32 widen exactly)."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)
