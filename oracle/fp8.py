"""Decode over an 8-bit floating-point KV cache (fp64, CPU).

Test infrastructure: only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may use it.

Source: "MHA, MQA và GQA" (coregenaihub ebook), the calculator's number-type selector
(fp32, bf16, fp8, int4) and its note that moving from bf16 to fp8 halves every byte count
while the savings ratio stays the same. The page fixes only the width (8 bits).

Readings: the 8-bit type is E4M3 without infinities (1 sign bit, 4 exponent bits with bias
7, 3 mantissa bits; exponent 0 holds the subnormals m/8·2⁻⁶; the all-ones exponent with
mantissa 7 is NaN; largest finite value 448), the usual KV-cache fp8. Each cached row
(sequence b, token t, KV head j) carries one fp32 scale for K and one for V; the cached
value is e4m3(byte)·scale. The query stays bf16. The decode itself is the GQA decode of
``oracle.attention`` over the dequantised caches, as the pages' attention is unchanged by
the number type.

Pinned by ``tests/test_oracle_pins.py``: all 256 codes against PyTorch's
``float8_e4m3fn`` conversion, the format's closed forms (1.0, 448, the smallest subnormal),
and decode identities (unit scales = decode over the decoded values; a uniform V scale
scales the output; a uniform K scale equals the same factor on the softmax scale).
"""

import numpy as np

from .attention import decode_gqa


def e4m3_to_float(codes):
    """Values of E4M3 codes (uint8 array) as float64, from the format's fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = sign * (1.0 + man / 8.0) * np.exp2(exp - 7.0)
    subnormal = sign * (man / 8.0) * 2.0 ** -6
    out = np.where(exp == 0, subnormal, normal)
    return np.where((exp == 0xF) & (man == 0x7), np.nan, out)


def dequantize(codes, scales):
    """Cached values e4m3(code)·scale: codes [..., D] uint8, scales [...] (one per row)."""
    return e4m3_to_float(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def decode_gqa_fp8(q, k_codes, v_codes, k_scale, v_scale, seq_lens, scale):
    """GQA decode over an E4M3 cache with per-row scales.

    q [B, Hq, D]; k_codes/v_codes [B, S_max, Hkv, D] uint8; k_scale/v_scale [B, S_max, Hkv].
    """
    return decode_gqa(q, dequantize(k_codes, k_scale), dequantize(v_codes, v_scale), seq_lens, scale)
