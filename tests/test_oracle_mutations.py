"""Plant plausible mistakes in the CPU oracle and show the pins catch each one.

Every mutation is applied with ``monkeypatch`` to the oracle's own module on the CPU for
the duration of one test; the pins of ``oracle_pins`` then have to fail.
"""

import numpy as np
import pytest

import oracle
from oracle import attention as oatt
from oracle import mla as omla
from tests import oracle_pins as pins


def _fails(check, *args):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check(*args)


def _decode_pins():
    return [
        (pins.check_decode_brute, oracle.decode_gqa),
        (pins.check_decode_sdpa, oracle.decode_gqa),
    ]


def _any_fails(checks):
    caught = 0
    for check, *args in checks:
        try:
            check(*args)
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught > 0, "no pin caught the planted mistake"


def test_interleaved_head_mapping_is_caught(monkeypatch):
    # h % Hkv instead of h // G
    def unit(q, k_cache, v_cache, seq_lens, scale, b, j):
        n_kv = k_cache.shape[2]
        s = int(seq_lens[b])
        heads = np.arange(q.shape[1])[np.arange(q.shape[1]) % n_kv == j]
        return oatt.attend(q[b, heads, :], k_cache[b, :s, j, :], v_cache[b, :s, j, :], scale)
    monkeypatch.setattr(oatt, "decode_gqa_unit", unit)
    _fails(pins.check_decode_brute, oracle.decode_gqa)
    _fails(pins.check_decode_sdpa, oracle.decode_gqa)


def test_dropped_scale_is_caught(monkeypatch):
    real = oatt.attend
    monkeypatch.setattr(oatt, "attend", lambda q, k, v, scale, allowed=None: real(q, k, v, 1.0, allowed))
    _any_fails(_decode_pins())
    _fails(pins.check_prefill_sdpa, oracle.prefill_gqa_causal)


def test_missing_normalisation_is_caught(monkeypatch):
    def attend(q_rows, keys, values, scale, allowed=None):
        s = float(scale) * (np.asarray(q_rows, float) @ np.asarray(keys, float).T)
        if allowed is not None:
            s = np.where(allowed, s, -np.inf)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        return e @ np.asarray(values, float)
    monkeypatch.setattr(oatt, "attend", attend)
    _any_fails(_decode_pins())


def test_causal_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "causal_allowed",
                        lambda q_len, k_len: np.arange(k_len)[None, :] < np.arange(q_len)[:, None] + (k_len - q_len))
    _fails(pins.check_prefill_brute, oracle.prefill_gqa_causal)
    _fails(pins.check_prefill_closed_forms, oracle.prefill_gqa_causal)


def test_anticausal_mask_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "causal_allowed",
                        lambda q_len, k_len: np.arange(k_len)[None, :] >= np.arange(q_len)[:, None])
    _fails(pins.check_prefill_sdpa, oracle.prefill_gqa_causal)


def test_last_token_dropped_is_caught(monkeypatch):
    real = oatt.decode_gqa_unit
    monkeypatch.setattr(oatt, "decode_gqa_unit",
                        lambda q, k, v, lens, scale, b, j: real(q, k, v, np.maximum(np.asarray(lens) - 1, 0), scale, b, j))
    _any_fails(_decode_pins())


def test_values_from_key_cache_is_caught(monkeypatch):
    real = oatt.decode_gqa_unit
    monkeypatch.setattr(oatt, "decode_gqa_unit",
                        lambda q, k, v, lens, scale, b, j: real(q, k, k, lens, scale, b, j))
    _any_fails(_decode_pins())


def test_lse_in_log2_is_caught():
    real = oatt.attend_partial

    def attend_partial(q_rows, keys, values, scale):
        o, lse = real(q_rows, keys, values, scale)
        return o, lse / np.log(2.0)
    _fails(pins.check_split_merge, oatt.attend, attend_partial, oatt.lse_merge)


def test_merge_without_max_weighting_is_caught():
    def bad_merge(o_parts, lse_parts):
        return np.asarray(o_parts).mean(axis=0)
    _fails(pins.check_split_merge, oatt.attend, oatt.attend_partial, bad_merge)


def test_mla_dropped_rope_term_is_caught(monkeypatch):
    real = omla.mla_decode_absorbed
    monkeypatch.setattr(omla, "mla_decode_absorbed",
                        lambda q_lat, q_rope, c, kr, lens, scale: real(q_lat, 0 * q_rope, c, kr, lens, scale))
    _fails(pins.check_mla_absorbed_equals_naive, omla.absorb_query, omla.mla_decode_absorbed,
           omla.apply_uv, omla.mla_decode_naive)
    _fails(pins.check_mla_is_mqa, omla.mla_decode_absorbed, oracle.decode_gqa)


def test_mla_wrong_absorption_operand_is_caught():
    def absorb_rows(q_nope, w_uk):   # contracts W_UK over r instead of d_nope (W·q, square case)
        q_nope = np.asarray(q_nope, float)
        w = np.asarray(w_uk, float)
        return np.einsum("hrn,bhn->bhr", w[:, :q_nope.shape[2], :q_nope.shape[2]], q_nope)
    _fails(pins.check_mla_absorbed_equals_naive, absorb_rows, omla.mla_decode_absorbed,
           omla.apply_uv, omla.mla_decode_naive)


def test_mla_naive_shared_rope_sign_error_is_caught(monkeypatch):
    real = omla.mla_decode_naive
    monkeypatch.setattr(omla, "mla_decode_naive",
                        lambda qn, qr, c, kr, wuk, wuv, lens, scale: real(qn, qr, c, -kr, wuk, wuv, lens, scale))
    _fails(pins.check_mla_naive_brute, omla.mla_decode_naive)


# ----------------------------------------------------------------------------- RoPE + append

def _rope_pins(rot):
    return [(pins.check_rope_complex, rot), (pins.check_rope_closed_forms, rot)]


def test_rope_sin_sign_is_caught():
    def rot(x, cis):
        x, cis = np.asarray(x, float), np.asarray(cis, float)
        c, s = cis[..., 0], cis[..., 1]
        re, im = x[..., 0::2] * c + x[..., 1::2] * s, -x[..., 0::2] * s + x[..., 1::2] * c
        return np.stack([re, im], -1).reshape(x.shape)
    _any_fails(_rope_pins(rot))


def test_rope_half_split_pairing_is_caught():
    def rot(x, cis):                 # pairs (j, j + W/2) instead of (2j, 2j+1)
        x, cis = np.asarray(x, float), np.asarray(cis, float)
        c, s = cis[..., 0], cis[..., 1]
        h = x.shape[-1] // 2
        return np.concatenate([x[..., :h] * c - x[..., h:] * s, x[..., :h] * s + x[..., h:] * c], -1)
    _any_fails(_rope_pins(rot))


def test_append_position_off_by_one_is_caught(monkeypatch):
    from oracle import rope as orope
    real = orope._append
    monkeypatch.setattr(orope, "_append", lambda q, kn, vn, pos, cis, kc, vc:
                        real(q, kn, vn, np.asarray(pos) + 1, cis, kc, vc))
    _fails(pins.check_append_brute, orope.kv_append_rope)
    _fails(pins.check_mla_append_brute, orope.mla_append_rope)


def test_append_rotating_the_value_is_caught():
    from oracle import rope as orope
    def bad(q, k_new, v_new, pos, cis, k, v):
        rv = [orope.rope_rotate(v_new[b], cis[min(max(int(p), 0), cis.shape[0] - 1)]) for b, p in enumerate(pos)]
        return orope.kv_append_rope(q, k_new, np.stack(rv), pos, cis, k, v)
    _fails(pins.check_append_brute, bad)


# ----------------------------------------------------------------------------- fp8 cache

def test_e4m3_exponent_bias_is_caught():
    from oracle import fp8 as ofp8
    def bad(codes):
        return ofp8.e4m3_to_float(codes) * 0.5          # bias 8 instead of 7
    _any_fails([(pins.check_e4m3_table, bad), (pins.check_e4m3_closed_forms, bad)])


def test_e4m3_subnormals_as_normals_is_caught():
    from oracle import fp8 as ofp8
    def bad(codes):
        c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
        v = ofp8.e4m3_to_float(codes)
        exp, man = (c >> 3) & 0xF, c & 7
        sign = np.where(c & 0x80, -1.0, 1.0)
        return np.where(exp == 0, sign * (1 + man / 8.0) * 2.0 ** -7, v)
    _any_fails([(pins.check_e4m3_table, bad), (pins.check_e4m3_closed_forms, bad)])


def test_fp8_dropped_value_scale_is_caught():
    from oracle import fp8 as ofp8
    def bad(q, kc, vc, ks, vs, lens, scale):
        return ofp8.decode_gqa_fp8(q, kc, vc, ks, np.ones_like(vs), lens, scale)
    _fails(pins.check_fp8_decode_identities, bad, ofp8.e4m3_to_float, oracle.decode_gqa)


# ----------------------------------------------------------------------------- chunked prefill

def test_chunked_top_left_mask_is_caught(monkeypatch):
    from oracle import chunked as och
    def top_left(q_len, k_len):      # is_causal's alignment: query i sees keys 0 .. i
        return np.arange(k_len)[None, :] <= np.arange(q_len)[:, None]
    monkeypatch.setattr(och, "causal_allowed", top_left)
    _fails(pins.check_chunked_sdpa, och.prefill_gqa_chunked)
    _fails(pins.check_mla_chunked, och.mla_prefill_absorbed, och.mla_prefill_naive, omla.absorb_query,
           omla.apply_uv, omla.mla_decode_absorbed)


def test_chunked_excluding_the_diagonal_is_caught(monkeypatch):
    from oracle import chunked as och
    def strict(q_len, k_len):
        off = k_len - q_len
        return np.arange(k_len)[None, :] < (np.arange(q_len)[:, None] + off) + (np.arange(k_len)[None, :] == 0)
    monkeypatch.setattr(och, "causal_allowed", strict)
    _fails(pins.check_chunked_ends, och.prefill_gqa_chunked, oracle.prefill_gqa_causal, oracle.decode_gqa)
