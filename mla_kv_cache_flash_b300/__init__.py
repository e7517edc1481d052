"""Python binding of libmlakv.so: KV-cache attention kernels for sm_103a.

Argument marshalling only. Each function checks the tensors' dtype, shape, device and
contiguity, allocates outputs/workspace with torch (so torch's caching allocator owns all
memory), and passes raw device pointers plus ``torch.cuda.current_stream()`` to the C ABI
declared in ``include/mlakv.h``. Every step of the computation runs in the library's CUDA
kernels; there is no host or PyTorch fallback. If the library is missing, or a call
returns an error, a ``RuntimeError`` carrying the library's message is raised.

Entry points (same names as the C ABI, without the ``attn_`` prefix):
  decode_gqa            GQA/MHA/MQA decode over a padded [B, S_max, Hkv, D] cache
  decode_mla_absorbed   MLA decode over the latent cache [c ‖ kr], W_UK absorbed in q_lat
  prefill_gqa_causal    causal GQA prefill over packed sequences (cu_seqlens)
  merge_partials        log-sum-exp merge of split partials
"""

import ctypes
import math
import os

import torch

__all__ = [
    "ATTN_F32", "ATTN_BF16", "ATTN_FP8_E4M3", "MlakvError", "decode_gqa_fp8", "lib", "lib_path", "decode_gqa", "decode_gqa_workspace_size",
    "decode_gqa_num_splits", "decode_gqa_noalloc", "decode_mla_absorbed", "decode_mla_workspace_size", "decode_mla_num_splits",
    "prefill_gqa_causal", "merge_partials", "check_status", "last_error", "version",
    "selftest_bounded_wait", "mla_absorb_query", "mla_apply_uv", "decode_mla", "kv_append_rope",
    "mla_append_rope", "prefill_gqa_chunked", "prefill_mla_chunked", "set_device_checks", "device_checks",
]

ATTN_F32 = 0
ATTN_BF16 = 1
ATTN_FP8_E4M3 = 2
ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_SHAPE, ATTN_ERR_UNSUPPORTED = 0, -1, -2, -3
ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT, ATTN_ERR_INPUT = -4, -5, -6, -7
_STATUS = {0: "ATTN_OK", -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_SHAPE", -3: "ATTN_ERR_UNSUPPORTED",
           -4: "ATTN_ERR_WORKSPACE", -5: "ATTN_ERR_CUDA", -6: "ATTN_ERR_TIMEOUT", -7: "ATTN_ERR_INPUT"}

lib_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmlakv.so")
_lib = None


class MlakvError(RuntimeError):
    def __init__(self, code, message):
        super().__init__(f"{_STATUS.get(code, code)}: {message}")
        self.code = code


_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

_SIGNATURES = {
    "attn_decode_gqa_workspace_size": (_c_size, [_c_int] * 6 + [_c_int]),
    "attn_decode_gqa_num_splits": (_c_int, [_c_int] * 7),
    "attn_decode_gqa": (_c_int, [_vp] * 5 + [_c_int] * 4 + [_c_float] + [_c_int] * 4 + [_vp, _c_size, _vp]),
    "attn_decode_gqa_noalloc_max_scratch": (_c_size, []),
    "attn_decode_gqa_noalloc": (_c_int, [_vp] * 5 + [_c_int] * 4 + [_c_float] + [_c_int] * 4 + [_vp]),
    "attn_decode_mla_workspace_size": (_c_size, [_c_int] * 6),
    "attn_decode_mla_num_splits": (_c_int, [_c_int] * 6),
    "attn_decode_mla_absorbed": (_c_int, [_vp] * 6 + [_c_int] * 4 + [_c_float] + [_c_int] * 3 + [_vp, _c_size, _vp]),
    "attn_decode_gqa_fp8": (_c_int, [_vp] * 7 + [_c_int] * 4 + [_c_float] + [_c_int] * 3 + [_vp, _c_size, _vp]),
    "attn_prefill_gqa_chunked_workspace_size": (_c_size, [_c_int] * 8),
    "attn_prefill_gqa_chunked": (_c_int, [_vp] * 6 + [_c_int] * 5 + [_c_float] + [_c_int] * 4 + [_vp, _c_size, _vp]),
    "attn_prefill_mla_chunked_workspace_size": (_c_size, [_c_int] * 5),
    "attn_prefill_mla_chunked": (_c_int, [_vp] * 7 + [_c_int] * 5 + [_c_float] + [_c_int] * 3 + [_vp, _c_size, _vp]),
    "attn_kv_append_rope": (_c_int, [_vp] * 9 + [_c_int] * 6 + [_vp]),
    "attn_mla_append_rope": (_c_int, [_vp] * 9 + [_c_int] * 5 + [_vp]),
    "attn_mla_absorb_query": (_c_int, [_vp] * 3 + [_c_int] * 4 + [_vp]),
    "attn_mla_apply_uv": (_c_int, [_vp] * 3 + [_c_int] * 4 + [_vp]),
    "attn_prefill_gqa_causal": (_c_int, [_vp] * 5 + [_c_int] * 4 + [_c_float] + [_c_int] * 2 + [_vp]),
    "attn_merge_partials": (_c_int, [_vp] * 3 + [_c_int] * 3 + [_vp]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_check_status": (_c_int, [_vp]),
    "attn_version": (ctypes.c_char_p, []),
    "attn_selftest_bounded_wait": (_c_int, [ctypes.c_longlong, _vp]),
    "attn_set_device_checks": (_c_int, [_c_int]),
    "attn_device_checks": (_c_int, []),
}


def lib():
    """The loaded library (loaded on first use; raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(
                f"{lib_path} is missing: build it with `python -m mla_kv_cache_flash_b300.build` "
                "(there is no fallback implementation)")
        handle = ctypes.CDLL(lib_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def last_error():
    return lib().attn_last_error().decode()


def version():
    return lib().attn_version().decode()


def set_device_checks(on):
    """Turn the device-side checks of seq_lens / cu_seqlens / cu_q / start_pos on or off (see
    attn_set_device_checks: a synchronising debugging aid); returns the previous setting."""
    return bool(lib().attn_set_device_checks(1 if on else 0))


def device_checks():
    return bool(lib().attn_device_checks())


def _check(rc):
    if rc != 0:
        raise MlakvError(rc, last_error())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, name, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def check_status():
    """Synchronise the current stream and raise if a kernel reported a device-side error."""
    _check(lib().attn_check_status(_stream()))


def selftest_bounded_wait(timeout_cycles=100_000):
    """Launch a kernel whose bounded wait runs out on purpose (see attn_selftest_bounded_wait);
    the next check_status() raises ATTN_ERR_TIMEOUT."""
    _check(lib().attn_selftest_bounded_wait(int(timeout_cycles), _stream()))


# ----------------------------------------------------------------------------- GQA decode

def decode_gqa_workspace_size(B, Hq, Hkv, D, max_s, dtype, n_split=0):
    return int(lib().attn_decode_gqa_workspace_size(B, Hq, Hkv, D, max_s, dtype, n_split))


def decode_gqa_num_splits(B, Hq, Hkv, D, max_s, dtype, n_split=0):
    n = lib().attn_decode_gqa_num_splits(B, Hq, Hkv, D, max_s, dtype, n_split)
    _check(min(n, 0))
    return n


def decode_gqa(q, k_cache, v_cache, seq_lens, out=None, scale=None, max_s=None, n_split=0, workspace=None):
    """out[b, h] = softmax(scale · q[b, h] · K[b, :S_b, h // G]ᵀ) · V[b, :S_b, h // G].

    q [B, Hq, D]; k_cache, v_cache [B, S_max, Hkv, D] (fp32 or bf16, same dtype as q);
    seq_lens [B] int32 on the device; returns out [B, Hq, D] fp32. ``max_s`` is a host-known
    bound on seq_lens (defaults to S_max); ``n_split`` = 0 lets the library choose. A
    ``workspace`` passed in must have been zero-filled before its first use (calls leave it so).
    """
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("q must be float32 or bfloat16")
    _need(q, "q", dt, 3)
    dev = q.device
    _need(k_cache, "k_cache", dt, 4, dev)
    _need(v_cache, "v_cache", dt, 4, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    _, S_max, Hkv, Dk = k_cache.shape
    if k_cache.shape[0] != B or Dk != D or v_cache.shape != k_cache.shape or seq_lens.shape[0] != B:
        raise ValueError("inconsistent shapes for q, k_cache, v_cache, seq_lens")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_s = S_max if max_s is None else int(max_s)
    code = ATTN_F32 if dt == torch.float32 else ATTN_BF16
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, 3, dev)
    need = decode_gqa_workspace_size(B, Hq, Hkv, D, max_s, code, n_split)
    if need and (workspace is None or workspace.numel() < need):
        # zero-filled: the library's per-segment counters start at zero and are left at zero
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_decode_gqa(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                                 B, Hq, Hkv, D, scale, S_max, max_s, code, n_split,
                                 _ptr(workspace), ws_bytes, _stream()))
    return out


def decode_gqa_fp8(q, k_cache, v_cache, k_scale, v_scale, seq_lens, out=None, scale=None, max_s=None, n_split=0,
                   workspace=None):
    """decode_gqa over an E4M3 cache: cached value = e4m3(code) · the row's scale.

    q [B, Hq, D] bf16; k_cache, v_cache [B, S_max, Hkv, D] uint8 codes (or float8_e4m3fn);
    k_scale, v_scale [B, S_max, Hkv] fp32; seq_lens [B] int32. Returns out [B, Hq, D] fp32.
    """
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    k_cache = k_cache.view(torch.uint8) if k_cache.dtype == torch.float8_e4m3fn else k_cache
    v_cache = v_cache.view(torch.uint8) if v_cache.dtype == torch.float8_e4m3fn else v_cache
    _need(k_cache, "k_cache", torch.uint8, 4, dev)
    _need(v_cache, "v_cache", torch.uint8, 4, dev)
    _need(k_scale, "k_scale", torch.float32, 3, dev)
    _need(v_scale, "v_scale", torch.float32, 3, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    _, S_max, Hkv, Dk = k_cache.shape
    if (k_cache.shape[0] != B or Dk != D or v_cache.shape != k_cache.shape or seq_lens.shape[0] != B
            or k_scale.shape != (B, S_max, Hkv) or v_scale.shape != k_scale.shape):
        raise ValueError("inconsistent shapes for q, k_cache, v_cache, k_scale, v_scale, seq_lens")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_s = S_max if max_s is None else int(max_s)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, 3, dev)
    need = decode_gqa_workspace_size(B, Hq, Hkv, D, max_s, ATTN_FP8_E4M3, n_split)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_decode_gqa_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                     _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, scale, S_max, max_s, n_split,
                                     _ptr(workspace), ws_bytes, _stream()))
    return out


def decode_gqa_noalloc(q, k_cache, v_cache, seq_lens, out, scale=None, max_s=None, n_split=0):
    """decode_gqa for callers that must not allocate device memory.

    The split scratch lives in a fixed array inside the library instead of a caller
    workspace, and ``out`` must be passed in, so the call allocates nothing. Calls whose
    kernels can overlap on the GPU share that array and must be ordered by the caller.
    """
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("q must be float32 or bfloat16")
    _need(q, "q", dt, 3)
    dev = q.device
    _need(k_cache, "k_cache", dt, 4, dev)
    _need(v_cache, "v_cache", dt, 4, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    _need(out, "out", torch.float32, 3, dev)
    B, Hq, D = q.shape
    _, S_max, Hkv, _ = k_cache.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_s = S_max if max_s is None else int(max_s)
    code = ATTN_F32 if dt == torch.float32 else ATTN_BF16
    _check(lib().attn_decode_gqa_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                                         B, Hq, Hkv, D, scale, S_max, max_s, code, n_split, _stream()))
    return out


# ----------------------------------------------------------------------------- MLA decode

def decode_mla_workspace_size(B, Hq, r, dr, max_s, n_split=0):
    return int(lib().attn_decode_mla_workspace_size(B, Hq, r, dr, max_s, n_split))


def decode_mla_num_splits(B, Hq, r, dr, max_s, n_split=0):
    n = lib().attn_decode_mla_num_splits(B, Hq, r, dr, max_s, n_split)
    _check(min(n, 0))
    return n


def decode_mla_absorbed(q_lat, q_rope, c_cache, krope_cache, seq_lens, scale, out_lat=None, max_s=None,
                        n_split=0, workspace=None):
    """out_lat[b, h] = Σ_t softmax_t(scale·(q_lat·c_t + q_rope·kr_t)) · c_t (bf16 in, fp32 out).

    q_lat [B, Hq, r], q_rope [B, Hq, dr], c_cache [B, S_max, r], krope_cache [B, S_max, dr],
    seq_lens [B] int32. The caller absorbs W_UK into q_lat and applies W_UV to out_lat.
    """
    bf = torch.bfloat16
    _need(q_lat, "q_lat", bf, 3)
    dev = q_lat.device
    _need(q_rope, "q_rope", bf, 3, dev)
    _need(c_cache, "c_cache", bf, 3, dev)
    _need(krope_cache, "krope_cache", bf, 3, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    B, Hq, r = q_lat.shape
    dr = q_rope.shape[2]
    S_max = c_cache.shape[1]
    if (q_rope.shape[:2] != (B, Hq) or c_cache.shape != (B, S_max, r) or krope_cache.shape != (B, S_max, dr)
            or seq_lens.shape[0] != B):
        raise ValueError("inconsistent shapes for q_lat, q_rope, c_cache, krope_cache, seq_lens")
    max_s = S_max if max_s is None else int(max_s)
    if out_lat is None:
        out_lat = torch.empty((B, Hq, r), dtype=torch.float32, device=dev)
    else:
        _need(out_lat, "out_lat", torch.float32, 3, dev)
    need = decode_mla_workspace_size(B, Hq, r, dr, max_s, n_split)
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_decode_mla_absorbed(_ptr(q_lat), _ptr(q_rope), _ptr(c_cache), _ptr(krope_cache),
                                          _ptr(seq_lens), _ptr(out_lat), B, Hq, r, dr, float(scale), S_max,
                                          max_s, n_split, _ptr(workspace), ws_bytes, _stream()))
    return out_lat


def mla_absorb_query(q_nope, w_uk, q_lat=None):
    """q_lat[b, h] = W_UK[h]ᵀ · q_nope[b, h], fp32 sums rounded to bf16.

    q_nope [B, Hq, d_nope] bf16, w_uk [Hq, d_nope, r] bf16. Returns q_lat [B, Hq, r] bf16.
    """
    bf = torch.bfloat16
    _need(q_nope, "q_nope", bf, 3)
    dev = q_nope.device
    _need(w_uk, "w_uk", bf, 3, dev)
    B, Hq, dn = q_nope.shape
    r = w_uk.shape[2]
    if w_uk.shape[:2] != (Hq, dn):
        raise ValueError("w_uk must be [Hq, d_nope, r] for q_nope [B, Hq, d_nope]")
    if q_lat is None:
        q_lat = torch.empty((B, Hq, r), dtype=bf, device=dev)
    else:
        _need(q_lat, "q_lat", bf, 3, dev)
        if q_lat.shape != (B, Hq, r):
            raise ValueError("q_lat must be [B, Hq, r]")
    _check(lib().attn_mla_absorb_query(_ptr(q_nope), _ptr(w_uk), _ptr(q_lat), B, Hq, dn, r, _stream()))
    return q_lat


def mla_apply_uv(o_lat, w_uv, out=None):
    """out[b, h] = W_UV[h] · o_lat[b, h] (fp32). o_lat [B, Hq, r] fp32, w_uv [Hq, d_v, r] bf16."""
    _need(o_lat, "o_lat", torch.float32, 3)
    dev = o_lat.device
    _need(w_uv, "w_uv", torch.bfloat16, 3, dev)
    B, Hq, r = o_lat.shape
    dv = w_uv.shape[1]
    if w_uv.shape != (Hq, dv, r):
        raise ValueError("w_uv must be [Hq, d_v, r] for o_lat [B, Hq, r]")
    if out is None:
        out = torch.empty((B, Hq, dv), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, 3, dev)
        if out.shape != (B, Hq, dv):
            raise ValueError("out must be [B, Hq, d_v]")
    _check(lib().attn_mla_apply_uv(_ptr(o_lat), _ptr(w_uv), _ptr(out), B, Hq, r, dv, _stream()))
    return out


def decode_mla(q_nope, q_rope, c_cache, krope_cache, w_uk, w_uv, seq_lens, scale, max_s=None, n_split=0,
               workspace=None):
    """One MLA decode step with both up-projections absorbed: W_UK into the query, the
    latent attention over [c ‖ kr], W_UV on its output. Three launches on the current stream.
    Returns out [B, Hq, d_v] fp32."""
    q_lat = mla_absorb_query(q_nope, w_uk)
    o_lat = decode_mla_absorbed(q_lat, q_rope, c_cache, krope_cache, seq_lens, scale, max_s=max_s,
                                n_split=n_split, workspace=workspace)
    return mla_apply_uv(o_lat, w_uv)


# ----------------------------------------------------------------------------- cache append + RoPE

def _cis(freqs_cis, s_max, w, dev):
    if freqs_cis.dtype == torch.complex64:
        freqs_cis = torch.view_as_real(freqs_cis)
    _need(freqs_cis, "freqs_cis", torch.float32, 3, dev)
    if freqs_cis.shape != (s_max, w // 2, 2):
        raise ValueError(f"freqs_cis must be [S_max={s_max}, {w // 2}, 2] (cos, sin), got {tuple(freqs_cis.shape)}")
    return freqs_cis


def kv_append_rope(q, k_new, v_new, positions, freqs_cis, k_cache, v_cache, q_out=None, new_lens=None):
    """Rotate the new token's q and k at positions[b], write k and v into row positions[b]
    of each sequence's cache. Returns (q_out, new_lens = positions + 1).

    q [B, Hq, D], k_new/v_new [B, Hkv, D], caches [B, S_max, Hkv, D] (all bf16 or all fp32),
    positions [B] int32, freqs_cis [S_max, D/2, 2] fp32 (cos, sin) or [S_max, D/2] complex64.
    """
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bf16 or fp32")
    _need(q, "q", dt, 3)
    dev = q.device
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, name, dt, 3, dev)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, dt, 4, dev)
    _need(positions, "positions", torch.int32, 1, dev)
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    S_max = k_cache.shape[1]
    if (k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape or k_cache.shape != (B, S_max, Hkv, D)
            or v_cache.shape != k_cache.shape or positions.shape[0] != B):
        raise ValueError("inconsistent shapes for q, k_new, v_new, k_cache, v_cache, positions")
    cis = _cis(freqs_cis, S_max, D, dev)
    q_out = torch.empty_like(q) if q_out is None else q_out
    _need(q_out, "q_out", dt, 3, dev)
    new_lens = torch.empty(B, dtype=torch.int32, device=dev) if new_lens is None else new_lens
    _need(new_lens, "new_lens", torch.int32, 1, dev)
    _check(lib().attn_kv_append_rope(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(cis), _ptr(q_out),
                                     _ptr(k_cache), _ptr(v_cache), _ptr(new_lens), B, Hq, Hkv, D, S_max,
                                     ATTN_BF16 if dt == torch.bfloat16 else ATTN_F32, _stream()))
    return q_out, new_lens


def mla_append_rope(q_rope, c_new, kr_new, positions, freqs_cis, c_cache, krope_cache, q_rope_out=None,
                    new_lens=None):
    """MLA decode step's cache write: rotate q_rope and kr_new at positions[b], write kr and
    the unrotated c_new into that row. Returns (q_rope_out, new_lens). All bf16."""
    bf = torch.bfloat16
    _need(q_rope, "q_rope", bf, 3)
    dev = q_rope.device
    _need(c_new, "c_new", bf, 2, dev)
    _need(kr_new, "kr_new", bf, 2, dev)
    _need(c_cache, "c_cache", bf, 3, dev)
    _need(krope_cache, "krope_cache", bf, 3, dev)
    _need(positions, "positions", torch.int32, 1, dev)
    B, Hq, dr = q_rope.shape
    r = c_new.shape[1]
    S_max = c_cache.shape[1]
    if (c_new.shape != (B, r) or kr_new.shape != (B, dr) or c_cache.shape != (B, S_max, r)
            or krope_cache.shape != (B, S_max, dr) or positions.shape[0] != B):
        raise ValueError("inconsistent shapes for q_rope, c_new, kr_new, c_cache, krope_cache, positions")
    cis = _cis(freqs_cis, S_max, dr, dev)
    q_rope_out = torch.empty_like(q_rope) if q_rope_out is None else q_rope_out
    _need(q_rope_out, "q_rope_out", bf, 3, dev)
    new_lens = torch.empty(B, dtype=torch.int32, device=dev) if new_lens is None else new_lens
    _need(new_lens, "new_lens", torch.int32, 1, dev)
    _check(lib().attn_mla_append_rope(_ptr(q_rope), _ptr(c_new), _ptr(kr_new), _ptr(positions), _ptr(cis),
                                      _ptr(q_rope_out), _ptr(c_cache), _ptr(krope_cache), _ptr(new_lens), B, Hq, r,
                                      dr, S_max, _stream()))
    return q_rope_out, new_lens


# ----------------------------------------------------------------------------- prefill

def prefill_gqa_causal(q, k, v, cu_seqlens, max_seqlen, out=None, scale=None):
    """Causal GQA attention of packed sequences over themselves (bf16 in, fp32 out).

    q [T, Hq, D], k/v [T, Hkv, D], cu_seqlens [B+1] int32 on the device, ``max_seqlen`` a
    host-known bound on the lengths. Returns out [T, Hq, D] fp32.
    """
    bf = torch.bfloat16
    _need(q, "q", bf, 3)
    dev = q.device
    _need(k, "k", bf, 3, dev)
    _need(v, "v", bf, 3, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, D) or v.shape != k.shape:
        raise ValueError("inconsistent shapes for q, k, v")
    B = cu_seqlens.shape[0] - 1
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, 3, dev)
    _check(lib().attn_prefill_gqa_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(out),
                                         B, Hq, Hkv, D, scale, int(max_seqlen), T, _stream()))
    return out


# ----------------------------------------------------------------------------- chunked prefill

def prefill_gqa_chunked(q, k_cache, v_cache, cu_q, start_pos, max_kv, out=None, scale=None, n_split=0,
                        workspace=None):
    """New tokens over an existing cache, bottom-right causal: packed row i of sequence b
    attends cache rows 0 .. start_pos[b] + i. q [T, Hq, D], caches [B, S_max, Hkv, D] (fp32 or
    bf16, as q) already holding the chunks, cu_q [B+1] and start_pos [B] int32 on the device,
    ``max_kv`` a host bound on start_pos + chunk length. Returns out [T, Hq, D] fp32."""
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("q must be float32 or bfloat16")
    _need(q, "q", dt, 3)
    dev = q.device
    _need(k_cache, "k_cache", dt, 4, dev)
    _need(v_cache, "v_cache", dt, 4, dev)
    _need(cu_q, "cu_q", torch.int32, 1, dev)
    _need(start_pos, "start_pos", torch.int32, 1, dev)
    T, Hq, D = q.shape
    B, S_max, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or cu_q.shape[0] != B + 1 or start_pos.shape[0] != B:
        raise ValueError("inconsistent shapes for q, k_cache, v_cache, cu_q, start_pos")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = ATTN_F32 if dt == torch.float32 else ATTN_BF16
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, 3, dev)
    if T == 0:
        return out                                   # nothing to attend (an empty tensor has no pointer)
    need = int(lib().attn_prefill_gqa_chunked_workspace_size(B, T, Hq, Hkv, D, int(max_kv), code, n_split))
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_prefill_gqa_chunked(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_q), _ptr(start_pos),
                                          _ptr(out), B, T, Hq, Hkv, D, scale, S_max, int(max_kv), code, n_split,
                                          _ptr(workspace), ws_bytes, _stream()))
    return out


def prefill_mla_chunked(q_lat, q_rope, c_cache, krope_cache, cu_q, start_pos, max_kv, scale, out_lat=None,
                        n_split=0, workspace=None):
    """MLA over an existing latent cache, bottom-right causal: packed row i of sequence b
    attends latent rows 0 .. start_pos[b] + i with key [c ‖ kr] and value c. q_lat [T, Hq, r],
    q_rope [T, Hq, dr], c_cache [B, S_max, r], krope_cache [B, S_max, dr] (bf16), cu_q [B+1],
    start_pos [B] int32. Returns out_lat [T, Hq, r] fp32."""
    bf = torch.bfloat16
    _need(q_lat, "q_lat", bf, 3)
    dev = q_lat.device
    _need(q_rope, "q_rope", bf, 3, dev)
    _need(c_cache, "c_cache", bf, 3, dev)
    _need(krope_cache, "krope_cache", bf, 3, dev)
    _need(cu_q, "cu_q", torch.int32, 1, dev)
    _need(start_pos, "start_pos", torch.int32, 1, dev)
    T, Hq, r = q_lat.shape
    dr = q_rope.shape[2]
    B, S_max, _ = c_cache.shape
    if (q_rope.shape[:2] != (T, Hq) or c_cache.shape != (B, S_max, r) or krope_cache.shape != (B, S_max, dr)
            or cu_q.shape[0] != B + 1 or start_pos.shape[0] != B):
        raise ValueError("inconsistent shapes for q_lat, q_rope, c_cache, krope_cache, cu_q, start_pos")
    if out_lat is None:
        out_lat = torch.empty((T, Hq, r), dtype=torch.float32, device=dev)
    else:
        _need(out_lat, "out_lat", torch.float32, 3, dev)
    if T == 0:
        return out_lat
    need = int(lib().attn_prefill_mla_chunked_workspace_size(B, T, Hq, int(max_kv), n_split))
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_prefill_mla_chunked(_ptr(q_lat), _ptr(q_rope), _ptr(c_cache), _ptr(krope_cache), _ptr(cu_q),
                                          _ptr(start_pos), _ptr(out_lat), B, T, Hq, r, dr, float(scale), S_max,
                                          int(max_kv), n_split, _ptr(workspace), ws_bytes, _stream()))
    return out_lat


# ----------------------------------------------------------------------------- merge

def merge_partials(o_part, lse_part, out=None):
    """out[row] = Σ_i e^{lse_i − M} o_i / Σ_i e^{lse_i − M}; o_part [rows, n, Dv], lse_part [rows, n]."""
    _need(o_part, "o_part", torch.float32, 3)
    dev = o_part.device
    _need(lse_part, "lse_part", torch.float32, 2, dev)
    rows, n, dv = o_part.shape
    if lse_part.shape != (rows, n):
        raise ValueError("lse_part must be [rows, n_split]")
    if out is None:
        out = torch.empty((rows, dv), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, 2, dev)
    _check(lib().attn_merge_partials(_ptr(o_part), _ptr(lse_part), _ptr(out), rows, n, dv, _stream()))
    return out
