"""Per-element error bounds of the MLA product path, derived from its arithmetic (shared by
the MLA parity tests; plain NumPy on the host).

  - q_lat = W_UKᵀ·q_nope from bf16 inputs: fp32 sums of d_nope products, then one bf16
    rounding, so |got − x| ≤ 2^-8·(|x| + γ) + γ with γ = d_nope·2^-24·Σ_n |q_n·w_n|.
  - the latent output against the decompress-then-attend oracle: the rounded q_lat moves
    each score by at most δ = scale·Σ_r |q_lat_r − x_r|·|c_r|, which moves the softmax
    average of the c rows by at most (e^{2δ} − 1)·max|c|; the decode itself adds its bf16
    tolerance; W_UV maps a latent error e to at most e·Σ_r |W_UV[h, v, r]| per output.
"""

import numpy as np

from workloads import to_f64

U_BF16 = 2.0 ** -8
U_F32 = 2.0 ** -24
DECODE_TOL = 3e-3      # the absorbed decode against the oracle on the same bf16 q_lat


def absorb_bound(qn, wuk, ref):
    """Bound on |q_lat − x| for q_lat formed in fp32 and rounded to bf16 (fp64 arrays)."""
    mag = np.einsum("hnr,bhn->bhr", np.abs(wuk), np.abs(qn))
    gamma = qn.shape[2] * U_F32 * mag
    return U_BF16 * (np.abs(ref) + gamma) + gamma + 1e-30


def full_step_tolerance(inp, scale, oracle):
    """Per-(b, h, v) bound on W_UV·(latent decode output) against the oracle's
    decompress-then-attend MLA, for a q_lat formed in fp32 and rounded to bf16."""
    q64, w64 = to_f64(inp["q_nope"]), to_f64(inp["w_uk"])
    x = oracle.absorb_query(q64, w64)                               # exact q_lat, [B,H,r]
    dq = absorb_bound(q64, w64, x)                                  # bound on |q_lat − x|
    c = to_f64(inp["c_cache"])                                      # [B,S,r]
    lens = inp["seq_lens"].cpu().numpy()
    B, H, r = x.shape
    wsum = np.abs(to_f64(inp["w_uv"])).sum(2)                       # [H, dv]
    tol = np.zeros((B, H, wsum.shape[1]))
    for b in range(B):
        s = int(lens[b])
        if s == 0:
            continue
        cb = np.abs(c[b, :s])                                       # [s, r]
        delta = scale * (cb @ dq[b].T).max(0)                       # [H]
        olat_tol = np.expm1(2 * delta) * cb.max() + DECODE_TOL      # [H]
        tol[b] = olat_tol[:, None] * wsum[None, :]
    return tol
