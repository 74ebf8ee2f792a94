"""SFA: sparse absorbed-MLA decode attention over the selected rows.

[GLM] §2.1: sparse flash attention runs only over the rows the indexer
selected. [TS] MLA section: the latent row (512 latent + 64 rope) is stored
once and serves as both K and V. So, for each query head h, over the k
selected rows K_j (576 values each):

    s_j   = scale * sum_{d < 576} q_h[d] * K_j[d]
    m     = max_j s_j,   p_j = exp(s_j - m),   Z = sum_j p_j
    out_h = sum_j p_j * K_j[0:512] / Z
    lse_h = m + ln Z

in float64 from the bf16 inputs; there is no mask (all selected rows are
history). `round_to_bf16_bits` rounds the float64 result once, to nearest
even, for comparison with a bf16 output.
"""
import numpy as np

D_LATENT = 512


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest, ties to even, done in one
    step from the float64 value (no intermediate float32 rounding)."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0) / 256.0          # 8 significant bits, ties to even
    y = np.ldexp(r, e)
    small = np.abs(y) < np.ldexp(1.0, -126)  # below bf16's normal range
    y = np.where(small, 0.0 * np.sign(y), y)
    return (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def sfa_decode(q_bits: np.ndarray, rows_bits: np.ndarray, scale: float):
    """q_bits uint16 [H][576], rows_bits uint16 [k][576] ->
    (out float64 [H][512], lse float64 [H])."""
    q = bf16_bits_to_f64(q_bits)
    K = bf16_bits_to_f64(rows_bits)
    s = scale * (q @ K.T)                       # [H][k]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    Z = p.sum(axis=1, keepdims=True)
    out = (p @ K[:, :D_LATENT]) / Z
    lse = m[:, 0] + np.log(Z[:, 0])
    return out, lse
