"""QJL two-term key score (oracle side; test infrastructure).

Restates "RotorQuant KV Cache Compression": The QJL Estimator Formula
(<q,k> ~ <q,k_mse> + ||r|| sqrt(pi/2)/m <S q, sign(S r)>), Implementation
Requirements 1-2 (store sign(S r) and ||r|| per key; k_mse is the
dequantised MSE key, r = k - k_mse) and 4 (score = (term1 + term2) * scale).

Readings: S is a Gaussian [m, 128] matrix with m = 128 (an input, seeded);
sign(0) = +1; the sign bits are stored one per dimension, 16 bytes per key,
bit j at byte j // 8, position j % 8, set when (S r)_j >= 0 (the page's
"packed bits ... as int8" is self-contradictory, so bits are packed); the
residual norm is stored as fp16 (round to nearest even from float64); k_mse
uses the fp16-rounded key norm, exactly as the dequantiser does; the
sign decision is taken in float32 (the value is rounded to float32 first).
"""

import numpy as np

from .codec import decode, fp16_rne, norm_value


def qjl_encode(k, k_idx, k_norm16, centroids, signs, S):
    """Returns (bits uint8 [N,16], rn16 uint16 [N], proj float64 [N,m])."""
    k = np.asarray(k, np.float64)
    k_mse = decode(k_idx, k_norm16, centroids, signs)
    r = k - k_mse
    rn16 = fp16_rne(np.sqrt(np.sum(r * r, axis=-1)))
    proj = r @ np.asarray(S, np.float64).T
    pos = proj.astype(np.float32) >= 0
    m = proj.shape[1]
    bits = np.zeros((k.shape[0], m // 8), np.uint8)
    for j in range(m):
        bits[:, j // 8] |= (pos[:, j].astype(np.uint8) << (j % 8))
    return bits, rn16, proj


def unpack_signs(bits, m=128):
    """Sign bits [..., m//8] -> +1/-1 float64 [..., m]."""
    bits = np.asarray(bits, np.uint8)
    out = np.empty(bits.shape[:-1] + (m,))
    for j in range(m):
        out[..., j] = np.where((bits[..., j // 8] >> (j % 8)) & 1, 1.0, -1.0)
    return out


def qjl_term2(q, bits, rn16, S):
    """term2_t = rn_t * sqrt(pi/2)/m * sum_j (S q)_j * sign_tj.

    q [128]; bits [T, m//8]; rn16 [T]; returns [T] float64 (before scale).
    """
    S = np.asarray(S, np.float64)
    m = S.shape[0]
    sq = S @ np.asarray(q, np.float64)
    return norm_value(rn16) * np.sqrt(np.pi / 2) / m * (unpack_signs(bits, m) @ sq)
