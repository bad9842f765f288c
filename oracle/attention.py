"""Decode attention over a packed cache (oracle side; test infrastructure).

``attention_dequantized`` is the plain definition: dequantise every cached key
and value ("TurboQuant KV Cache Compression — Spec", Quantize / Dequantize and
Attention with TurboQuant cache: dequantise the cached K, V, then standard
attention), score s_t = scale * <q, k_hat_t> (+ the QJL correction of
"RotorQuant KV Cache Compression", Fused Kernel Logic, when given), softmax
with max subtraction, o = sum_t p_t v_hat_t; all in float64.

``attention_rotated`` restates the spec's "Optimization: Fused dequant-dot":
rotate q once, score against n_t * c[idx] in the rotated domain, accumulate
values there, rotate the output back once.  It is exactly equal to the plain
definition (R is orthogonal) and exists only so tests can check that identity.

Readings: grouped-query heads map query head h to KV head h // G with
G = Hq / Hkv (contiguous groups); a per-sequence length L_b means tokens
[0, L_b) of that sequence are attended.
"""

import numpy as np

from .codec import decode, decode_rotated
from .rotation import rotate, rotate_inverse


def _softmax_weights(s):
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_dequantized(q, k_hat, v_hat, scale, seq_lens=None, term2=None):
    """Plain attention over dequantised caches.

    q [B, Hq, 128]; k_hat, v_hat [B, Hkv, T, 128] (float64 reconstructions);
    term2 optional [B, Hq, T] additive key-score correction (before scale).
    Returns o [B, Hq, 128] float64.
    """
    q = np.asarray(q, np.float64)
    B, Hq, d = q.shape
    Hkv, T = k_hat.shape[1], k_hat.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = T if seq_lens is None else int(seq_lens[b])
        for h in range(Hq):
            kv = h // G
            s = k_hat[b, kv, :L] @ q[b, h]
            if term2 is not None:
                s = s + term2[b, h, :L]
            p = _softmax_weights(scale * s)
            out[b, h] = p @ v_hat[b, kv, :L]
    return out


def dequantize_cache(idx, norm16, centroids, signs):
    """Cache codes [B, Hkv, T, 128] + norms [B, Hkv, T] -> float64 [B,Hkv,T,128]."""
    B, H, T, d = idx.shape
    flat = decode(idx.reshape(-1, d), norm16.reshape(-1), centroids, signs)
    return flat.reshape(B, H, T, d)


def attention_rotated(q, k_idx, k_norm16, kc, v_idx, v_norm16, vc, signs, scale,
                      seq_lens=None):
    """Fused dequant-dot form of the same attention (identity check only)."""
    q = np.asarray(q, np.float64)
    B, Hq, d = q.shape
    Hkv, T = k_idx.shape[1], k_idx.shape[2]
    G = Hq // Hkv
    q_rot = rotate(q.reshape(-1, d), signs).reshape(B, Hq, d)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = T if seq_lens is None else int(seq_lens[b])
        for h in range(Hq):
            kv = h // G
            kr = decode_rotated(k_idx[b, kv, :L], k_norm16[b, kv, :L], kc)
            vr = decode_rotated(v_idx[b, kv, :L], v_norm16[b, kv, :L], vc)
            p = _softmax_weights(scale * (kr @ q_rot[b, h]))
            out[b, h] = rotate_inverse((p @ vr)[None, :], signs)[0]
    return out


def attention_causal(q, k_hat, v_hat, scale, seq_lens=None):
    """Attention of several new query tokens per sequence over the cache
    that already holds them (a prefill chunk, or the draft tokens of a
    speculative verify step): the plain definition above with a causal mask.

    The fork page's section 2 (Requirements) routes every quantised-KV
    attention through the fused flash-attention path, prefill included; the
    spec's Integration Points write each new token into the cache before the
    attention over it.  Reading: the M query tokens of sequence b are the
    last M tokens of its L_b cached ones, so query token i sits at position
    p = L_b - M + i and attends to the keys at positions 0..p (p + 1 keys);
    a query whose position is negative (L_b < M) attends to nothing and its
    output is zero.

    q [B, M, Hq, 128]; k_hat, v_hat [B, Hkv, T, 128] float64; seq_lens [B]
    (None: T).  Returns o [B, M, Hq, 128] float64.
    """
    q = np.asarray(q, np.float64)
    B, M, Hq, d = q.shape
    Hkv, T = k_hat.shape[1], k_hat.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, M, Hq, d))
    for b in range(B):
        L = T if seq_lens is None else int(seq_lens[b])
        for i in range(M):
            p = L - M + i
            if p < 0:
                continue
            for h in range(Hq):
                kv = h // G
                s = k_hat[b, kv, :p + 1] @ q[b, i, h]
                out[b, i, h] = _softmax_weights(scale * s) @ v_hat[b, kv, :p + 1]
    return out
