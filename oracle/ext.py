"""Further block formats of the TurboQuant family (oracle side; test
infrastructure): the norm-corrected encode, the dense 8-in-3 packing of
3-bit codes, and the 8-bit turboq8 codec.

Restates:

* "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", section 4, Encode
  pipeline step 4 (corrected norm): the L2 norm of the reconstructed
  centroids, recon_norm, is computed and grp_norm / recon_norm is stored as
  the block norm, pre-compensating for the codebook's approximation error;
  "lmcache.v1.distributed.serde.turboquant", Configuration (the `_nc` presets
  enable norm correction).
* "TurboQuant KV Cache Compression — Spec", Algorithm Detail Step 3: 3-bit
  codes may be packed eight values into three bytes, with no waste.
* "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", At a glance and the
  turboq8 paragraph: the FWHT rotation followed by a uniform 256-level grid,
  centroid[i] = (i - 127.5) / 127.5, with a per-block absmax scale; 8.125
  bits per weight, 130-byte blocks.

Readings (where the pages leave a step open):

* Norm correction: recon_norm = ||c[idx]||_2 over the block's 128 codes, in
  the rotated domain (the rotation is orthogonal, so it is also the norm of
  the reconstruction before scaling); the stored fp16 norm is
  fp16(||x|| / recon_norm), rounded once from float64.  The codes are those
  of the plain encode (the correction changes only the stored norm), and
  decoding is unchanged: x_hat = n16 * R^T c[idx], so ||x_hat|| = ||x|| up to
  the fp16 rounding of the norm.  A zero row stores 0.
* 8-in-3 packing: the codes of elements 8g .. 8g + 7 form the 24-bit
  little-endian word at bytes 2 + 3g .. 2 + 3g + 2, element 8g + p in bits
  3p .. 3p + 2; the fp16 norm stays in bytes 0..1 (50-byte blocks, as the
  split-plane 3-bit block).
* turboq8: u = R x = H (D x) / sqrt(128) (not normalised); a = max_j |u_j|;
  the stored scale is fp16(a) (rounded once from float64); code
  i_j = floor(127.5 (u_j / a + 1) + 1/2) clamped to [0, 255], the nearest
  level (ties to the upper one), the decision taken in float32 like the
  other codecs' (u_j / a rounded to float32 first); a zero row stores scale
  0 and code 128 everywhere.  Decode: x_hat = R^T (s16 (i - 127.5) / 127.5).
  Block: [fp16 scale][128 code bytes], element j at byte 2 + j.
"""

import numpy as np

from .codec import D, encode, fp16_rne, norm_value, quantize
from .rotation import rotate, rotate_inverse


def recon_norm(idx: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """||c[idx]||_2 of each row of codes [N, 128] (float64)."""
    c = np.asarray(centroids, np.float64)[np.asarray(idx, np.int64)]
    return np.sqrt(np.sum(c * c, axis=-1))


def encode_nc(x: np.ndarray, signs: np.ndarray, centroids: np.ndarray, boundaries32: np.ndarray):
    """Norm-corrected encode: the plain encode's codes, stored norm
    fp16(||x|| / ||c[idx]||).  Returns (idx, norm16, y, corrected norm float64)."""
    x = np.asarray(x, np.float64)
    idx, _, y = encode(x, signs, boundaries32)
    n = np.sqrt(np.sum(x * x, axis=-1))
    r = recon_norm(idx, centroids)
    v = np.where(n > 0, n / np.where(r > 0, r, 1.0), 0.0)
    return idx, fp16_rne(v), y, v


def pack_dense3(idx: np.ndarray, norm16: np.ndarray) -> np.ndarray:
    """3-bit codes [N, 128] and fp16 norm bits [N] -> 50-byte blocks, eight
    codes per three bytes."""
    idx = np.asarray(idx, np.uint32)
    n = idx.shape[0]
    out = np.zeros((n, 50), np.uint8)
    nb = np.asarray(norm16, np.uint16)
    out[:, 0] = nb & 0xFF
    out[:, 1] = nb >> 8
    for g in range(16):
        word = np.zeros(n, np.uint32)
        for p in range(8):
            word |= (idx[:, 8 * g + p] & 7) << (3 * p)
        for k in range(3):
            out[:, 2 + 3 * g + k] = (word >> (8 * k)) & 0xFF
    return out


def unpack_dense3(blocks: np.ndarray):
    """Inverse of pack_dense3: -> (idx [N, 128] uint8, norm16 [N])."""
    b = np.asarray(blocks, np.uint8)
    norm16 = b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8)
    idx = np.zeros((b.shape[0], D), np.uint8)
    for g in range(16):
        word = (b[:, 2 + 3 * g].astype(np.uint32) | (b[:, 3 + 3 * g].astype(np.uint32) << 8) |
                (b[:, 4 + 3 * g].astype(np.uint32) << 16))
        for p in range(8):
            idx[:, 8 * g + p] = (word >> (3 * p)) & 7
    return idx, norm16


Q8_BLOCK = 130


def q8_levels() -> np.ndarray:
    """The 256 turboq8 levels (i - 127.5) / 127.5 (float64)."""
    return (np.arange(256, dtype=np.float64) - 127.5) / 127.5


def encode_q8(x: np.ndarray, signs: np.ndarray):
    """turboq8 encode of rows x [N, 128]: (codes uint8 [N, 128], scale16
    uint16 [N], t float64 [N, 128]) with t = 127.5 (u / a + 1), the code
    coordinate whose distance to a half-integer measures how close a
    decision was."""
    x = np.asarray(x, np.float64)
    u = rotate(x, signs)
    a = np.max(np.abs(u), axis=-1)
    safe = np.where(a > 0, a, 1.0)
    y = np.where(a[..., None] > 0, u / safe[..., None], 0.0)
    y32 = y.astype(np.float32).astype(np.float64)
    t = 127.5 * (y32 + 1.0)
    idx = np.clip(np.floor(t + 0.5), 0, 255).astype(np.uint8)
    return idx, fp16_rne(a), t


def decode_q8(idx: np.ndarray, scale16: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x_hat = R^T (s16 * (i - 127.5) / 127.5) ([N, 128] float64)."""
    lv = q8_levels()[np.asarray(idx, np.int64)]
    return rotate_inverse(norm_value(scale16)[:, None] * lv, signs)


def pack_q8(idx: np.ndarray, scale16: np.ndarray) -> np.ndarray:
    idx = np.asarray(idx, np.uint8)
    out = np.zeros((idx.shape[0], Q8_BLOCK), np.uint8)
    s = np.asarray(scale16, np.uint16)
    out[:, 0] = s & 0xFF
    out[:, 1] = s >> 8
    out[:, 2:] = idx
    return out


def unpack_q8(blocks: np.ndarray):
    b = np.asarray(blocks, np.uint8)
    return b[:, 2:].copy(), b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8)
