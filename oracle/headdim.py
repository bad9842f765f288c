"""The codec at head dims other than 128 (oracle side; test infrastructure).

Restates "TurboQuant KV Cache Compression — Spec":

* Types / Codebook Generation: target dimensions 64, 96, 128 and 160; the
  codebook of dimension d is the Lloyd-Max quantiser of Beta(d/2, d/2)
  (mapped to [-1, 1]), bit widths 2, 3, 4.
* Hadamard Transform Detail: the transform needs d a power of two; for
  other d the page offers padding and truncation, or "a dense random
  orthogonal matrix".
* Algorithm Detail steps 1-3 and As-Built Notes, as for d = 128: normalise
  by the L2 norm, rotate, level index from the boundaries, bit packing.

Readings (where the pages leave a step open):

* The rotation is a dense orthogonal matrix R (d x d) that both sides take as
  an input: y = R x / ||x||, x_hat = n16 R^T c[idx].  Pad-and-truncate is not
  used: with truncation the rotation is no longer orthogonal, so x_hat would
  not reconstruct x and the norm would not be preserved.  For a power of two
  d, R = H_d D / sqrt(d) (Sylvester-Hadamard matrix, random signs D) is one
  such matrix (``hadamard_rotation``); for 96 and 160 any orthogonal matrix
  serves (tests draw one from a seeded QR factorisation).
* Block layout generalised from the 128-element block: [fp16 norm] then the
  codes, 2-bit four per byte, 4-bit two per byte, 3-bit as a 2-bit low plane
  of d / 4 bytes followed by a 1-bit high plane of d / 8 bytes; lowest
  element in the lowest bits.  Block bytes 2 + d * bits / 8 (d a multiple
  of 8).
* Decisions as for d = 128: y in float64, rounded to float32, compared with
  the float32 boundaries; the norm rounded once to fp16 from float64; a zero
  row stores norm 0 and code L/2 everywhere.
"""

import numpy as np

from .codec import fp16_rne, norm_value, quantize
from .rotation import hadamard

HEAD_DIMS = (64, 96, 128, 160)


def block_bytes_d(d: int, bits: int) -> int:
    if d % 8 or d <= 0:
        raise ValueError("d must be a positive multiple of 8")
    if bits not in (2, 3, 4):
        raise ValueError("bits must be 2, 3 or 4")
    return 2 + d * bits // 8


def hadamard_rotation(d: int, signs: np.ndarray) -> np.ndarray:
    """R = H_d D / sqrt(d) for a power of two d (signs: the first d of a
    sign diagonal), float64 [d, d]."""
    s = np.asarray(signs, np.float64)[:d]
    return hadamard(d) * s[None, :] / np.sqrt(d)


def encode_d(x: np.ndarray, R: np.ndarray, boundaries32: np.ndarray):
    """Rows x [N, d] -> (codes uint8 [N, d], norm16 uint16 [N], y float64 [N, d]),
    y = R x / ||x||."""
    x = np.asarray(x, np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1))
    w = x @ np.asarray(R, np.float64).T
    safe = np.where(n > 0, n, 1.0)
    y = np.where(n[:, None] > 0, w / safe[:, None], 0.0)
    return quantize(y, boundaries32), fp16_rne(n), y


def decode_d(idx: np.ndarray, norm16: np.ndarray, centroids: np.ndarray, R: np.ndarray) -> np.ndarray:
    """x_hat = n16 R^T c[idx] ([N, d] float64)."""
    c = np.asarray(centroids, np.float64)[np.asarray(idx, np.int64)]
    return (norm_value(norm16)[:, None] * c) @ np.asarray(R, np.float64)


def pack_d(idx: np.ndarray, norm16: np.ndarray, bits: int) -> np.ndarray:
    """Codes [N, d] and fp16 norm bits [N] -> blocks [N, block_bytes_d]."""
    idx = np.asarray(idx, np.uint8)
    n, d = idx.shape
    out = np.zeros((n, block_bytes_d(d, bits)), np.uint8)
    nb = np.asarray(norm16, np.uint16)
    out[:, 0] = nb & 0xFF
    out[:, 1] = nb >> 8
    for j in range(d):
        v = idx[:, j]
        if bits == 2:
            out[:, 2 + j // 4] |= (v & 3) << (2 * (j % 4))
        elif bits == 4:
            out[:, 2 + j // 2] |= (v & 15) << (4 * (j % 2))
        else:
            out[:, 2 + j // 4] |= (v & 3) << (2 * (j % 4))
            out[:, 2 + d // 4 + j // 8] |= ((v >> 2) & 1) << (j % 8)
    return out


def unpack_d(blocks: np.ndarray, d: int, bits: int):
    """Inverse of pack_d: -> (codes [N, d] uint8, norm16 [N])."""
    b = np.asarray(blocks, np.uint8)
    norm16 = b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8)
    idx = np.zeros((b.shape[0], d), np.uint8)
    for j in range(d):
        if bits == 2:
            idx[:, j] = (b[:, 2 + j // 4] >> (2 * (j % 4))) & 3
        elif bits == 4:
            idx[:, j] = (b[:, 2 + j // 2] >> (4 * (j % 2))) & 15
        else:
            lo = (b[:, 2 + j // 4] >> (2 * (j % 4))) & 3
            hi = (b[:, 2 + d // 4 + j // 8] >> (j % 8)) & 1
            idx[:, j] = lo | (hi << 2)
    return idx, norm16
