"""Quantise-on-insert, bit packing and dequantisation (oracle side; test
infrastructure).

Restates:

* "TurboQuant KV Cache Compression — Spec": As-Built Notes (signs before the
  Hadamard transform; normalise by the vector's L2 norm), Algorithm Detail
  Step 2 (binary search of boundaries[] gives the level index; centroids[]
  gives the reconstruction value) and Step 3 (bit packing), Overview
  (dequantise = look up centroids, rotate back).
* "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", section 4, Block
  structures: 128-element blocks, an fp16 norm in the first two bytes, 2-bit
  codes four per byte, 3-bit codes as a 2-bit low plane plus a 1-bit high
  plane eight per byte, 4-bit codes nibble-packed.

Readings:

* Block bytes are 2 + 16*bits: 34 (2-bit), 50 (3-bit), 66 (4-bit).  The
  fork's 4-bit block is 68 bytes because it also stores an rnorm that only
  its legacy QJL mode uses; this codec has no rnorm.
* Within a byte, the lowest-numbered element sits in the lowest bits.
* The level index of y is the number of boundaries b_i with b_i <= y (an
  exact tie goes to the upper cell), in ascending level order.
* The index decision is taken in float32, the precision of the pages'
  tables and vectors: y is computed in float64, rounded to float32 and
  compared with the float32 boundary table.
* A zero vector has n = 0; its y is taken as 0 (every index is L/2) and its
  stored norm is 0, so it decodes to exactly 0.
* The norm is stored as IEEE fp16, rounded to nearest-even directly from the
  float64 norm (no float32 step).
"""

import numpy as np

from .rotation import rotate, rotate_inverse

D = 128


def block_bytes(bits: int) -> int:
    """Bytes of one 128-element block: fp16 norm + 128*bits/8 code bytes."""
    if bits not in (2, 3, 4):
        raise ValueError("bits must be 2, 3 or 4")
    return 2 + (D * bits) // 8


def fp16_rne(x) -> np.ndarray:
    """float64 -> IEEE binary16 bit patterns (uint16), round to nearest even."""
    with np.errstate(over="ignore"):       # overflow to +inf is the IEEE result
        return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def quantize(y: np.ndarray, boundaries32: np.ndarray) -> np.ndarray:
    """Level index #{i : b_i <= y}, decided in float32 (see module notes)."""
    y32 = np.asarray(y, np.float64).astype(np.float32)
    b32 = np.asarray(boundaries32, np.float32)
    return np.searchsorted(b32, y32, side="right").astype(np.uint8)


def encode(x: np.ndarray, signs: np.ndarray, boundaries32: np.ndarray):
    """Encode rows of x ([N, 128], exact input values) into codes and norms.

    n = ||x||_2;  y = H (D x) / (sqrt(d) n);  idx = quantize(y);
    norm16 = fp16(n).  Returns (idx uint8 [N,128], norm16 uint16 [N],
    y float64 [N,128]); y is returned so that tests can measure how close a
    coordinate lies to a boundary.
    """
    x = np.asarray(x, np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1))
    w = rotate(x, signs)
    safe = np.where(n > 0, n, 1.0)
    y = np.where(n[..., None] > 0, w / safe[..., None], 0.0)
    return quantize(y, boundaries32), fp16_rne(n), y


def pack_block(idx: np.ndarray, norm16: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes [N,128] and fp16 norm bits [N] into blocks [N, block_bytes]."""
    idx = np.asarray(idx, np.uint8)
    n = idx.shape[0]
    out = np.zeros((n, block_bytes(bits)), np.uint8)
    nb = np.asarray(norm16, np.uint16)
    out[:, 0] = nb & 0xFF
    out[:, 1] = nb >> 8
    for j in range(D):
        v = idx[:, j].astype(np.uint8)
        if bits == 2:
            out[:, 2 + j // 4] |= (v & 3) << (2 * (j % 4))
        elif bits == 4:
            out[:, 2 + j // 2] |= (v & 15) << (4 * (j % 2))
        else:
            out[:, 2 + j // 4] |= (v & 3) << (2 * (j % 4))
            out[:, 34 + j // 8] |= ((v >> 2) & 1) << (j % 8)
    return out


def unpack_block(blocks: np.ndarray, bits: int):
    """Inverse of pack_block: blocks [N, block_bytes] -> (idx [N,128], norm16 [N])."""
    blocks = np.asarray(blocks, np.uint8)
    norm16 = blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8)
    idx = np.zeros((blocks.shape[0], D), np.uint8)
    for j in range(D):
        if bits == 2:
            idx[:, j] = (blocks[:, 2 + j // 4] >> (2 * (j % 4))) & 3
        elif bits == 4:
            idx[:, j] = (blocks[:, 2 + j // 2] >> (4 * (j % 2))) & 15
        else:
            lo = (blocks[:, 2 + j // 4] >> (2 * (j % 4))) & 3
            hi = (blocks[:, 34 + j // 8] >> (j % 8)) & 1
            idx[:, j] = lo | (hi << 2)
    return idx, norm16


def norm_value(norm16: np.ndarray) -> np.ndarray:
    """fp16 bit patterns -> float64 values."""
    return np.asarray(norm16, np.uint16).view(np.float16).astype(np.float64)


def decode_rotated(idx: np.ndarray, norm16: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """Rotated-domain reconstruction n16 * c[idx] ([N,128] float64)."""
    c = np.asarray(centroids, np.float64)
    return norm_value(norm16)[:, None] * c[np.asarray(idx, np.int64)]


def decode(idx: np.ndarray, norm16: np.ndarray, centroids: np.ndarray,
           signs: np.ndarray) -> np.ndarray:
    """x_hat = n16 * R^T c[idx] ([N,128] float64)."""
    return rotate_inverse(decode_rotated(idx, norm16, centroids), signs)
