"""Randomized Hadamard rotation (oracle side; test infrastructure).

Restates "TurboQuant KV Cache Compression — Spec": Algorithm Detail, Step 1
(a fixed random orthogonal rotation built from a Walsh-Hadamard matrix H and a
diagonal D of random signs), As-Built Notes (signs applied before the
transform: H (D x)), and Hadamard Transform Detail (scale 1/sqrt(d)).

The oracle writes the definition out: H is the d x d Sylvester-Hadamard
matrix, H[i, j] = (-1)^popcount(i & j), applied as a dense float64 product.

Reading: R x = H (D x) / sqrt(d).  The page calls the inverse "the same
operation", which holds only with the factors reversed: R^-1 = R^T =
D H / sqrt(d) (H is symmetric and H H = d I, D D = I).
"""

import functools

import numpy as np


@functools.lru_cache(maxsize=None)
def _hadamard(d: int) -> np.ndarray:
    i = np.arange(d)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    h = np.where(pc % 2 == 0, 1.0, -1.0)
    h.setflags(write=False)
    return h


def hadamard(d: int = 128) -> np.ndarray:
    """Sylvester-Hadamard matrix of order d (d a power of two), float64."""
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    return _hadamard(d)


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R x = H (D x) / sqrt(d) for each row of x ([..., d])."""
    d = x.shape[-1]
    return (np.asarray(x, np.float64) * signs) @ hadamard(d).T / np.sqrt(d)


def rotate_inverse(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R^T y = D (H y) / sqrt(d) for each row of y ([..., d])."""
    d = y.shape[-1]
    return (np.asarray(y, np.float64) @ hadamard(d).T / np.sqrt(d)) * signs
