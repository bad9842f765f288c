"""Lloyd-Max scalar codebooks (oracle side; test infrastructure).

Restates "TurboQuant KV Cache Compression — Spec", Algorithm Detail, Step 2
(one optimal codebook per (head_dim, bits) for the Beta(d/2, d/2) coordinate
law, boundaries + centroids, levels = 2**bits) and the Codebook Generation
section (centroids are conditional expectations of their cells, boundaries
are midpoints of adjacent centroids, iterate to convergence).

Readings (the pages leave these open or get them wrong):

* Domain.  The spec shifts rotated coordinates to [0, 1].  The codebook is
  kept in the unshifted unit-sphere coordinate y = 2u - 1 in [-1, 1], where
  u ~ Beta(d/2, d/2); a boundary b in u is 2b - 1 in y.  Same decisions.
* Start.  The spec starts from uniform boundaries in [0, 1] and iterates
  about 20 times.  For Beta(64, 64) most uniform cells carry no mass (0/0)
  at 3 and 4 bits, and 20 steps are far from a fixed point, so the iteration
  starts from the law's quantiles and runs until the centroids move by less
  than 1e-15.
* Symmetry.  The law is symmetric about 0, so after every step the centroids
  are made exactly antisymmetric; the middle boundary is then exactly 0.
"""

import numpy as np
from scipy import special


def lloyd_max(mass, moment, init_centroids, lo, hi, tol=1e-15, max_iter=200000):
    """Generic Lloyd iteration on a 1-D law given by its cell integrals.

    ``mass(a, b)`` is P(a < Y < b); ``moment(a, b)`` is E[Y 1{a < Y < b}].
    Returns (centroids, boundaries, iterations).  Boundaries are midpoints of
    adjacent centroids; each centroid becomes its cell's conditional mean.
    """
    c = np.array(init_centroids, dtype=np.float64)
    it = 0
    for it in range(1, max_iter + 1):
        b = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([lo], b, [hi]))
        new = np.array([moment(edges[i], edges[i + 1]) / mass(edges[i], edges[i + 1])
                        for i in range(len(c))])
        new = 0.5 * (new - new[::-1])           # exact antisymmetry
        delta = np.max(np.abs(new - c))
        c = new
        if delta < tol:
            break
    b = 0.5 * (c[:-1] + c[1:])
    return c, b, it


def _beta_pieces(alpha):
    """Cell integrals of y = 2u - 1, u ~ Beta(alpha, alpha), via I_x(a, b)."""
    def cdf_u(a, x):
        return special.betainc(a, alpha, x)

    def mass(ya, yb):
        return cdf_u(alpha, (yb + 1) / 2) - cdf_u(alpha, (ya + 1) / 2)

    def moment_u(ya, yb):
        # E[u 1{cell}] = E[u] * (I(alpha+1, alpha) difference); E[u] = 1/2
        return 0.5 * (cdf_u(alpha + 1, (yb + 1) / 2) - cdf_u(alpha + 1, (ya + 1) / 2))

    def moment(ya, yb):
        return 2.0 * moment_u(ya, yb) - mass(ya, yb)

    def second_u(ya, yb):
        # E[u^2 1{cell}] = E[u^2] * (I(alpha+2, alpha) difference)
        eu2 = alpha * (alpha + 1) / ((2 * alpha) * (2 * alpha + 1))
        return eu2 * (cdf_u(alpha + 2, (yb + 1) / 2) - cdf_u(alpha + 2, (ya + 1) / 2))

    def second(ya, yb):
        # y^2 = 4u^2 - 4u + 1
        return 4 * second_u(ya, yb) - 4 * moment_u(ya, yb) + mass(ya, yb)

    return mass, moment, second


def beta_codebook(d: int = 128, bits: int = 4, tol=1e-15):
    """Lloyd-Max codebook of the Beta(d/2, d/2) coordinate law, in y units.

    Returns (centroids[2**bits], boundaries[2**bits - 1], iterations), float64,
    ascending.  Start: the law's (i + 1/2)/L quantiles.
    """
    alpha = d / 2.0
    levels = 1 << bits
    mass, moment, _ = _beta_pieces(alpha)
    q = (np.arange(levels) + 0.5) / levels
    init = 2.0 * special.betaincinv(alpha, alpha, q) - 1.0
    return lloyd_max(mass, moment, init, -1.0, 1.0, tol=tol)


def gaussian_codebook(bits: int, sigma: float = 1.0, tol=1e-15):
    """Lloyd-Max codebook of N(0, sigma^2) (used only as a pin and for the
    llama.cpp fork's N(0, 1/128) statement in its encode pipeline, step 3)."""
    levels = 1 << bits

    def mass(a, b):
        return special.ndtr(b) - special.ndtr(a)

    def pdf(x):
        return np.exp(-0.5 * x * x) / np.sqrt(2 * np.pi) if np.isfinite(x) else 0.0

    def moment(a, b):
        return pdf(a) - pdf(b)

    q = (np.arange(levels) + 0.5) / levels
    init = special.ndtri(q)
    c, b, it = lloyd_max(mass, moment, init, -np.inf, np.inf, tol=tol)
    return c * sigma, b * sigma, it


def beta_law_moments(centroids, boundaries, alpha):
    """Per-coordinate mean squared error E[(y - Q(y))^2] of a codebook under
    y = 2u - 1, u ~ Beta(alpha, alpha) (closed form via incomplete beta)."""
    mass, moment, second = _beta_pieces(alpha)
    edges = np.concatenate(([-1.0], np.asarray(boundaries, np.float64), [1.0]))
    total = 0.0
    for i, c in enumerate(np.asarray(centroids, np.float64)):
        a, b = edges[i], edges[i + 1]
        total += second(a, b) - 2 * c * moment(a, b) + c * c * mass(a, b)
    return total
