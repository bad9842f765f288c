"""Pins of the oracle's codec at head dims 64, 96 and 160 (oracle.headdim).

Each check ties the oracle to something other than itself: scipy's Hadamard
matrix and numerical integration of the Beta density, the already pinned
d = 128 codec, exhaustive pack / unpack identities, norm preservation of an
orthogonal rotation, and the distortion the Lloyd-Max codebook predicts."""

import numpy as np
import pytest
from scipy import integrate, linalg, stats

import oracle
from oracle import codec, headdim
from turboquant_bit_kv_gb300 import workloads


def _orthogonal(d, seed):
    """A seeded random orthogonal matrix (QR of a Gaussian matrix, signs fixed)."""
    a = np.random.default_rng(seed).standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))[None, :]


def _rows(n, d, seed):
    return np.random.default_rng(seed).standard_normal((n, d))


def test_hadamard_rotation_is_scipy_hadamard_with_signs():
    s = oracle.sign_diagonal(workloads.SIGN_SEED)
    for d in (64, 128):
        R = headdim.hadamard_rotation(d, s)
        ref = linalg.hadamard(d) * s[:d][None, :] / np.sqrt(d)
        assert np.array_equal(R, ref)
        assert np.allclose(R @ R.T, np.eye(d), atol=1e-12)


def test_d128_reduces_to_the_pinned_codec():
    """With R = H D / sqrt(128) the general-d encode is the d = 128 codec."""
    s = oracle.sign_diagonal(workloads.SIGN_SEED)
    R = headdim.hadamard_rotation(128, s)
    x = _rows(300, 128, 1)
    for bits in (2, 3, 4):
        c, b64, _ = oracle.beta_codebook(128, bits)
        b32 = b64.astype(np.float32)
        i1, n1, y1 = codec.encode(x, s, b32)
        i2, n2, y2 = headdim.encode_d(x, R, b32)
        assert np.array_equal(n1, n2)
        # codes agree except where float64 sums of a different order straddle a boundary
        close = np.abs(y1 - y2) > 0
        assert np.array_equal(i1[~close], i2[~close])
        assert np.mean(i1 != i2) < 1e-4
        assert np.array_equal(headdim.pack_d(i1, n1, bits), codec.pack_block(i1, n1, bits))


@pytest.mark.parametrize("d", headdim.HEAD_DIMS)
@pytest.mark.parametrize("bits", (2, 3, 4))
def test_pack_unpack_identity(d, bits):
    rng = np.random.default_rng(d * 10 + bits)
    idx = rng.integers(0, 1 << bits, (64, d)).astype(np.uint8)
    n16 = rng.integers(0, 1 << 16, 64).astype(np.uint16)
    blk = headdim.pack_d(idx, n16, bits)
    assert blk.shape == (64, 2 + d * bits // 8)
    i2, n2 = headdim.unpack_d(blk, d, bits)
    assert np.array_equal(i2, idx) and np.array_equal(n2, n16)
    # every code bit lands in exactly one block bit: a single set code bit sets a single block bit
    one = np.zeros((1, d), np.uint8)
    one[0, d - 1] = 1 << (bits - 1)
    assert np.unpackbits(headdim.pack_d(one, np.zeros(1, np.uint16), bits)).sum() == 1


@pytest.mark.parametrize("d", headdim.HEAD_DIMS)
@pytest.mark.parametrize("bits", (2, 3, 4))
def test_code_bytes_are_the_pages_packed_size(d, bits):
    """The spec's Memory Layout gives ceil(head_dim * bits / 8) packed bytes per
    head; a block adds the fp16 norm."""
    assert headdim.block_bytes_d(d, bits) - 2 == -(-(d * bits) // 8)


@pytest.mark.parametrize("d", (64, 96, 160))
@pytest.mark.parametrize("bits", (2, 4))
def test_codebook_is_the_beta_lloyd_max_fixed_point(d, bits):
    """Centroids are the conditional means of Beta(d/2, d/2) on [-1, 1] between
    the boundaries, and boundaries the midpoints (scipy quadrature)."""
    c, b, _ = oracle.beta_codebook(d, bits)
    law = stats.beta(d / 2, d / 2, loc=-1, scale=2)
    edges = np.concatenate([[-1.0], b, [1.0]])
    for i in range(len(c)):
        m0 = integrate.quad(law.pdf, edges[i], edges[i + 1], epsabs=1e-14)[0]
        m1 = integrate.quad(lambda y: y * law.pdf(y), edges[i], edges[i + 1], epsabs=1e-14)[0]
        assert abs(m1 / m0 - c[i]) < 1e-9
    assert np.allclose(b, 0.5 * (c[1:] + c[:-1]), atol=1e-12)


@pytest.mark.parametrize("d", (64, 96, 160))
def test_orthogonal_rotation_preserves_the_norm(d):
    """||x_hat|| = n16 ||c[idx]|| for any orthogonal R (a transposed or
    non-orthogonal rotation would break it), and x_hat lies near x."""
    R = _orthogonal(d, d) if d != 64 else headdim.hadamard_rotation(64, oracle.sign_diagonal(workloads.SIGN_SEED))
    x = _rows(500, d, d + 1)
    c, b64, _ = oracle.beta_codebook(d, 4)
    idx, n16, _ = headdim.encode_d(x, R, b64.astype(np.float32))
    xh = headdim.decode_d(idx, n16, c, R)
    lhs = np.linalg.norm(xh, axis=1)
    rhs = codec.norm_value(n16) * np.linalg.norm(c[idx], axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-12)
    cos = np.sum(xh * x, axis=1) / (np.linalg.norm(xh, axis=1) * np.linalg.norm(x, axis=1))
    assert np.min(cos) > 0.97   # 4-bit: about 0.995 on average


@pytest.mark.parametrize("d", (64, 96, 160))
@pytest.mark.parametrize("bits", (2, 3, 4))
def test_distortion_matches_the_codebook(d, bits):
    """Mean squared error per coordinate of y against the codebook's predicted
    distortion under its own law (the coordinates of R x / ||x|| follow
    Beta((d-1)/2, (d-1)/2), close to the Beta(d/2, d/2) the page fixes)."""
    R = _orthogonal(d, 3 * d)
    x = _rows(4000, d, 2 * d)
    c, b, _ = oracle.beta_codebook(d, bits)
    idx, n16, y = headdim.encode_d(x, R, b.astype(np.float32))
    mse = np.mean((y - c[idx]) ** 2)
    law = stats.beta(d / 2, d / 2, loc=-1, scale=2)
    edges = np.concatenate([[-1.0], b, [1.0]])
    pred = sum(integrate.quad(lambda t, ci=ci: (t - ci) ** 2 * law.pdf(t), lo, hi)[0]
               for ci, lo, hi in zip(c, edges[:-1], edges[1:]))
    assert abs(mse / pred - 1) < 0.08


def test_zero_row():
    d = 96
    R = _orthogonal(d, 5)
    c, b64, _ = oracle.beta_codebook(d, 3)
    idx, n16, _ = headdim.encode_d(np.zeros((2, d)), R, b64.astype(np.float32))
    assert np.all(n16 == 0) and np.all(idx == 4)
    assert np.all(headdim.decode_d(idx, n16, c, R) == 0)
