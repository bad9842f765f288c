"""Pins of the CPU oracle against values fixed outside it: published test
vectors, textbook tables, library routines, closed forms, invariants and
brute force.  CPU only."""

import os

import numpy as np
import pytest
import scipy.linalg
import scipy.stats
from scipy import integrate

import oracle
from oracle import codec, qjl
from turboquant_bit_kv_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


@pytest.fixture(scope="module")
def books():
    out = {}
    for b in (2, 3, 4):
        c, bd, _ = oracle.beta_codebook(D, b)
        out[b] = (c, bd)
    return out


# ---------------------------------------------------------------- signs

def test_splitmix64_published_vectors():
    want = [int(x, 16) for x in _golden_lines("splitmix64_seed0.txt")]
    assert oracle.splitmix64(0, 3) == want


def test_sign_diagonal_deterministic_and_balanced():
    s1 = oracle.sign_diagonal(1)
    assert np.array_equal(s1, oracle.sign_diagonal(1))
    assert not np.array_equal(s1, oracle.sign_diagonal(2))
    assert set(np.unique(s1)) <= {-1.0, 1.0}
    assert 30 < np.sum(s1 < 0) < 98


# ---------------------------------------------------------------- rotation

def test_hadamard_matches_scipy():
    for d in (2, 8, 64, 128):
        assert np.array_equal(oracle.hadamard(d), scipy.linalg.hadamard(d).astype(float))


def test_hadamard_closed_form():
    H = oracle.hadamard(D)
    assert np.array_equal(H @ H, D * np.eye(D))


def test_rotation_orthogonal_and_inverse():
    rng = np.random.default_rng(5)
    s = oracle.sign_diagonal(1)
    x = rng.standard_normal((64, D))
    y = oracle.rotate(x, s)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    assert np.max(np.abs(oracle.rotate_inverse(y, s) - x)) < 1e-12
    R = oracle.rotate(np.eye(D), s).T            # columns are R e_j
    assert np.max(np.abs(R @ R.T - np.eye(D))) < 1e-12
    assert np.max(np.abs(R.T @ R - np.eye(D))) < 1e-12
    Hn = oracle.hadamard(D) / np.sqrt(D)          # the unsigned transform is self-inverse
    assert np.max(np.abs(Hn @ Hn - np.eye(D))) < 1e-12
    # R e_1 = D_11 * H e_1 / sqrt(d): every entry has magnitude 1/sqrt(d)
    assert np.allclose(np.abs(R[:, 0]), 1 / np.sqrt(D), rtol=0, atol=1e-15)


def test_rotation_sign_order_is_signs_first():
    # H (D x) differs from D (H x) for a generic x; the as-built order applies
    # the signs to x before the transform.
    s = oracle.sign_diagonal(1)
    x = np.arange(D, dtype=float)
    H = oracle.hadamard(D)
    assert np.allclose(oracle.rotate(x[None], s)[0], H @ (s * x) / np.sqrt(D))
    assert not np.allclose(oracle.rotate(x[None], s)[0], s * (H @ x) / np.sqrt(D))


# ---------------------------------------------------------------- codebook

def _beta_cell_mean_quad(a, b, alpha):
    pdf = lambda y: scipy.stats.beta.pdf((y + 1) / 2, alpha, alpha) / 2
    m0 = integrate.quad(pdf, a, b, epsabs=0, epsrel=1e-13, limit=200)[0]
    m1 = integrate.quad(lambda y: y * pdf(y), a, b, epsabs=0, epsrel=1e-13, limit=200)[0]
    return m1 / m0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_lloyd_fixed_point_by_quadrature(books, bits):
    c, b = books[bits]
    assert len(c) == 1 << bits and len(b) == (1 << bits) - 1
    assert np.all(np.diff(c) > 0)
    edges = np.concatenate(([-1.0], b, [1.0]))
    for i in range(len(c)):
        # conditional mean of the cell by adaptive quadrature of the Beta pdf
        assert abs(_beta_cell_mean_quad(edges[i], edges[i + 1], D / 2) - c[i]) < 1e-9
    assert np.max(np.abs(b - 0.5 * (c[:-1] + c[1:]))) < 1e-15
    assert np.array_equal(c, -c[::-1])
    assert b[len(b) // 2] == 0.0


def test_codebook_two_bit_matches_printed_centroids(books):
    printed = np.array([float(v) for v in _golden_lines("turboq2_centroids.txt")])
    assert np.array_equal(np.round(books[2][0], 3), printed)
    # the fork states its law as N(0, 1/128); its levels (0.0400, 0.1335)
    # agree with the printed three decimals up to truncation of the last one
    cg, _, _ = oracle.gaussian_codebook(2, sigma=1 / np.sqrt(128))
    assert np.max(np.abs(cg - printed)) < 1e-3


def test_generic_lloyd_reproduces_max_table():
    for ln in _golden_lines("max1960_gaussian.txt"):
        levels, vals = ln.split(":")
        want = np.array([float(v) for v in vals.split()])
        bits = int(levels).bit_length() - 1
        c, _, _ = oracle.gaussian_codebook(bits)
        got = c[len(c) // 2:]
        assert np.max(np.abs(got - want) / want) < 4e-4, (levels, got, want)


def test_beta_codebook_approaches_gaussian_limit(books):
    # y = 2u - 1, u ~ Beta(d/2, d/2) has variance 1/(d+1) and tends to normal.
    for bits in (2, 3, 4):
        cg, _, _ = oracle.gaussian_codebook(bits)
        cb = books[bits][0] * np.sqrt(D + 1)
        assert np.max(np.abs(cb - cg) / np.abs(cg)) < 0.02


# ---------------------------------------------------------------- codec

def test_fp16_rounds_directly_from_float64():
    assert codec.fp16_rne(1 + 2**-11)[()] == 0x3C00          # tie -> even
    assert codec.fp16_rne(1 + 2**-11 + 2**-40)[()] == 0x3C01  # no float32 step
    assert codec.fp16_rne(65504.0)[()] == 0x7BFF
    assert codec.fp16_rne(65520.0)[()] == 0x7C00              # overflow -> +inf
    assert codec.fp16_rne(0.0)[()] == 0


def test_block_sizes_match_pages():
    for ln in _golden_lines("block_sizes.txt"):
        bits, nbytes, bpw = ln.split()
        assert codec.block_bytes(int(bits)) == int(nbytes)
        assert codec.block_bytes(int(bits)) * 8 / D == float(bpw)
    assert codec.block_bytes(4) == 66


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_unpack_exhaustive(bits):
    L = 1 << bits
    nb = codec.block_bytes(bits)
    for v in range(L):
        idx = np.zeros((D, D), np.uint8)
        idx[np.arange(D), np.arange(D)] = v         # row j holds v at position j
        norms = np.arange(D, dtype=np.uint16) * 513
        blk = codec.pack_block(idx, norms, bits)
        assert blk.shape == (D, nb)
        back, n16 = codec.unpack_block(blk, bits)
        assert np.array_equal(back, idx) and np.array_equal(n16, norms)
        assert np.array_equal(blk[:, 0] | (blk[:, 1].astype(np.uint16) << 8), norms)
        for j in range(D):
            body = blk[j, 2:]
            # where the single non-zero code lands (lowest element in lowest bits)
            expect = np.zeros(nb - 2, np.uint8)
            if bits == 2:
                expect[j // 4] = v << (2 * (j % 4))
            elif bits == 4:
                expect[j // 2] = v << (4 * (j % 2))
            else:
                expect[j // 4] = (v & 3) << (2 * (j % 4))
                expect[32 + j // 8] = (v >> 2) << (j % 8)
            assert np.array_equal(body, expect), (bits, v, j)
    rng = np.random.default_rng(0)
    idx = rng.integers(0, L, (500, D)).astype(np.uint8)
    n16 = rng.integers(0, 1 << 16, 500).astype(np.uint16)
    back, nn = codec.unpack_block(codec.pack_block(idx, n16, bits), bits)
    assert np.array_equal(back, idx) and np.array_equal(nn, n16)


def test_quantize_tie_goes_up_and_zero_vector(books):
    c, b = books[4]
    b32 = b.astype(np.float32)
    y = np.array(b32, np.float64)[None, :]
    assert np.array_equal(codec.quantize(y, b32)[0], np.arange(1, 16))
    s = oracle.sign_diagonal(1)
    idx, n16, _ = codec.encode(np.zeros((1, D)), s, b32)
    assert np.all(idx == 8) and n16[0] == 0
    assert np.array_equal(codec.decode(idx, n16, c, s), np.zeros((1, D)))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_encode_scale_invariance_and_edge_magnitudes(books, bits):
    c, b = books[bits]
    b32 = b.astype(np.float32)
    s = oracle.sign_diagonal(1)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, D))
    i0, n0, _ = codec.encode(x, s, b32)
    for f in (2.0**-20, 2.0**-4, 2.0**10):     # exact power-of-two scalings
        i1, n1, _ = codec.encode(x * f, s, b32)
        assert np.array_equal(i0, i1)
        want = codec.fp16_rne(np.linalg.norm(x, axis=1) * f)
        assert np.array_equal(n1, want)
    same = np.full((1, D), 3.0)                  # all-same vector
    i2, n2, y2 = codec.encode(same, s, b32)
    assert n2[0] == codec.fp16_rne(3.0 * np.sqrt(D))
    assert np.allclose(np.sum(y2 * y2), 1.0)


def test_encode_deterministic_by_seed(books):
    b32 = books[4][1].astype(np.float32)
    x = workloads.single_head(T=256)["k"].numpy().astype(np.float64)
    a = codec.encode(x, oracle.sign_diagonal(1), b32)[0]
    assert np.array_equal(a, codec.encode(x, oracle.sign_diagonal(1), b32)[0])
    assert not np.array_equal(a, codec.encode(x, oracle.sign_diagonal(7), b32)[0])


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_roundtrip_mse_matches_closed_form(books, bits):
    # Isotropic Gaussian rows are uniform on the sphere after normalising;
    # a coordinate of the unit sphere in R^d is 2 Beta((d-1)/2, (d-1)/2) - 1.
    c, b = books[bits]
    x = workloads.single_head(T=4096)["k"].numpy().astype(np.float64)
    s = oracle.sign_diagonal(workloads.SIGN_SEED)
    idx, n16, _ = codec.encode(x, s, b.astype(np.float32))
    xh = codec.decode(idx, n16, c, s)
    rel = np.mean(np.sum((x - xh) ** 2, 1) / np.sum(x * x, 1))
    pred = D * oracle.beta_law_moments(c, b, (D - 1) / 2)
    assert abs(rel / pred - 1) < 0.02, (rel, pred)


def test_dot_product_preservation(books):
    c, b = books[4]
    s = oracle.sign_diagonal(1)
    rng = np.random.default_rng(3)
    k = rng.standard_normal((2000, D))
    q = rng.standard_normal(D)
    idx, n16, _ = codec.encode(k, s, b.astype(np.float32))
    kh = codec.decode(idx, n16, c, s)
    err = (kh - k) @ q
    # error std per dot ~ ||q|| ||k|| sqrt(D_4) / sqrt(d) ... bounded well below ||q|| ||k||
    assert np.sqrt(np.mean(err**2)) < 0.12 * np.sqrt(D) * np.linalg.norm(q) / np.sqrt(D)


# ---------------------------------------------------------------- attention

def _small_cache(books, kb, vb, B=2, Hq=8, Hkv=2, T=37, seed=0):
    rng = np.random.default_rng(seed)
    s = oracle.sign_diagonal(1)
    k = rng.standard_normal((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    q = rng.standard_normal((B, Hq, D))
    kc, kbd = books[kb]
    vc, vbd = books[vb]
    ki, kn, _ = codec.encode(k.reshape(-1, D), s, kbd.astype(np.float32))
    vi, vn, _ = codec.encode(v.reshape(-1, D), s, vbd.astype(np.float32))
    sh = (B, Hkv, T)
    return dict(q=q, ki=ki.reshape(*sh, D), kn=kn.reshape(sh), kc=kc,
                vi=vi.reshape(*sh, D), vn=vn.reshape(sh), vc=vc, s=s)


def _deq(cache):
    from oracle.attention import dequantize_cache
    return (dequantize_cache(cache["ki"], cache["kn"], cache["kc"], cache["s"]),
            dequantize_cache(cache["vi"], cache["vn"], cache["vc"], cache["s"]))


def test_attention_fused_form_equals_definition(books):
    c = _small_cache(books, 4, 2)
    kh, vh = _deq(c)
    scale = 1 / np.sqrt(D)
    lens = np.array([37, 11])
    a = oracle.attention_dequantized(c["q"], kh, vh, scale, seq_lens=lens)
    r = oracle.attention_rotated(c["q"], c["ki"], c["kn"], c["kc"], c["vi"], c["vn"],
                                 c["vc"], c["s"], scale, seq_lens=lens)
    assert np.max(np.abs(a - r)) < 1e-12


def test_attention_matches_torch_sdpa(books):
    import torch
    c = _small_cache(books, 3, 3, T=53)
    kh, vh = _deq(c)
    scale = 1 / np.sqrt(D)
    a = oracle.attention_dequantized(c["q"], kh, vh, scale)
    G = c["q"].shape[1] // kh.shape[1]
    kt = torch.from_numpy(np.repeat(kh, G, axis=1))
    vt = torch.from_numpy(np.repeat(vh, G, axis=1))
    qt = torch.from_numpy(c["q"])[:, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    assert np.max(np.abs(ref[:, :, 0].numpy() - a)) < 1e-12


def test_attention_special_cases(books):
    c = _small_cache(books, 4, 2, T=9)
    kh, vh = _deq(c)
    G = 4
    # one token: output is that token's value
    o1 = oracle.attention_dequantized(c["q"], kh[:, :, :1], vh[:, :, :1], 0.3)
    assert np.allclose(o1, np.repeat(vh[:, :, 0], G, axis=1), atol=1e-14)
    # identical keys: uniform weights, output is the mean value
    same = np.repeat(kh[:, :, :1], 9, axis=2)
    o2 = oracle.attention_dequantized(c["q"], same, vh, 0.3)
    assert np.allclose(o2, np.repeat(vh.mean(axis=2), G, axis=1), atol=1e-13)
    # zero scale: uniform weights as well
    o3 = oracle.attention_dequantized(c["q"], kh, vh, 0.0)
    assert np.allclose(o3, np.repeat(vh.mean(axis=2), G, axis=1), atol=1e-13)


def test_causal_attention_matches_torch_sdpa_with_mask(books):
    """Multi-token (causal) attention against torch's scaled_dot_product_attention
    with an explicit boolean mask built from the query positions, per
    sequence, for ragged lengths."""
    import torch
    c = _small_cache(books, 4, 3, B=2, Hq=8, Hkv=2, T=41, seed=4)
    kh, vh = _deq(c)
    scale = 1 / np.sqrt(D)
    M = 6
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, M, 8, D))
    lens = np.array([41, 17])
    got = oracle.attention_causal(q, kh, vh, scale, seq_lens=lens)
    for b in range(2):
        L = int(lens[b])
        pos = L - M + np.arange(M)
        mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])          # [M, L]
        kt = torch.from_numpy(np.repeat(kh[b, :, :L], 4, axis=0))               # [Hq, L, D]
        vt = torch.from_numpy(np.repeat(vh[b, :, :L], 4, axis=0))
        qt = torch.from_numpy(q[b].transpose(1, 0, 2))                           # [Hq, M, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        assert np.max(np.abs(ref.numpy().transpose(1, 0, 2) - got[b])) < 1e-12


def test_causal_attention_special_cases(books):
    c = _small_cache(books, 4, 2, B=2, Hq=8, Hkv=2, T=12, seed=5)
    kh, vh = _deq(c)
    scale = 0.2
    rng = np.random.default_rng(2)
    M = 12
    q = rng.standard_normal((2, M, 8, D))
    o = oracle.attention_causal(q, kh, vh, scale)
    # the first position sees only the first key: its output is that value
    assert np.allclose(o[:, 0], np.repeat(vh[:, :, 0], 4, axis=1), atol=1e-14)
    # the last query token sees the whole cache: the decode attention of that token
    dec = oracle.attention_dequantized(q[:, -1], kh, vh, scale)
    assert np.allclose(o[:, -1], dec, atol=1e-14)
    # causality: changing keys / values after a query's position leaves its output unchanged
    kh2, vh2 = kh.copy(), vh.copy()
    kh2[:, :, 7:] = rng.standard_normal(kh2[:, :, 7:].shape)
    vh2[:, :, 7:] = rng.standard_normal(vh2[:, :, 7:].shape)
    o2 = oracle.attention_causal(q, kh2, vh2, scale)
    assert np.array_equal(o2[:, :7], o[:, :7])
    assert not np.allclose(o2[:, 7:], o[:, 7:])
    # fewer cached tokens than query tokens: the leading queries have no keys and give zeros
    o3 = oracle.attention_causal(q, kh, vh, scale, seq_lens=np.array([5, 12]))
    assert np.all(o3[0, :7] == 0) and np.allclose(o3[0, 7:], oracle.attention_causal(
        q[:1, 7:], kh[:1, :, :5], vh[:1, :, :5], scale)[0], atol=1e-14)


def test_attention_cosine_matches_pages_soft(books):
    # The spec's measured quality table (synthetic Gaussian): soft band 0.015.
    rng = np.random.default_rng(11)
    s = oracle.sign_diagonal(1)
    T = 4096
    k = rng.standard_normal((T, D))
    v = rng.standard_normal((T, D))
    cosines = []
    for ln in _golden_lines("attention_cosine.txt"):
        kb, vb, want = ln.split()
        kc, kbd = books[int(kb)]
        vc, vbd = books[int(vb)]
        ki, kn, _ = codec.encode(k, s, kbd.astype(np.float32))
        vi, vn, _ = codec.encode(v, s, vbd.astype(np.float32))
        kh = codec.decode(ki, kn, kc, s)[None, None]
        vh = codec.decode(vi, vn, vc, s)[None, None]
        q = rng.standard_normal((1, 16, D))
        o = oracle.attention_dequantized(q, k[None, None], v[None, None], 1 / np.sqrt(D))
        oh = oracle.attention_dequantized(q, kh, vh, 1 / np.sqrt(D))
        cos = np.mean(np.sum(o * oh, -1) / np.linalg.norm(o, axis=-1) / np.linalg.norm(oh, axis=-1))
        cosines.append(cos)
        assert abs(cos - float(want)) < 0.015, (kb, vb, cos)


# ---------------------------------------------------------------- QJL

def test_qjl_identity_sketch_closed_form(books):
    c, b = books[3]
    s = oracle.sign_diagonal(1)
    rng = np.random.default_rng(4)
    k = rng.standard_normal((20, D))
    q = rng.standard_normal(D)
    idx, n16, _ = codec.encode(k, s, b.astype(np.float32))
    bits, rn16, proj = oracle.qjl_encode(k, idx, n16, c, s, np.eye(D))
    r = k - codec.decode(idx, n16, c, s)
    assert np.allclose(proj, r, atol=0)
    t2 = oracle.qjl_term2(q, bits, rn16, np.eye(D))
    rn = codec.norm_value(rn16)
    want = rn * np.sqrt(np.pi / 2) / D * (np.where(r >= 0, 1.0, -1.0) @ q)
    assert np.allclose(t2, want, rtol=1e-14, atol=0)


def test_qjl_zero_residual(books):
    c, b = books[3]
    s = oracle.sign_diagonal(1)
    idx = np.full((3, D), 5, np.uint8)
    n16 = codec.fp16_rne(np.array([1.0, 2.0, 0.5]))
    k = codec.decode(idx, n16, c, s)                 # keys equal to their own k_mse
    S = np.random.default_rng(0).standard_normal((D, D))
    bits, rn16, _ = oracle.qjl_encode(k, idx, n16, c, s, S)
    assert np.all(rn16 == 0)
    assert np.all(oracle.qjl_term2(np.ones(D), bits, rn16, S) == 0)


def test_qjl_term2_unbiased(books):
    # E_S[term2] = <q, r> for Gaussian S (QJL estimator).  Use the exact
    # residual norm here: the fp16 rounding of ||r|| is a separate, tiny bias.
    rng = np.random.default_rng(9)
    q = rng.standard_normal(D)
    r = rng.standard_normal(D) * 0.3
    est = []
    for _ in range(3000):
        S = rng.standard_normal((D, D))
        sgn = np.where(S @ r >= 0, 1.0, -1.0)
        est.append(np.linalg.norm(r) * np.sqrt(np.pi / 2) / D * (sgn @ (S @ q)))
    est = np.array(est)
    se = est.std() / np.sqrt(len(est))
    assert abs(est.mean() - q @ r) < 4 * se
    # and the oracle's packed path gives the same estimator for one S
    bits = np.zeros((1, 16), np.uint8)
    for j in range(D):
        bits[0, j // 8] |= (int(sgn[j] > 0) << (j % 8))
    rn16 = codec.fp16_rne(np.linalg.norm(r))
    t2 = oracle.qjl_term2(q, bits, rn16[None], S)[0]
    assert np.isclose(t2, codec.norm_value(rn16) * np.sqrt(np.pi / 2) / D * (sgn @ (S @ q)))


# ---------------------------------------------------------------- serde

@pytest.mark.parametrize("L,sf,sl,want", [(32, 2, 2, (2, 30)), (3, 2, 2, (2, 2)),
                                          (4, 0, 0, (0, 4)), (5, 9, 0, (5, 5)),
                                          (6, 1, 9, (1, 1))])
def test_serde_compressed_range_rule(L, sf, sl, want):
    assert oracle.serde_ranges(L, sf, sl) == want


@pytest.mark.parametrize("L,T,bs,sf,sl", [(5, 24, 8, 2, 2), (5, 21, 8, 1, 1), (3, 16, 16, 2, 2)])
def test_serde_roundtrip_and_size(books, L, T, bs, sf, sl):
    import torch
    hidden = 256
    x = workloads.storage_kv(L=L, T=T, hidden=hidden, seed=3)["kv"]
    values = x.to(torch.float64).numpy()
    raw = x.view(torch.uint8).numpy().reshape(2, L, T, hidden * 2)
    s = oracle.sign_diagonal(1)
    (kc, kb), (vc, vb) = books[4], books[4]
    buf = oracle.serialize((values, raw), bs, sf, sl, 4, 4, s,
                           kb.astype(np.float32), vb.astype(np.float32))
    assert len(buf) == oracle.serde_size(L, T, hidden, D, bs, sf, sl, 4, 4)
    rraw, rec, (qs, qe) = oracle.deserialize(buf, L, T, hidden, bs, sf, sl, 4, 4, s,
                                             kc, vc, np.uint16)
    for l in list(range(qs)) + list(range(qe, L)):
        assert np.array_equal(rraw[:, l], raw[:, l])
    pred = D * oracle.beta_law_moments(kc, kb, (D - 1) / 2)
    for l in range(qs, qe):
        rel = np.sum((rec[:, l] - values[:, l]) ** 2) / np.sum(values[:, l] ** 2)
        assert abs(rel / pred - 1) < 0.25
