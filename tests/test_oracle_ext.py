"""Pins of the oracle's further block formats (norm correction, 8-in-3
packing, turboq8) against values fixed outside it: the pages' block sizes,
closed forms, brute force and a dense Hadamard matrix from scipy.  CPU only."""

import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from oracle import codec, ext

D = 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    out = {}
    with open(os.path.join(GOLDEN, "turboq8_and_dense3.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                k, v = ln.split()
                out[k] = float(v)
    return out


@pytest.fixture(scope="module")
def s():
    return oracle.sign_diagonal(1)


def _rows(n, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal((n, D)) * scale


# ---------------------------------------------------------------- norm correction

@pytest.mark.parametrize("bits", [2, 3, 4])
def test_norm_correction_restores_the_norm(s, bits):
    """Before the fp16 rounding the corrected block reconstructs a vector of
    exactly the input's norm (the rotation, taken here as a dense matrix, is
    orthogonal); after it, within one fp16 half-ulp; the plain encode's
    reconstruction is shorter by the codebook's distortion."""
    c, bd, _ = oracle.beta_codebook(D, bits)
    x = _rows(500, bits, scale=3.0)
    idx, n16, _, v = ext.encode_nc(x, s, c, bd.astype(np.float32))
    R = scipy.linalg.hadamard(D) * s[None, :] / np.sqrt(D)       # R = H D / sqrt(d)
    xhat_exact = (v[:, None] * c[idx]) @ R                        # R^T (v c[idx]) as row vectors
    nx = np.linalg.norm(x, axis=1)
    assert np.max(np.abs(np.linalg.norm(xhat_exact, axis=1) / nx - 1)) < 1e-12
    xhat16 = codec.decode(idx, n16, c, s)
    assert np.max(np.abs(np.linalg.norm(xhat16, axis=1) / nx - 1)) <= 2.0**-11 * (1 + 1e-9)
    # the plain norm's reconstruction is shorter by about sqrt(1 - distortion)
    _, n16p, _ = codec.encode(x, s, bd.astype(np.float32))
    plain = np.linalg.norm(codec.decode(idx, n16p, c, s), axis=1) / nx
    assert np.mean(plain) < 1 - 1e-3
    assert np.all(np.abs(plain - 1) > np.abs(np.linalg.norm(xhat16, axis=1) / nx - 1) - 2.0**-11)


def test_norm_correction_zero_row_and_codes(s):
    c, bd, _ = oracle.beta_codebook(D, 3)
    x = _rows(20, 7)
    x[3] = 0.0
    idx, n16, _, v = ext.encode_nc(x, s, c, bd.astype(np.float32))
    assert n16[3] == 0 and v[3] == 0.0
    assert np.all(idx[3] == 4)                    # y := 0 -> the upper of the middle cells
    # the stored value is fp16(||x|| / ||c[idx]||) rounded once
    r = np.sqrt(np.sum(c[idx] ** 2, axis=1))
    want = (np.linalg.norm(x, axis=1) / r).astype(np.float16).view(np.uint16)
    assert np.array_equal(np.delete(n16, 3), np.delete(want, 3))


# ---------------------------------------------------------------- 8-in-3 packing

def test_dense3_block_size_and_worked_example():
    g = _golden()
    idx = np.zeros((1, D), np.uint8)
    idx[0, int(g["dense3_example_element"])] = int(g["dense3_example_code"])
    blk = ext.pack_dense3(idx, np.array([0x3C00], np.uint16))
    assert blk.shape[1] - 2 == int(g["dense3_code_bytes"]) == D * 3 // 8
    assert blk[0, int(g["dense3_example_byte"])] == int(g["dense3_example_value"])
    assert np.count_nonzero(blk[0, 2:]) == 1
    assert blk[0, 0] == 0x00 and blk[0, 1] == 0x3C


def test_dense3_pack_unpack_identity_exhaustive():
    # every code value at every position, and random blocks
    for v in range(8):
        for j in range(D):
            idx = np.zeros((1, D), np.uint8)
            idx[0, j] = v
            got, n = ext.unpack_dense3(ext.pack_dense3(idx, np.array([1234], np.uint16)))
            assert np.array_equal(got, idx) and n[0] == 1234
    idx = np.random.default_rng(3).integers(0, 8, (257, D)).astype(np.uint8)
    n16 = np.random.default_rng(4).integers(0, 65536, 257).astype(np.uint16)
    got, n = ext.unpack_dense3(ext.pack_dense3(idx, n16))
    assert np.array_equal(got, idx) and np.array_equal(n, n16)
    # the same codes as the split-plane block, in another arrangement
    gi, gn = codec.unpack_block(codec.pack_block(idx, n16, 3), 3)
    assert np.array_equal(gi, got) and np.array_equal(gn, n)


# ---------------------------------------------------------------- turboq8

def test_q8_levels_and_block_size():
    g = _golden()
    lv = ext.q8_levels()
    assert len(lv) == int(g["q8_levels"])
    assert lv[0] == g["q8_level0"] and lv[255] == g["q8_level255"]
    assert np.allclose(np.diff(lv), 2 / 255, rtol=0, atol=1e-15)
    assert ext.Q8_BLOCK == int(g["q8_block_bytes"])
    assert ext.Q8_BLOCK * 8 / D == g["q8_bpw"]


def test_q8_decision_is_the_nearest_level_by_brute_force():
    # the closed-form decision against an argmin over all 256 levels (ties: upper)
    y = np.concatenate([np.linspace(-1, 1, 20001), np.random.default_rng(5).uniform(-1, 1, 5000)])
    t = 127.5 * (y.astype(np.float32).astype(np.float64) + 1.0)
    got = np.clip(np.floor(t + 0.5), 0, 255)
    lv = ext.q8_levels()
    y32 = y.astype(np.float32).astype(np.float64)
    d = np.abs(y32[:, None] - lv[None, :])
    best = np.argmin(d - 1e-15 * np.arange(256)[None, :], axis=1)   # ties to the upper level
    assert np.array_equal(got, best)


def test_q8_roundtrip_bound_extremes_and_zero(s):
    x = _rows(300, 9, scale=2.0)
    x[5] = 0.0
    idx, s16, _ = ext.encode_q8(x, s)
    R = scipy.linalg.hadamard(D) * s[None, :] / np.sqrt(D)
    u = x @ R.T                                             # R x, from a dense Hadamard matrix
    a = np.max(np.abs(u), axis=1)
    # the block's largest coordinate lands on an end level
    j = np.argmax(np.abs(u), axis=1)
    ends = idx[np.arange(300), j]
    ok = np.arange(300) != 5
    assert np.all((ends[ok] == 0) | (ends[ok] == 255))
    # every coordinate within half a step, plus the fp16 scale's rounding
    sv = codec.norm_value(s16)
    rec = sv[:, None] * ext.q8_levels()[idx]
    err = np.abs(rec - u)
    bound = a[:, None] / 255 * (1 + 1e-9) + np.abs(a - sv)[:, None] + 1e-12
    assert np.all(err <= bound)
    # decode is the inverse rotation of that reconstruction
    assert np.allclose(ext.decode_q8(idx, s16, s), rec @ R, atol=1e-12)
    # zero row: scale 0, code 128, decodes to exactly 0
    assert s16[5] == 0 and np.all(idx[5] == 128) and np.all(ext.decode_q8(idx[5:6], s16[5:6], s) == 0)
    got_i, got_s = ext.unpack_q8(ext.pack_q8(idx, s16))
    assert np.array_equal(got_i, idx) and np.array_equal(got_s, s16)
