"""Comparison rules shared by the GPU parity tests.

* Codes: bit-exact, except coordinates whose float64 y lies within 1e-5 of a
  decision boundary; such mismatches are counted and must stay below 1e-4 of
  all coordinates.
* Norms (fp16): bit-exact, except where the float64 norm lies within 2^-22
  (relative) of an fp16 rounding boundary; counted, below 1e-4 of vectors.
* QJL sign bits: bit-exact, except where |(S r)_j| <= 1e-5 * ||S_j|| * ||r||.
  QJL residual norms: equal, or one fp16 step apart where the float64 norm
  lies within 4e-6 (relative) of an fp16 rounding boundary (the residual is a
  float32 quantity on the GPU: its relative error is a few 1e-7, see design
  notes).
* Attention outputs: per output vector, max_i |o_i - o_ref_i| / max_i |o_ref_i|
  <= 1e-3 (float32 accumulate), on identical packed caches made by the oracle.
"""

import numpy as np

import oracle
from oracle import codec

CODE_TOL_Y = 1e-5
CODE_FRAC = 1e-4
ATTN_TOL = 1e-3

# One entry per comparison made by check_codes / record(): the counts the
# parity rule asks to be reported (printed at the end of the pytest session).
RECORDS = []


def record(label, **counts):
    RECORDS.append(dict(label=label, **counts))


def fp16_tie_distance(n):
    """Relative distance of float64 n (>= 0) to the nearest fp16 rounding
    boundary around fp16(n)."""
    n = np.asarray(n, np.float64)
    h = n.astype(np.float16)
    hv = h.astype(np.float64)
    lo = np.nextafter(h, np.float16(0)).astype(np.float64)
    hi = np.nextafter(h, np.float16(np.inf)).astype(np.float64)
    d1 = np.abs(n - 0.5 * (lo + hv))
    d2 = np.abs(n - 0.5 * (hv + hi))
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(n > 0, np.minimum(d1, d2) / n, np.inf)


def check_counted(label, idx_g, idx_o, dist_y, n_g, n_o, exact, tie=2.0**-21):
    """The codes rule for given per-coordinate distances to a decision point
    (dist_y) and a scale or norm whose exact float64 value is `exact`: codes
    bit-exact except within CODE_TOL_Y, the stored fp16 bit-exact except within
    `tie` (relative) of an fp16 rounding boundary; mismatches counted."""
    mism = idx_g != idx_o
    assert np.all(dist_y[mism] < CODE_TOL_Y), (label, np.sum(mism & (dist_y >= CODE_TOL_Y)))
    assert mism.mean() < CODE_FRAC, (label, mism.mean())
    nm = n_g != n_o
    assert np.all(fp16_tie_distance(exact[nm]) < tie), (label, exact[nm][:4])
    assert nm.mean() < CODE_FRAC
    record(label, coords=int(mism.size), near_boundary=int((dist_y < CODE_TOL_Y).sum()),
           code_mismatch=int(mism.sum()), vectors=int(nm.size), norm_mismatch=int(nm.sum()))


def check_codes(gpu_blocks, bits, x, signs, b32, label=""):
    """Compare GPU blocks [N, bb] (uint8) with the oracle's encoding of x."""
    x = np.asarray(x, np.float64)
    idx_o, n16_o, y = codec.encode(x, signs, b32)
    idx_g, n16_g = codec.unpack_block(np.asarray(gpu_blocks), bits)
    mism = idx_g != idx_o
    bd = np.asarray(b32, np.float64)
    near = np.zeros(y.shape, bool)
    for b in bd:
        near |= np.abs(y - b) < CODE_TOL_Y
    n = np.sqrt(np.sum(x * x, axis=-1))
    norm_near = fp16_tie_distance(n) < 2.0**-22
    nm = n16_g != n16_o
    record(label, bits=bits, coords=int(mism.size), near_boundary=int(near.sum()), code_mismatch=int(mism.sum()),
           vectors=int(nm.size), norm_near_tie=int(norm_near.sum()), norm_mismatch=int(nm.sum()))
    if mism.any():
        ym = y[mism]
        dist = np.min(np.abs(ym[:, None] - np.asarray(b32, np.float64)[None, :]), axis=-1)
        far = dist >= CODE_TOL_Y
        assert not far.any(), "%s: %d code mismatches far from a boundary, e.g. y=%s" % (
            label, far.sum(), ym[far][:4])
    assert mism.mean() < CODE_FRAC, "%s: code mismatch fraction %.2e" % (label, mism.mean())
    if nm.any():
        assert np.all(fp16_tie_distance(n[nm]) < 2.0**-22), "%s: norm mismatch away from a tie" % label
    assert nm.mean() < CODE_FRAC, "%s: norm mismatch fraction %.2e" % (label, nm.mean())
    return int(mism.sum()), int(nm.sum())


def ulp_of(x, dtype):
    """Spacing of the torch float type `dtype` (bf16 / fp16) at |x| (float64)."""
    import torch
    mant = {torch.bfloat16: 7, torch.float16: 10}[dtype]
    tiny = {torch.bfloat16: 2.0**-133, torch.float16: 2.0**-24}[dtype]
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.maximum(2.0 ** (e - mant), tiny), tiny)


def rne(x, dtype):
    """Round float64 x to the torch float type `dtype` (bf16 / fp16), nearest
    even, in one step (no float32 intermediate); no overflow handling."""
    x = np.asarray(x, np.float64)
    q = ulp_of(x, dtype)
    return np.round(x / q) * q


def attn_rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref), axis=-1)
    num = np.max(np.abs(got - ref), axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)


def oracle_books():
    out = {}
    for b in (2, 3, 4):
        c, bd, _ = oracle.beta_codebook(128, b)
        out[b] = (c, bd, bd.astype(np.float32))
    return out
