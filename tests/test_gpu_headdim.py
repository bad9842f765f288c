"""GPU parity of the codec and the decode attention at head dims 64, 96, 128
and 160 (a dense orthogonal rotation as an input), against oracle.headdim
and the oracle's plain attention, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
from oracle import codec, headdim
from parity_util import ATTN_TOL, CODE_FRAC, CODE_TOL_Y, attn_rel_err, fp16_tie_distance, record
from turboquant_bit_kv_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    tq.lib()
    return dict(tq=tq, dev=torch.device("cuda:0"))


def _rotation(env, d):
    """d = 64: the library's H D / 8; other d: a seeded random orthogonal matrix."""
    tq = env["tq"]
    if d == 64:
        R = tq.tq_rotation_hadamard(64, tq.tq_signs_from_seed(workloads.SIGN_SEED)).double().numpy()
    else:
        a = np.random.default_rng(1000 + d).standard_normal((d, d))
        q, r = np.linalg.qr(a)
        R = q * np.sign(np.diag(r))[None, :]
    R32 = R.astype(np.float32)
    # both sides use the same float32 matrix
    return R32.astype(np.float64), torch.from_numpy(R32).to(env["dev"])


def _check(label, bits, idx_g, idx_o, y, b32, n16_g, n16_o, x):
    """The parity rule of the 128-element codec: codes bit-exact except within
    1e-5 of a boundary, norms except within 2^-22 of an fp16 tie; counted."""
    mism = idx_g != idx_o
    near = np.zeros(y.shape, bool)
    for b in np.asarray(b32, np.float64):
        near |= np.abs(y - b) < CODE_TOL_Y
    n = np.sqrt(np.sum(np.asarray(x, np.float64) ** 2, axis=-1))
    nm = n16_g != n16_o
    record(label, bits=bits, coords=int(mism.size), near_boundary=int(near.sum()), code_mismatch=int(mism.sum()),
           vectors=int(nm.size), norm_near_tie=int((fp16_tie_distance(n) < 2.0**-22).sum()), norm_mismatch=int(nm.sum()))
    assert not (mism & ~near).any(), "%s: code mismatches away from a boundary" % label
    assert mism.mean() < CODE_FRAC
    assert np.all(fp16_tie_distance(n[nm]) < 2.0**-22) and nm.mean() < CODE_FRAC


def _books(d, bits):
    c, b, _ = oracle.beta_codebook(d, bits)
    return c.astype(np.float32).astype(np.float64), b.astype(np.float32)


@pytest.mark.parametrize("d", (64, 96, 128, 160))
@pytest.mark.parametrize("bits", (2, 3, 4))
@pytest.mark.parametrize("dtype", (torch.float32, torch.bfloat16))
def test_encode_decode_match_oracle(env, d, bits, dtype):
    tq, dev = env["tq"], env["dev"]
    R, Rd = _rotation(env, d)
    c, b32 = _books(d, bits)
    cb = tq.tq_codebook_load(d, bits)
    n = 1000
    x = torch.randn((n, d), generator=torch.Generator().manual_seed(d + bits), dtype=torch.float32).to(dtype)
    x[3] = 0                                  # a zero row
    x[5] *= 1e-3
    xd = x.to(dev)
    bb = tq.tq_block_bytes_d(d, bits)
    blocks = torch.full((n + 2, bb), 0xA5, dtype=torch.uint8, device=dev)
    tq.tq_encode_kv_d(xd, cb, Rd, blocks[1:n + 1])
    torch.cuda.synchronize()
    got = blocks.cpu().numpy()
    assert np.all(got[0] == 0xA5) and np.all(got[-1] == 0xA5)   # nothing written outside
    idx, n16 = headdim.unpack_d(got[1:n + 1], d, bits)
    ridx, rn16, y = headdim.encode_d(x.double().numpy(), R, b32)
    _check("head dim %d" % d, bits, idx, ridx, y, b32, n16, rn16, x.double().numpy())
    assert np.all(idx[3] == (1 << bits) // 2) and n16[3] == 0
    # decode the library's own blocks; float32 arithmetic, one rounding
    out = torch.empty((n, d), dtype=torch.float32, device=dev)
    tq.tq_decode_kv_d(blocks[1:n + 1], n, cb, Rd, out)
    torch.cuda.synchronize()
    ref = headdim.decode_d(idx, n16, c, R)
    nrm = codec.norm_value(n16)[:, None]
    assert np.max(np.abs(out.double().cpu().numpy() - ref) / np.maximum(nrm, 1e-30)) < 1e-5


@pytest.mark.parametrize("d", (64, 96, 128, 160))
@pytest.mark.parametrize("bits", (2, 3, 4))
@pytest.mark.parametrize("dtype", (torch.bfloat16, torch.float16))
def test_encode_tensor_core_rows_match_oracle(env, d, bits, dtype):
    """More than 1024 bf16 / fp16 rows take the tensor-core encode (R as two
    16-bit terms): a ragged last tile, a zero row, rows whose float32 sum of
    squares leaves the safe range (bf16) or is small (fp16), into a 16-byte
    aligned block array (bulk stores) and into one that is only 2-byte
    aligned (2-byte stores)."""
    tq, dev = env["tq"], env["dev"]
    R, Rd = _rotation(env, d)
    c, b32 = _books(d, bits)
    cb = tq.tq_codebook_load(d, bits)
    n = 128 * 23 + 37
    x = torch.randn((n, d), generator=torch.Generator().manual_seed(7 * d + bits), dtype=torch.float32)
    x[7] = 0
    if dtype == torch.bfloat16:
        x[300] *= 1e-22      # squares underflow float32
        x[301] *= 1e17       # squares overflow float32
    else:
        x[300] *= 1e-3
        x[301] *= 1000.0
    x = x.to(dtype)
    xd = x.to(dev)
    bb = tq.tq_block_bytes_d(d, bits)
    ridx, rn16, y = headdim.encode_d(x.double().numpy(), R, b32)
    aligned = torch.empty((n, bb), dtype=torch.uint8, device=dev)
    padded = torch.full((n + 2, bb), 0xA5, dtype=torch.uint8, device=dev)
    tq.tq_encode_kv_d(xd, cb, Rd, aligned)
    tq.tq_encode_kv_d(xd, cb, Rd, padded[1:n + 1])
    torch.cuda.synchronize()
    got_p = padded.cpu().numpy()
    assert np.all(got_p[0] == 0xA5) and np.all(got_p[-1] == 0xA5)   # nothing written outside
    for label, got in (("aligned", aligned.cpu().numpy()), ("2-byte aligned", got_p[1:n + 1])):
        idx, n16 = headdim.unpack_d(got, d, bits)
        _check("tensor-core head dim %d %s %s" % (d, str(dtype), label), bits, idx, ridx, y, b32, n16, rn16,
               x.double().numpy())
        assert np.all(idx[7] == (1 << bits) // 2) and n16[7] == 0
    assert np.array_equal(aligned.cpu().numpy(), got_p[1:n + 1])


def _near_tie_pairs(rng, k):
    """fp16 pairs (a, b) whose norm sqrt(a^2 + b^2) lies within 2^-20 (relative)
    of an fp16 rounding boundary, but not within 2^-30."""
    out = []
    while len(out) < k:
        a = rng.uniform(0.5, 2.0, 200000).astype(np.float16).astype(np.float64)
        b = rng.uniform(0.5, 2.0, 200000).astype(np.float16).astype(np.float64)
        dist = fp16_tie_distance(np.sqrt(a * a + b * b))
        sel = (dist < 2.0**-20) & (dist > 2.0**-30)
        out.extend(zip(a[sel], b[sel]))
    return np.array(out[:k])


@pytest.mark.parametrize("d", (64, 160))
def test_encode_tensor_core_norms_near_fp16_ties(env, d):
    """Rows whose norm lies within 2^-20 of an fp16 rounding boundary take the
    exact norm (listed in the main loop, rewritten after it): nine rows in ten
    here, so most CTAs' lists (512 rows) overflow and every row of such a CTA
    is redone; the norms must still be the correctly rounded ones."""
    tq, dev = env["tq"], env["dev"]
    R, Rd = _rotation(env, d)
    c, b32 = _books(d, 4)
    rng = np.random.default_rng(d)
    n = 152 * 5 * 128
    x = np.zeros((n, d))
    pairs = _near_tie_pairs(rng, n)
    rows = np.arange(n)
    i = rows % d
    j = (i + 1 + rows % (d - 1)) % d
    sg = rng.choice([-1.0, 1.0], (n, 2))
    x[rows, i] = pairs[:, 0] * sg[:, 0]
    x[rows, j] = pairs[:, 1] * sg[:, 1]
    plain = rng.random(n) < 0.1
    x[plain] = rng.standard_normal((int(plain.sum()), d))
    xt = torch.from_numpy(x).to(torch.float16)
    blocks = torch.empty((n, tq.tq_block_bytes_d(d, 4)), dtype=torch.uint8, device=dev)
    tq.tq_encode_kv_d(xt.to(dev), tq.tq_codebook_load(d, 4), Rd, blocks)
    torch.cuda.synchronize()
    idx, n16 = headdim.unpack_d(blocks.cpu().numpy(), d, 4)
    ridx, rn16, y = headdim.encode_d(xt.double().numpy(), R, b32)
    nn = np.sqrt(np.sum(xt.double().numpy() ** 2, axis=1))
    assert np.mean(fp16_tie_distance(nn) < 2.0**-20) > 0.85      # the rows are where they should be
    _check("near-tie norms head dim %d" % d, 4, idx, ridx, y, b32, n16, rn16, xt.double().numpy())


@pytest.mark.parametrize("d,kbits,vbits,B,Hq,Hkv,T,lens", [
    # up to four heads per KV head: one n-tile of 4 heads x (hi, lo)
    (64, 4, 2, 3, 8, 2, 700, [700, 1, 333]),
    (160, 4, 4, 2, 4, 4, 520, [0, 517]),
    (64, 2, 2, 2, 4, 2, 1000, None),
    (96, 3, 4, 2, 6, 2, 777, [777, 31]),
    (128, 4, 2, 4, 16, 4, 2100, [2100, 0, 1, 1057]),
    (160, 3, 2, 2, 12, 4, 1500, [33, 1500]),
    (160, 2, 4, 1, 2, 2, 3000, None),
    (96, 4, 3, 2, 8, 2, 600, [600, 599]),
    (64, 3, 3, 3, 3, 3, 1100, [1, 1100, 40]),
    (160, 4, 3, 2, 16, 4, 1300, [1300, 777]),
    (128, 2, 3, 1, 2, 1, 2600, None),
    # five to eight heads per KV head: the eight-head n-tile (hi and lo as separate products)
    (96, 3, 3, 2, 14, 2, 1000, None),
    (128, 2, 3, 1, 8, 1, 4096, None),
    (64, 4, 2, 1, 16, 2, 900, [900]),
    (160, 4, 4, 2, 20, 4, 1100, [1100, 613]),
    (64, 2, 3, 3, 18, 3, 700, [0, 700, 31]),
    (128, 3, 2, 2, 16, 2, 1500, [1, 1500]),
    # a short batch over a long context: many splits per (sequence, KV head)
    (64, 4, 2, 1, 4, 1, 16384, None),
    (160, 3, 3, 2, 16, 2, 12000, [12000, 9001]),
])
def test_attention_matches_oracle(env, d, kbits, vbits, B, Hq, Hkv, T, lens):
    tq, dev = env["tq"], env["dev"]
    R, Rd = _rotation(env, d)
    T_cap = (T + 15) // 8 * 8   # a multiple of 8 past T
    rng = np.random.default_rng(d + T)
    k = rng.standard_normal((B, Hkv, T, d))
    v = rng.standard_normal((B, Hkv, T, d))
    q = torch.from_numpy(rng.standard_normal((B, Hq, d))).to(torch.bfloat16)
    hats, blks = {}, {}
    for name, x, bits in (("k", k, kbits), ("v", v, vbits)):
        c, b32 = _books(d, bits)
        idx, n16, _ = headdim.encode_d(x.reshape(-1, d), R, b32)
        hats[name] = headdim.decode_d(idx, n16, c, R).reshape(B, Hkv, T, d)
        blk = np.zeros((B, Hkv, T_cap, tq.tq_block_bytes_d(d, bits)), np.uint8)
        blk[:, :, :T] = headdim.pack_d(idx, n16, bits).reshape(B, Hkv, T, -1)
        blks[name] = torch.from_numpy(blk).to(dev)
    out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes_d(B, Hq, Hkv, T_cap, d), dtype=torch.uint8, device=dev)
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    scale = 1 / np.sqrt(d)
    tq.tq_attn_decode_d(q.to(dev), blks["k"], tq.tq_codebook_load(d, kbits), blks["v"], tq.tq_codebook_load(d, vbits),
                        Rd, out, ws, T, scale, seq_lens=sl)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    keep = list(range(B)) if lens is None else [i for i, L in enumerate(lens) if L > 0]
    if lens is not None:
        assert np.all(got[[i for i, L in enumerate(lens) if L == 0]] == 0)
    ref = oracle.attention_dequantized(q.double().numpy()[keep], hats["k"][keep], hats["v"][keep], scale,
                                       seq_lens=None if lens is None else [lens[i] for i in keep])
    err = attn_rel_err(got[keep], ref)
    assert np.all(err < ATTN_TOL), err.max()
