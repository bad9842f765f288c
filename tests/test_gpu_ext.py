"""GPU parity of the further block formats (tq_encode_kv_ex / tq_decode_kv_ex):
the norm-corrected encode, the dense 8-in-3 3-bit layout and turboq8, against
the oracle on the same seeded rows.

Rules: codes bit-exact except coordinates within 1e-5 (in y = u / n or
u / a) of a decision boundary, below 1e-4 of all coordinates; stored fp16
norms and scales bit-exact except where the exact value lies within 2^-21
(relative) of an fp16 rounding boundary; decode as the plain decode test
(float32 within 1e-6 of the norm, 16-bit outputs the correct rounding of a
value within 2e-7 of the norm of the exact one)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import codec, ext
from turboquant_bit_kv_gb300 import workloads

from parity_util import check_counted as _check, rne

pytestmark = pytest.mark.gpu

D = 128
NC, DENSE3 = 1, 2


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    tq.lib()
    books = {}
    for b in (2, 3, 4):
        c, bd, _ = oracle.beta_codebook(D, b)
        books[b] = (c.astype(np.float32).astype(np.float64), bd.astype(np.float32))
    return dict(tq=tq, dev=torch.device("cuda:0"), books=books,
                cbs={b: tq.tq_codebook_load(128, b) for b in (2, 3, 4, 8)},
                signs=tq.tq_signs_from_seed(workloads.SIGN_SEED), s=oracle.sign_diagonal(workloads.SIGN_SEED))


def _rows(n, seed, dtype):
    x = workloads.qwen_outlier(B=1, Hq=1, Hkv=1, T=n, seed=seed)["k"].reshape(-1, D).float()
    x[5] = 0.0                                   # a zero row
    x[7] *= 2.0 ** -30                           # a tiny one
    return x.to(dtype)


def _nc_norm(x, idx, c):
    """Corrected norm ||x|| / ||c[idx]|| of rows with the given codes, and its fp16 bits."""
    r = ext.recon_norm(idx, c)
    n = np.linalg.norm(x, axis=1)
    v = np.where(n > 0, n / np.where(r > 0, r, 1.0), 0.0)
    return v, codec.fp16_rne(v)


def _encode(env, x, bits, flags, n_extra=0, **kw):
    tq, dev = env["tq"], env["dev"]
    n = x.shape[0]
    bb = tq.tq_block_bytes_ex(bits, flags)
    out = torch.full((n * bb + 64,), 0xA5, dtype=torch.uint8, device=dev)
    tq.tq_encode_kv_ex(x.to(dev), env["cbs"][bits], env["signs"], out[32:32 + n * bb], flags=flags, **kw)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.all(o[:32] == 0xA5) and np.all(o[-32:] == 0xA5)
    return o[32:32 + n * bb].reshape(n, bb)


@pytest.mark.parametrize("n", [1000, 2600])      # (2600 bf16 / fp16 rows: the tensor-core encode)
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_norm_corrected_encode(env, bits, dtype, n):
    x = _rows(n, bits, dtype)
    g = _encode(env, x, bits, NC)
    xd = x.double().numpy()
    c, b32 = env["books"][bits]
    idx_o, n_o, y, v = ext.encode_nc(xd, env["s"], c, b32)
    idx_g, n_g = codec.unpack_block(g, bits)
    dist = np.min(np.abs(y[..., None] - b32.astype(np.float64)[None, None, :]), axis=-1)
    # the stored norm is checked against the block's own codes (a code allowed to differ at a
    # boundary changes the recon norm too)
    v_g, n_og = _nc_norm(xd, idx_g, c)
    _check("nc %d %s" % (bits, dtype), idx_g, idx_o, dist, n_g, n_og, v_g)
    # the corrected norm gives a reconstruction of the input's norm (to fp16)
    nx = np.linalg.norm(xd, axis=1)
    rec = np.linalg.norm(codec.decode(idx_g, n_g, c, env["s"]), axis=1)
    ok = nx > 1e-3          # (the tiny row's norm is an fp16 subnormal)
    assert np.all(np.abs(rec[ok] / nx[ok] - 1) <= 2.0**-11 + 1e-9)


@pytest.mark.parametrize("n", [777, 2600])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("flags", [DENSE3, DENSE3 | NC])
def test_dense3_encode(env, dtype, flags, n):
    x = _rows(n, 11, dtype)
    g = _encode(env, x, 3, flags)
    xd = x.double().numpy()
    c, b32 = env["books"][3]
    idx_o, n_o, y = codec.encode(xd, env["s"], b32)
    exact = np.linalg.norm(xd, axis=1)
    idx_g, n_g = ext.unpack_dense3(g)
    if flags & NC:
        exact, n_o = _nc_norm(xd, idx_g, c)
    dist = np.min(np.abs(y[..., None] - b32.astype(np.float64)[None, None, :]), axis=-1)
    _check("dense3 %d" % flags, idx_g, idx_o, dist, n_g, n_o, exact)


@pytest.mark.parametrize("bits,flags", [(4, NC), (3, DENSE3 | NC), (8, 0)])
def test_tensor_core_encode_strided_rows_unaligned_blocks(env, bits, flags):
    """The tensor-core encode with rows 272 bytes apart (a strided view) into
    a block array that starts 2 bytes past a 16-byte boundary (2-byte stores
    instead of bulk copies): the same blocks as the contiguous, aligned call."""
    tq, dev = env["tq"], env["dev"]
    n = 2100
    x = _rows(n, 17, torch.bfloat16)
    wide = torch.zeros((n, 136), dtype=torch.bfloat16)
    wide[:, :D] = x
    xs = wide.to(dev)[:, :D]                      # row stride 136 elements
    assert xs.stride(0) == 136
    bb = tq.tq_block_bytes_ex(bits, flags)
    ref = _encode(env, x, bits, flags)
    out = torch.full((n * bb + 64,), 0xA5, dtype=torch.uint8, device=dev)
    tq.tq_encode_kv_ex(xs, env["cbs"][bits], env["signs"], out[34:34 + n * bb], flags=flags)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.all(o[:34] == 0xA5) and np.all(o[34 + n * bb:] == 0xA5)
    assert np.array_equal(o[34:34 + n * bb].reshape(n, bb), ref)


def _decode(env, blocks, bits, flags, dtype, stride=None, offset=0):
    tq, dev = env["tq"], env["dev"]
    n, bb = blocks.shape
    st = stride or bb
    buf = np.full((n, st), 0x5A, np.uint8)
    buf[:, offset:offset + bb] = blocks
    out = torch.empty((n, D), dtype=dtype, device=dev)
    tq.tq_decode_kv_ex(torch.from_numpy(buf.reshape(-1)).to(dev), n, env["cbs"][bits], env["signs"], out,
                       block_stride_bytes=st, block_offset=offset, flags=flags)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def _check_decode(got, ref, nrm, dtype):
    if dtype == torch.float32:
        assert np.max(np.abs(got - ref) / np.maximum(nrm, 1e-30)) < 1e-6
    else:
        delta = 2e-7 * nrm
        assert np.all((got >= rne(ref - delta, dtype)) & (got <= rne(ref + delta, dtype)))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_dense3_decode(env, dtype):
    x = _rows(555, 12, torch.float32).double().numpy()
    c, b32 = env["books"][3]
    idx, n16, _ = codec.encode(x, env["s"], b32)
    got = _decode(env, ext.pack_dense3(idx, n16), 3, DENSE3, dtype, stride=70, offset=6)
    _check_decode(got, codec.decode(idx, n16, c, env["s"]), codec.norm_value(n16)[:, None], dtype)


@pytest.mark.parametrize("n", [700, 2600])       # (bf16 / fp16 rows beyond 1024: the tensor-core encode)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_turboq8_encode(env, dtype, n):
    x = _rows(n, 13, dtype)
    tq, dev = env["tq"], env["dev"]
    g = _encode(env, x, 8, 0)
    xd = x.double().numpy()
    idx_o, s_o, t = ext.encode_q8(xd, env["s"])
    idx_g, s_g = ext.unpack_q8(g)
    dist_y = np.abs(t - np.floor(t) - 0.5) / 127.5         # y-distance to a rounding midpoint
    a = np.max(np.abs(oracle.rotate(xd, env["s"])), axis=1)
    _check("turboq8 %s %d" % (dtype, n), idx_g, idx_o, dist_y, s_g, s_o, a)
    # the plain entry point takes a turboq8 codebook as well, and a destination index (the
    # CUDA-core kernel: its codes may differ from the tensor-core ones only at a rounding midpoint)
    dst = torch.randperm(n + 10, generator=torch.Generator().manual_seed(2))[:n]
    slots = torch.zeros((n + 10, 140), dtype=torch.uint8, device=dev)
    tq.tq_encode_kv(x.to(dev), env["cbs"][8], env["signs"], slots, block_stride_bytes=140,
                    dst_index=dst.to(dev))
    torch.cuda.synchronize()
    idx_d, s_d = ext.unpack_q8(slots.cpu().numpy()[dst.numpy(), :130])
    _check("turboq8 %s %d, destination index" % (dtype, n), idx_d, idx_o, dist_y, s_d, s_o, a)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_turboq8_decode(env, dtype):
    x = _rows(640, 14, torch.float32).double().numpy()
    idx, s16, _ = ext.encode_q8(x, env["s"])
    got = _decode(env, ext.pack_q8(idx, s16), 8, 0, dtype, stride=134, offset=2)
    ref = ext.decode_q8(idx, s16, env["s"])
    # errors relative to the vector's norm (the scale is only its largest rotated coordinate)
    nrm = np.linalg.norm(ref, axis=1, keepdims=True)
    _check_decode(got, ref, nrm, dtype)
    # and through the plain entry point
    tq, dev = env["tq"], env["dev"]
    out = torch.empty((x.shape[0], D), dtype=torch.float32, device=dev)
    tq.tq_decode_kv(torch.from_numpy(ext.pack_q8(idx, s16)).to(dev), x.shape[0], env["cbs"][8], env["signs"], out)
    torch.cuda.synchronize()
    _check_decode(out.double().cpu().numpy(), ref, nrm, torch.float32)


def test_ext_argument_errors(env):
    tq = env["tq"]
    assert tq.tq_block_bytes_ex(8, 0) == 130 and tq.tq_block_bytes_ex(3, DENSE3) == 50
    assert tq.tq_block_bytes_ex(4, DENSE3) == 0 and tq.tq_block_bytes_ex(8, NC) == 0
    x = torch.zeros((4, D), dtype=torch.bfloat16, device=env["dev"])
    blk = torch.zeros((4, 66), dtype=torch.uint8, device=env["dev"])
    with pytest.raises(tq.TQError):
        tq.tq_encode_kv_ex(x, env["cbs"][4], env["signs"], blk, flags=DENSE3)
    with pytest.raises(tq.TQError):
        tq.tq_encode_kv_ex(x, env["cbs"][4], env["signs"], blk, flags=8)
