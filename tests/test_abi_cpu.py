"""C-ABI library checks that need no GPU: it builds, loads, exports every
function include/tq.h declares, its host-only functions agree with the
oracle, and argument validation fails before anything is enqueued."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    from turboquant_bit_kv_gb300 import build_lib, tq as mod
    build_lib.build()
    mod.lib()
    return mod


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_expected_calls():
    names = _declared_functions()
    for n in ("tq_codebook_load", "tq_encode_kv", "tq_decode_kv", "tq_attn_decode", "tq_qjl_encode"):
        assert n in names


def test_library_exports_every_declared_symbol(tq):
    L = tq.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_library_codebook_equals_oracle(tq, bits):
    cb = tq.tq_codebook_load(128, bits)
    c, b, _ = oracle.beta_codebook(128, bits)
    assert cb.head_dim == 128 and cb.bits == bits and cb.levels == 1 << bits
    got_c = np.array(cb.centroids[:1 << bits], np.float32)
    got_b = np.array(cb.boundaries[:(1 << bits) - 1], np.float32)
    # two independent Lloyd-Max implementations, both rounded to float32
    assert np.array_equal(got_c, c.astype(np.float32))
    assert np.array_equal(got_b, b.astype(np.float32))


def test_library_signs_equal_oracle(tq):
    for seed in (0, 1, 2, 12345, 2**63 + 7):
        s = tq.tq_signs_from_seed(seed)
        bits = np.array([(s.w[j // 32] >> (j % 32)) & 1 for j in range(128)])
        want = oracle.sign_diagonal(seed)
        assert np.array_equal(np.where(bits == 1, -1.0, 1.0), want)


def test_block_bytes(tq):
    assert [tq.tq_block_bytes(b) for b in (1, 2, 3, 4, 5)] == [0, 34, 50, 66, 0]


@pytest.mark.parametrize("L,T,hidden,bs,sf,sl,kb,vb", [
    (32, 65536, 1024, 16, 2, 2, 4, 4), (5, 21, 256, 8, 1, 1, 4, 2), (3, 16, 128, 16, 2, 2, 3, 3),
    (4, 100, 512, 32, 0, 0, 2, 4), (6, 7, 128, 16, 9, 0, 4, 4)])
def test_serde_size_equals_oracle(tq, L, T, hidden, bs, sf, sl, kb, vb):
    assert tq.tq_serde_size(L, T, hidden, bs, sf, sl, kb, vb) == \
        oracle.serde_size(L, T, hidden, 128, bs, sf, sl, kb, vb)


def test_workspace_bytes(tq):
    assert tq.tq_attn_workspace_bytes(16, 32, 8, 8192) > 0
    assert tq.tq_attn_workspace_bytes(1, 3, 2, 64) == 0
    assert tq.tq_attn_workspace_bytes(0, 8, 8, 64) == 0
    # grows with context until the split count saturates
    assert tq.tq_attn_workspace_bytes(1, 1, 1, 64) <= tq.tq_attn_workspace_bytes(1, 1, 1, 4096)


def _noalloc_limit():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    m = re.search(r"#define TQ_ATTN_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    return int(m.group(1)) << int(m.group(2))


@pytest.mark.parametrize("sms", [148, 152, 160])
def test_noalloc_scratch_covers_the_documented_shapes(tq, sms):
    """The shapes the header says fit tq_attn_decode_noalloc's fixed array
    do fit (at short and very long contexts), and the one it says is
    refused does not."""
    f = tq.lib().tq_attn_workspace_bytes_sms
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 5
    limit = _noalloc_limit()
    assert limit == 16 << 20
    for B, Hq, Hkv in ((64, 28, 4), (64, 32, 8), (128, 32, 8), (16, 32, 8), (8, 32, 8)):
        for T_cap in (4096, 32776, 1 << 20):
            need = f(B, Hq, Hkv, T_cap, sms)
            assert 0 < need <= limit, (B, Hq, Hkv, T_cap, need)
    assert f(256, 32, 8, 4096, sms) > limit
    # the figures quoted in the header, to 0.1 MiB
    for (B, Hq, Hkv), mib in (((64, 28, 4), 11.4), ((64, 32, 8), 9.2), ((128, 32, 8), 14.3), ((256, 32, 8), 24.4)):
        assert abs(f(B, Hq, Hkv, 32776, sms) / 2**20 - mib) < 0.1


def test_status_strings(tq):
    for s in (0, -1, -2, -3, -4, -5, -6, 7):
        assert isinstance(tq.tq_status_string(s), str) and tq.tq_status_string(s)


def test_argument_errors_return_before_enqueue(tq):
    """Each call below fails host validation; the fake device addresses are
    never dereferenced and nothing reaches the GPU."""
    L = tq.lib()
    cb4 = tq.tq_codebook_load(128, 4)
    sg = tq.tq_signs_from_seed(1)
    A = ctypes.c_void_p(0x10000)          # 16-byte aligned fake address
    U = ctypes.c_void_p(0x10002)          # misaligned fake address
    st = ctypes.c_void_p(0)
    assert L.tq_codebook_load(128, 5, ctypes.byref(tq.tq_codebook())) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_codebook_load(80, 4, ctypes.byref(tq.tq_codebook())) == tq.TQ_ERR_UNSUPPORTED   # not a target dim
    assert L.tq_signs_from_seed(1, 96, ctypes.byref(tq.tq_signs())) == tq.TQ_ERR_UNSUPPORTED
    # encode
    assert L.tq_encode_kv(None, 1, 10, 128, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_ERR_ARG
    assert L.tq_encode_kv(A, 1, -1, 128, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_ERR_ARG
    assert L.tq_encode_kv(A, 7, 10, 128, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_encode_kv(U, 1, 10, 128, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_ERR_ALIGN
    assert L.tq_encode_kv(A, 1, 10, 100, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_ERR_ARG
    assert L.tq_encode_kv(A, 1, 10, 132, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_ERR_ALIGN
    assert L.tq_encode_kv(A, 1, 10, 128, ctypes.byref(cb4), sg, A, 65, None, st) == tq.TQ_ERR_ARG
    assert L.tq_encode_kv(A, 1, 10, 128, ctypes.byref(cb4), sg, A, 67, None, st) == tq.TQ_ERR_ALIGN
    assert L.tq_encode_kv(A, 1, 0, 128, ctypes.byref(cb4), sg, A, 66, None, st) == tq.TQ_OK  # no-op
    bad = tq.tq_codebook_load(128, 4)
    bad.levels = 8
    assert L.tq_encode_kv(A, 1, 10, 128, ctypes.byref(bad), sg, A, 66, None, st) == tq.TQ_ERR_UNSUPPORTED
    # decode
    assert L.tq_decode_kv(A, 66, 10, ctypes.byref(cb4), sg, U, 0, 128, st) == tq.TQ_ERR_ALIGN
    assert L.tq_decode_kv(A, 64, 10, ctypes.byref(cb4), sg, A, 0, 128, st) == tq.TQ_ERR_ARG
    # attention
    ws = tq.tq_attn_workspace_bytes(2, 8, 2, 64)

    def attn(**kw):
        a = dict(q=A, qd=1, k=A, kcb=ctypes.byref(cb4), v=A, vcb=ctypes.byref(cb4), sl=None, B=2, Hq=8, Hkv=2,
                 Tc=64, T=64, scale=0.1, bits=None, rn=None, S=None, out=A, ws=A, wsb=ws)
        a.update(kw)
        return L.tq_attn_decode(a["q"], a["qd"], a["k"], a["kcb"], a["v"], a["vcb"], a["sl"], a["B"], a["Hq"],
                                a["Hkv"], a["Tc"], a["T"], ctypes.c_float(a["scale"]), sg, a["bits"], a["rn"],
                                a["S"], a["out"], a["ws"], a["wsb"], st)
    assert attn(T=65) == tq.TQ_ERR_ARG
    assert attn(T=0) == tq.TQ_ERR_ARG
    assert attn(Tc=60, T=60) == tq.TQ_ERR_ARG
    assert attn(Hq=7) == tq.TQ_ERR_ARG
    assert attn(Hq=18) == tq.TQ_ERR_UNSUPPORTED
    assert attn(wsb=ws - 1) == tq.TQ_ERR_WORKSPACE
    assert attn(k=U) == tq.TQ_ERR_ALIGN
    assert attn(bits=A) == tq.TQ_ERR_ARG              # QJL needs all three buffers
    assert attn(scale=float("nan")) == tq.TQ_ERR_ARG
    assert attn(q=None) == tq.TQ_ERR_ARG
    # serde
    assert L.tq_serde_serialize(A, 1, 4, 16, 200, 128, 16, 1, 1, ctypes.byref(cb4), ctypes.byref(cb4), sg, A,
                                st) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_serde_serialize(A, 0, 4, 16, 256, 128, 16, 1, 1, ctypes.byref(cb4), ctypes.byref(cb4), sg, A,
                                st) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_serde_serialize(U, 1, 4, 16, 256, 128, 16, 1, 1, ctypes.byref(cb4), ctypes.byref(cb4), sg, A,
                                st) == tq.TQ_ERR_ALIGN


@pytest.mark.parametrize("d", (64, 96, 160))
@pytest.mark.parametrize("bits", (2, 3, 4))
def test_library_codebook_other_head_dims(tq, d, bits):
    """Codebooks of the spec's other target dims: the library's Lloyd-Max of
    Beta(d/2, d/2) equals the oracle's in float32."""
    cb = tq.tq_codebook_load(d, bits)
    c, b, _ = oracle.beta_codebook(d, bits)
    assert cb.head_dim == d and cb.levels == 1 << bits
    assert np.array_equal(np.array(cb.centroids[:1 << bits], np.float32), c.astype(np.float32))
    assert np.array_equal(np.array(cb.boundaries[:(1 << bits) - 1], np.float32), b.astype(np.float32))
    assert tq.tq_block_bytes_d(d, bits) == 2 + d * bits // 8
    with pytest.raises(tq.TQError):
        tq.tq_codebook_load(80, bits)


def test_library_hadamard_rotation(tq):
    from oracle import headdim
    from turboquant_bit_kv_gb300 import workloads
    s = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    sd = oracle.sign_diagonal(workloads.SIGN_SEED)
    for d in (64, 128):
        R = tq.tq_rotation_hadamard(d, s).double().numpy()
        assert np.allclose(R, headdim.hadamard_rotation(d, sd), rtol=0, atol=1e-7)
    with pytest.raises(tq.TQError):
        tq.tq_rotation_hadamard(96, s)


def test_head_dim_calls_validate_before_launching(tq):
    """Argument errors of the head-dim calls come from the host checks (no GPU needed)."""
    import ctypes
    L = tq.lib()
    cb = tq.tq_codebook_load(96, 3)
    fake = ctypes.c_void_p(1 << 20)
    assert L.tq_encode_kv_d(fake, tq.TQ_F32, 4, 80, ctypes.byref(cb), fake, fake, None) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_encode_kv_d(fake, tq.TQ_F32, 4, 64, ctypes.byref(cb), fake, fake, None) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_encode_kv_d(fake, tq.TQ_F32, 0, 96, ctypes.byref(cb), fake, fake, None) == tq.TQ_OK
    assert L.tq_encode_kv_d(fake, tq.TQ_F32, 4, 96, ctypes.byref(cb), ctypes.c_void_p((1 << 20) + 4), fake,
                            None) == tq.TQ_ERR_ALIGN
    assert L.tq_attn_workspace_bytes_d(2, 8, 2, 1000, 96) > 0
    assert L.tq_attn_workspace_bytes_d(2, 8, 3, 1000, 96) == 0
    # decode attention: T_cap a multiple of 8, block arrays 16-byte aligned
    f = lambda off=0: ctypes.c_void_p((1 << 20) + off)
    big = 1 << 40

    def attn(T_cap, k_off=0, v_off=0):
        return L.tq_attn_decode_d(f(), tq.TQ_F32, f(k_off), ctypes.byref(cb), f(v_off), ctypes.byref(cb), None, 2, 8,
                                  2, T_cap, 50, 96, ctypes.c_float(0.1), f(), f(), f(), big, None)
    assert attn(100) == tq.TQ_ERR_ARG
    assert attn(104, k_off=2) == tq.TQ_ERR_ALIGN
    assert attn(104, v_off=8) == tq.TQ_ERR_ALIGN
