"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs (small and ragged sizes; full sizes are in
test_gpu_fullsize.py)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import codec
from turboquant_bit_kv_gb300 import workloads

from parity_util import ATTN_TOL, attn_rel_err, check_codes, oracle_books, fp16_tie_distance, rne

pytestmark = pytest.mark.gpu

D = 128
GUARD = 64


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    tq.lib()
    dev = torch.device("cuda:0")
    return dict(tq=tq, dev=dev, books=oracle_books(),
                cbs={b: tq.tq_codebook_load(128, b) for b in (2, 3, 4)},
                signs=tq.tq_signs_from_seed(workloads.SIGN_SEED),
                s=oracle.sign_diagonal(workloads.SIGN_SEED))


def _guarded(nbytes, dev, fill=0xA5):
    """uint8 buffer with guard bytes on both sides; returns (full, inner)."""
    full = torch.full((nbytes + 2 * GUARD,), fill, dtype=torch.uint8, device=dev)
    return full, full[GUARD:GUARD + nbytes]


def _guards_intact(full, fill=0xA5):
    g = torch.cat([full[:GUARD], full[-GUARD:]]).cpu().numpy()
    return bool(np.all(g == fill))


def _encode_gpu(env, x, bits, **kw):
    tq = env["tq"]
    n = x.shape[0]
    bb = tq.tq_block_bytes(bits)
    full, blk = _guarded(n * bb, env["dev"])
    tq.tq_encode_kv(x, env["cbs"][bits], env["signs"], blk, **kw)
    torch.cuda.synchronize()
    assert _guards_intact(full)
    return blk.view(n, bb).cpu().numpy()


# ------------------------------------------------------------------ encode

@pytest.mark.parametrize("bits", [2, 3, 4])
def test_encode_single_head_fp32(env, bits):
    w = workloads.single_head(T=4096, seed=0)
    for name in ("k", "v"):
        x = w[name]
        g = _encode_gpu(env, x.to(env["dev"]), bits)
        check_codes(g, bits, x.double().numpy(), env["s"], env["books"][bits][2], "single_head %s" % name)


@pytest.mark.parametrize("bits,src", [(4, "llama"), (2, "llama"), (3, "qwen"), (4, "qwen")])
def test_encode_bf16_workloads_ragged(env, bits, src):
    if src == "llama":
        w = workloads.llama_decode(B=2, Hq=8, Hkv=2, T=1000, seed=3)
    else:
        w = workloads.qwen_outlier(B=2, Hq=14, Hkv=2, T=777, seed=4)
    for name in ("k", "v"):
        x = w[name].reshape(-1, D)          # 4000 / 3108 rows: several tiles + ragged tail
        g = _encode_gpu(env, x.to(env["dev"]), bits)
        check_codes(g, bits, x.double().numpy(), env["s"], env["books"][bits][2], "%s %s" % (src, name))


# Calls of up to 1024 rows use the mma.sync encode kernel, larger ones the
# tcgen05 kernel: the layout and edge-case tests run at both sizes.
SMALL_AND_TC = [333, 2333]


@pytest.mark.parametrize("n", SMALL_AND_TC)
def test_encode_fp16_and_strided_rows(env, n):
    tq = env["tq"]
    gen = torch.Generator().manual_seed(11)
    base = torch.randn((n, 2 * D), generator=gen).to(torch.float16)
    x = base[:, 64:64 + D]                   # row stride 256 elements, offset 64 (128 B)
    g = _encode_gpu(env, base.to(env["dev"])[:, 64:64 + D], 3)
    check_codes(g, 3, x.double().numpy(), env["s"], env["books"][3][2], "fp16 strided")
    assert tq.tq_block_bytes(3) == g.shape[1]


@pytest.mark.parametrize("pad", [0, 2048])
def test_encode_edge_vectors(env, pad):
    rows = [np.zeros(D), np.full(D, 3.0), np.full(D, -0.5), np.eye(D)[5] * 7.0, np.eye(D)[127] * -2.0,
            np.linspace(-1, 1, D) * 1e4, np.linspace(-1, 1, D) * 2.0**-100,
            np.where(np.arange(D) % 2 == 0, 1.0, -1.0), np.r_[np.ones(64), np.zeros(64)]]
    rows += list(np.random.default_rng(13).standard_normal((pad, D)))   # pad: through the tcgen05 kernel
    x = torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16)
    for bits in (2, 3, 4):
        g = _encode_gpu(env, x.to(env["dev"]), bits)
        check_codes(g, bits, x.double().numpy(), env["s"], env["books"][bits][2], "edge")
        idx, n16 = codec.unpack_block(g[:1], bits)
        assert n16[0] == 0 and np.all(idx == (1 << bits) // 2)      # zero vector


def test_encode_listed_rows_in_full_groups(env):
    """Zero, tiny and huge rows scattered through full 32-row groups (whose
    blocks leave by bulk copy before the listed rows are finished); a tensor
    of zero rows with a few random ones; and a tensor of tiny rows, which
    overflows every CTA's list of rows to finish."""
    gen = np.random.default_rng(11)
    x = gen.standard_normal((4096, D))
    special = gen.choice(4096, 200, replace=False)
    x[special[:80]] = 0.0
    x[special[80:140]] *= 2.0**-110
    x[special[140:]] *= 2.0**60
    xt = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)
    for bits in (2, 3, 4):
        g = _encode_gpu(env, xt.to(env["dev"]), bits)
        check_codes(g, bits, xt.double().numpy(), env["s"], env["books"][bits][2], "listed rows")
    z = np.zeros((128 * 700, D))
    z[::997] = gen.standard_normal((z[::997].shape[0], D))
    zt = torch.tensor(z, dtype=torch.float32).to(torch.bfloat16)
    for bits in (3, 4):
        g = _encode_gpu(env, zt.to(env["dev"]), bits)
        check_codes(g, bits, zt.double().numpy(), env["s"], env["books"][bits][2], "zero rows")
    # every row tiny: more listed rows than a CTA's list holds (each CTA rechecks all of its rows)
    t = gen.standard_normal((128 * 400, D)) * 2.0**-110
    tt = torch.tensor(t, dtype=torch.float32).to(torch.bfloat16)
    g = _encode_gpu(env, tt.to(env["dev"]), 2)
    check_codes(g, 2, tt.double().numpy(), env["s"], env["books"][2][2], "tiny rows")


@pytest.mark.parametrize("n,slots", [(37, 100), (1500, 2000)])
def test_encode_scatter_dst_index_and_slot_stride(env, n, slots):
    """Append-style scatter into a slot layout (K block then V block per slot)."""
    tq = env["tq"]
    dev = env["dev"]
    slot = tq.tq_block_bytes(4) + tq.tq_block_bytes(2)
    gen = torch.Generator().manual_seed(5)
    k = torch.randn((n, D), generator=gen).to(torch.bfloat16)
    v = torch.randn((n, D), generator=gen).to(torch.bfloat16)
    dst = torch.randperm(slots, generator=gen)[:n].to(torch.int64)
    full, buf = _guarded(slots * slot, dev, fill=0x3C)
    tq.tq_encode_kv(k.to(dev), env["cbs"][4], env["signs"], buf, block_stride_bytes=slot,
                    dst_index=dst.to(dev))
    tq.tq_encode_kv(v.to(dev), env["cbs"][2], env["signs"], buf, block_stride_bytes=slot,
                    dst_index=dst.to(dev), block_offset=tq.tq_block_bytes(4))
    torch.cuda.synchronize()
    assert _guards_intact(full, 0x3C)
    b = buf.view(slots, slot).cpu().numpy()
    check_codes(b[dst.numpy(), :66], 4, k.double().numpy(), env["s"], env["books"][4][2], "scatter k")
    check_codes(b[dst.numpy(), 66:], 2, v.double().numpy(), env["s"], env["books"][2][2], "scatter v")
    untouched = np.setdiff1d(np.arange(slots), dst.numpy())
    assert np.all(b[untouched] == 0x3C)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("reps", [1, 8])
def test_encode_dst_index_runs(env, bits, reps):
    """Destination indices mixing 32-row groups that form one aligned run of
    consecutive slots (stored in bulk), an unaligned run, a run with one pair
    swapped, a reversed group and a ragged tail: every block lands in its own
    slot and no other slot changes."""
    tq = env["tq"]
    dev = env["dev"]
    bb = tq.tq_block_bytes(bits)
    slots = 600 * reps
    runs = []
    for r in range(reps):                      # reps = 8: 1336 rows, through the tcgen05 kernel
        o = 600 * r
        runs += [np.arange(64, 96) + o,        # aligned run (64 * bb is a multiple of 16)
                 np.arange(101, 133) + o,      # consecutive but unaligned
                 np.r_[np.arange(200, 216), 217, 216, np.arange(218, 232)] + o,   # one pair swapped
                 np.arange(300, 332)[::-1] + o,   # reversed
                 np.arange(400, 432) + o]      # aligned run
    runs.append(np.arange(500, 507) + 600 * (reps - 1))   # ragged tail
    dst = torch.from_numpy(np.concatenate(runs).astype(np.int64))
    n = dst.numel()
    gen = torch.Generator().manual_seed(11 + bits)
    x = torch.randn((n, D), generator=gen).to(torch.bfloat16)
    full, buf = _guarded(slots * bb, dev, fill=0x3C)
    tq.tq_encode_kv(x.to(dev), env["cbs"][bits], env["signs"], buf, dst_index=dst.to(dev))
    torch.cuda.synchronize()
    assert _guards_intact(full, 0x3C)
    b = buf.view(slots, bb).cpu().numpy()
    check_codes(b[dst.numpy()], bits, x.double().numpy(), env["s"], env["books"][bits][2], "runs")
    untouched = np.setdiff1d(np.arange(slots), dst.numpy())
    assert np.all(b[untouched] == 0x3C)


def test_encode_empty_is_noop(env):
    tq = env["tq"]
    full, blk = _guarded(66, env["dev"])
    tq.tq_encode_kv(torch.empty((0, D), dtype=torch.bfloat16, device=env["dev"]), env["cbs"][4],
                    env["signs"], blk)
    torch.cuda.synchronize()
    assert np.all(full.cpu().numpy() == 0xA5)


def test_encode_deterministic(env):
    x = workloads.llama_decode(B=1, Hq=4, Hkv=1, T=300, seed=9)["k"].reshape(-1, D).to(env["dev"])
    a = _encode_gpu(env, x, 4)
    b = _encode_gpu(env, x, 4)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_decode_matches_oracle(env, bits, out_dtype):
    tq = env["tq"]
    dev = env["dev"]
    c, _, b32 = env["books"][bits]
    x = workloads.qwen_outlier(B=1, Hq=7, Hkv=1, T=555, seed=2)["k"].reshape(-1, D).double().numpy()
    idx, n16, _ = codec.encode(x, env["s"], b32)
    blocks = torch.from_numpy(codec.pack_block(idx, n16, bits)).to(dev)
    ref = codec.decode(idx, n16, c, env["s"])
    out = torch.empty((x.shape[0], D), dtype=out_dtype, device=dev)
    tq.tq_decode_kv(blocks, x.shape[0], env["cbs"][bits], env["signs"], out)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    nrm = codec.norm_value(n16)[:, None]
    if out_dtype == torch.float32:
        assert np.max(np.abs(got - ref) / np.maximum(nrm, 1e-30)) < 1e-6
    else:
        # the GPU value must be the correct rounding (nearest even) of some
        # value within the float32 arithmetic error (2e-7 of the vector norm)
        # of the exact one
        delta = 2e-7 * nrm
        lo = rne(ref - delta, out_dtype)
        hi = rne(ref + delta, out_dtype)
        assert np.all((got >= lo) & (got <= hi))


@pytest.mark.parametrize("bits,slot,offset,n,out_dtype", [
    (4, 132, 66, 80, torch.float32),      # V halves of 132-byte storage slots (a 2-byte aligned start)
    (4, 132, 0, 3001, torch.float32),     # K halves: many tiles per warp, a ragged last tile
    (4, 132, 66, 3001, torch.bfloat16),   # the storage layer's bf16 output from V halves
    (4, 132, 0, 777, torch.bfloat16),     # ... and from K halves
    (3, 144, 6, 1000, torch.float32),     # the longest stride staged as one byte span per tile
    (2, 70, 2, 777, torch.float32),       # a short stride: tiles that start at every 2-byte offset in 16
    (2, 146, 10, 500, torch.float32),     # just above the span limit: per-block word staging
    (3, 1024, 512, 300, torch.float32),   # a long stride
])
def test_decode_slot_stride(env, bits, slot, offset, n, out_dtype):
    tq = env["tq"]
    dev = env["dev"]
    c, _, b32 = env["books"][bits]
    x = workloads.qwen_outlier(B=1, Hq=7, Hkv=1, T=n, seed=11 + bits)["k"].reshape(-1, D).double().numpy()
    idx, n16, _ = codec.encode(x, env["s"], b32)
    bb = 2 + 16 * bits
    buf = np.full((n, slot), 0xA5, np.uint8)   # bytes outside the blocks hold a pattern, not zeros
    buf[:, offset:offset + bb] = codec.pack_block(idx, n16, bits)
    out = torch.empty((n, D), dtype=out_dtype, device=dev)
    tq.tq_decode_kv(torch.from_numpy(buf.reshape(-1)).to(dev), n, env["cbs"][bits], env["signs"], out,
                    block_stride_bytes=slot, block_offset=offset)
    torch.cuda.synchronize()
    ref = codec.decode(idx, n16, c, env["s"])
    nrm = codec.norm_value(n16)[:, None]
    got = out.double().cpu().numpy()
    if out_dtype == torch.float32:
        assert np.max(np.abs(got - ref) / np.maximum(nrm, 1e-30)) < 1e-6
    else:
        delta = 2e-7 * nrm
        assert np.all((got >= rne(ref - delta, out_dtype)) & (got <= rne(ref + delta, out_dtype)))


# ------------------------------------------------------------------ attention

def _oracle_cache(env, k, v, kbits, vbits):
    """Oracle-encoded caches: k, v float64 [B, Hkv, T, 128]."""
    B, H, T, _ = k.shape
    out = {}
    for name, x, bits in (("k", k, kbits), ("v", v, vbits)):
        c, _, b32 = env["books"][bits]
        idx, n16, _ = codec.encode(x.reshape(-1, D), env["s"], b32)
        out[name] = (idx.reshape(B, H, T, D), n16.reshape(B, H, T))
        out[name + "_hat"] = codec.decode(idx, n16, c, env["s"]).reshape(B, H, T, D)
        out[name + "_blk"] = codec.pack_block(idx, n16, bits).reshape(B, H, T, -1)
    return out


def _run_attn(env, q, kblk, vblk, kbits, vbits, T, T_cap, scale, seq_lens=None, qjl=None, v_raw=None, vcb=None):
    tq = env["tq"]
    dev = env["dev"]
    B, Hkv = kblk.shape[:2]
    Hq = q.shape[1]
    kb = torch.zeros((B, Hkv, T_cap, kblk.shape[-1]), dtype=torch.uint8)
    kb[:, :, :T] = torch.from_numpy(kblk)
    kb = kb.to(dev)
    if v_raw is None:
        vb = torch.zeros((B, Hkv, T_cap, vblk.shape[-1]), dtype=torch.uint8)
        vb[:, :, :T] = torch.from_numpy(vblk)
        vcb = env["cbs"][vbits] if vcb is None else vcb
    else:
        vb = torch.zeros((B, Hkv, T_cap, D), dtype=torch.float16)
        vb[:, :, :T] = v_raw
        vcb = None
    vb = vb.to(dev)
    out_full = torch.full((B * Hq * D + 2 * 16,), 7.0, dtype=torch.float32, device=dev)
    out = out_full[16:16 + B * Hq * D].view(B, Hq, D)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap), dtype=torch.uint8, device=dev)
    extra = {}
    if qjl is not None:
        bits, rn, S = qjl
        bt = torch.zeros((B, Hkv, T_cap, 16), dtype=torch.uint8)
        bt[:, :, :T] = torch.from_numpy(bits)
        rt = torch.zeros((B, Hkv, T_cap), dtype=torch.int16)
        rt[:, :, :T] = torch.from_numpy(rn.view(np.int16))
        extra = dict(qjl_bits=bt.to(dev), res_norm_f16=rt.to(dev), S=torch.from_numpy(S).float().to(dev))
    sl = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device=dev)
    tq.tq_attn_decode(q.to(dev), kb, env["cbs"][kbits], vb, vcb, out, ws, T, scale, env["signs"], seq_lens=sl,
                      **extra)
    torch.cuda.synchronize()
    o = out_full.cpu().numpy()
    assert np.all(o[:16] == 7.0) and np.all(o[-16:] == 7.0)
    return out.double().cpu().numpy()


@pytest.mark.parametrize("kbits,vbits", [(4, 2), (4, 3), (4, 4), (3, 2)])
def test_attention_single_head(env, kbits, vbits):
    w = workloads.single_head(T=4096, seed=0)
    k = w["k"].double().numpy()[None, None]
    v = w["v"].double().numpy()[None, None]
    q = w["q"][None, None]
    cache = _oracle_cache(env, k, v, kbits, vbits)
    scale = 1 / np.sqrt(D)
    got = _run_attn(env, q, cache["k_blk"], cache["v_blk"], kbits, vbits, 4096, 4096, scale)
    ref = oracle.attention_dequantized(q.double().numpy(), cache["k_hat"], cache["v_hat"], scale)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()


@pytest.mark.parametrize("B,Hq,Hkv,T,T_cap,kbits,vbits,lens", [
    (3, 8, 2, 1000, 1008, 4, 2, [1000, 1, 513]),     # GQA 4:1, ragged lengths
    (2, 14, 2, 300, 304, 3, 3, None),               # GQA 7:1
    (2, 2, 2, 65, 72, 2, 4, None),                  # G = 1
    (1, 4, 2, 130, 136, 4, 4, [129]),               # G = 2
    (2, 16, 2, 200, 200, 2, 2, [0, 200]),           # G = 8, an empty sequence
    (1, 4, 1, 1, 8, 4, 2, None),                    # a single token
    # many short segments: warp chunk ranges span several (sequence, KV head) segments,
    # random lengths with empty sequences among them
    (500, 8, 8, 20, 24, 4, 2, "random"),            # G = 1, one chunk per segment
    (300, 32, 8, 70, 72, 3, 3, "random"),           # G = 4, three chunks per segment
    (100, 56, 8, 45, 48, 3, 3, "random"),           # G = 7 (two n-tiles)
    # few long segments: more than 32 partials per segment, merged by two to four slot groups
    (2, 8, 2, 9000, 9008, 3, 3, [9000, 4500]),      # 58 slots, a ragged second sequence
    (1, 4, 1, 20000, 20000, 4, 2, None),            # 126 slots
    (1, 8, 2, 32768, 32768, 4, 2, None),            # 206 slots: two rounds per group
])
def test_attention_gqa_ragged(env, B, Hq, Hkv, T, T_cap, kbits, vbits, lens):
    if lens == "random":
        lens = [int(x) for x in np.random.default_rng(B).integers(0, T + 1, B)]
        lens[0], lens[-1] = 0, T
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=21)
    k = w["k"].double().numpy()
    v = w["v"].double().numpy()
    cache = _oracle_cache(env, k, v, kbits, vbits)
    scale = 1 / np.sqrt(D)
    got = _run_attn(env, w["q"], cache["k_blk"], cache["v_blk"], kbits, vbits, T, T_cap, scale, seq_lens=lens)
    if lens is not None and 0 in lens:
        zero = [i for i, l in enumerate(lens) if l == 0]
        assert np.all(got[zero] == 0)
        keep = [i for i, l in enumerate(lens) if l > 0]
        ref = oracle.attention_dequantized(w["q"].double().numpy()[keep], cache["k_hat"][keep],
                                           cache["v_hat"][keep], scale, seq_lens=[lens[i] for i in keep])
        got = got[keep]
    else:
        ref = oracle.attention_dequantized(w["q"].double().numpy(), cache["k_hat"], cache["v_hat"], scale,
                                           seq_lens=lens)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()


def test_attention_asymmetric_value_codebook(env):
    """A caller's own value codebook (here the library's 3-bit one with one
    centroid moved, so it is no longer symmetric) is looked up as given: the
    decode matches the oracle decoded with the same centroids."""
    from turboquant_bit_kv_gb300 import tq as tqm
    B, Hq, Hkv, T, T_cap = 2, 14, 2, 300, 304
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=23)
    k = w["k"].double().numpy()
    v = w["v"].double().numpy()
    cache = _oracle_cache(env, k, v, 4, 3)
    moved = np.asarray(env["books"][3][0], np.float32).copy()
    moved[7] = np.float32(moved[7] * 1.25)
    vcb = tqm.tq_codebook.from_buffer_copy(env["cbs"][3])
    vcb.centroids[7] = float(moved[7])
    idx, n16 = cache["v"]
    v_hat = codec.decode(idx.reshape(-1, D), n16.reshape(-1), moved.astype(np.float64),
                         env["s"]).reshape(v.shape)
    scale = 1 / np.sqrt(D)
    got = _run_attn(env, w["q"], cache["k_blk"], cache["v_blk"], 4, 3, T, T_cap, scale, vcb=vcb)
    ref = oracle.attention_dequantized(w["q"].double().numpy(), cache["k_hat"], v_hat, scale)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()
    # the library codebook gives a different result (the moved centroid matters)
    lib = _run_attn(env, w["q"], cache["k_blk"], cache["v_blk"], 4, 3, T, T_cap, scale)
    assert attn_rel_err(lib, got).max() > 10 * ATTN_TOL


def test_attention_identical_keys_give_mean_value(env):
    """All keys equal: the weights are uniform and o is the mean value."""
    B, Hq, Hkv, T = 1, 4, 1, 97
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=5)
    k = np.repeat(w["k"].double().numpy()[:, :, :1], T, axis=2)
    cache = _oracle_cache(env, k, w["v"].double().numpy(), 4, 2)
    got = _run_attn(env, w["q"], cache["k_blk"], cache["v_blk"], 4, 2, T, 104, 1 / np.sqrt(D))
    mean = cache["v_hat"].mean(axis=2)
    assert np.max(attn_rel_err(got, np.repeat(mean, Hq, axis=1))) < ATTN_TOL


def test_attention_qjl_two_term(env):
    B, Hq, Hkv, T, T_cap = 2, 8, 2, 500, 512
    w = workloads.qjl_keys(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=8)
    k = w["k"].double().numpy()
    S = w["S"].double().numpy()
    c3, _, b32 = env["books"][3]
    idx, n16, _ = codec.encode(k.reshape(-1, D), env["s"], b32)
    bits, rn16, _ = oracle.qjl_encode(k.reshape(-1, D), idx, n16, c3, env["s"], S)
    kblk = codec.pack_block(idx, n16, 3).reshape(B, Hkv, T, -1)
    k_hat = codec.decode(idx, n16, c3, env["s"]).reshape(B, Hkv, T, D)
    q = w["q"].double().numpy()
    G = Hq // Hkv
    term2 = np.zeros((B, Hq, T))
    bits4 = bits.reshape(B, Hkv, T, 16)
    rn4 = rn16.reshape(B, Hkv, T)
    for b in range(B):
        for h in range(Hq):
            term2[b, h] = oracle.qjl_term2(q[b, h], bits4[b, h // G], rn4[b, h // G], S)
    v_raw = w["v"]
    scale = 1 / np.sqrt(D)
    got = _run_attn(env, w["q"], kblk, None, 3, None, T, T_cap, scale, qjl=(bits4, rn4, S), v_raw=v_raw)
    ref = oracle.attention_dequantized(q, k_hat, v_raw.double().numpy(), scale, term2=term2)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()


@pytest.mark.parametrize("kbits", [3, 4])
def test_attention_raw_fp16_values(env, kbits):
    B, Hq, Hkv, T, T_cap = 2, 8, 2, 300, 304
    w = workloads.qjl_keys(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=13)
    k = w["k"].double().numpy()
    c, _, b32 = env["books"][kbits]
    idx, n16, _ = codec.encode(k.reshape(-1, D), env["s"], b32)
    kblk = codec.pack_block(idx, n16, kbits).reshape(B, Hkv, T, -1)
    k_hat = codec.decode(idx, n16, c, env["s"]).reshape(B, Hkv, T, D)
    scale = 1 / np.sqrt(D)
    got = _run_attn(env, w["q"], kblk, None, kbits, None, T, T_cap, scale, v_raw=w["v"])
    ref = oracle.attention_dequantized(w["q"].double().numpy(), k_hat, w["v"].double().numpy(), scale)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()


def test_attention_qjl_with_packed_values(env):
    B, Hq, Hkv, T, T_cap = 1, 4, 1, 200, 200
    w = workloads.qjl_keys(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=14)
    k = w["k"].double().numpy()
    v = w["v"].double().numpy()
    S = w["S"].double().numpy()
    c3, _, b32 = env["books"][3]
    idx, n16, _ = codec.encode(k.reshape(-1, D), env["s"], b32)
    bits, rn16, _ = oracle.qjl_encode(k.reshape(-1, D), idx, n16, c3, env["s"], S)
    cache = _oracle_cache(env, k, v, 3, 2)
    q = w["q"].double().numpy()
    term2 = np.stack([oracle.qjl_term2(q[0, h], bits, rn16, S) for h in range(Hq)])[None]
    scale = 1 / np.sqrt(D)
    got = _run_attn(env, w["q"], cache["k_blk"], cache["v_blk"], 3, 2, T, T_cap, scale,
                    qjl=(bits.reshape(B, Hkv, T, 16), rn16.reshape(B, Hkv, T), S))
    ref = oracle.attention_dequantized(q, cache["k_hat"], cache["v_hat"], scale, term2=term2)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()


# ------------------------------------------------------------------ QJL encode

def _check_qjl(env, k, bits, k_row_stride=None, block_pad=0):
    """tq_qjl_encode on keys k (CPU tensor [n, 128]) and oracle-made blocks
    against the oracle: bits may differ only where |(S r)_j| <= 1e-5 ||S_j|| ||r||,
    the fp16 residual norm by one step only within 4e-6 of an fp16 tie."""
    tq = env["tq"]
    dev = env["dev"]
    S = workloads.qjl_keys(B=1, Hq=1, Hkv=1, T=1, seed=0)["S"]
    c, _, b32 = env["books"][bits]
    kx = k.double().numpy()
    n = kx.shape[0]
    idx, n16, _ = codec.encode(kx, env["s"], b32)
    packed = codec.pack_block(idx, n16, bits)
    bb = packed.shape[1]
    stride = bb + block_pad
    blk_host = np.zeros((n, stride), dtype=np.uint8)
    blk_host[:, :bb] = packed
    blk = torch.from_numpy(blk_host.reshape(-1)).to(dev)
    kd = k.to(dev)
    if k_row_stride is not None:
        wide = torch.zeros((n, k_row_stride), dtype=k.dtype, device=dev)
        wide[:, :D] = kd
        kd = wide[:, :D]
    fb, bits_t = _guarded(n * 16, dev)
    fr, rn_b = _guarded(n * 2, dev)
    rn = rn_b.view(torch.int16)
    tq.tq_qjl_encode(kd, blk, env["cbs"][bits], env["signs"], S.to(dev), bits_t, rn, block_stride_bytes=stride)
    torch.cuda.synchronize()
    assert _guards_intact(fb) and _guards_intact(fr)
    ob, orn, proj = oracle.qjl_encode(kx, idx, n16, c, env["s"], S.double().numpy())
    gbits = np.unpackbits(bits_t.view(n, 16).cpu().numpy(), axis=1, bitorder="little")
    obits = np.unpackbits(ob, axis=1, bitorder="little")
    mism = gbits != obits
    r = kx - codec.decode(idx, n16, c, env["s"])
    scale = np.linalg.norm(S.double().numpy(), axis=1)[None, :] * np.linalg.norm(r, axis=1)[:, None]
    assert np.all(np.abs(proj[mism]) <= 1e-5 * scale[mism]), "%d sign bits differ beyond the bound" % (
        np.sum(np.abs(proj[mism]) > 1e-5 * scale[mism]))
    grn = rn.cpu().numpy().view(np.uint16)
    diff = grn.astype(np.int64) - orn.astype(np.int64)
    assert np.all(np.abs(diff) <= 1)
    if np.any(diff != 0):
        assert np.all(fp16_tie_distance(np.linalg.norm(r, axis=1)[diff != 0]) < 4e-6)


def test_qjl_encode_matches_oracle(env):
    w = workloads.qjl_keys(B=1, Hq=4, Hkv=2, T=700, seed=6)
    _check_qjl(env, w["k"].reshape(-1, D), 3)


@pytest.mark.parametrize("bits,dtype,n,row_stride,block_pad", [
    (2, torch.bfloat16, 129, None, 0),        # one full tile + 1 row
    (4, torch.float16, 128, None, 0),         # exactly one tile
    (3, torch.float16, 1, None, 0),           # a single key
    (4, torch.bfloat16, 40000, None, 0),      # several tiles per CTA (the producer / epilogue pipeline)
    (3, torch.bfloat16, 40001, None, 0),      # back-to-back 3-bit blocks: 16-byte staging, ragged last group
    (2, torch.float16, 5000, None, 2),        # padded 2-bit slots: 16-bit staging, pair lookups
    (3, torch.bfloat16, 1000, 192, 4),        # strided key rows, padded block slots (2-byte offsets)
    (2, torch.float32, 300, None, 2),         # float32 keys: CUDA-core kernel
])
def test_qjl_encode_widths_dtypes_layouts(env, bits, dtype, n, row_stride, block_pad):
    w = workloads.qjl_keys(B=1, Hq=1, Hkv=1, T=n, seed=7 + bits)
    _check_qjl(env, w["k"].reshape(-1, D).to(dtype), bits, k_row_stride=row_stride, block_pad=block_pad)


def test_qjl_encode_outlier_keys(env):
    # keys with a few large channels and widely spread norms
    w = workloads.qwen_outlier(B=1, Hq=7, Hkv=1, T=1500, seed=9)
    _check_qjl(env, w["k"].reshape(-1, D), 4)
    _check_qjl(env, w["k"].reshape(-1, D), 2)


# ------------------------------------------------------------------ serde

@pytest.mark.parametrize("L,T,hidden,bs,sf,sl,special", [
    (6, 32, 256, 16, 2, 2, False), (5, 40, 256, 16, 1, 1, False), (3, 16, 128, 16, 2, 2, False),
    # whole 128-row tiles of slots (one paired launch), with zero, tiny and huge rows in both halves
    (4, 64, 1024, 16, 1, 1, True)])
def test_serde_roundtrip_matches_oracle(env, L, T, hidden, bs, sf, sl, special):
    tq = env["tq"]
    dev = env["dev"]
    x = workloads.storage_kv(L=L, T=T, hidden=hidden, seed=12)["kv"]
    if special:
        rows = x.view(2, L, T, hidden // D, D)
        rng = np.random.default_rng(5)
        for kv in (0, 1):
            for l in range(sf, L - sl):
                t = rng.choice(T, 6, replace=False)
                rows[kv, l, t[0:2]] = 0.0
                rows[kv, l, t[2:4]] *= 2.0**-110
                rows[kv, l, t[4:6]] *= 2.0**60
    values = x.double().numpy()
    raw = x.view(torch.uint8).numpy().reshape(2, L, T, hidden * 2)
    (kc, _, kb32), (vc, _, vb32) = env["books"][4], env["books"][4]
    ref = oracle.serialize((values, raw), bs, sf, sl, 4, 4, env["s"], kb32, vb32)
    size = tq.tq_serde_size(L, T, hidden, bs, sf, sl, 4, 4)
    assert size == len(ref)
    full, dst = _guarded(size, dev)
    tq.tq_serde_serialize(x.to(dev), env["cbs"][4], env["cbs"][4], env["signs"], dst, block_size=bs,
                          skip_first=sf, skip_last=sl)
    torch.cuda.synchronize()
    assert _guards_intact(full)
    got = dst.cpu().numpy()
    qs, qe = oracle.serde_ranges(L, sf, sl)
    n_first = 2 * qs * T * hidden * 2
    assert np.array_equal(got[:n_first], ref[:n_first])
    n_comp = (qe - qs) * -(-T // bs) * bs * (hidden // D) * 132
    assert np.array_equal(got[n_first + n_comp:], ref[n_first + n_comp:])
    gc = got[n_first:n_first + n_comp].reshape(qe - qs, -(-T // bs) * bs, hidden // D, 132)
    rc = ref[n_first:n_first + n_comp].reshape(qe - qs, -(-T // bs) * bs, hidden // D, 132)
    assert np.array_equal(gc[:, T:], rc[:, T:])          # zero padding slots
    for li, l in enumerate(range(qs, qe)):
        for kv, off in ((0, 0), (1, 66)):
            blk = gc[li, :T, :, off:off + 66].reshape(-1, 66)
            check_codes(blk, 4, values[kv, l].reshape(-1, D), env["s"], kb32, "serde l%d" % l)
    # deserialise the oracle's bytes on the GPU
    out_full = torch.full((2 * L * T * hidden + 64,), 3.0, dtype=torch.bfloat16, device=dev)
    out = out_full[32:32 + 2 * L * T * hidden].view(2, L, T, hidden)
    tq.tq_serde_deserialize(torch.from_numpy(ref).to(dev), env["cbs"][4], env["cbs"][4], env["signs"], out,
                            block_size=bs, skip_first=sf, skip_last=sl)
    torch.cuda.synchronize()
    o = out_full.float().cpu().numpy()
    assert np.all(o[:32] == 3.0) and np.all(o[-32:] == 3.0)
    rraw, rec, _ = oracle.deserialize(ref, L, T, hidden, bs, sf, sl, 4, 4, env["s"], kc, vc, np.uint16)
    gbytes = out.cpu().view(torch.uint8).numpy().reshape(2, L, T, hidden * 2)
    for l in list(range(qs)) + list(range(qe, L)):
        assert np.array_equal(gbytes[:, l], rraw[:, l])
    grec = out.double().cpu().numpy()
    # each bf16 output must be the correct rounding (nearest even) of some
    # value within the float32 arithmetic error (2e-7 of the block's norm) of
    # the exact one, as in the decode test; the norms come from the slots
    slots = ref[n_first:n_first + n_comp].reshape(qe - qs, -(-T // bs) * bs, hidden // D, 132)[:, :T]
    H = hidden // D
    for li, l in enumerate(range(qs, qe)):
        for kv, off in ((0, 0), (1, 66)):
            n16 = slots[li, :, :, off:off + 2].copy().view(np.uint16)[..., 0]
            nrm = np.repeat(codec.norm_value(n16).reshape(T, H), D, axis=1)
            r = rec[kv, l]
            g = grec[kv, l]
            fin = np.isfinite(r)   # rows whose fp16 norm overflowed decode to inf / NaN on both sides
            delta = 2e-7 * nrm[fin]
            lo = rne(r[fin] - delta, torch.bfloat16)
            hi = rne(r[fin] + delta, torch.bfloat16)
            assert np.all((g[fin] >= lo) & (g[fin] <= hi)), (l, kv)
            assert not np.isfinite(g[~fin]).any()   # the inf / NaN mix depends on the summation order


@pytest.mark.parametrize("kbits,packed_v", [(4, False), (2, True)])
def test_attention_qjl_other_key_widths(env, kbits, packed_v):
    """QJL with 4-bit keys and raw values, or 2-bit keys and 4-bit values
    (the CUDA-core split kernel; the tensor-core kernel covers 3-bit keys)."""
    B, Hq, Hkv, T, T_cap = 2, 6, 2, 150, 152
    w = workloads.qjl_keys(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=15)
    k = w["k"].double().numpy()
    S = w["S"].double().numpy()
    c, _, b32 = env["books"][kbits]
    idx, n16, _ = codec.encode(k.reshape(-1, D), env["s"], b32)
    bits, rn16, _ = oracle.qjl_encode(k.reshape(-1, D), idx, n16, c, env["s"], S)
    kblk = codec.pack_block(idx, n16, kbits).reshape(B, Hkv, T, -1)
    k_hat = codec.decode(idx, n16, c, env["s"]).reshape(B, Hkv, T, D)
    q = w["q"].double().numpy()
    G = Hq // Hkv
    bits4, rn4 = bits.reshape(B, Hkv, T, 16), rn16.reshape(B, Hkv, T)
    term2 = np.zeros((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            term2[b, h] = oracle.qjl_term2(q[b, h], bits4[b, h // G], rn4[b, h // G], S)
    scale = 1 / np.sqrt(D)
    if packed_v:
        cache = _oracle_cache(env, k, w["v"].double().numpy(), kbits, 4)
        got = _run_attn(env, w["q"], kblk, cache["v_blk"], kbits, 4, T, T_cap, scale, qjl=(bits4, rn4, S))
        v_hat = cache["v_hat"]
    else:
        got = _run_attn(env, w["q"], kblk, None, kbits, None, T, T_cap, scale, qjl=(bits4, rn4, S), v_raw=w["v"])
        v_hat = w["v"].double().numpy()
    ref = oracle.attention_dequantized(q, k_hat, v_hat, scale, term2=term2)
    err = attn_rel_err(got, ref)
    assert np.all(err < ATTN_TOL), err.max()
