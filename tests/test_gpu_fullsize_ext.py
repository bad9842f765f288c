"""GPU parity at full size for the further decode workloads (the asymmetric
turboq8 / 4-bit norm-corrected pair, the paged cache, head dims 160 and 128
through a dense rotation), each in
the launch configuration the benchmark times.  As in the other full-size
tests, the oracle checks sampled outputs one by one:

* encode: codes and stored norms or scales of sampled rows;
* attention: a few sampled (sequence, KV head) slices of the cache are
  overwritten with oracle-made blocks before the full-size launch, so those
  slices hold identical packed caches on both sides, and their query heads
  are compared with the oracle's brute-force attention.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import codec, ext, headdim
from turboquant_bit_kv_gb300 import workloads

from parity_util import ATTN_TOL, attn_rel_err, check_codes, check_counted, oracle_books

pytestmark = pytest.mark.gpu

D = 128
B, HQ, HKV, T = 16, 32, 8, 8192          # the Llama-3-8B-shaped decode workloads
G = HQ // HKV
# sampled (sequence, KV head) slices: first and last, and slices in between
SLICES = [(0, 0), (3, 5), (7, 7), (8, 0), (12, 3), (15, 7)]


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    tq.lib()
    return dict(tq=tq, dev=torch.device("cuda:0"), books=oracle_books(),
                cbs={b: tq.tq_codebook_load(128, b) for b in (2, 3, 4, 8)},
                signs=tq.tq_signs_from_seed(workloads.SIGN_SEED), s=oracle.sign_diagonal(workloads.SIGN_SEED))


def _sample_rows(n_rows, n, seed):
    return np.sort(np.random.default_rng(seed).choice(n_rows, size=n, replace=False))


def _compare_heads(q, out, b, h, k_hat, v_hat, scale):
    qs = q[b, h * G:(h + 1) * G].double().cpu().numpy()[None]
    ref = oracle.attention_dequantized(qs, k_hat[None, None], v_hat[None, None], scale)
    err = attn_rel_err(out[b, h * G:(h + 1) * G].double().cpu().numpy()[None], ref)
    assert np.all(err < ATTN_TOL), (b, h, err.max())


def _q8_check(env, blocks, x, label):
    """turboq8 rows: codes exact except at a rounding midpoint, scales except at an fp16 tie."""
    idx_o, s_o, t = ext.encode_q8(x, env["s"])
    idx_g, s_g = ext.unpack_q8(blocks)
    dist_y = np.abs(t - np.floor(t) - 0.5) / 127.5
    a = np.max(np.abs(oracle.rotate(x, env["s"])), axis=1)
    check_counted(label, idx_g, idx_o, dist_y, s_g, s_o, a)


def _nc_check(env, blocks, x, bits, label):
    """Norm-corrected rows: codes as the plain codec, the stored norm ||x|| / ||c[idx]|| of the
    block's own codes."""
    c, _, b32 = env["books"][bits]
    c = c.astype(np.float32).astype(np.float64)        # the library's float32 codebook
    idx_o, _, y, _ = ext.encode_nc(x, env["s"], c, b32)
    idx_g, n_g = codec.unpack_block(blocks, bits)
    dist = np.min(np.abs(y[..., None] - b32.astype(np.float64)[None, None, :]), axis=-1)
    r = ext.recon_norm(idx_g, c)
    nx = np.linalg.norm(x, axis=1)
    exact = np.where(nx > 0, nx / np.where(r > 0, r, 1.0), 0.0)
    check_counted(label, idx_g, idx_o, dist, n_g, codec.fp16_rne(exact), exact)


def test_turboq8_pair_fullsize(env):
    """Batch 16, 32/8 heads, context 8192, bf16 K/V: turboq8 keys (130-byte
    blocks) and 4-bit norm-corrected values through tq_encode_kv_ex (the
    tensor-core encodes), one decode step on the split-K kernels."""
    tq, dev = env["tq"], env["dev"]
    w = workloads.llama_decode(B=B, Hq=HQ, Hkv=HKV, T=T, seed=0, device=dev)
    k, v, q = w["k"], w["v"], w["q"]
    nvec = B * HKV * T
    kb = torch.empty((B, HKV, T, 130), dtype=torch.uint8, device=dev)
    vb = torch.empty((B, HKV, T, 66), dtype=torch.uint8, device=dev)
    tq.tq_encode_kv_ex(k.view(-1, D), env["cbs"][8], env["signs"], kb)
    tq.tq_encode_kv_ex(v.view(-1, D), env["cbs"][4], env["signs"], vb, flags=tq.TQ_FMT_NORM_CORRECT)
    torch.cuda.synchronize()
    rows = torch.from_numpy(_sample_rows(nvec, 8192, 21)).to(dev)
    _q8_check(env, kb.view(nvec, -1)[rows].cpu().numpy(), k.view(-1, D)[rows].double().cpu().numpy(),
              "turboq8 pair K (full size)")
    rows = torch.from_numpy(_sample_rows(nvec, 8192, 22)).to(dev)
    _nc_check(env, vb.view(nvec, -1)[rows].cpu().numpy(), v.view(-1, D)[rows].double().cpu().numpy(), 4,
              "turboq8 pair V nc (full size)")

    hats = {}
    c4 = env["books"][4][0].astype(np.float32).astype(np.float64)
    for b, h in SLICES:
        xk = k[b, h].double().cpu().numpy()
        idx, s16, _ = ext.encode_q8(xk, env["s"])
        kb[b, h] = torch.from_numpy(ext.pack_q8(idx, s16)).to(dev)
        khat = ext.decode_q8(idx, s16, env["s"])
        xv = v[b, h].double().cpu().numpy()
        vidx, vn16, _, _ = ext.encode_nc(xv, env["s"], c4, env["books"][4][2])
        vb[b, h] = torch.from_numpy(codec.pack_block(vidx, vn16, 4)).to(dev)
        hats[(b, h)] = (khat, codec.decode(vidx, vn16, c4, env["s"]))
    out = torch.empty((B, HQ, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, HQ, HKV, T), dtype=torch.uint8, device=dev)
    scale = 1 / np.sqrt(D)
    tq.tq_attn_decode(q, kb, env["cbs"][8], vb, env["cbs"][4], out, ws, T, scale, env["signs"])
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    for b, h in SLICES:
        _compare_heads(q, out, b, h, *hats[(b, h)], scale)


def test_paged_decode_fullsize(env):
    """Batch 16, 32/8 heads, context 8192, K4/V2 in a pool of 32-token pages
    assigned in a seeded shuffled order: every token encoded into its page
    slot through a destination index, one decode step through the block
    table on the split-K kernels."""
    tq, dev = env["tq"], env["dev"]
    P = 32
    per = T // P
    w = workloads.llama_decode(B=B, Hq=HQ, Hkv=HKV, T=T, seed=0, device=dev)
    k, v, q = w["k"], w["v"], w["q"]
    table = torch.randperm(B * per, generator=torch.Generator().manual_seed(7)).view(B, per).to(torch.int32).to(dev)
    t = torch.arange(T, device=dev)
    pg = table.long()[:, None, t // P]
    dst = ((pg * HKV + torch.arange(HKV, device=dev)[None, :, None]) * P + (t % P)[None, None, :]).reshape(-1)
    kp = torch.empty((B * per, HKV, P, 66), dtype=torch.uint8, device=dev)
    vp = torch.empty((B * per, HKV, P, 34), dtype=torch.uint8, device=dev)
    tq.tq_encode_kv(k.view(-1, D), env["cbs"][4], env["signs"], kp.view(-1, 66), dst_index=dst)
    tq.tq_encode_kv(v.view(-1, D), env["cbs"][2], env["signs"], vp.view(-1, 34), dst_index=dst)
    torch.cuda.synchronize()
    nvec = B * HKV * T
    for name, x, pool, bits, seed in (("K", k, kp, 4, 23), ("V", v, vp, 2, 24)):
        rows = torch.from_numpy(_sample_rows(nvec, 8192, seed)).to(dev)
        got = pool.view(-1, pool.shape[-1])[dst[rows]].cpu().numpy()
        check_codes(got, bits, x.view(-1, D)[rows].double().cpu().numpy(), env["s"], env["books"][bits][2],
                    "paged %s (full size)" % name)

    hats = {}
    tab = table.cpu().numpy()
    for b, h in SLICES:
        pair = []
        for x, pool, bits in ((k, kp, 4), (v, vp, 2)):
            c, _, b32 = env["books"][bits]
            idx, n16, _ = codec.encode(x[b, h].double().cpu().numpy(), env["s"], b32)
            blk = torch.from_numpy(codec.pack_block(idx, n16, bits)).to(dev).view(per, P, -1)
            for p in range(per):
                pool[int(tab[b, p]), h] = blk[p]
            pair.append(codec.decode(idx, n16, c, env["s"]))
        hats[(b, h)] = tuple(pair)
    out = torch.empty((B, HQ, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, HQ, HKV, T), dtype=torch.uint8, device=dev)
    scale = 1 / np.sqrt(D)
    tq.tq_attn_decode_paged(q, kp, env["cbs"][4], vp, env["cbs"][2], table, P, out, T, scale, env["signs"],
                            workspace=ws)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    for b, h in SLICES:
        _compare_heads(q, out, b, h, *hats[(b, h)], scale)


@pytest.mark.parametrize("d,Hq", [(160, 32), (128, 64)])
def test_headdim_fullsize(env, d, Hq):
    """Batch 8, 8 KV heads, context 8192, bf16 K/V, K4/V2 through a seeded
    dense orthogonal rotation: head dim 160 with 32 query heads (4 per KV
    head) and head dim 128 with 64 (8 per KV head: the attention kernel's
    eight-head variant); the tensor-core encodes and one decode step (prep,
    tensor-core attention, combine)."""
    tq, dev = env["tq"], env["dev"]
    Bh = 8
    Gh = Hq // HKV
    a = np.random.default_rng(d).standard_normal((d, d))
    qm, r = np.linalg.qr(a)
    R32 = (qm * np.sign(np.diag(r))[None, :]).astype(np.float32)
    R = R32.astype(np.float64)
    Rd = torch.from_numpy(R32).to(dev)
    g = torch.Generator(device=dev).manual_seed(d)
    k = torch.randn((Bh, HKV, T, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((Bh, HKV, T, d), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((Bh, Hq, d), generator=g, device=dev).to(torch.bfloat16)
    books = {}
    for bits in (2, 4):
        c, bd, _ = oracle.beta_codebook(d, bits)
        books[bits] = (c.astype(np.float32).astype(np.float64), bd.astype(np.float32))
    nvec = Bh * HKV * T
    blocks = {}
    for name, x, bits, seed in (("K", k, 4, 25), ("V", v, 2, 26)):
        blk = torch.empty((Bh, HKV, T, tq.tq_block_bytes_d(d, bits)), dtype=torch.uint8, device=dev)
        tq.tq_encode_kv_d(x.view(-1, d), tq.tq_codebook_load(d, bits), Rd, blk.view(nvec, -1))
        torch.cuda.synchronize()
        rows = torch.from_numpy(_sample_rows(nvec, 8192, seed)).to(dev)
        xs = x.view(-1, d)[rows].double().cpu().numpy()
        idx_o, n16_o, y = headdim.encode_d(xs, R, books[bits][1])
        idx_g, n16_g = headdim.unpack_d(blk.view(nvec, -1)[rows].cpu().numpy(), d, bits)
        dist = np.min(np.abs(y[..., None] - books[bits][1].astype(np.float64)[None, None, :]), axis=-1)
        check_counted("head dim %d %s (full size)" % (d, name), idx_g, idx_o, dist, n16_g, n16_o,
                      np.linalg.norm(xs, axis=1), tie=2.0**-22)
        blocks[name] = blk

    hats = {}
    for b, h in ((0, 0), (3, 5), (5, 2), (7, 7)):
        pair = []
        for name, x, bits in (("K", k, 4), ("V", v, 2)):
            idx, n16, _ = headdim.encode_d(x[b, h].double().cpu().numpy(), R, books[bits][1])
            blocks[name][b, h] = torch.from_numpy(headdim.pack_d(idx, n16, bits)).to(dev)
            pair.append(headdim.decode_d(idx, n16, books[bits][0], R))
        hats[(b, h)] = tuple(pair)
    out = torch.empty((Bh, Hq, d), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes_d(Bh, Hq, HKV, T, d), dtype=torch.uint8, device=dev)
    scale = 1 / np.sqrt(d)
    tq.tq_attn_decode_d(q, blocks["K"], tq.tq_codebook_load(d, 4), blocks["V"], tq.tq_codebook_load(d, 2), Rd, out,
                        ws, T, scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    for (b, h), (k_hat, v_hat) in hats.items():
        qs = q[b, h * Gh:(h + 1) * Gh].double().cpu().numpy()[None]
        ref = oracle.attention_dequantized(qs, k_hat[None, None], v_hat[None, None], scale)
        err = attn_rel_err(out[b, h * Gh:(h + 1) * Gh].double().cpu().numpy()[None], ref)
        assert np.all(err < ATTN_TOL), (b, h, err.max())
