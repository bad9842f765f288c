"""GPU parity of the multi-token (causal) attention over packed caches
(tq_attn_prefill, tensor cores): the oracle's brute-force causal attention
on identical packed caches made by the oracle's encoder, per output vector
max |o - o_ref| / max |o_ref| <= 1e-3."""

import numpy as np
import pytest
import torch

import oracle
from oracle import codec, ext
from turboquant_bit_kv_gb300 import workloads

from parity_util import ATTN_TOL, attn_rel_err, oracle_books

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    tq.lib()
    return dict(tq=tq, dev=torch.device("cuda:0"), books=oracle_books(),
                cbs={b: tq.tq_codebook_load(128, b) for b in (2, 3, 4, 8)},
                signs=tq.tq_signs_from_seed(workloads.SIGN_SEED), s=oracle.sign_diagonal(workloads.SIGN_SEED))


def _cache(env, x, bits):
    """Oracle blocks and reconstructions of x float64 [B, H, T, 128]."""
    B, H, T, _ = x.shape
    if bits == 8:
        idx, s16, _ = ext.encode_q8(x.reshape(-1, D), env["s"])
        return (ext.pack_q8(idx, s16).reshape(B, H, T, -1),
                ext.decode_q8(idx, s16, env["s"]).reshape(B, H, T, D))
    c, _, b32 = env["books"][bits]
    idx, n16, _ = codec.encode(x.reshape(-1, D), env["s"], b32)
    return (codec.pack_block(idx, n16, bits).reshape(B, H, T, -1),
            codec.decode(idx, n16, c, env["s"]).reshape(B, H, T, D))


def _run(env, q, kblk, vblk, kbits, vbits, T, T_cap, scale, lens=None):
    tq, dev = env["tq"], env["dev"]
    B, Hkv = kblk.shape[:2]
    M, Hq = q.shape[1], q.shape[2]
    kb = torch.zeros((B, Hkv, T_cap, kblk.shape[-1]), dtype=torch.uint8)
    kb[:, :, :T] = torch.from_numpy(kblk)
    vb = torch.zeros((B, Hkv, T_cap, vblk.shape[-1]), dtype=torch.uint8)
    vb[:, :, :T] = torch.from_numpy(vblk)
    n = B * M * Hq * D
    out_full = torch.full((n + 32,), 7.0, dtype=torch.float32, device=dev)
    out = out_full[16:16 + n].view(B, M, Hq, D)
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    tq.tq_attn_prefill(q.to(dev), kb.to(dev), env["cbs"][kbits], vb.to(dev), env["cbs"][vbits], out, T, scale,
                       env["signs"], seq_lens=sl)
    torch.cuda.synchronize()
    o = out_full.cpu().numpy()
    assert np.all(o[:16] == 7.0) and np.all(o[-16:] == 7.0)
    return out.double().cpu().numpy()


@pytest.mark.parametrize("B,M,Hq,Hkv,T,T_cap,kbits,vbits,lens,qdt", [
    (2, 16, 8, 2, 300, 304, 4, 2, None, torch.float32),            # one row tile, a ragged key tile
    (2, 16, 8, 2, 300, 304, 4, 2, [300, 150], torch.bfloat16),     # ragged lengths
    (1, 24, 28, 4, 257, 264, 3, 3, None, torch.bfloat16),          # 7 heads per KV head: 168 rows, two row tiles
    (3, 20, 8, 4, 200, 200, 4, 4, [200, 7, 64], torch.float16),    # a sequence shorter than M: zero rows
    (2, 1, 32, 8, 129, 136, 3, 2, [129, 65], torch.bfloat16),      # one query token: the decode case
    (1, 64, 32, 8, 1000, 1000, 4, 2, None, torch.bfloat16),        # 256 rows per KV head, 16 key tiles
    (2, 16, 8, 2, 300, 304, 8, 4, [300, 99], torch.bfloat16),      # turboq8 keys, 4-bit values
    (1, 24, 28, 4, 257, 264, 8, 2, None, torch.float16),           # turboq8 keys, 2-bit values, 7 heads
    (2, 12, 8, 4, 150, 152, 4, 8, [150, 40], torch.float32),       # 4-bit keys, turboq8 values
])
def test_prefill_matches_oracle(env, B, M, Hq, Hkv, T, T_cap, kbits, vbits, lens, qdt):
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=30 + M)
    kblk, khat = _cache(env, w["k"].double().numpy(), kbits)
    vblk, vhat = _cache(env, w["v"].double().numpy(), vbits)
    q = torch.randn((B, M, Hq, D), generator=torch.Generator().manual_seed(M + Hq), dtype=torch.float32).to(qdt)
    scale = 1 / np.sqrt(D)
    got = _run(env, q, kblk, vblk, kbits, vbits, T, T_cap, scale, lens)
    ref = oracle.attention_causal(q.double().numpy(), khat, vhat, scale, seq_lens=lens)
    err = attn_rel_err(got.reshape(-1, D), ref.reshape(-1, D))
    assert np.all(err < ATTN_TOL), err.max()
    if lens is not None:
        for b, L in enumerate(lens):
            assert np.all(got[b, :max(0, M - L)] == 0)   # queries before the first cached token


def test_prefill_decode_agreement(env):
    """With one query token the causal attention is the decode attention:
    the two entry points agree on the same cache."""
    tq, dev = env["tq"], env["dev"]
    B, Hq, Hkv, T = 2, 16, 4, 777
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=3)
    kblk, _ = _cache(env, w["k"].double().numpy(), 4)
    vblk, _ = _cache(env, w["v"].double().numpy(), 2)
    scale = 1 / np.sqrt(D)
    got = _run(env, w["q"][:, None], kblk, vblk, 4, 2, T, 784, scale)
    kb = torch.zeros((B, Hkv, 784, 66), dtype=torch.uint8)
    kb[:, :, :T] = torch.from_numpy(kblk)
    vb = torch.zeros((B, Hkv, 784, 34), dtype=torch.uint8)
    vb[:, :, :T] = torch.from_numpy(vblk)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, 784), dtype=torch.uint8, device=dev)
    tq.tq_attn_decode(w["q"].to(dev), kb.to(dev), env["cbs"][4], vb.to(dev), env["cbs"][2], out, ws, T, scale,
                      env["signs"])
    torch.cuda.synchronize()
    err = attn_rel_err(got[:, 0].reshape(-1, D), out.double().cpu().numpy().reshape(-1, D))
    assert np.all(err < 2 * ATTN_TOL), err.max()


@pytest.mark.parametrize("kbits,vbits,Hq,ws_full", [
    (8, 4, 12, True), (8, 3, 12, True), (8, 2, 12, True), (4, 8, 12, True),   # split-K tensor-core path, G = 4
    (8, 4, 21, True), (4, 8, 21, True),                                      # G = 7 (the eight-head n-tile)
    (8, 4, 12, False), (4, 8, 21, False),                                    # no workspace: the causal kernel
])
def test_decode_attention_turboq8_pairs(env, kbits, vbits, Hq, ws_full):
    """tq_attn_decode over turboq8 keys or values (the asymmetric pairs): the
    oracle's attention on identical packed caches, on the split-K decode path
    (a full workspace) and on the one-token causal kernel (a workspace too
    small for the split-K partials)."""
    tq, dev = env["tq"], env["dev"]
    B, Hkv, T, T_cap = 3, 3, 500, 504
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=50 + kbits + vbits)
    kblk, khat = _cache(env, w["k"].double().numpy(), kbits)
    vblk, vhat = _cache(env, w["v"].double().numpy(), vbits)
    kb = torch.zeros((B, Hkv, T_cap, kblk.shape[-1]), dtype=torch.uint8)
    kb[:, :, :T] = torch.from_numpy(kblk)
    vb = torch.zeros((B, Hkv, T_cap, vblk.shape[-1]), dtype=torch.uint8)
    vb[:, :, :T] = torch.from_numpy(vblk)
    lens = [500, 123, 1]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap) if ws_full else 16, dtype=torch.uint8, device=dev)
    scale = 1 / np.sqrt(D)
    tq.tq_attn_decode(w["q"].to(dev), kb.to(dev), env["cbs"][kbits], vb.to(dev), env["cbs"][vbits], out, ws, T,
                      scale, env["signs"], seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    ref = oracle.attention_dequantized(w["q"].double().numpy(), khat, vhat, scale, seq_lens=lens)
    err = attn_rel_err(out.double().cpu().numpy().reshape(-1, D), ref.reshape(-1, D))
    assert np.all(err < ATTN_TOL), err.max()


def _paged(kblk, vblk, page, rng):
    """Scatter contiguous caches [B, Hkv, T, bytes] into shuffled pages of a
    pool [pages, Hkv, page, bytes]; returns (k_pool, v_pool, table int32)."""
    B, Hkv, T = kblk.shape[:3]
    per = -(-T // page)
    n_pages = B * per + 3                         # spare pages nothing points to
    order = rng.permutation(n_pages)[:B * per].reshape(B, per)
    kp = np.full((n_pages, Hkv, page, kblk.shape[-1]), 0xEE, np.uint8)
    vp = np.full((n_pages, Hkv, page, vblk.shape[-1]), 0xEE, np.uint8)
    for b in range(B):
        for p in range(per):
            t0, t1 = p * page, min(T, (p + 1) * page)
            kp[order[b, p], :, :t1 - t0] = kblk[b, :, t0:t1]
            vp[order[b, p], :, :t1 - t0] = vblk[b, :, t0:t1]
    table = np.concatenate([order, np.full((B, 2), 10**6)], axis=1).astype(np.int32)   # unused tail entries
    return kp, vp, table


@pytest.mark.parametrize("page,M,kbits,vbits,lens", [
    (16, 16, 4, 2, [300, 77]),     # vLLM-sized pages, ragged lengths
    (40, 24, 3, 3, [299, 300]),    # a page size that is no power of two
    (64, 1, 8, 4, [300, 5]),       # decode over a paged turboq8 / 4-bit cache
])
def test_paged_matches_oracle(env, page, M, kbits, vbits, lens):
    tq, dev = env["tq"], env["dev"]
    B, Hq, Hkv, T = 2, 8, 2, 300
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=70 + page)
    kblk, khat = _cache(env, w["k"].double().numpy(), kbits)
    vblk, vhat = _cache(env, w["v"].double().numpy(), vbits)
    kp, vp, table = _paged(kblk, vblk, page, np.random.default_rng(page))
    scale = 1 / np.sqrt(D)
    q = torch.randn((B, M, Hq, D), generator=torch.Generator().manual_seed(page), dtype=torch.float32).to(
        torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    args = (torch.from_numpy(kp).to(dev), env["cbs"][kbits], torch.from_numpy(vp).to(dev), env["cbs"][vbits],
            torch.from_numpy(table).to(dev), page)
    if M == 1:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
        tq.tq_attn_decode_paged(q[:, 0].to(dev), *args, out, T, scale, env["signs"], seq_lens=sl)
        got = out.double().cpu().numpy()[:, None]
    else:
        out = torch.empty((B, M, Hq, D), dtype=torch.float32, device=dev)
        tq.tq_attn_prefill_paged(q.to(dev), *args, out, T, scale, env["signs"], seq_lens=sl)
        got = out.double().cpu().numpy()
    torch.cuda.synchronize()
    ref = oracle.attention_causal(q.double().numpy(), khat, vhat, scale, seq_lens=lens)
    err = attn_rel_err(got.reshape(-1, D), ref.reshape(-1, D))
    assert np.all(err < ATTN_TOL), err.max()


def test_circular_cache_and_eviction(env):
    """The spec's Integration Points: a circular cache written at
    pos % T_cap (through a destination index) holds the last T_cap tokens,
    and attention over the full window is the attention over those tokens;
    evicting the oldest tokens by moving packed bytes (a device memmove)
    keeps every remaining block's value."""
    tq, dev = env["tq"], env["dev"]
    B, Hq, Hkv, T_cap, total = 1, 8, 2, 256, 400
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=total, seed=81)
    k, v = w["k"].to(dev), w["v"].to(dev)
    kb = torch.zeros((B, Hkv, T_cap, 66), dtype=torch.uint8, device=dev)
    vb = torch.zeros((B, Hkv, T_cap, 34), dtype=torch.uint8, device=dev)
    for h in range(Hkv):
        pos = torch.arange(total, device=dev)
        dst = h * T_cap + pos % T_cap                # later positions overwrite the oldest slots
        # positions are written in order, so the last write to a slot is the newest token
        for start in range(0, total, T_cap):
            sel = slice(start, min(total, start + T_cap))
            tq.tq_encode_kv(k[0, h, sel].contiguous(), env["cbs"][4], env["signs"], kb.view(-1, 66),
                            dst_index=dst[sel].contiguous())
            tq.tq_encode_kv(v[0, h, sel].contiguous(), env["cbs"][2], env["signs"], vb.view(-1, 34),
                            dst_index=dst[sel].contiguous())
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap), dtype=torch.uint8, device=dev)
    scale = 1 / np.sqrt(D)
    tq.tq_attn_decode(w["q"].to(dev), kb, env["cbs"][4], vb, env["cbs"][2], out, ws, T_cap, scale, env["signs"])
    torch.cuda.synchronize()
    # the oracle over the last T_cap tokens (attention does not depend on their slot order)
    last = slice(total - T_cap, total)
    khat = _cache(env, w["k"][:, :, last].double().numpy(), 4)[1]
    vhat = _cache(env, w["v"][:, :, last].double().numpy(), 2)[1]
    ref = oracle.attention_dequantized(w["q"].double().numpy(), khat, vhat, scale)
    assert np.all(attn_rel_err(out.double().cpu().numpy().reshape(-1, D), ref.reshape(-1, D)) < ATTN_TOL)
    # eviction: drop the 100 oldest tokens of a linear cache by moving the packed bytes down
    lin_k = torch.zeros((B, Hkv, T_cap, 66), dtype=torch.uint8, device=dev)
    lin_v = torch.zeros((B, Hkv, T_cap, 34), dtype=torch.uint8, device=dev)
    for h in range(Hkv):
        tq.tq_encode_kv(k[0, h, :T_cap].contiguous(), env["cbs"][4], env["signs"], lin_k[0, h])
        tq.tq_encode_kv(v[0, h, :T_cap].contiguous(), env["cbs"][2], env["signs"], lin_v[0, h])
    before = torch.empty((T_cap - 100, D), dtype=torch.float32, device=dev)
    tq.tq_decode_kv(lin_k[0, 1, 100:], T_cap - 100, env["cbs"][4], env["signs"], before)
    kept = lin_k[:, :, 100:].clone()
    lin_k[:, :, :T_cap - 100] = kept
    lin_v[:, :, :T_cap - 100] = lin_v[:, :, 100:].clone()
    after = torch.empty((T_cap - 100, D), dtype=torch.float32, device=dev)
    tq.tq_decode_kv(lin_k[0, 1, :T_cap - 100], T_cap - 100, env["cbs"][4], env["signs"], after)
    torch.cuda.synchronize()
    assert torch.equal(before, after)             # moved bytes decode to the same values
    tq.tq_attn_decode(w["q"].to(dev), lin_k, env["cbs"][4], lin_v, env["cbs"][2], out, ws, T_cap - 100, scale,
                      env["signs"])
    torch.cuda.synchronize()
    khat = _cache(env, w["k"][:, :, 100:T_cap].double().numpy(), 4)[1]
    vhat = _cache(env, w["v"][:, :, 100:T_cap].double().numpy(), 2)[1]
    ref = oracle.attention_dequantized(w["q"].double().numpy(), khat, vhat, scale)
    assert np.all(attn_rel_err(out.double().cpu().numpy().reshape(-1, D), ref.reshape(-1, D)) < ATTN_TOL)


@pytest.mark.parametrize("page,kbits,vbits,Hq,Hkv,lens", [
    (32, 4, 2, 16, 4, [700, 333, 32]),      # the split-K decode kernels through the block table
    (64, 3, 3, 28, 4, [700, 701, 1]),       # 7 heads per KV head (two n-tiles), a one-token sequence
    (96, 2, 4, 8, 8, [650, 96, 95]),        # page boundaries at 96-token steps
])
def test_paged_decode_split_k(env, page, kbits, vbits, Hq, Hkv, lens):
    tq, dev = env["tq"], env["dev"]
    B, T = 3, 701
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=90 + page)
    kblk, khat = _cache(env, w["k"].double().numpy(), kbits)
    vblk, vhat = _cache(env, w["v"].double().numpy(), vbits)
    kp, vp, table = _paged(kblk, vblk, page, np.random.default_rng(page + 1))
    scale = 1 / np.sqrt(D)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, (T + 7) // 8 * 8), dtype=torch.uint8, device=dev)
    tq.tq_attn_decode_paged(w["q"].to(dev), torch.from_numpy(kp).to(dev), env["cbs"][kbits],
                            torch.from_numpy(vp).to(dev), env["cbs"][vbits], torch.from_numpy(table).to(dev), page,
                            out, T, scale, env["signs"], seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev),
                            workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.attention_dequantized(w["q"].double().numpy(), khat, vhat, scale, seq_lens=lens)
    err = attn_rel_err(out.double().cpu().numpy().reshape(-1, D), ref.reshape(-1, D))
    assert np.all(err < ATTN_TOL), err.max()
