"""tq_attn_decode_noalloc: the attention entry point for callers that cannot
allocate device memory (for example an engine whose memory all sits in its
own pre-reserved pool, or a plugin that is handed only its input and output
buffers).  It keeps its split-K scratch in a fixed device array inside the
library.  Checked here through the C ABI against tq_attn_decode (which takes a
caller-allocated workspace) on two calls in a row, with the attention
tolerance the other parity tests use.  This file is collected last so that a
run stopping at the first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

from turboquant_bit_kv_gb300 import workloads

pytestmark = pytest.mark.gpu

ATTN_TOL = 1e-3


def _rel(got, ref):
    den = np.max(np.abs(ref), axis=-1)
    return np.max(np.abs(got - ref), axis=-1) / np.where(den > 0, den, 1.0)


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    L = tq.lib()
    L.tq_attn_decode_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.POINTER(tq.tq_codebook), ctypes.c_void_p,
                                         ctypes.POINTER(tq.tq_codebook), ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                         tq.tq_signs, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]
    dev = torch.device("cuda:0")
    B, Hq, Hkv, T, T_cap = 4, 16, 4, 3000, 3008
    kcb, vcb = tq.tq_codebook_load(128, 4), tq.tq_codebook_load(128, 2)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    stream = torch.cuda.current_stream(dev)
    scale = 1 / np.sqrt(128)
    outs_ref, outs_new = [], []
    for call in range(2):
        w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=40 + call, device=dev)
        kb = torch.zeros((B, Hkv, T_cap, 66), dtype=torch.uint8, device=dev)
        vb = torch.zeros((B, Hkv, T_cap, 34), dtype=torch.uint8, device=dev)
        for b in range(B):
            for h in range(Hkv):
                tq.tq_encode_kv(w["k"][b, h], kcb, signs, kb[b, h])
                tq.tq_encode_kv(w["v"][b, h], vcb, signs, vb[b, h])
        lens = torch.tensor([T, T - 1, 1, 1234 + call], dtype=torch.int32, device=dev)
        ref = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
        ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap), dtype=torch.uint8, device=dev)
        tq.tq_attn_decode(w["q"], kb, kcb, vb, vcb, ref, ws, T, scale, signs, seq_lens=lens)
        new = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
        st = L.tq_attn_decode_noalloc(ctypes.c_void_p(w["q"].data_ptr()), tq.TQ_BF16,
                                      ctypes.c_void_p(kb.data_ptr()), ctypes.byref(kcb),
                                      ctypes.c_void_p(vb.data_ptr()), ctypes.byref(vcb),
                                      ctypes.c_void_p(lens.data_ptr()), B, Hq, Hkv, T_cap, T,
                                      ctypes.c_float(scale), signs, None, None, None,
                                      ctypes.c_void_p(new.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        torch.cuda.synchronize(dev)
        outs_ref.append(ref.double().cpu().numpy())
        outs_new.append(new.double().cpu().numpy())
    for r, n in zip(outs_ref, outs_new):
        assert np.all(np.isfinite(n))
        assert np.all(_rel(n, r) <= ATTN_TOL)
    # the two calls saw different inputs, so the shared scratch was reused
    assert not np.allclose(outs_new[0], outs_new[1])
    # a shape whose scratch would not fit is refused before any launch
    big = L.tq_attn_decode_noalloc(ctypes.c_void_p(w["q"].data_ptr()), tq.TQ_BF16,
                                   ctypes.c_void_p(kb.data_ptr()), ctypes.byref(kcb),
                                   ctypes.c_void_p(vb.data_ptr()), ctypes.byref(vcb), None, 4096, 32, 8, 8192,
                                   8192, ctypes.c_float(scale), signs, None, None, None,
                                   ctypes.c_void_p(new.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert big == tq.TQ_ERR_WORKSPACE


def test_noalloc_split_path_qjl_twice():
    """The same comparison on a shape served by the CUDA-core split kernels
    (QJL two-term score with 3-bit keys, 8 query heads per KV head, raw fp16
    values) and their combine, so those partials also go through the shared
    array; the two calls use different inputs and sequence lengths."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    L = tq.lib()
    L.tq_attn_decode_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.POINTER(tq.tq_codebook), ctypes.c_void_p,
                                         ctypes.POINTER(tq.tq_codebook), ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                         tq.tq_signs, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]
    dev = torch.device("cuda:0")
    B, Hq, Hkv, T, T_cap = 2, 16, 2, 700, 704
    plan = (ctypes.c_int64 * 8)()
    assert L.tq_attn_plan(B, Hq, Hkv, T, 3, 16, 1, 0, plan) == tq.TQ_ERR_UNSUPPORTED   # the split path
    cb = tq.tq_codebook_load(128, 3)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    stream = torch.cuda.current_stream(dev)
    scale = 1 / np.sqrt(128)
    outs_ref, outs_new = [], []
    for call in range(2):
        w = workloads.qjl_keys(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=60 + call, device=dev)
        kb = torch.zeros((B, Hkv, T_cap, 50), dtype=torch.uint8, device=dev)
        bits = torch.zeros((B, Hkv, T_cap, 16), dtype=torch.uint8, device=dev)
        rn = torch.zeros((B, Hkv, T_cap), dtype=torch.int16, device=dev)
        v = torch.zeros((B, Hkv, T_cap, 128), dtype=torch.float16, device=dev)
        v[:, :, :T] = w["v"]
        for b in range(B):
            for h in range(Hkv):
                tq.tq_encode_kv(w["k"][b, h], cb, signs, kb[b, h, :T])
                tq.tq_qjl_encode(w["k"][b, h], kb[b, h, :T], cb, signs, w["S"], bits[b, h, :T], rn[b, h, :T])
        lens = torch.tensor([T - 5 * call, 333 + call], dtype=torch.int32, device=dev)
        ref = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
        ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap), dtype=torch.uint8, device=dev)
        tq.tq_attn_decode(w["q"], kb, cb, v, None, ref, ws, T, scale, signs, seq_lens=lens, qjl_bits=bits,
                          res_norm_f16=rn, S=w["S"])
        new = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
        st = L.tq_attn_decode_noalloc(ctypes.c_void_p(w["q"].data_ptr()), tq.TQ_BF16,
                                      ctypes.c_void_p(kb.data_ptr()), ctypes.byref(cb),
                                      ctypes.c_void_p(v.data_ptr()), None,
                                      ctypes.c_void_p(lens.data_ptr()), B, Hq, Hkv, T_cap, T,
                                      ctypes.c_float(scale), signs, ctypes.c_void_p(bits.data_ptr()),
                                      ctypes.c_void_p(rn.data_ptr()), ctypes.c_void_p(w["S"].data_ptr()),
                                      ctypes.c_void_p(new.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        torch.cuda.synchronize(dev)
        outs_ref.append(ref.double().cpu().numpy())
        outs_new.append(new.double().cpu().numpy())
    for r, n in zip(outs_ref, outs_new):
        assert np.all(np.isfinite(n))
        assert np.all(_rel(n, r) <= ATTN_TOL)
    assert not np.allclose(outs_new[0], outs_new[1])
