"""The library's calls are stream-ordered and allocate nothing, so a decode
step (append-encode of the new rows, then the split-K decode attention with
its query prep and combine, chained as programmatic dependents) can be
captured in a CUDA graph and replayed: the replay gives bit-identical
results to the calls issued one by one, on new inputs written into the
captured buffers between replays."""

import numpy as np
import pytest
import torch

from turboquant_bit_kv_gb300 import workloads

pytestmark = pytest.mark.gpu


def test_decode_step_in_a_cuda_graph():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    dev = torch.device("cuda:0")
    B, Hq, Hkv, T, T_cap = 4, 28, 4, 600, 608
    cb = tq.tq_codebook_load(128, 3)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    s = torch.cuda.Stream(dev)
    w = workloads.qwen_outlier(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=5, device=dev)
    kb = torch.zeros((B, Hkv, T_cap, 50), dtype=torch.uint8, device=dev)
    vb = torch.zeros_like(kb)
    bh = torch.arange(B * Hkv, device=dev, dtype=torch.int64)
    dst_pre = (bh[:, None] * T_cap + torch.arange(T - 1, device=dev, dtype=torch.int64)[None, :]).reshape(-1)
    dst_new = bh * T_cap + (T - 1)
    with torch.cuda.stream(s):
        tq.tq_encode_kv(w["k"][:, :, :T - 1].contiguous().view(-1, 128), cb, signs, kb, dst_index=dst_pre, stream=s)
        tq.tq_encode_kv(w["v"][:, :, :T - 1].contiguous().view(-1, 128), cb, signs, vb, dst_index=dst_pre, stream=s)
    knew = w["k"][:, :, T - 1].contiguous().view(-1, 128).clone()
    vnew = w["v"][:, :, T - 1].contiguous().view(-1, 128).clone()
    q = w["q"].clone()
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap), dtype=torch.uint8, device=dev)
    scale = 1 / np.sqrt(128)

    def step():
        tq.tq_encode_kv(knew, cb, signs, kb, dst_index=dst_new, stream=s)
        tq.tq_encode_kv(vnew, cb, signs, vb, dst_index=dst_new, stream=s)
        tq.tq_attn_decode(q, kb, cb, vb, cb, out, ws, T, scale, signs, stream=s)

    with torch.cuda.stream(s):
        step()   # first calls (kernel attributes, tensor maps) before the capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    g = torch.Generator(device=dev).manual_seed(11)
    for _ in range(2):
        # new inputs into the captured buffers
        knew.copy_(torch.randn(knew.shape, generator=g, device=dev).to(knew.dtype))
        vnew.copy_(torch.randn(vnew.shape, generator=g, device=dev).to(vnew.dtype))
        q.copy_(torch.randn(q.shape, generator=g, device=dev).to(q.dtype))
        torch.cuda.synchronize(dev)
        graph.replay()
        torch.cuda.synchronize(dev)
        got_out, got_k, got_v = out.clone(), kb.clone(), vb.clone()
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize(dev)
        assert torch.equal(got_k, kb) and torch.equal(got_v, vb)
        assert torch.equal(got_out, out)
        assert torch.isfinite(out).all()
