"""Bounded waits: a kernel whose wait for a copy runs out finishes, records
the event, and the caller reads it through tq_device_status; the context
stays usable.  The failure is made by the library's test hook
(tq_debug_drop_copies: the kernels issue none of their bulk / TMA copies, so
their first wait is on a phase that nothing completes and runs out after
about 0.1 s), not by a fault."""

import numpy as np
import pytest
import torch

import oracle
from oracle import codec
from turboquant_bit_kv_gb300 import workloads

from parity_util import ATTN_TOL, attn_rel_err, check_codes, oracle_books

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from turboquant_bit_kv_gb300 import tq
    tq.lib()
    yield dict(tq=tq, dev=torch.device("cuda:0"), books=oracle_books(),
               cbs={b: tq.tq_codebook_load(128, b) for b in (2, 3, 4)},
               signs=tq.tq_signs_from_seed(workloads.SIGN_SEED), s=oracle.sign_diagonal(workloads.SIGN_SEED))
    tq.tq_debug_drop_copies(False)


def _calls(env, x, q, S, kb, vb, bits, qb, rn, out, ws, T):
    """The three kernels with bounded waits: tensor-core encode (more than
    1024 rows), tensor-core QJL encode, tensor-core attention."""
    tq = env["tq"]
    tq.tq_encode_kv(x.view(-1, D), env["cbs"][4], env["signs"], kb.view(-1, 66))
    tq.tq_qjl_encode(x.view(-1, D), kb.view(-1, 66), env["cbs"][4], env["signs"], S, qb.view(-1, 16), rn.view(-1))
    tq.tq_attn_decode(q, kb, env["cbs"][4], vb, env["cbs"][2], out, ws, T, 1 / np.sqrt(D), env["signs"])


def test_wait_that_runs_out_is_reported(env):
    tq, dev = env["tq"], env["dev"]
    B, Hq, Hkv, T = 2, 8, 2, 1536
    w = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=21, device=dev)
    S = workloads.qjl_keys(B=1, Hq=1, Hkv=1, T=8, seed=21, device=dev)["S"]
    x, q = w["k"], w["q"]
    kb = torch.zeros((B, Hkv, T, 66), dtype=torch.uint8, device=dev)
    vb = torch.zeros((B, Hkv, T, 34), dtype=torch.uint8, device=dev)
    tq.tq_encode_kv(w["v"].view(-1, D), env["cbs"][2], env["signs"], vb.view(-1, 34))
    qb = torch.zeros((B, Hkv, T, 16), dtype=torch.uint8, device=dev)
    rn = torch.zeros((B, Hkv, T), dtype=torch.int16, device=dev)
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    assert tq.tq_attn_plan(B, Hq, Hkv, T, 4, 2)["W"] > 0      # the tensor-core attention path
    tq.tq_device_status(clear=True)

    # every call completes normally: no event
    _calls(env, x, q, S, kb, vb, 4, qb, rn, out, ws, T)
    assert tq.tq_device_status() == tq.TQ_OK
    good = kb.cpu().numpy().copy()
    good_out = out.cpu().numpy().copy()

    # each kernel with its copies dropped: it returns (no hang), and the event is recorded
    for which in range(5):
        tq.tq_debug_drop_copies(True)
        try:
            if which == 0:
                tq.tq_encode_kv(x.view(-1, D), env["cbs"][4], env["signs"], kb.view(-1, 66))
            elif which == 1:
                tq.tq_qjl_encode(x.view(-1, D), torch.from_numpy(good).to(dev).view(-1, 66), env["cbs"][4],
                                 env["signs"], S, qb.view(-1, 16), rn.view(-1))
            elif which == 2:
                kb.copy_(torch.from_numpy(good))
                tq.tq_attn_decode(q, kb, env["cbs"][4], vb, env["cbs"][2], out, ws, T, 1 / np.sqrt(D), env["signs"])
            elif which == 3:
                # the tensor-core encode at another head dim (bf16 rows, more than 1024)
                R = torch.eye(64, dtype=torch.float32, device=dev)
                hb = torch.empty((x.numel() // 64, tq.tq_block_bytes_d(64, 4)), dtype=torch.uint8, device=dev)
                tq.tq_encode_kv_d(x.reshape(-1, 64), tq.tq_codebook_load(64, 4), R, hb)
            else:
                # the same kernel's turboq8 mode (bf16 rows, more than 1024)
                q8 = torch.empty((x.numel() // D, 130), dtype=torch.uint8, device=dev)
                tq.tq_encode_kv_ex(x.view(-1, D), tq.tq_codebook_load(128, 8), env["signs"], q8)
        finally:
            tq.tq_debug_drop_copies(False)
        assert tq.tq_device_status(clear=True) == tq.TQ_ERR_TIMEOUT, which
        assert tq.tq_device_status() == tq.TQ_OK        # cleared
        if which == 2:
            assert not torch.isfinite(out).all()          # the failed partials are marked

    # the context is still usable: the same calls give the same, correct results again
    _calls(env, x, q, S, kb, vb, 4, qb, rn, out, ws, T)
    assert tq.tq_device_status() == tq.TQ_OK
    assert np.array_equal(kb.cpu().numpy(), good)
    check_codes(good.reshape(-1, 66), 4, x.view(-1, D).double().cpu().numpy(), env["s"], env["books"][4][2],
                "after timeouts")
    assert np.allclose(out.cpu().numpy(), good_out, rtol=0, atol=0)
