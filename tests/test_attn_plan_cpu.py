"""The tensor-core attention path's work partition (tq_attn_plan, host only),
checked by brute force against its definition: chunks of 32 tokens ordered by
(sequence, KV head, position), worker w owning chunks [w Ctot / W,
(w + 1) Ctot / W), Smax bounding the worker ranges that meet one (sequence,
KV head) segment, and the cap on workers per segment for small problems."""

import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def tq():
    from turboquant_bit_kv_gb300 import build_lib, tq as t
    build_lib.build()
    t.lib()
    return t


SHAPES = [
    # B, Hq, Hkv, T, key bits, value bits (16: raw fp16), QJL
    (16, 32, 8, 8192, 4, 2, False),      # the decode workload
    (64, 28, 4, 32769, 3, 3, False),     # the 3-bit append workload (two n-tiles)
    (8, 32, 8, 16384, 3, 16, True),      # the QJL workload (raw values)
    (1, 1, 1, 4096, 4, 2, False),        # one head
    (1, 32, 8, 8192, 4, 2, False),       # batch 1
    (1, 32, 8, 32768, 4, 2, False),
    (1, 32, 8, 2048, 4, 2, False),
    (4, 32, 8, 4096, 4, 2, False),
    (2, 28, 4, 4096, 3, 3, False),
    (1, 4, 1, 20000, 4, 2, False),
    (2, 8, 2, 9000, 3, 3, False),
    (500, 8, 8, 20, 4, 2, False),        # many one-chunk segments
    (300, 32, 8, 70, 3, 3, False),
    (1, 4, 1, 1, 4, 2, False),           # a single token
    (3, 8, 2, 1000, 4, 2, False),
    (2, 2, 2, 65, 2, 4, False),
    (7, 56, 8, 777, 2, 2, False),
    (5, 40, 5, 3333, 4, 4, False),
]


def _check(p, B, Hkv, T):
    C = math.ceil(T / 32)
    Ctot = B * Hkv * C
    W, P, Smax = p["W"], p["P"], p["Smax"]
    assert p["C"] == C and p["Ctot"] == Ctot
    assert 1 <= P <= W <= Ctot
    assert W <= P * p["warps"]
    # every worker range is non-empty
    w = np.arange(W, dtype=np.int64)
    lo, hi = w * Ctot // W, (w + 1) * Ctot // W
    assert np.all(hi > lo) and lo[0] == 0 and hi[-1] == Ctot and np.all(lo[1:] == hi[:-1])
    # ranges meeting each segment, by brute force, against Smax and the combine's slot count
    segs = B * Hkv
    meets = np.zeros(segs, dtype=np.int64)
    for a, b in zip(lo // C, (hi - 1) // C):
        meets[a:b + 1] += 1
    assert meets.max() <= Smax <= C
    j = np.arange(segs, dtype=np.int64)
    first = ((j * C + 1) * W - 1) // Ctot                 # the worker owning the segment's first chunk
    last = (((j + 1) * C) * W - 1) // Ctot               # ... and its last chunk
    assert np.array_equal(last - first + 1, meets)
    # the owner of a chunk is the largest w with floor(w Ctot / W) <= chunk
    for x in np.unique(np.linspace(0, Ctot - 1, 50).astype(np.int64)):
        owner = ((x + 1) * W - 1) // Ctot
        assert lo[owner] <= x < hi[owner]
    # combine slot groups: one per 32 slots, at most four
    assert p["combine_groups"] == min(4, max(1, math.ceil(Smax / 32)))
    return C, Ctot, segs


@pytest.mark.parametrize("sms", [1, 16, 148, 152])
@pytest.mark.parametrize("shape", SHAPES)
def test_plan_partition(tq, shape, sms):
    B, Hq, Hkv, T, kb, vb, qjl = shape
    p = tq.tq_attn_plan(B, Hq, Hkv, T, kb, vb, qjl=qjl, sms=sms)
    C, Ctot, segs = _check(p, B, Hkv, T)
    # small problems: at most 31 workers per segment while each keeps 5 chunks or fewer
    full = min(Ctot, p["P"] * p["warps"])
    if p["W"] < full:
        assert p["W"] == max(31 * segs, math.ceil(Ctot / 5))
        assert p["Smax"] <= 32 or math.ceil(Ctot / p["W"]) <= 5


def test_plan_large_workloads_use_every_warp(tq):
    # the decode workload on 152 SMs: 12 warps per SM, every warp a worker, at most 16 partials
    p = tq.tq_attn_plan(16, 32, 8, 8192, 4, 2, sms=152)
    assert p["P"] == 152 and p["W"] == 152 * p["warps"] and p["Smax"] <= 32 and p["combine_groups"] == 1


def test_plan_rejects_split_path_and_bad_shapes(tq):
    with pytest.raises(tq.TQError):
        tq.tq_attn_plan(1, 3, 2, 64, 4, 2)                 # Hq not a multiple of Hkv
    with pytest.raises(tq.TQError):
        tq.tq_attn_plan(1, 8, 8, 0, 4, 2)                  # no tokens
    with pytest.raises(tq.TQError):
        tq.tq_attn_plan(1, 8, 8, 64, 5, 2)                 # bits
    for args in ((1, 8, 1, 64, 3, 16), (1, 4, 1, 64, 2, 16), (1, 4, 1, 64, 3, 3)):
        with pytest.raises(tq.TQError) as e:                # QJL shapes served by the CUDA-core path
            tq.tq_attn_plan(*args, qjl=True)
        assert e.value.status == tq.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,Hkv,T,slots", [
    (8, 8, 8192, 456),        # the head-dim-160 workload: 3 CTAs per SM on 152 SMs
    (8, 8, 8192, 304),        # 2 CTAs per SM (4-bit values at d = 160)
    (1, 1, 16384, 456),       # one long sequence: many splits
    (2, 4, 32, 456),          # one chunk: one split
    (3, 2, 700, 456),
    (64, 8, 32768, 456),      # more segments than slots: several waves
    (1, 1, 1, 1),
])
def test_headdim_split_plan_matches_its_definition(tq, B, Hkv, T, slots):
    """tq_attn_plan_d against its stated rule, by brute force: of s = 1 .. max(1, C / 16)
    (C = ceil(T / 32) chunks), the first s with the fewest waves x (steps per warp + 1); then
    whole chunks per split and no empty split."""
    warps = 4
    splits, tps, smax = tq.tq_attn_plan_d(B, Hkv, T, slots, warps)
    C = -(-T // 32)
    assert smax == max(1, C // 16)
    costs = [(-(-B * Hkv * s // slots)) * (-(-(-(-C // s)) // warps) + 1) for s in range(1, smax + 1)]
    best = 1 + costs.index(min(costs))
    assert tps == -(-C // best) * 32 and tps % 32 == 0
    assert splits == -(-T // tps)
    assert 1 <= splits <= best <= smax
    assert splits * tps >= T and (splits - 1) * tps < T     # every split holds tokens
    with pytest.raises(Exception):
        tq.tq_attn_plan_d(B, Hkv, 0, slots, warps)
