"""Benchmark of the TurboQuant KV hot path on GB300.

Default workload (``--workload qwen25_7b_append``, the largest decode
configuration): batch 64, 28 query heads, 4 KV heads, head_dim 128, context
32768 bf16 K/V with 1% outlier channels, K3/V3.  One step = quantise-on-
insert of the whole 32768-token K and V prefix into a [B, Hkv, T_cap] cache
through a destination index (tq_encode_kv), the append of one new token per
sequence, and one fused decode-attention step over the 32769 tokens
(tq_attn_decode).

Other workloads (one JSON line each, same keys):

* ``llama3_8b_decode``   -- batch 16, 32/8 heads, context 8192, bf16 K/V with
                            log-normal channel scales and AR(1) correlation
                            0.9, K4/V2: encode the cache, one decode step;
* ``single_head_fp32``   -- one head, 4096 fp32 K/V rows, K4/V2, one query;
* ``qjl_two_term``       -- batch 8, 32/8 heads, context 16384: K3 encode,
                            QJL sign bits + residual norms, attention with the
                            two-term score and raw fp16 values;
* ``storage_roundtrip``  -- [2, 32, 65536, 1024] bf16: serialise (4 raw
                            layers, 28 layers K4/V4 in 132-byte slots) and
                            deserialise.

`value` is the metric's decode-attention throughput: the attention call's
algorithmic bytes (packed K/V blocks with their norms, the query and the
output; QJL side data where used) over the call's device time inside the
timed steps, in GB/s (for the storage round trip, which has no attention
call, the serialise + deserialise bytes over their time).
`dtype` is the arithmetic type of the path (float32: every product exact or
split into fp16 hi / lo parts, every sum in float32), `io_dtype` that of the
inputs.  `encode_gvec_s` / `encode_frac_hbm` give the prefix encode's vectors per
second and its bytes over time as a fraction of the HBM peak (`frac_hbm` and
`encode_frac_hbm` against the measured copy bandwidth, the `_nominal`
fields against the nominal 8 TB/s); `parts` has
every call of the step.  `e2e` measures the metric through the C ABI from
pinned host buffers: each step copies the step's new inputs (the query and
the appended token's K/V rows) from the host, runs the append and the
attention call against the cache resident in HBM, and reads the output
back; `e2e.full_step` runs the whole step (the prefix K/V rows copied from
the host too) and reports the step's bytes over its time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                       [--workload NAME]
Under torchrun each rank runs an independent replica on its own GPU (weak
scaling; the path has no exchange step); rank 0 prints one JSON line.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode-attention GB/s & % HBM peak; encode Gvec/s (1xGB300)"
DEFAULT_WORKLOAD = "qwen25_7b_append"
WORKLOADS = {
    "llama3_8b_decode": dict(B=16, Hq=32, Hkv=8, T=8192, head_dim=128, key_bits=4, value_bits=2,
                             kv_dtype="bf16", scale="1/sqrt(128)"),
    "single_head_fp32": dict(B=1, Hq=1, Hkv=1, T=4096, head_dim=128, key_bits=4, value_bits=2,
                             kv_dtype="fp32", scale="1/sqrt(128)"),
    "qwen25_7b_append": dict(B=64, Hq=28, Hkv=4, T=32769, T_cap=32776, head_dim=128, key_bits=3, value_bits=3,
                             kv_dtype="bf16", outlier_channels="5 of 512 x20", append_tokens=1,
                             scale="1/sqrt(128)"),
    "qjl_two_term": dict(B=8, Hq=32, Hkv=8, T=16384, head_dim=128, key_bits=3, value="fp16 raw", qjl_m=128,
                         kv_dtype="bf16 keys / fp16 values", scale="1/sqrt(128)"),
    "llama3_8b_prefill": dict(B=16, Hq=32, Hkv=8, T=8192, M=64, head_dim=128, key_bits=4, value_bits=2,
                              kv_dtype="bf16", query="64 new tokens per sequence, causal",
                              scale="1/sqrt(128)"),
    "llama3_8b_turboq8_pair": dict(B=16, Hq=32, Hkv=8, T=8192, head_dim=128, key_format="turboq8 (130 B)",
                                   value_format="4-bit norm-corrected (66 B)", kv_dtype="bf16",
                                   scale="1/sqrt(128)"),
    "llama3_8b_paged_decode": dict(B=16, Hq=32, Hkv=8, T=8192, head_dim=128, key_bits=4, value_bits=2,
                                   page_tokens=32, kv_dtype="bf16", scale="1/sqrt(128)"),
    "headdim_160_decode": dict(B=8, Hq=32, Hkv=8, T=8192, head_dim=160, key_bits=4, value_bits=2, kv_dtype="bf16",
                               rotation="seeded random orthogonal 160 x 160 (QR), float32", scale="1/sqrt(160)"),
    "headdim_128_g8_decode": dict(B=8, Hq=64, Hkv=8, T=8192, head_dim=128, key_bits=4, value_bits=2,
                                  kv_dtype="bf16", rotation="seeded random orthogonal 128 x 128 (QR), float32",
                                  scale="1/sqrt(128)"),
    "storage_roundtrip": dict(layout="[2, 32, 65536, 1024]", L=32, T=65536, hidden=1024, head_dim=128,
                              block_size=16, skip_first=2, skip_last=2, key_bits=4, value_bits=4, slot_bytes=132,
                              kv_dtype="bf16"),
}
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # the part's nominal HBM3e bandwidth (8 TB/s), reported beside the measured peak
CSRC = os.path.join(ROOT, "turboquant_bit_kv_gb300", "csrc")
# the sources each kernel group is built from (profiled DRAM traffic is only
# reported while these are unchanged since the capture)
KERNEL_SOURCES = {
    "encode": ["tq_encode.cu", "tq_tc.cuh", "tq_device.cuh"],
    "ext_encode": ["tq_ext.cu", "tq_headdim_tc.cu", "tq_tc.cuh", "tq_device.cuh"],
    "append": ["tq_encode.cu", "tq_tc.cuh", "tq_device.cuh"],
    "prefill": ["tq_attn_prefill.cu", "tq_tc.cuh", "tq_device.cuh"],
    "pair_attention": ["tq_attn.cu", "tq_attn.cuh", "tq_attn_mma.cu", "tq_attn_mma.h", "tq_attn_mma.cuh",
                       "tq_attn_mma_k4.cu", "tq_attn_mma_k8.cu", "tq_device.cuh"],
    "paged_attention": ["tq_attn.cu", "tq_attn.cuh", "tq_attn_mma.cu", "tq_attn_mma.h", "tq_attn_mma.cuh",
                        "tq_attn_mma_k2.cu", "tq_attn_mma_k3.cu", "tq_attn_mma_k4.cu", "tq_device.cuh"],
    "attention": ["tq_attn.cu", "tq_attn.cuh", "tq_attn_mma.cu", "tq_attn_mma.h", "tq_attn_mma.cuh",
                  "tq_attn_mma_k2.cu", "tq_attn_mma_k3.cu", "tq_attn_mma_k4.cu", "tq_attn_g1.cu",
                  "tq_attn_g2.cu", "tq_attn_g4.cu", "tq_attn_g8.cu", "tq_device.cuh"],
    "qjl": ["tq_qjl.cu", "tq_tc.cuh", "tq_codec.cu", "tq_device.cuh"],
    "hd_encode": ["tq_headdim.cu", "tq_headdim.cuh", "tq_headdim_tc.cu", "tq_tc.cuh", "tq_device.cuh"],
    "hd_attention": ["tq_headdim.cu", "tq_headdim.cuh", "tq_headdim_mma.cuh", "tq_headdim_mma.cu", "tq_device.cuh"],
    "hd_attention_g8": ["tq_headdim.cu", "tq_headdim.cuh", "tq_headdim_mma.cuh", "tq_headdim_mma.cu",
                        "tq_headdim_mma8.cu", "tq_device.cuh"],
    "serialize": ["tq_encode.cu", "tq_tc.cuh", "tq_codec.cu", "tq_device.cuh"],
    "deserialize": ["tq_decode.cu", "tq_codec.cu", "tq_device.cuh"],
}
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.md")


def step_bytes(B, Hq, Hkv, T, kbits=4, vbits=2):
    """Algorithmic bytes of the decode step: encode K and V (bf16 rows in,
    blocks out) and one attention step (blocks, bf16 q in, fp32 out)."""
    nvec = B * Hkv * T
    kbb, vbb = 2 + 16 * kbits, 2 + 16 * vbits
    enc_k = nvec * 128 * 2 + nvec * kbb
    enc_v = nvec * 128 * 2 + nvec * vbb
    attn = nvec * (kbb + vbb) + B * Hq * 128 * 2 + B * Hq * 128 * 4
    return dict(enc_k=enc_k, enc_v=enc_v, attn=attn, nvec=2 * nvec, total=enc_k + enc_v + attn)


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Measured dense 16-bit tensor throughput (TFLOP/s): the burst figure of
    MEASURED_PEAKS.json (fp16 and bf16 run at the same rate), else the
    fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 same rate)"
    except Exception:
        return 1900.0, "fallback"


def source_sha(group):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[group]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, group):
    """DRAM bytes (read + write) per step of a kernel group, from the ncu
    table under profiles/, or None when absent or when the group's sources
    changed since the capture."""
    try:
        with open(TRAFFIC_TABLE) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    for line in lines:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == workload and cells[1] == group:
            try:
                val = int(cells[2].replace(",", ""))
            except ValueError:
                return None
            return val if cells[3] == source_sha(group) else None
    return None


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def reduce_max(x, world):
    """Max of a float over ranks (identity when world == 1)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload plans (GPU arm)

class Op:
    """One call of the path inside a step: `fn()` launches it on the bench
    stream; `nbytes` is its algorithmic bytes, `launches` the kernels of this
    library it launches, `nvec` the 128-element vectors it encodes/decodes."""

    def __init__(self, name, group, fn, nbytes, launches, nvec=0):
        self.name, self.group, self.fn, self.nbytes, self.launches, self.nvec = \
            name, group, fn, nbytes, launches, nvec
        self.flops = 0


def _pinned(t):
    return t.cpu().pin_memory()


class _CopyPipe:
    """Host-to-device copies of an end-to-end step, issued in chunks on a
    side stream; the bench stream waits for a chunk right before the call that
    reads it, so the kernels run while the remaining bytes cross the host link
    (the link's bandwidth bounds the step; more copy streams do not add to it).
    Steps alternate between `nbuf` sets of device input buffers, so the copies
    of the next step run while this step's last kernels finish."""

    def __init__(self, stream, nbuf=2):
        self.main = stream
        self.side = torch.cuda.Stream(device=stream.device)
        self.free = [None] * nbuf   # per buffer set: its last reader on the bench stream has run
        self.n = 0

    def begin(self):
        """Start a step; returns the index of the buffer set its copies fill."""
        i = self.n % len(self.free)
        self.n += 1
        ev = self.free[i]
        if ev is None:
            ev = torch.cuda.Event()
            ev.record(self.main)
        self.side.wait_event(ev)
        return i

    def release(self, i):
        """Buffer set i has been read by everything enqueued so far on the bench stream."""
        ev = torch.cuda.Event()
        ev.record(self.main)
        self.free[i] = ev

    def copy(self, dst, src):
        with torch.cuda.stream(self.side):
            dst.copy_(src, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(self.side)
        return ev

    def wait(self, ev):
        self.main.wait_event(ev)


def _chunks(n, parts, align=1024):
    """`parts` row ranges covering [0, n), boundaries on multiples of `align` rows."""
    size = -(-n // parts)
    size = -(-size // align) * align
    return [slice(a, min(n, a + size)) for a in range(0, n, size)]


def plan_llama(tq, wl, dev, stream, seed, batch):
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS["llama3_8b_decode"]
    B, Hq, Hkv, T = batch or W["B"], W["Hq"], W["Hkv"], W["T"]
    nb = step_bytes(B, Hq, Hkv, T)
    kcb, vcb = tq.tq_codebook_load(128, 4), tq.tq_codebook_load(128, 2)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=seed, device=dev)
    k, v, q = data["k"], data["v"], data["q"]
    kb = torch.empty((B, Hkv, T, tq.tq_block_bytes(4)), dtype=torch.uint8, device=dev)
    vb = torch.empty((B, Hkv, T, tq.tq_block_bytes(2)), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(128.0)
    nvec = B * Hkv * T

    def attn(qq=q):
        tq.tq_attn_decode(qq, kb, kcb, vb, vcb, out, ws, T, scale, signs, stream=stream)

    ops = [Op("encode_k", "encode", lambda: tq.tq_encode_kv(k.view(-1, 128), kcb, signs, kb, stream=stream),
              nb["enc_k"], 1, nvec),
           Op("encode_v", "encode", lambda: tq.tq_encode_kv(v.view(-1, 128), vcb, signs, vb, stream=stream),
              nb["enc_v"], 1, nvec),
           Op("attention", "attention", attn, nb["attn"], 3)]

    def e2e():
        hk, hv, hq = _pinned(k).view(-1, 128), _pinned(v).view(-1, 128), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        bufs = [[torch.empty_like(t, device=dev) for t in (hk, hv, hq)] for _ in range(2)]
        kb2, vb2 = kb.view(nvec, -1), vb.view(nvec, -1)
        pipe, parts = _CopyPipe(stream), _chunks(nvec, 4)

        def step():
            i = pipe.begin()
            dk, dv, dq = bufs[i]
            eq = pipe.copy(dq, hq)
            ek = [pipe.copy(dk[r], hk[r]) for r in parts]
            ev = [pipe.copy(dv[r], hv[r]) for r in parts]
            for r, e in zip(parts, ek):
                pipe.wait(e)
                tq.tq_encode_kv(dk[r], kcb, signs, kb2[r], stream=stream)
            for r, e in zip(parts, ev):
                pipe.wait(e)
                tq.tq_encode_kv(dv[r], vcb, signs, vb2[r], stream=stream)
            pipe.wait(eq)
            attn(dq)
            pipe.release(i)
            hout.copy_(out, non_blocking=True)
        return step, k.numel() * 2 + v.numel() * 2 + q.numel() * 2, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 2, out.numel() * 4

    def sample():
        rng = np.random.default_rng(3)
        res = []
        for name, x, blk, bits in (("K", k, kb, 4), ("V", v, vb, 2)):
            pick = torch.from_numpy(np.sort(rng.choice(nvec, 4096, replace=False))).to(dev)
            res.append((name, bits, x.view(-1, 128)[pick].double().cpu().numpy(),
                        blk.view(nvec, -1)[pick].cpu().numpy()))
        return res

    cfg = dict(W, B=B, l2="inputs (537 MB) larger than L2 (129 MB); attention also timed after an L2 flush")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, sample=sample, config=cfg,
                dtype="bf16")


def plan_single_head(tq, wl, dev, stream, seed, batch):
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS["single_head_fp32"]
    T = W["T"]
    kcb, vcb = tq.tq_codebook_load(128, 4), tq.tq_codebook_load(128, 2)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.single_head(T=T, seed=seed, device=dev)
    k, v = data["k"], data["v"]
    q = data["q"].view(1, 1, 128)
    kb = torch.empty((1, 1, T, 66), dtype=torch.uint8, device=dev)
    vb = torch.empty((1, 1, T, 34), dtype=torch.uint8, device=dev)
    out = torch.empty((1, 1, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(1, 1, 1, T), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(128.0)

    def attn(qq=q):
        tq.tq_attn_decode(qq, kb, kcb, vb, vcb, out, ws, T, scale, signs, stream=stream)

    ops = [Op("encode_k", "encode", lambda: tq.tq_encode_kv(k, kcb, signs, kb, stream=stream), T * (512 + 66),
              1, T),
           Op("encode_v", "encode", lambda: tq.tq_encode_kv(v, vcb, signs, vb, stream=stream), T * (512 + 34),
              1, T),
           Op("attention", "attention", attn, T * 100 + 512 + 512, 3)]

    def e2e():
        hk, hv, hq = _pinned(k), _pinned(v), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dk, dv, dq = torch.empty_like(k), torch.empty_like(v), torch.empty_like(q)

        def step():
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            tq.tq_encode_kv(dk, kcb, signs, kb, stream=stream)
            tq.tq_encode_kv(dv, vcb, signs, vb, stream=stream)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, (k.numel() + v.numel() + q.numel()) * 4, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 4, out.numel() * 4

    def sample():
        return [("K", 4, k.double().cpu().numpy(), kb.view(T, -1).cpu().numpy()),
                ("V", 2, v.double().cpu().numpy(), vb.view(T, -1).cpu().numpy())]

    cfg = dict(W, l2="inputs (4.6 MB) fit in L2: launch-bound, report microseconds")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, sample=sample, config=cfg,
                dtype="f32")


def plan_qwen(tq, wl, dev, stream, seed, batch):
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS["qwen25_7b_append"]
    B, Hq, Hkv, T, T_cap = batch or W["B"], W["Hq"], W["Hkv"], W["T"], W["T_cap"]
    cb = tq.tq_codebook_load(128, 3)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.qwen_outlier(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=seed, device=dev)
    q = data["q"]
    pre = {n: data[n][:, :, :T - 1].contiguous().view(-1, 128) for n in ("k", "v")}
    new = {n: data[n][:, :, T - 1].contiguous().view(-1, 128) for n in ("k", "v")}
    del data
    torch.cuda.empty_cache()
    bh = torch.arange(B * Hkv, device=dev, dtype=torch.int64)
    dst_pre = (bh[:, None] * T_cap + torch.arange(T - 1, device=dev, dtype=torch.int64)[None, :]).reshape(-1)
    dst_new = bh * T_cap + (T - 1)
    blk = {n: torch.zeros((B, Hkv, T_cap, 50), dtype=torch.uint8, device=dev) for n in ("k", "v")}
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T_cap), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(128.0)
    n_pre, n_new = B * Hkv * (T - 1), B * Hkv

    def enc(x, n, dst):
        return lambda: tq.tq_encode_kv(x, cb, signs, blk[n], dst_index=dst, stream=stream)

    def attn(qq=q):
        tq.tq_attn_decode(qq, blk["k"], cb, blk["v"], cb, out, ws, T, scale, signs, stream=stream)

    ops = [Op("encode_k", "encode", enc(pre["k"], "k", dst_pre), n_pre * (256 + 50), 1, n_pre),
           Op("encode_v", "encode", enc(pre["v"], "v", dst_pre), n_pre * (256 + 50), 1, n_pre),
           Op("append_k", "append", enc(new["k"], "k", dst_new), n_new * (256 + 50), 1, n_new),
           Op("append_v", "append", enc(new["v"], "v", dst_new), n_new * (256 + 50), 1, n_new),
           Op("attention", "attention", attn, B * Hkv * T * 100 + B * Hq * 128 * (2 + 4), 3)]

    def e2e():
        hk, hv = _pinned(pre["k"]), _pinned(pre["v"])
        hnk, hnv, hq = _pinned(new["k"]), _pinned(new["v"]), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        bufs = [[torch.empty_like(t) for t in (pre["k"], pre["v"], new["k"], new["v"], q)] for _ in range(2)]

        pipe, parts = _CopyPipe(stream), _chunks(n_pre, 4)

        def step():
            i = pipe.begin()
            dk, dv, dnk, dnv, dq = bufs[i]
            small = [pipe.copy(d, h) for d, h in ((dnk, hnk), (dnv, hnv), (dq, hq))]
            ek = [pipe.copy(dk[r], hk[r]) for r in parts]
            ev = [pipe.copy(dv[r], hv[r]) for r in parts]
            for n, d, evs in (("k", dk, ek), ("v", dv, ev)):
                for r, e in zip(parts, evs):
                    pipe.wait(e)
                    enc(d[r], n, dst_pre[r])()
            for e in small:
                pipe.wait(e)
            enc(dnk, "k", dst_new)()
            enc(dnv, "v", dst_new)()
            attn(dq)
            pipe.release(i)
            hout.copy_(out, non_blocking=True)
        return step, (2 * (n_pre + n_new) * 128 + q.numel()) * 2, out.numel() * 4

    def decode_e2e():
        hnk, hnv, hq = _pinned(new["k"]), _pinned(new["v"]), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dnk, dnv, dq = torch.empty_like(new["k"]), torch.empty_like(new["v"]), torch.empty_like(q)

        def step():
            dnk.copy_(hnk, non_blocking=True)
            dnv.copy_(hnv, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            enc(dnk, "k", dst_new)()
            enc(dnv, "v", dst_new)()
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, (2 * n_new * 128 + q.numel()) * 2, out.numel() * 4

    def sample():
        rng = np.random.default_rng(3)
        res = []
        for n in ("k", "v"):
            pick = torch.from_numpy(np.sort(rng.choice(n_pre, 4096, replace=False))).to(dev)
            res.append(("prefix " + n.upper(), 3, pre[n][pick].double().cpu().numpy(),
                        blk[n].view(-1, 50)[dst_pre[pick]].cpu().numpy()))
            res.append(("append " + n.upper(), 3, new[n].double().cpu().numpy(),
                        blk[n].view(-1, 50)[dst_new].cpu().numpy()))
        return res

    cfg = dict(W, B=B, l2="inputs (4.3 GB) larger than L2; attention also timed after an L2 flush",
               note="destination-index reads (8 B per vector) are not counted as algorithmic bytes")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, sample=sample, config=cfg,
                dtype="bf16")


def plan_qjl(tq, wl, dev, stream, seed, batch):
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS["qjl_two_term"]
    B, Hq, Hkv, T = batch or W["B"], W["Hq"], W["Hkv"], W["T"]
    cb = tq.tq_codebook_load(128, 3)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.qjl_keys(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=seed, device=dev)
    k, v, q, S = data["k"], data["v"], data["q"], data["S"]
    n = B * Hkv * T
    kb = torch.empty((B, Hkv, T, 50), dtype=torch.uint8, device=dev)
    bits = torch.empty((B, Hkv, T, 16), dtype=torch.uint8, device=dev)
    rn = torch.empty((B, Hkv, T), dtype=torch.int16, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(128.0)

    def enc(kk):
        tq.tq_encode_kv(kk.view(-1, 128), cb, signs, kb, stream=stream)

    def qjl(kk):
        tq.tq_qjl_encode(kk.view(-1, 128), kb.view(-1, 50), cb, signs, S, bits.view(-1, 16), rn.view(-1),
                         stream=stream)

    def attn(qq=q, vv=v):
        tq.tq_attn_decode(qq, kb, cb, vv, None, out, ws, T, scale, signs, qjl_bits=bits, res_norm_f16=rn, S=S,
                          stream=stream)

    ops = [Op("encode_k", "encode", lambda: enc(k), n * (256 + 50), 1, n),
           Op("qjl_encode", "qjl", lambda: qjl(k), n * (256 + 50 + 16 + 2) + 128 * 128 * 4, 1, n),
           Op("attention", "attention", attn, n * (50 + 16 + 2 + 256) + B * Hq * 128 * (2 + 4) + 128 * 128 * 4, 3)]

    def e2e():
        hk, hv, hq = _pinned(k).view(-1, 128), _pinned(v), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        bufs = [[torch.empty_like(t, device=dev) for t in (hk, hv, hq)] for _ in range(2)]
        kb2, bits2, rn2 = kb.view(n, 50), bits.view(n, 16), rn.view(n)
        pipe, parts = _CopyPipe(stream), _chunks(n, 4)

        def step():
            i = pipe.begin()
            dk, dv, dq = bufs[i]
            ek = [pipe.copy(dk[r], hk[r]) for r in parts]
            ev = pipe.copy(dv, hv)
            eq = pipe.copy(dq, hq)
            for r, e in zip(parts, ek):
                pipe.wait(e)
                tq.tq_encode_kv(dk[r], cb, signs, kb2[r], stream=stream)
                tq.tq_qjl_encode(dk[r], kb2[r], cb, signs, S, bits2[r], rn2[r], stream=stream)
            pipe.wait(ev)
            pipe.wait(eq)
            attn(dq, dv)
            pipe.release(i)
            hout.copy_(out, non_blocking=True)
        return step, (k.numel() + v.numel() + q.numel()) * 2, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 2, out.numel() * 4

    def sample():
        rng = np.random.default_rng(3)
        pick = torch.from_numpy(np.sort(rng.choice(n, 4096, replace=False))).to(dev)
        return [("K", 3, k.view(-1, 128)[pick].double().cpu().numpy(), kb.view(n, 50)[pick].cpu().numpy())]

    cfg = dict(W, B=B, l2="inputs (537 MB) larger than L2; attention also timed after an L2 flush",
               note="QJL sketch S: seeded 128x128 N(0,1) float32; resident on the device")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, sample=sample, config=cfg,
                dtype="bf16")


def prefill_flops(B, M, Hq, T):
    """Algorithmic FLOPs of causal attention of M query tokens per sequence
    over T cached tokens: query token i (position T - M + i) meets T - M + i + 1
    keys; 2 * 128 FLOPs for its score and 2 * 128 for its value sum each."""
    keys = sum(T - M + i + 1 for i in range(M))
    return B * Hq * keys * 4 * 128


def plan_prefill(tq, wl, dev, stream, seed, batch):
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS["llama3_8b_prefill"]
    B, Hq, Hkv, T, M = batch or W["B"], W["Hq"], W["Hkv"], W["T"], W["M"]
    kcb, vcb = tq.tq_codebook_load(128, 4), tq.tq_codebook_load(128, 2)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=seed, device=dev)
    k, v = data["k"], data["v"]
    g = torch.Generator(device=dev).manual_seed(seed + 101)
    q = torch.randn((B, M, Hq, 128), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    kb = torch.empty((B, Hkv, T, 66), dtype=torch.uint8, device=dev)
    vb = torch.empty((B, Hkv, T, 34), dtype=torch.uint8, device=dev)
    out = torch.empty((B, M, Hq, 128), dtype=torch.float32, device=dev)
    scale = 1.0 / np.sqrt(128.0)
    nvec = B * Hkv * T
    nb = step_bytes(B, Hq, Hkv, T)
    # the prefill reads the cache once per 128-row tile of (query token, head) rows
    attn_bytes = nvec * 100 + q.numel() * 2 + out.numel() * 4
    flops = prefill_flops(B, M, Hq, T)

    def attn(qq=q):
        tq.tq_attn_prefill(qq, kb, kcb, vb, vcb, out, T, scale, signs, stream=stream)

    ops = [Op("encode_k", "encode", lambda: tq.tq_encode_kv(k.view(-1, 128), kcb, signs, kb, stream=stream),
              nb["enc_k"], 1, nvec),
           Op("encode_v", "encode", lambda: tq.tq_encode_kv(v.view(-1, 128), vcb, signs, vb, stream=stream),
              nb["enc_v"], 1, nvec),
           Op("attention", "prefill", attn, attn_bytes, 1)]
    ops[-1].flops = flops

    def e2e():
        hk, hv, hq = _pinned(k).view(-1, 128), _pinned(v).view(-1, 128), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dk, dv, dq = torch.empty_like(hk, device=dev), torch.empty_like(hv, device=dev), torch.empty_like(q)

        def step():
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            tq.tq_encode_kv(dk, kcb, signs, kb.view(nvec, -1), stream=stream)
            tq.tq_encode_kv(dv, vcb, signs, vb.view(nvec, -1), stream=stream)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, (k.numel() + v.numel() + q.numel()) * 2, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 2, out.numel() * 4

    def sample():
        rng = np.random.default_rng(3)
        res = []
        for name, x, blk, bits in (("K", k, kb, 4), ("V", v, vb, 2)):
            pick = torch.from_numpy(np.sort(rng.choice(nvec, 4096, replace=False))).to(dev)
            res.append((name, bits, x.view(-1, 128)[pick].double().cpu().numpy(),
                        blk.view(nvec, -1)[pick].cpu().numpy()))
        return res

    cfg = dict(W, B=B, l2="inputs (537 MB) larger than L2 (129 MB); attention also timed after an L2 flush",
               note="attention bytes: packed K/V blocks + q + out once; flops: 4 * 128 per (query row, visible "
                    "key)")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, sample=sample, config=cfg,
                dtype="bf16", tensor="prefill")


def plan_turboq8_pair(tq, wl, dev, stream, seed, batch):
    """Llama-shaped decode step with the fork's high-precision asymmetric pair:
    turboq8 keys, 4-bit norm-corrected values (encode the cache, one decode
    step on the split-K tensor-core decode kernels: query prep, attention,
    combine)."""
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS[wl]
    B, Hq, Hkv, T = batch or W["B"], W["Hq"], W["Hkv"], W["T"]
    k8, v4 = tq.tq_codebook_load(128, 8), tq.tq_codebook_load(128, 4)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=seed, device=dev)
    k, v, q = data["k"], data["v"], data["q"]
    nvec = B * Hkv * T
    kb = torch.empty((B, Hkv, T, 130), dtype=torch.uint8, device=dev)
    vb = torch.empty((B, Hkv, T, 66), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(128.0)

    def attn(qq=q):
        tq.tq_attn_decode(qq, kb, k8, vb, v4, out, ws, T, scale, signs, stream=stream)

    ops = [Op("encode_k", "ext_encode", lambda: tq.tq_encode_kv_ex(k.view(-1, 128), k8, signs, kb, stream=stream),
              nvec * (256 + 130), 1, nvec),
           Op("encode_v", "ext_encode", lambda: tq.tq_encode_kv_ex(v.view(-1, 128), v4, signs, vb,
                                                                flags=tq.TQ_FMT_NORM_CORRECT, stream=stream),
              nvec * (256 + 66), 1, nvec),
           Op("attention", "pair_attention", attn, nvec * (130 + 66) + q.numel() * 2 + out.numel() * 4, 3)]

    def e2e():
        hk, hv, hq = _pinned(k).view(-1, 128), _pinned(v).view(-1, 128), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dk, dv, dq = torch.empty_like(hk, device=dev), torch.empty_like(hv, device=dev), torch.empty_like(q)

        def step():
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            tq.tq_encode_kv_ex(dk, k8, signs, kb.view(nvec, -1), stream=stream)
            tq.tq_encode_kv_ex(dv, v4, signs, vb.view(nvec, -1), flags=tq.TQ_FMT_NORM_CORRECT, stream=stream)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, (k.numel() + v.numel() + q.numel()) * 2, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 2, out.numel() * 4

    cfg = dict(W, B=B, l2="inputs (537 MB) larger than L2; attention also timed after an L2 flush")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, config=cfg, dtype="bf16")


def plan_paged(tq, wl, dev, stream, seed, batch):
    """Llama-shaped decode step over a paged cache: the cache lives in a pool
    of 32-token pages assigned to sequences in a seeded shuffled order; the
    step encodes every token into its page slot (through a destination index)
    and runs one decode step through the block table."""
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS[wl]
    B, Hq, Hkv, T, P = batch or W["B"], W["Hq"], W["Hkv"], W["T"], W["page_tokens"]
    kcb, vcb = tq.tq_codebook_load(128, 4), tq.tq_codebook_load(128, 2)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=seed, device=dev)
    k, v, q = data["k"], data["v"], data["q"]
    per = T // P
    g = torch.Generator(device="cpu").manual_seed(seed + 7)
    table = torch.randperm(B * per, generator=g).view(B, per).to(torch.int32).to(dev)
    # destination slot of token t of (b, kvh): (page * Hkv + kvh) * P + t % P
    t = torch.arange(T, device=dev)
    pg = table.long()[:, None, t // P]                                   # [B, 1, T]
    dst = ((pg * Hkv + torch.arange(Hkv, device=dev)[None, :, None]) * P + (t % P)[None, None, :]).reshape(-1)
    nvec = B * Hkv * T
    kp = torch.empty((B * per, Hkv, P, 66), dtype=torch.uint8, device=dev)
    vp = torch.empty((B * per, Hkv, P, 34), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    scale = 1.0 / np.sqrt(128.0)
    nb = step_bytes(B, Hq, Hkv, T)

    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T), dtype=torch.uint8, device=dev)

    def attn(qq=q):
        tq.tq_attn_decode_paged(qq, kp, kcb, vp, vcb, table, P, out, T, scale, signs, workspace=ws, stream=stream)

    ops = [Op("encode_k", "encode", lambda: tq.tq_encode_kv(k.view(-1, 128), kcb, signs, kp.view(-1, 66),
                                                            dst_index=dst, stream=stream), nb["enc_k"], 1, nvec),
           Op("encode_v", "encode", lambda: tq.tq_encode_kv(v.view(-1, 128), vcb, signs, vp.view(-1, 34),
                                                            dst_index=dst, stream=stream), nb["enc_v"], 1, nvec),
           Op("attention", "paged_attention", attn, nb["attn"], 3)]

    def e2e():
        hk, hv, hq = _pinned(k).view(-1, 128), _pinned(v).view(-1, 128), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dk, dv, dq = torch.empty_like(hk, device=dev), torch.empty_like(hv, device=dev), torch.empty_like(q)

        def step():
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            tq.tq_encode_kv(dk, kcb, signs, kp.view(-1, 66), dst_index=dst, stream=stream)
            tq.tq_encode_kv(dv, vcb, signs, vp.view(-1, 34), dst_index=dst, stream=stream)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, (k.numel() + v.numel() + q.numel()) * 2, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 2, out.numel() * 4

    cfg = dict(W, B=B, l2="inputs (537 MB) larger than L2; attention also timed after an L2 flush",
               note="destination-index and block-table reads are not counted as algorithmic bytes")
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, config=cfg, dtype="bf16")


def plan_storage(tq, wl, dev, stream, seed, batch):
    from turboquant_bit_kv_gb300 import workloads
    W = WORKLOADS["storage_roundtrip"]
    L, T, hidden, bs, sf, sl = W["L"], W["T"], W["hidden"], W["block_size"], W["skip_first"], W["skip_last"]
    if batch:
        T = batch * 1024                  # smaller cases for profiling
    cb = tq.tq_codebook_load(128, 4)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    x = workloads.storage_kv(L=L, T=T, hidden=hidden, seed=seed, device=dev)["kv"]
    size = tq.tq_serde_size(L, T, hidden, bs, sf, sl, 4, 4)
    buf = torch.empty(size, dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    Lc = L - sf - sl
    nvec = 2 * Lc * T * (hidden // 128)
    each_way = x.numel() * 2 + size

    def ser(src=x):
        tq.tq_serde_serialize(src, cb, cb, signs, buf, block_size=bs, skip_first=sf, skip_last=sl, stream=stream)

    def des(dst=y):
        tq.tq_serde_deserialize(buf, cb, cb, signs, dst, block_size=bs, skip_first=sf, skip_last=sl,
                                stream=stream)

    ops = [Op("serialize", "serialize", ser, each_way, 2, nvec),
           Op("deserialize", "deserialize", des, each_way, 2 if T % bs == 0 else 2 * Lc, nvec)]

    def e2e():
        hx = _pinned(x)
        hy = torch.empty_like(x, device="cpu").pin_memory()
        dx, dy = torch.empty_like(x), torch.empty_like(x)

        def step():
            dx.copy_(hx, non_blocking=True)
            ser(dx)
            des(dy)
            hy.copy_(dy, non_blocking=True)
        return step, x.numel() * 2, x.numel() * 2

    H = hidden // 128
    qs = sf
    comp_off = 2 * qs * T * hidden * 2

    def sample():
        rng = np.random.default_rng(3)
        layer = (sf + L - sl) // 2
        ti = torch.from_numpy(np.sort(rng.choice(T, 512, replace=False))).to(dev)
        comp = buf[comp_off:comp_off + Lc * (-(-T // bs) * bs) * H * 132].view(Lc, -1, H, 132)
        res = []
        for kv, off in ((0, 0), (1, 66)):
            rows = x[kv, layer].view(T, H, 128)[ti].reshape(-1, 128)
            blocks = comp[layer - qs][ti][:, :, off:off + 66].reshape(-1, 66)
            res.append(("layer %d %s" % (layer, "KV"[kv]), 4, rows.double().cpu().numpy(), blocks.cpu().numpy()))
        return res

    def mse_per_layer():
        """Round-trip MSE of every layer (relative to the layer's mean square), K and V."""
        ser()
        des()
        torch.cuda.synchronize(dev)
        out = {"K": [], "V": []}
        for layer in range(L):
            for kv in (0, 1):
                xd = x[kv, layer].float()
                m = float(((y[kv, layer].float() - xd) ** 2).mean() / (xd * xd).mean())
                out["KV"[kv]].append(round(m, 6))
        return out

    cfg = dict(W, T=T, l2="inputs (8.6 GB) larger than L2",
               note="raw layers are device-to-device copies; per way: tensor bytes + serialised bytes")
    return dict(ops=ops, cold=None, e2e=e2e, decode_e2e=None, sample=sample, mse=mse_per_layer, config=cfg,
                dtype="bf16")


def _rotation_d(d):
    """A seeded (seed d) random orthogonal d x d matrix (QR of a Gaussian matrix), float32."""
    a = np.random.default_rng(d).standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return (q * np.sign(np.diag(r))[None, :]).astype(np.float32)


def plan_headdim(tq, wl, dev, stream, seed, batch):
    """Decode step at another head dim through the caller's dense rotation:
    head dim 160 (a spec target dim that is not a power of two) with 4
    query heads per KV head, or head dim 128 with 8 (the attention kernel's
    eight-head variant): encode K (4-bit) and V (2-bit), then one decode
    attention step."""
    W = WORKLOADS[wl]
    B, Hq, Hkv, T, d = batch or W["B"], W["Hq"], W["Hkv"], W["T"], W["head_dim"]
    kcb, vcb = tq.tq_codebook_load(d, W["key_bits"]), tq.tq_codebook_load(d, W["value_bits"])
    R = torch.from_numpy(_rotation_d(d)).to(dev)
    g = torch.Generator(device=dev).manual_seed(seed + d)
    k = torch.randn((B, Hkv, T, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B, Hkv, T, d), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((B, Hq, d), generator=g, device=dev).to(torch.bfloat16)
    kbb, vbb = tq.tq_block_bytes_d(d, W["key_bits"]), tq.tq_block_bytes_d(d, W["value_bits"])
    kb = torch.empty((B, Hkv, T, kbb), dtype=torch.uint8, device=dev)
    vb = torch.empty((B, Hkv, T, vbb), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes_d(B, Hq, Hkv, T, d), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(d)
    nvec = B * Hkv * T

    def attn(qq=q):
        tq.tq_attn_decode_d(qq, kb, kcb, vb, vcb, R, out, ws, T, scale, stream=stream)

    ops = [Op("encode_k", "hd_encode", lambda: tq.tq_encode_kv_d(k.view(-1, d), kcb, R, kb.view(nvec, -1),
                                                                 stream=stream), nvec * (2 * d + kbb), 1, nvec),
           Op("encode_v", "hd_encode", lambda: tq.tq_encode_kv_d(v.view(-1, d), vcb, R, vb.view(nvec, -1),
                                                                 stream=stream), nvec * (2 * d + vbb), 1, nvec),
           Op("attention", "hd_attention" if Hq // Hkv <= 4 else "hd_attention_g8", attn,
              nvec * (kbb + vbb) + q.numel() * 2 + out.numel() * 4, 3)]

    def e2e():
        hk, hv, hq = _pinned(k).view(-1, d), _pinned(v).view(-1, d), _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dk, dv, dq = torch.empty_like(hk, device=dev), torch.empty_like(hv, device=dev), torch.empty_like(q)

        def step():
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            tq.tq_encode_kv_d(dk, kcb, R, kb.view(nvec, -1), stream=stream)
            tq.tq_encode_kv_d(dv, vcb, R, vb.view(nvec, -1), stream=stream)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, (k.numel() + v.numel() + q.numel()) * 2, out.numel() * 4

    def decode_e2e():
        hq = _pinned(q)
        hout = torch.empty_like(out, device="cpu").pin_memory()
        dq = torch.empty_like(q)

        def step():
            dq.copy_(hq, non_blocking=True)
            attn(dq)
            hout.copy_(out, non_blocking=True)
        return step, q.numel() * 2, out.numel() * 4

    cfg = dict(W, B=B, l2="inputs (%d MB) larger than L2 (129 MB); attention also timed after an L2 flush" %
               ((k.numel() + v.numel()) * 2 // 10**6))
    return dict(ops=ops, cold="attention", e2e=e2e, decode_e2e=decode_e2e, config=cfg, dtype="bf16")


PLANS = {"llama3_8b_decode": plan_llama, "single_head_fp32": plan_single_head, "qwen25_7b_append": plan_qwen,
         "qjl_two_term": plan_qjl, "llama3_8b_prefill": plan_prefill, "llama3_8b_turboq8_pair": plan_turboq8_pair,
         "llama3_8b_paged_decode": plan_paged, "storage_roundtrip": plan_storage, "headdim_160_decode": plan_headdim,
         "headdim_128_g8_decode": plan_headdim}


def _mean_ms(evs, a, b):
    return statistics.mean(e[a].elapsed_time(e[b]) for e in evs)


def run_gpu(args, rank, world, local_rank):
    from turboquant_bit_kv_gb300 import tq

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    # a stream of our own (CUDA graphs cannot be captured on the legacy default stream)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    plan = PLANS[args.workload](tq, args.workload, dev, stream, args.seed + rank, args.batch)
    ops = plan["ops"]

    def step():
        for op in ops:
            op.fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if args.profile_only:
        # profiling mode (for ncu): a few plain steps, no timing or extras
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
        return None

    # the step as one CUDA graph (the library's calls, captured as they are issued), with a timing
    # event between the calls, so that the device time of each call excludes the host's launch
    # overhead; without graph support (or with --eager) the calls are issued one by one
    graph = None
    gev = None
    if not args.eager:
        try:
            gev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(ops) + 1)]
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                gev[0].record(stream)
                for j, op in enumerate(ops):
                    op.fn()
                    gev[j + 1].record(stream)
            for _ in range(2):
                graph.replay()
            torch.cuda.synchronize(dev)
        except Exception as exc:   # (an older torch without external events, or a capture error)
            print("bench: CUDA graph capture unavailable (%s); timing eager calls" % exc, file=sys.stderr)
            graph = None
            torch.cuda.synchronize(dev)

    # timed region: an event after every call, on the launching stream
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if graph is not None:
        # one replay per step; the events inside are read back after each replay
        per_op = [[] for _ in ops]
        step_ms = []
        t0.record(stream)
        for i in range(args.steps):
            graph.replay()
            gev[-1].synchronize()
            for j in range(len(ops)):
                per_op[j].append(gev[j].elapsed_time(gev[j + 1]))
            step_ms.append(gev[0].elapsed_time(gev[-1]))
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        clk = clocks.stop()
        ms_step = reduce_max(statistics.mean(step_ms), world)
        op_ms = [statistics.mean(v) for v in per_op]
    else:
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(args.steps)]
        t0.record(stream)
        for i in range(args.steps):
            e = evs[i]
            e[0].record(stream)
            for j, op in enumerate(ops):
                op.fn()
                e[j + 1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        clk = clocks.stop()
        ms_step = reduce_max(t0.elapsed_time(t1) / args.steps, world)
        op_ms = [_mean_ms(evs, j, j + 1) for j in range(len(ops))]

    # the attention call alone with a cold L2 (the cache was just written by
    # the encode, so the in-step time partly reads L2)
    cold_ms = None
    if plan["cold"]:
        cop = next(op for op in ops if op.name == plan["cold"])
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cold = []
        for _ in range(min(max(3, args.steps), 50)):
            flush.zero_()
            a0.record(stream)
            cop.fn()
            a1.record(stream)
            torch.cuda.synchronize(dev)
            cold.append(a0.elapsed_time(a1))
        cold_ms = statistics.median(cold)
        del flush

    def timed_e2e(make):
        step, h2d, d2h = make()
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        n_iter = max(3, min(args.steps, 200, int(2e10 // max(1, h2d + d2h))))
        barrier(world)
        t0.record(stream)
        for _ in range(n_iter):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        return reduce_max(t0.elapsed_time(t1) / n_iter, world), n_iter, h2d, d2h

    # end to end through the C ABI from pinned host buffers: the decode step
    # (new inputs from the host, cache resident) and the whole step
    full_ms, n_full, full_h2d, full_d2h = timed_e2e(plan["e2e"])
    dec = timed_e2e(plan["decode_e2e"]) if plan.get("decode_e2e") else None

    extra = {}
    if plan.get("mse"):
        extra["roundtrip_mse_per_layer"] = plan["mse"]()
    samples = plan["sample"]() if plan.get("sample") else []

    peak, peak_kind = hbm_peak()
    total = sum(op.nbytes for op in ops)
    parts, groups = {}, {}
    for op, ms in zip(ops, op_ms):
        gbs = op.nbytes / (ms * 1e-3) / 1e9
        p = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4),
             "bytes": op.nbytes}
        if op.nvec:
            p["gvec_s"] = round(op.nvec / (ms * 1e-3) / 1e9, 3)
        if op.name == plan["cold"]:
            cg = op.nbytes / (cold_ms * 1e-3) / 1e9
            p.update(cold_l2_us=round(cold_ms * 1e3, 2), cold_l2_gbs=round(cg, 1),
                     cold_l2_frac_hbm=round(cg / peak, 4))
        parts[op.name] = p
        g = groups.setdefault(op.group, {"ms": 0.0, "bytes": 0, "launches": 0, "nvec": 0})
        g["ms"] += ms
        g["bytes"] += op.nbytes
        g["launches"] += op.launches
        g["nvec"] += op.nvec

    def roofline(name):
        g = groups[name]
        ach = g["bytes"] / (g["ms"] * 1e-3) / 1e9
        tr = profiled_traffic(args.workload, name)
        if plan.get("tensor") == name:
            # a dense contraction: useful FLOPs against the measured dense 16-bit tensor peak
            tf, tkind = tensor_peak()
            fl = sum(op.flops for op in ops if op.group == name)
            at = fl / (g["ms"] * 1e-3) / 1e12
            return {"bound": "tensor", "kernel": name, "launches_per_step": g["launches"], "achieved": round(at, 2),
                    "peak": tf, "peak_kind": tkind, "unit": "TFLOP/s", "frac": round(at / tf, 4), "traffic": tr,
                    "algorithmic_flops": fl, "algorithmic_bytes": g["bytes"], "gbs": round(ach, 1)}
        return {"bound": "hbm", "kernel": name, "launches_per_step": g["launches"], "achieved": round(ach, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(ach / peak, 4),
                "traffic": tr, "algorithmic_bytes": g["bytes"]}

    # the metric: the decode-attention call's bytes over its time (per call,
    # averaged over the timed steps); without an attention call, the step's
    attn = next((op for op in ops if op.name == "attention"), None)
    if attn is not None:
        a_ms = op_ms[ops.index(attn)]
        value = world * attn.nbytes / (a_ms * 1e-3) / 1e9
        head = attn.group
        if attn.flops:
            parts[attn.name]["tflops"] = round(attn.flops / (a_ms * 1e-3) / 1e12, 2)
    else:
        value = world * total / (ms_step * 1e-3) / 1e9
        head = max(groups, key=lambda n: groups[n]["ms"])
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "dtype_note": "float32 arithmetic: exact 16-bit tensor-core products (encode), fp16 hi / lo operand splits "
                      "(attention) and every sum in float32; inputs %s, codes packed bytes" % plan["dtype"],
        "io_dtype": plan["dtype"], "data": "synthetic (seeded; no dataset or model weights)",
        "config": dict(plan["config"], workload=args.workload,
                       launch="cuda_graph (one replay per step)" if graph is not None else "eager calls",
                       parallelism="replicas" if world > 1 else "single GPU"),
        "frac_hbm": round(value / world / peak, 4),
        "frac_hbm_nominal": round(value / world / NOMINAL_HBM_GBS, 4),
    }
    enc_group = next((n for n in ("encode", "ext_encode", "hd_encode") if n in groups), None)
    if enc_group is not None:
        g = groups[enc_group]
        res["encode_gvec_s"] = round(world * g["nvec"] / (g["ms"] * 1e-3) / 1e9, 3)
        res["encode_gbs"] = round(g["bytes"] / (g["ms"] * 1e-3) / 1e9, 1)
        res["encode_frac_hbm"] = round(res["encode_gbs"] / peak, 4)
        res["encode_frac_hbm_nominal"] = round(res["encode_gbs"] / NOMINAL_HBM_GBS, 4)
    res.update({
        "step_gbs": round(world * total / (ms_step * 1e-3) / 1e9, 2),
        "parts": parts,
        "roofline": roofline(head),
        "roofline_by_kernel": {n: roofline(n) for n in groups},
    })
    full = {"value": round(world * total / (full_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "what": "the whole step's algorithmic bytes over the step run from pinned host buffers",
            "ms_per_step": round(full_ms, 4), "steps": n_full, "h2d_bytes_per_step": full_h2d,
            "d2h_bytes_per_step": full_d2h}
    if dec is not None:
        d_ms, d_n, d_h2d, d_d2h = dec
        res["e2e"] = {"value": round(world * attn.nbytes / (d_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                      "what": "attention bytes over a decode step through the C ABI: new query (and appended "
                              "K/V rows) copied from pinned host memory, append + attention against the "
                              "HBM-resident cache, output read back",
                      "ms_per_step": round(d_ms, 4), "steps": d_n, "h2d_bytes_per_step": d_h2d,
                      "d2h_bytes_per_step": d_d2h, "full_step": full}
    else:
        res["e2e"] = full
    res.update(extra)
    res["gpu_launches"] = sum(op.launches for op in ops) * args.steps
    res["clocks"] = clk
    res["_samples"] = samples
    return res


# ---------------------------------------------------------------- oracle (CPU) arm

def _oracle_books():
    import oracle
    return {b: oracle.beta_codebook(128, b)[:2] for b in (2, 3, 4)}


def _oracle_roundtrip(codec, x, s, c, bd, bits):
    """Oracle encode + pack + unpack + decode of rows x (float64 [N, 128])."""
    idx, n16, _ = codec.encode(x, s, bd.astype(np.float32))
    blk = codec.pack_block(idx, n16, bits)
    idx, n16 = codec.unpack_block(blk, bits)
    return codec.decode(idx, n16, c, s), idx, n16


_SAMPLE_INPUTS = {}


def _sample_inputs(key, make):
    """Seeded inputs of an oracle sample, drawn once per key (the draw is not
    part of the timed oracle work)."""
    if key not in _SAMPLE_INPUTS:
        _SAMPLE_INPUTS.clear()
        _SAMPLE_INPUTS[key] = make()
    return _SAMPLE_INPUTS[key]


def oracle_sample(workload, groups, seed=0, frac=1.0):
    """Time the oracle on a bounded sample of `workload`: `groups` (sequence,
    KV head) slices over the first `frac` of the context (or, for the storage
    round trip, groups of 1024 tokens x 8 heads of one compressed layer).
    Returns (seconds, algorithmic bytes of the sample, description)."""
    import oracle
    from oracle import codec
    from turboquant_bit_kv_gb300 import workloads

    W = WORKLOADS[workload]
    s = oracle.sign_diagonal(workloads.SIGN_SEED)
    books = _oracle_books()
    scale = 1 / np.sqrt(128)
    T = max(64, int(W["T"] * frac)) if "Hq" in W else 0
    if workload in ("llama3_8b_turboq8_pair", "llama3_8b_paged_decode"):
        workload = "llama3_8b_decode"
        W = WORKLOADS[workload]
    if workload in ("llama3_8b_decode", "single_head_fp32", "qwen25_7b_append"):
        G = W["Hq"] // W["Hkv"]
        kbits, vbits = W["key_bits"], W["value_bits"]
        key = (workload, groups, T, seed)
        if workload == "llama3_8b_decode":
            data = _sample_inputs(key, lambda: workloads.llama_decode(B=1, Hq=G * groups, Hkv=groups, T=T,
                                                                      seed=seed))
        elif workload == "qwen25_7b_append":
            data = _sample_inputs(key, lambda: workloads.qwen_outlier(B=1, Hq=G * groups, Hkv=groups, T=T,
                                                                      seed=seed))
        else:
            groups = 1
            d = _sample_inputs(key, lambda: workloads.single_head(T=T, seed=seed))
            data = {"k": d["k"][None, None], "v": d["v"][None, None], "q": d["q"].view(1, 1, 128)}
        k = data["k"][0].double().numpy()
        v = data["v"][0].double().numpy()
        q = data["q"].double().numpy()
        t0 = time.perf_counter()
        kh = [_oracle_roundtrip(codec, k[g], s, *books[kbits], kbits)[0] for g in range(groups)]
        vh = [_oracle_roundtrip(codec, v[g], s, *books[vbits], vbits)[0] for g in range(groups)]
        oracle.attention_dequantized(q, np.stack(kh)[None], np.stack(vh)[None], scale)
        secs = time.perf_counter() - t0
        ib = 4 if workload == "single_head_fp32" else 2
        kbb, vbb = 2 + 16 * kbits, 2 + 16 * vbits
        n = groups * T
        nbytes = n * (128 * ib * 2 + kbb + vbb) + n * (kbb + vbb) + G * groups * 128 * (ib + 4)
        desc = "%d (sequence, KV head) slice(s) at T=%d: encode K/V rows, attend %d query heads" % (groups, T, G)
        return secs, nbytes, desc
    if workload.startswith("headdim_"):
        from oracle import headdim
        G, d = W["Hq"] // W["Hkv"], W["head_dim"]
        R = _rotation_d(d).astype(np.float64)
        rng = np.random.default_rng(seed)
        k = rng.standard_normal((groups, T, d))
        v = rng.standard_normal((groups, T, d))
        q = rng.standard_normal((1, G * groups, d))
        kbits, vbits = W["key_bits"], W["value_bits"]
        ck, bk, _ = oracle.beta_codebook(d, kbits)
        cv, bv, _ = oracle.beta_codebook(d, vbits)
        t0 = time.perf_counter()
        kh, vh = [], []
        for g in range(groups):
            i, n16, _ = headdim.encode_d(k[g], R, bk.astype(np.float32))
            kh.append(headdim.decode_d(i, n16, ck, R))
            i, n16, _ = headdim.encode_d(v[g], R, bv.astype(np.float32))
            vh.append(headdim.decode_d(i, n16, cv, R))
        oracle.attention_dequantized(q, np.stack(kh)[None], np.stack(vh)[None], 1 / np.sqrt(d))
        secs = time.perf_counter() - t0
        n = groups * T
        kbb, vbb = 2 + d * kbits // 8, 2 + d * vbits // 8
        nbytes = n * (2 * d * 2 + kbb + vbb) + n * (kbb + vbb) + G * groups * d * 6
        return secs, nbytes, "%d (sequence, KV head) slice(s) at T=%d, head dim %d: encode K/V rows, attend %d query heads" % (
            groups, T, d, G)
    if workload == "llama3_8b_prefill":
        G, M = W["Hq"] // W["Hkv"], W["M"]
        data = _sample_inputs((workload, groups, T, seed),
                              lambda: workloads.llama_decode(B=1, Hq=G * groups, Hkv=groups, T=T, seed=seed))
        k = data["k"][0].double().numpy()
        v = data["v"][0].double().numpy()
        q = np.random.default_rng(seed).standard_normal((1, M, G * groups, 128))
        t0 = time.perf_counter()
        kh = [_oracle_roundtrip(codec, k[g], s, *books[4], 4)[0] for g in range(groups)]
        vh = [_oracle_roundtrip(codec, v[g], s, *books[2], 2)[0] for g in range(groups)]
        oracle.attention_causal(q, np.stack(kh)[None], np.stack(vh)[None], scale)
        secs = time.perf_counter() - t0
        n = groups * T
        nbytes = n * (256 * 2 + 100) + n * 100 + M * G * groups * 128 * 6
        desc = "%d (sequence, KV head) slice(s) at T=%d: encode K/V rows, causal attention of %d tokens x %d " \
               "heads" % (groups, T, M, G)
        return secs, nbytes, desc
    if workload == "qjl_two_term":
        G = W["Hq"] // W["Hkv"]
        data = _sample_inputs((workload, groups, T, seed),
                              lambda: workloads.qjl_keys(B=1, Hq=G * groups, Hkv=groups, T=T, seed=seed))
        k = data["k"][0].double().numpy()
        v = data["v"][0].double().numpy()
        q = data["q"].double().numpy()
        S = data["S"].double().numpy()
        c3 = books[3][0]
        t0 = time.perf_counter()
        kh, t2 = [], np.zeros((1, G * groups, T))
        for g in range(groups):
            khat, idx, n16 = _oracle_roundtrip(codec, k[g], s, *books[3], 3)
            bits, rn16, _ = oracle.qjl_encode(k[g], idx, n16, c3, s, S)
            for h in range(G):
                t2[0, g * G + h] = oracle.qjl_term2(q[0, g * G + h], bits, rn16, S)
            kh.append(khat)
        oracle.attention_dequantized(q, np.stack(kh)[None], v[None], scale, term2=t2)
        secs = time.perf_counter() - t0
        n = groups * T
        nbytes = n * 306 + n * 324 + n * 324 + G * groups * 128 * 6 + 2 * 65536
        desc = "%d (sequence, KV head) slice(s) at T=%d: K3 encode, QJL encode, two-term attention of %d " \
               "query heads" % (groups, T, G)
        return secs, nbytes, desc
    # storage round trip: encode + decode of 1024-token x 8-head groups of K and V rows
    x = _sample_inputs((workload, groups, seed),
                       lambda: workloads.storage_kv(L=1, T=1024 * groups, hidden=1024, seed=seed))["kv"]
    rows = x.double().numpy().reshape(2, -1, 128)
    c4, b4 = books[4]
    t0 = time.perf_counter()
    for kv in range(2):
        _oracle_roundtrip(codec, rows[kv], s, c4, b4, 4)
    secs = time.perf_counter() - t0
    n = rows.shape[1] * 2
    nbytes = 2 * n * (256 + 66)
    return secs, nbytes, "%d K+V rows of a compressed layer: serialise + deserialise" % n


CPU_GROUPS = {"llama3_8b_decode": 128, "single_head_fp32": 1, "qwen25_7b_append": 24, "qjl_two_term": 32,
              "llama3_8b_prefill": 8, "llama3_8b_turboq8_pair": 128, "llama3_8b_paged_decode": 128,
              "storage_roundtrip": 64, "headdim_160_decode": 32, "headdim_128_g8_decode": 32}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def busy_threads(fn):
    """fn() and the threads it kept busy on average: the process's user + system CPU time over
    the wall time of the call (the oracle's elementwise numpy work runs on one thread, its matrix
    products on as many as the BLAS library starts)."""
    import resource
    r0, w0 = resource.getrusage(resource.RUSAGE_SELF), time.perf_counter()
    out = fn()
    r1, w1 = resource.getrusage(resource.RUSAGE_SELF), time.perf_counter()
    cpu = (r1.ru_utime - r0.ru_utime) + (r1.ru_stime - r0.ru_stime)
    return out, round(cpu / max(w1 - w0, 1e-9), 1)


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores; each step is a
    bounded sample sized so that warm-up + steps stay near a minute and a half."""
    if rank != 0:
        return None
    wl = args.workload
    t1, _, _ = oracle_sample(wl, 1)            # warms caches (codebooks, Hadamard) and calibrates
    t1, _, _ = oracle_sample(wl, 1)
    per_step = 90.0 / max(1, args.steps + args.warmup)
    groups = args.cpu_groups or CPU_GROUPS[wl]
    groups = max(1, min(groups, int(per_step / max(t1, 1e-3))))
    frac = 1.0
    if groups == 1 and t1 > per_step and "Hq" in WORKLOADS[wl]:
        frac = max(1.0 / 64, per_step / t1)   # a leading part of one slice's context
    for _ in range(args.warmup):
        oracle_sample(wl, groups, frac=frac)
    times, nbytes, desc, busy = [], 0, "", []
    for _ in range(args.steps):
        (secs, nbytes, desc), b = busy_threads(lambda: oracle_sample(wl, groups, frac=frac))
        times.append(secs)
        busy.append(b)
    sec = statistics.mean(times)
    val = nbytes / sec / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": dict(WORKLOADS[wl], workload=wl),
        "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "cores": max(busy), "cores_available": cpu_cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def parity_counts(samples):
    """Codes and norms of sampled rows of the benchmarked step against the
    oracle's encoding of the same rows: coordinates within 1e-5 of a decision
    boundary, code mismatches (allowed only there, below 1e-4 of the
    coordinates), norms within 2^-22 of an fp16 rounding tie, norm mismatches."""
    import oracle
    from oracle import codec
    from turboquant_bit_kv_gb300 import workloads

    s = oracle.sign_diagonal(workloads.SIGN_SEED)
    books = {b: oracle.beta_codebook(128, b)[1].astype(np.float32) for b in (2, 3, 4)}
    rows, tot = [], {"coords": 0, "near_boundary": 0, "code_mismatch": 0, "far_mismatch": 0, "vectors": 0,
                     "norm_near_tie": 0, "norm_mismatch": 0}
    for label, bits, x, blocks in samples:
        b32 = books[bits]
        idx_o, n16_o, y = codec.encode(x, s, b32)
        idx_g, n16_g = codec.unpack_block(blocks, bits)
        near = np.zeros(y.shape, bool)
        for b in b32.astype(np.float64):
            near |= np.abs(y - b) < 1e-5
        mism = idx_g != idx_o
        n = np.sqrt(np.sum(x * x, axis=-1))
        h = n.astype(np.float16)
        mids = [0.5 * (np.nextafter(h, np.float16(0)).astype(np.float64) + h.astype(np.float64)),
                0.5 * (np.nextafter(h, np.float16(np.inf)).astype(np.float64) + h.astype(np.float64))]
        with np.errstate(divide="ignore", invalid="ignore"):
            tie = np.where(n > 0, np.minimum(np.abs(n - mids[0]), np.abs(n - mids[1])) / n, np.inf) < 2.0**-22
        r = {"sample": label, "bits": bits, "coords": int(mism.size), "near_boundary": int(near.sum()),
             "code_mismatch": int(mism.sum()), "far_mismatch": int((mism & ~near).sum()), "vectors": int(n.size),
             "norm_near_tie": int(tie.sum()), "norm_mismatch": int((n16_g != n16_o).sum())}
        rows.append(r)
        for k in tot:
            tot[k] += r[k]
    out = dict(tot, code_mismatch_frac=tot["code_mismatch"] / max(1, tot["coords"]),
               norm_mismatch_frac=tot["norm_mismatch"] / max(1, tot["vectors"]), samples=rows)
    return out


def cpu_baseline(workload, groups):
    oracle_sample(workload, 1)
    (secs, nbytes, desc), busy = busy_threads(lambda: oracle_sample(workload, groups or CPU_GROUPS[workload]))
    return {"value": round(nbytes / secs / 1e9, 6), "unit": "GB/s", "cores": busy, "cores_available": cpu_cores(),
            "kind": "oracle", "sample": "%s, %.1f s" % (desc, secs), "single_thread": single_thread_baseline(workload)}


def single_thread_baseline(workload):
    """The oracle on one (sequence, KV head) slice of the workload with every thread pool of
    numpy's libraries held to one thread (a child process: the pools are sized when numpy loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; bench.oracle_sample(%r, 1); "
            "r, b = bench.busy_threads(lambda: bench.oracle_sample(%r, 1)); "
            "print(json.dumps([r[0], r[1], r[2], b]))" % (ROOT, workload, workload))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        secs, nbytes, desc, busy = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:   # (reported, not fatal: the baseline is context, not a result)
        return {"unavailable": "%s" % type(e).__name__}
    return {"value": round(nbytes / secs / 1e9, 6), "unit": "GB/s", "cores": busy,
            "sample": "%s, %.2f s" % (desc, secs)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-groups", type=int, default=0, help="oracle sample size (0: the workload's default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller cases for profiling)")
    ap.add_argument("--eager", action="store_true", help="time the calls as issued one by one (no CUDA graph)")
    ap.add_argument("--profile-only", action="store_true",
                    help="run warm-up + steps without timing or extras (for ncu captures)")
    args = ap.parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference" and rank != 0:
        return                       # the oracle arm runs on rank 0 only
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_gpu(args, rank, world, local_rank)
        samples = res.pop("_samples", []) if res is not None else []
        if rank == 0 and res is not None and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_groups)
            if samples:
                res["parity_counts"] = parity_counts(samples)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
