"""Benchmark of the TurboQuant KV hot path on GB300.

One step = quantise-on-insert of the whole K and V cache (tq_encode_kv: K
4-bit, V 2-bit) followed by one fused decode-attention step over it
(tq_attn_decode), on the Llama-3-8B-shaped decode workload: batch 16,
32 query heads, 8 KV heads, head_dim 128, context 8192, bf16 K/V with
log-normal channel scales and AR(1) token correlation 0.9.

`value` is the algorithmic bytes of a step (K/V bf16 in + packed blocks out,
packed blocks + q in + fp32 out) over the device time of a step, in GB/s.
`e2e` is the same bytes over the time of a step run through the C ABI from
pinned host buffers (host->device copy of K, V and q, the step, and the
device->host copy of the output inside the timed region).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs an independent replica on its own GPU (weak
scaling; the path has no exchange step); rank 0 prints one JSON line.
"""

import argparse
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
WORKLOAD = dict(workload="llama3_8b_decode", B=16, Hq=32, Hkv=8, T=8192, head_dim=128,
                key_bits=4, value_bits=2, kv_dtype="bf16", scale="1/sqrt(128)")
FALLBACK_HBM_GBS = 6800.0


def step_bytes(B, Hq, Hkv, T, kbits=4, vbits=2):
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


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world, local_rank):
    from turboquant_bit_kv_gb300 import tq, workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    W = WORKLOAD
    B, Hq, Hkv, T = args.batch or W["B"], W["Hq"], W["Hkv"], W["T"]
    nb = step_bytes(B, Hq, Hkv, T)
    kcb, vcb = tq.tq_codebook_load(128, 4), tq.tq_codebook_load(128, 2)
    signs = tq.tq_signs_from_seed(workloads.SIGN_SEED)
    data = workloads.llama_decode(B=B, Hq=Hq, Hkv=Hkv, T=T, seed=args.seed + rank, device=dev)
    k, v, q = data["k"], data["v"], data["q"]
    kb = torch.empty((B, Hkv, T, tq.tq_block_bytes(4)), dtype=torch.uint8, device=dev)
    vb = torch.empty((B, Hkv, T, tq.tq_block_bytes(2)), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attn_workspace_bytes(B, Hq, Hkv, T), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(128.0)
    stream = torch.cuda.current_stream(dev)
    kf, vf = k.view(-1, 128), v.view(-1, 128)

    def step():
        tq.tq_encode_kv(kf, kcb, signs, kb, stream=stream)
        tq.tq_encode_kv(vf, vcb, signs, vb, stream=stream)
        tq.tq_attn_decode(q, kb, kcb, vb, vcb, out, ws, T, scale, signs, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if args.profile_only:
        # profiling mode (for ncu): a few plain steps, no timing or extras
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
        return None

    # timed region: per-kernel events on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        e = evs[i]
        e[0].record(stream)
        tq.tq_encode_kv(kf, kcb, signs, kb, stream=stream)
        e[1].record(stream)
        tq.tq_encode_kv(vf, vcb, signs, vb, stream=stream)
        e[2].record(stream)
        tq.tq_attn_decode(q, kb, kcb, vb, vcb, out, ws, T, scale, signs, stream=stream)
        e[3].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ms_step = reduce_max(ms_total / args.steps, world)
    enc_k_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    enc_v_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    attn_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    # attention alone with a cold L2 (the cache was just written by the encode)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cold = []
    for _ in range(min(max(3, args.steps), 50)):
        flush.zero_()
        a0.record(stream)
        tq.tq_attn_decode(q, kb, kcb, vb, vcb, out, ws, T, scale, signs, stream=stream)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        cold.append(a0.elapsed_time(a1))
    attn_cold_ms = statistics.median(cold)
    del flush

    # end to end through the C ABI from pinned host buffers
    hk = k.cpu().pin_memory()
    hv = v.cpu().pin_memory()
    hq = q.cpu().pin_memory()
    hout = torch.empty_like(out, device="cpu").pin_memory()
    dk, dv, dq = torch.empty_like(k), torch.empty_like(v), torch.empty_like(q)

    def e2e_step():
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        tq.tq_encode_kv(dk.view(-1, 128), kcb, signs, kb, stream=stream)
        tq.tq_encode_kv(dv.view(-1, 128), vcb, signs, vb, stream=stream)
        tq.tq_attn_decode(dq, kb, kcb, vb, vcb, out, ws, T, scale, signs, stream=stream)
        hout.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    n_e2e = min(args.steps, 200)
    t0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(t0.elapsed_time(t1) / n_e2e, world)

    peak, peak_kind = hbm_peak()
    enc_bytes = nb["enc_k"] + nb["enc_v"]
    enc_gbs = enc_bytes / ((enc_k_ms + enc_v_ms) * 1e-3) / 1e9
    attn_gbs = nb["attn"] / (attn_ms * 1e-3) / 1e9
    attn_cold_gbs = nb["attn"] / (attn_cold_ms * 1e-3) / 1e9
    value = world * nb["total"] / (ms_step * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; no dataset or model weights)",
        "config": dict(WORKLOAD, l2="inputs (537 MB) larger than L2 (129 MB); attention also timed after an "
                       "L2 flush", parallelism="replicas" if world > 1 else "single GPU"),
        "parts": {
            "encode": {"us": round((enc_k_ms + enc_v_ms) * 1e3, 2), "gbs": round(enc_gbs, 1),
                       "gvec_s": round(nb["nvec"] / ((enc_k_ms + enc_v_ms) * 1e-3) / 1e9, 3),
                       "frac_hbm": round(enc_gbs / peak, 4)},
            "attention": {"us": round(attn_ms * 1e3, 2), "gbs": round(attn_gbs, 1),
                          "frac_hbm": round(attn_gbs / peak, 4), "cold_l2_us": round(attn_cold_ms * 1e3, 2),
                          "cold_l2_gbs": round(attn_cold_gbs, 1),
                          "cold_l2_frac_hbm": round(attn_cold_gbs / peak, 4)},
        },
        "roofline": {"bound": "hbm", "kernel": "encode_kernel (K 4-bit + V 2-bit launches)",
                     "achieved": round(enc_gbs, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(enc_gbs / peak, 4), "traffic": None},
        "e2e": {"value": round(world * nb["total"] / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": k.numel() * 2 + v.numel() * 2 + q.numel() * 2,
                "d2h_bytes_per_step": out.numel() * 4},
        "gpu_launches": 4 * args.steps,
        "clocks": clk,
    }
    return res


# ---------------------------------------------------------------- oracle (CPU) arm

def oracle_sample(groups, seed=0):
    """Time the oracle on `groups` (sequence, KV head) slices of the workload:
    encode their K and V rows, then decode attention for their query heads.
    Returns (seconds, algorithmic bytes of the sample)."""
    import oracle
    from oracle import codec
    from turboquant_bit_kv_gb300 import workloads

    W = WORKLOAD
    T, G = W["T"], W["Hq"] // W["Hkv"]
    data = workloads.llama_decode(B=1, Hq=G * groups, Hkv=groups, T=T, seed=seed)
    k = data["k"][0].double().numpy()
    v = data["v"][0].double().numpy()
    q = data["q"].double().numpy()
    s = oracle.sign_diagonal(workloads.SIGN_SEED)
    kc, kbd, _ = oracle.beta_codebook(128, 4)
    vc, vbd, _ = oracle.beta_codebook(128, 2)
    t0 = time.perf_counter()
    kh, vh = [], []
    for g in range(groups):
        ki, kn, _ = codec.encode(k[g], s, kbd.astype(np.float32))
        vi, vn, _ = codec.encode(v[g], s, vbd.astype(np.float32))
        kblk, vblk = codec.pack_block(ki, kn, 4), codec.pack_block(vi, vn, 2)
        ki, kn = codec.unpack_block(kblk, 4)
        vi, vn = codec.unpack_block(vblk, 2)
        kh.append(codec.decode(ki, kn, kc, s))
        vh.append(codec.decode(vi, vn, vc, s))
    oracle.attention_dequantized(q, np.stack(kh)[None], np.stack(vh)[None], 1 / np.sqrt(128))
    secs = time.perf_counter() - t0
    nb = step_bytes(1, G * groups, groups, T)
    return secs, nb["total"]


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return None
    groups = args.cpu_groups
    oracle_sample(1)                  # warm caches (codebook iteration, Hadamard matrix)
    times, nbytes = [], 0
    for _ in range(args.warmup):
        oracle_sample(groups)
    for _ in range(args.steps):
        secs, nbytes = oracle_sample(groups)
        times.append(secs)
    sec = statistics.mean(times)
    val = nbytes / sec / 1e9
    sample = "%d of 128 (sequence, KV head) slices per step: encode their K/V rows (T=8192) and attend " \
             "their 4 query heads" % groups
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": dict(WORKLOAD), "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "cores": cpu_cores(),
                                                   "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(groups):
    oracle_sample(1)
    secs, nbytes = oracle_sample(groups)
    return {"value": round(nbytes / secs / 1e9, 6), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "%d of 128 (sequence, KV head) slices of the step (encode K/V rows, attend 4 query "
                      "heads), %.1f s" % (groups, secs)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-groups", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller cases for profiling)")
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
        if args.cpu_groups == 128:
            args.cpu_groups = 4
        res = run_reference(args, rank, world)
    else:
        res = run_gpu(args, rank, world, local_rank)
        if rank == 0 and res is not None and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.cpu_groups)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
