"""Host logic of the multi-process benchmark on CPU (gloo, world size 2):
the max-over-ranks timing reduction and the barrier, and the reference arm's
rank handling under torchrun (rank 0 alone runs; the others exit 0)."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        m = bench.reduce_max(1.5 + rank, world)       # rank 1 is the slower one
        m2 = bench.reduce_max(-3.0 * (rank + 1), world)
        q.put((rank, m, m2))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5, -3.0), (1, 2.5, -3.0)]


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(4.25, 1) == 4.25
    bench.barrier(1)


def test_step_bytes_of_the_decode_workload():
    """Bytes counted per step: K/V bf16 rows in, 66 + 34 B blocks out, then
    the blocks, the bf16 query and the fp32 output of the attention step."""
    sys.path.insert(0, ROOT)
    import bench
    nb = bench.step_bytes(16, 32, 8, 8192)
    nvec = 16 * 8 * 8192
    assert nb["enc_k"] == nvec * (256 + 66)
    assert nb["enc_v"] == nvec * (256 + 34)
    assert nb["attn"] == nvec * 100 + 16 * 32 * 128 * (2 + 4)
    assert nb["attn"] == 105250816


def test_reference_arm_under_torchrun_prints_one_line():
    """Two ranks: rank 0 times the oracle on a tiny sample and prints the
    JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-groups", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("n,parts", [(1048576, 4), (8388608, 4), (5000, 4), (1000, 4), (1, 4), (4096, 1)])
def test_end_to_end_chunks_cover_rows_once(n, parts):
    # the chunked host-to-device copies of an end-to-end step: every row exactly once, in order,
    # at most `parts` chunks, boundaries on multiples of 1024 rows (16-byte aligned block offsets)
    sys.path.insert(0, ROOT)
    import bench
    ch = bench._chunks(n, parts)
    assert 1 <= len(ch) <= parts
    assert ch[0].start == 0 and ch[-1].stop == n
    for a, b in zip(ch, ch[1:]):
        assert a.stop == b.start
    for c in ch:
        assert c.start < c.stop and c.start % 1024 == 0


def test_every_workload_has_a_plan_an_oracle_sample_and_kernel_sources():
    """Each workload the bench accepts has a plan, an oracle sample size for
    the CPU baseline, and every traffic row names a workload and a kernel
    group whose sources the bench can hash."""
    sys.path.insert(0, ROOT)
    import bench
    assert set(bench.PLANS) == set(bench.WORKLOADS) == set(bench.CPU_GROUPS)
    assert bench.DEFAULT_WORKLOAD in bench.WORKLOADS
    for group, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(bench.CSRC, f)), (group, f)
    rows = [l.split("|")[1:3] for l in open(bench.TRAFFIC_TABLE) if l.startswith("| ") and l.count("|") >= 8]
    rows = [(w.strip(), g.strip()) for w, g in rows if w.strip() not in ("workload", "---")]
    assert rows
    for w, g in rows:
        assert w in bench.WORKLOADS and g in bench.KERNEL_SOURCES, (w, g)


def test_cpu_baseline_reports_busy_threads_and_a_single_thread_figure():
    """The oracle's CPU baseline carries the threads it kept busy (CPU time
    over wall time) and a figure with numpy's thread pools held to one."""
    sys.path.insert(0, ROOT)
    import bench
    (out, busy) = bench.busy_threads(lambda: sum(i * i for i in range(200000)))
    assert out > 0 and 0.5 <= busy <= 1.5          # a pure-Python loop keeps one thread busy
    st = bench.single_thread_baseline("single_head_fp32")
    assert "unavailable" not in st, st
    assert st["cores"] <= 1.2 and st["value"] > 0 and st["unit"] == "GB/s"
