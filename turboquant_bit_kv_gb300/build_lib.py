"""Build libtq.so in-tree with nvcc for sm_103a (translation units compiled in
parallel, then linked as one shared library next to this file)."""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtq.so")

SOURCES = ["tq_host.cpp", "tq_encode.cu", "tq_decode.cu", "tq_codec.cu", "tq_qjl.cu", "tq_attn.cu", "tq_attn_g1.cu", "tq_attn_g2.cu",
           "tq_attn_g4.cu", "tq_attn_g8.cu", "tq_attn_noalloc.cu", "tq_attn_plan.cu", "tq_attn_mma.cu", "tq_attn_mma_k2.cu",
           "tq_attn_mma_k3.cu", "tq_attn_mma_k4.cu", "tq_attn_mma_k8.cu", "tq_status.cu",
           "tq_attn_prefill.cu", "tq_ext.cu", "tq_headdim.cu", "tq_headdim_tc.cu", "tq_headdim_mma.cu",
           "tq_headdim_mma8.cu"]
HEADERS = ["tq_device.cuh", "tq_tc.cuh", "tq_attn.cuh", "tq_attn_mma.h", "tq_attn_mma.cuh", "tq_internal.h", "tq_headdim.cuh",
           "tq_headdim_mma.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include"),
         "-I" + CSRC]


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def _compile(src):
    obj = os.path.join(BUILD, src + ".o")
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in HEADERS] + \
        [os.path.join(ROOT, "include", "tq.h")]
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest(deps):
        return obj
    cmd = [NVCC] + ARCH + FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj


def build(verbose=False):
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest(objs):
        return LIB
    tmp = LIB + ".tmp"
    cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    if verbose:
        print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
