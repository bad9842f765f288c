"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the method: it only draws the inputs that
both the CUDA path and the CPU oracle consume.  Every generator uses its own
``torch.Generator`` seeded from ``seed`` on the requested device, draws in a
fixed order, computes in float32 and casts to the stored dtype (round to
nearest even).  The same seed on CPU and on CUDA gives different numbers;
a test always generates once and hands the same bytes to both sides.

Workloads (head_dim 128 throughout):

* ``single_head``      -- one head, K and V [T, 128] float32 i.i.d. N(0, 1),
                          one float32 N(0, 1) query (T = 4096).
* ``llama_decode``     -- K, V [B, Hkv, T, 128] bf16 with a per-(KV head,
                          channel) LogNormal(0, 0.5) scale (drawn separately
                          for K and V) over AR(1) token series of correlation
                          0.9 with unit stationary variance; q [B, Hq, 128]
                          bf16 N(0, 1).  (B 16, Hq 32, Hkv 8, T 8192.)
* ``qwen_outlier``     -- K, V [B, Hkv, T, 128] bf16 N(0, 1) where 1% of the
                          Hkv*128 KV channels (rounded) are multiplied by 20;
                          the same channels for K and V; q bf16 N(0, 1).
                          (B 64, Hq 28, Hkv 4, T 32768 + 1 appended token.)
* ``qjl_keys``         -- K bf16 N(0, 1), V fp16 N(0, 1) [B, Hkv, T, 128],
                          q bf16 N(0, 1), Gaussian sketch S [128, 128] float32
                          N(0, 1) from its own seed.  (B 8, Hq 32, Hkv 8,
                          T 16384.)
* ``storage_kv``       -- [2, L, T, hidden] bf16 N(0, 1).  (L 32, T 65536,
                          hidden 1024.)

The pages measure quality on public datasets and real model activations; none
of those are used here -- these draws stand in for them.
"""

import torch

SIGN_SEED = 1      # seed of the sign diagonal D (splitmix64 on both sides)
SKETCH_SEED = 2    # seed of the QJL sketch S


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, chunk_rows=1 << 20):
    """float32 N(0, 1) of the given shape, drawn in row chunks of the first
    dimension to bound temporaries."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    flat = out.view(shape[0], -1)
    per = max(1, chunk_rows * 128 // max(1, flat.shape[1]))
    for i in range(0, shape[0], per):
        flat[i:i + per] = torch.randn(flat[i:i + per].shape, generator=g,
                                      device=device, dtype=torch.float32)
    return out


def single_head(T=4096, seed=0, device="cpu"):
    g = _gen(device, seed)
    k = torch.randn((T, 128), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((T, 128), generator=g, device=device, dtype=torch.float32)
    q = torch.randn((128,), generator=g, device=device, dtype=torch.float32)
    return {"k": k, "v": v, "q": q}


def _ar1(B, H, T, rho, g, device):
    """AR(1) series along T: z_0 ~ N(0,1), z_t = rho z_{t-1} + sqrt(1-rho^2) e_t."""
    e = torch.randn((B, H, T, 128), generator=g, device=device, dtype=torch.float32)
    c = (1.0 - rho * rho) ** 0.5
    z = torch.empty_like(e)
    z[:, :, 0] = e[:, :, 0]
    for t in range(1, T):
        torch.add(z[:, :, t - 1] * rho, e[:, :, t], alpha=c, out=z[:, :, t])
    return z


def llama_decode(B=16, Hq=32, Hkv=8, T=8192, rho=0.9, seed=0, device="cpu"):
    g = _gen(device, seed)
    out = {}
    for name in ("k", "v"):
        scale = torch.exp(0.5 * torch.randn((Hkv, 128), generator=g, device=device,
                                            dtype=torch.float32))
        z = _ar1(B, Hkv, T, rho, g, device)
        out[name] = (z * scale[None, :, None, :]).to(torch.bfloat16)
        del z
    out["q"] = torch.randn((B, Hq, 128), generator=g, device=device,
                           dtype=torch.float32).to(torch.bfloat16)
    return out


def qwen_outlier(B=64, Hq=28, Hkv=4, T=32769, outlier_frac=0.01, factor=20.0,
                 seed=0, device="cpu"):
    g = _gen(device, seed)
    n_ch = Hkv * 128
    n_out = int(round(outlier_frac * n_ch))
    perm = torch.randperm(n_ch, generator=g, device=device)
    ch = torch.sort(perm[:n_out]).values
    mult = torch.ones(n_ch, device=device, dtype=torch.float32)
    mult[ch] = factor
    mult = mult.view(Hkv, 128)
    out = {"outlier_channels": ch.cpu()}
    for name in ("k", "v"):
        x = torch.empty((B, Hkv, T, 128), dtype=torch.bfloat16, device=device)
        for b in range(B):
            r = torch.randn((Hkv, T, 128), generator=g, device=device, dtype=torch.float32)
            x[b] = (r * mult[:, None, :]).to(torch.bfloat16)
        out[name] = x
    out["q"] = torch.randn((B, Hq, 128), generator=g, device=device,
                           dtype=torch.float32).to(torch.bfloat16)
    return out


def qjl_keys(B=8, Hq=32, Hkv=8, T=16384, seed=0, device="cpu"):
    g = _gen(device, seed)
    k = _randn((B, Hkv, T, 128), g, device).to(torch.bfloat16)
    v = _randn((B, Hkv, T, 128), g, device).to(torch.float16)
    q = torch.randn((B, Hq, 128), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    gs = _gen(device, SKETCH_SEED)
    S = torch.randn((128, 128), generator=gs, device=device, dtype=torch.float32)
    return {"k": k, "v": v, "q": q, "S": S}


def storage_kv(L=32, T=65536, hidden=1024, seed=0, device="cpu"):
    g = _gen(device, seed)
    x = torch.empty((2, L, T, hidden), dtype=torch.bfloat16, device=device)
    for kv in range(2):
        for l in range(L):
            x[kv, l] = torch.randn((T, hidden), generator=g, device=device,
                                   dtype=torch.float32).to(torch.bfloat16)
    return {"kv": x}
