// Decode attention: split-combine kernel and the C-ABI entry points
// tq_attn_workspace_bytes / tq_attn_decode.  The split-pass kernels live in
// tq_attn.cuh and are instantiated in tq_attn_g{1,2,4,8}.cu.
#include <cmath>

#include "tq_attn.cuh"
#include "tq_attn_mma.h"
#include "tq_internal.h"

namespace tq {

int launch_attn_split_g1(int kb, int vb, const AttnArgs &a, dim3 grid, int smem, cudaStream_t st);
int launch_attn_split_g2(int kb, int vb, const AttnArgs &a, dim3 grid, int smem, cudaStream_t st);
int launch_attn_split_g4(int kb, int vb, const AttnArgs &a, dim3 grid, int smem, cudaStream_t st);
int launch_attn_split_g8(int kb, int vb, const AttnArgs &a, dim3 grid, int smem, cudaStream_t st);

// Merge the splits of one (sequence, query head).  When the values were
// packed (accumulated in the rotated domain) the result is rotated back:
// o = D H (acc / l) / sqrt(128); raw values were accumulated as they are.
__global__ void __launch_bounds__(kAttnThreads) attn_combine_kernel(const float *ws, int splits, int rotate_back,
                                                                    uint32_t s0, uint32_t s1, uint32_t s2,
                                                                    uint32_t s3, float *out) {
    __shared__ float buf[kD];
    const int d = threadIdx.x;
    const float *base = ws + (int64_t)blockIdx.x * splits * kPartialFloats;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, base[s * kPartialFloats]);
    float l = 0.f, acc = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float m = base[s * kPartialFloats];
            if (m == -INFINITY) continue;
            const float w = exp2f(m - M);
            l = fmaf(w, base[s * kPartialFloats + 1], l);
            acc = fmaf(w, base[s * kPartialFloats + 4 + d], acc);
        }
    }
    const float o = l > 0.f ? acc / l : 0.f;
    if (!rotate_back) {
        out[(int64_t)blockIdx.x * kD + d] = o;
        return;
    }
    buf[d] = o;
    __syncthreads();
    smem_fwht_rows<1>(buf);
    const uint32_t sw[4] = {s0, s1, s2, s3};
    const float v = buf[d] * 0.08838834764831845f;
    out[(int64_t)blockIdx.x * kD + d] = ((sw[d >> 5] >> (d & 31)) & 1u) ? -v : v;
}

// Merge for the tensor-core kernel's partition: the slots of segment
// j = (sequence, KV head) are the CTAs that touched it.  Launched as a
// programmatic dependent of the attention kernel: its CTAs may start while
// the attention kernel drains and wait here until its writes are visible.
__global__ void __launch_bounds__(kAttnThreads) attn_combine_mma_kernel(const float *ws, MmaPlan plan, int Hq,
                                                                        int Hkv, int rotate_back, uint32_t s0,
                                                                        uint32_t s1, uint32_t s2, uint32_t s3,
                                                                        float *out) {
    __shared__ float buf[kD];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int d = threadIdx.x;
    const int b = blockIdx.x / Hq, h = blockIdx.x % Hq;
    const int G = Hq / Hkv;
    const int64_t j = (int64_t)b * Hkv + h / G;
    const int64_t first = mma_cta_of_chunk(j * plan.C, plan);
    const int nslots = (int)(mma_cta_of_chunk((j + 1) * plan.C - 1, plan) - first + 1);
    const float *base = ws + (int64_t)blockIdx.x * plan.Smax * kPartialFloats;
    float M = -INFINITY;
    for (int s = 0; s < nslots; ++s) M = fmaxf(M, base[s * kPartialFloats]);
    float l = 0.f, acc = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < nslots; ++s) {
            const float m = base[s * kPartialFloats];
            if (m == -INFINITY) continue;
            const float w = exp2f(m - M);
            l = fmaf(w, base[s * kPartialFloats + 1], l);
            acc = fmaf(w, base[s * kPartialFloats + 4 + d], acc);
        }
    }
    const float o = l > 0.f ? acc / l : 0.f;
    if (!rotate_back) {
        out[(int64_t)blockIdx.x * kD + d] = o;
        return;
    }
    buf[d] = o;
    __syncthreads();
    smem_fwht_rows<1>(buf);
    const uint32_t sw[4] = {s0, s1, s2, s3};
    const float v = buf[d] * 0.08838834764831845f;
    out[(int64_t)blockIdx.x * kD + d] = ((sw[d >> 5] >> (d & 31)) & 1u) ? -v : v;
}

static int attn_smem_bytes(int kb, int vb) {
    const int head = (1040 * 2 + 8 * kD + kTT * 8 + 8 * 4 + 32) * 4;
    const int kbb = 2 + 16 * kb, vbb = vb == 16 ? 256 : 2 + 16 * vb;
    const int stage = ((kTT * kbb + 15) & ~15) + ((kTT * vbb + 15) & ~15) + kTT * 16 + kTT * 2;
    return head + 2 * stage;
}

}  // namespace tq

using namespace tq;

extern "C" size_t tq_attn_workspace_bytes(int B, int Hq, int Hkv, int T_cap) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || T_cap <= 0 || Hq % Hkv) return 0;
    int splits, tps;
    attn_split_plan(B, Hkv, T_cap, &splits, &tps);
    const int ms = mma_max_slots(B, Hkv, T_cap);
    const int slots = splits > ms ? splits : ms;
    return (size_t)B * Hq * slots * kPartialFloats * sizeof(float);
}

extern "C" int tq_attn_decode(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                              const void *v, const tq_codebook *vcb, const int32_t *seq_lens, int B, int Hq,
                              int Hkv, int T_cap, int T, float scale, tq_signs signs, const uint8_t *qjl_bits,
                              const uint16_t *res_norm_f16, const float *S, float *out, void *workspace,
                              size_t workspace_bytes, void *stream) {
    if (!q || !k_blocks || !kcb || !v || !out || !workspace) return TQ_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T_cap <= 0 || T < 1 || T > T_cap || (T_cap & 7))
        return TQ_ERR_ARG;
    if (!std::isfinite(scale)) return TQ_ERR_ARG;
    const int G = Hq / Hkv;
    if (G > 8 || dtype_bytes(q_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (kcb->head_dim != kD || kcb->bits < 2 || kcb->bits > 4 || kcb->levels != (1 << kcb->bits))
        return TQ_ERR_UNSUPPORTED;
    if (vcb && (vcb->head_dim != kD || vcb->bits < 2 || vcb->bits > 4 || vcb->levels != (1 << vcb->bits)))
        return TQ_ERR_UNSUPPORTED;
    const bool qjl = qjl_bits || res_norm_f16 || S;
    if (qjl && !(qjl_bits && res_norm_f16 && S)) return TQ_ERR_ARG;
    if (!aligned(q, dtype_bytes(q_dtype)) || !aligned(k_blocks, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(workspace, 16) || (qjl && (!aligned(qjl_bits, 16) || !aligned(res_norm_f16, 16) || !aligned(S, 4))))
        return TQ_ERR_ALIGN;
    if (workspace_bytes < tq_attn_workspace_bytes(B, Hq, Hkv, T_cap)) return TQ_ERR_WORKSPACE;

    AttnArgs a;
    a.q = q;
    a.q_dtype = q_dtype;
    a.k = k_blocks;
    a.v = static_cast<const uint8_t *>(v);
    a.seq_lens = seq_lens;
    a.qjl_bits = qjl ? qjl_bits : nullptr;
    a.rn = qjl ? res_norm_f16 : nullptr;
    a.S = qjl ? S : nullptr;
    a.ws = static_cast<float *>(workspace);
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.T_cap = T_cap;
    a.T = T;
    attn_split_plan(B, Hkv, T, &a.splits, &a.tiles_per_split);
    a.qscale = scale * 1.4426950408889634f;
    for (int i = 0; i < 16; ++i) {
        a.kc[i] = kcb->centroids[i];
        a.vc[i] = vcb ? vcb->centroids[i] : 0.f;
    }
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];

    const int kb = kcb->bits, vb = vcb ? vcb->bits : 16;
    const int smem = attn_smem_bytes(kb, vb);
    cudaStream_t st = (cudaStream_t)stream;
    dim3 grid(a.splits, Hkv, B);
    if (attn_mma_supported(kb, vb, qjl, G)) {
        MmaPlan mp = mma_plan(B, Hkv, T, kb, vb, qjl, G);
        int r = launch_attn_mma(a, mp, kb, vb, qjl, st);
        if (r != TQ_OK) return r;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(B * Hq));
        cfg.blockDim = dim3(kAttnThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, attn_combine_mma_kernel, (const float *)a.ws, mp, Hq, Hkv, vcb ? 1 : 0,
                               signs.w[0], signs.w[1], signs.w[2], signs.w[3], out) != cudaSuccess)
            return TQ_ERR_CUDA;
        return launch_status();
    }
    int r;
    if (G == 1) r = launch_attn_split_g1(kb, vb, a, grid, smem, st);
    else if (G == 2) r = launch_attn_split_g2(kb, vb, a, grid, smem, st);
    else if (G <= 4) r = launch_attn_split_g4(kb, vb, a, grid, smem, st);
    else r = launch_attn_split_g8(kb, vb, a, grid, smem, st);
    if (r != TQ_OK) return r;
    attn_combine_kernel<<<B * Hq, kAttnThreads, 0, st>>>(a.ws, a.splits, vcb ? 1 : 0, signs.w[0], signs.w[1],
                                                          signs.w[2], signs.w[3], out);
    return launch_status();
}
