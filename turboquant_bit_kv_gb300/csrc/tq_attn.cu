// Decode attention: split-combine kernel and the C-ABI entry points
// tq_attn_workspace_bytes / tq_attn_decode.  The split-pass kernels live in
// tq_attn.cuh and are instantiated in tq_attn_g{1,2,4,8}.cu.
#include <algorithm>
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

// (hi, lo) fp16 halves of x packed as one half2: x = hi + lo to about 2^-22.
__device__ __forceinline__ uint32_t prep_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Query prep of the tensor-core kernel, once per (sequence, KV head)
// segment j: the rotated query R q = H (D q) / sqrt(128) of each of its G
// heads times scale * log2(e) ("TurboQuant KV Cache Compression — Spec",
// Optimization: Fused dequant-dot: the query is rotated once), and for the
// two-term score the sketched raw query S q times scale * log2(e) *
// sqrt(pi / 2) / m ("RotorQuant KV Cache Compression", The QJL Estimator
// Formula), m = 128.  Each is split x = hi + lo into fp16 halves and stored
// as the B fragments of the m16n8k16 products: part p (n-tiles 0, 1 of the
// rotated query; 2: S q), lane (g, t), k-step ks -> words 2 ks, 2 ks + 1 =
// rows {2t, 2t+1}, {2t+8, 2t+9} <-> dims 32t + 4ks + {0, 1}, {2, 3} of
// column g = (head 4p + g / 2, part g & 1: hi / lo).
__global__ void __launch_bounds__(kAttnThreads) attn_prep_mma_kernel(const __grid_constant__ AttnArgs a,
                                                                     MmaPlan plan, int qjl) {
    __shared__ __align__(16) float qs[8 * kD];
    __shared__ __align__(16) float raw[8 * kD];   // two-term score: scaled raw queries, then S q
    asm volatile("griddepcontrol.launch_dependents;");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t j = blockIdx.x;
    const int b = (int)(j / a.Hkv), kvh = (int)(j % a.Hkv);
    for (int h = warp; h < 8; h += 4) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (h < a.G) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                v[k] = load_q(a.q, a.q_dtype, ((int64_t)b * a.Hq + kvh * a.G + h) * kD + 4 * lane + k);
        }
        if (qjl) {
            const float f = a.qscale * (1.2533141373155003f / 128.f);   // sqrt(pi / 2) / m, m = 128
            reinterpret_cast<float4 *>(raw + h * kD)[lane] = make_float4(v[0] * f, v[1] * f, v[2] * f, v[3] * f);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = 4 * lane + k;
            if ((a.signs[d >> 5] >> (d & 31)) & 1u) v[k] = -v[k];
        }
        const float x0 = v[0] + v[1], x1 = v[0] - v[1], x2 = v[2] + v[3], x3 = v[2] - v[3];
        v[0] = x0 + x2;
        v[2] = x0 - x2;
        v[1] = x1 + x3;
        v[3] = x1 - x3;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float o = __shfl_xor_sync(0xffffffffu, v[k], m);
                v[k] = (lane & m) ? (o - v[k]) : (v[k] + o);
            }
        }
        const float f = a.qscale * 0.08838834764831845f;
        reinterpret_cast<float4 *>(qs + h * kD)[lane] = make_float4(v[0] * f, v[1] * f, v[2] * f, v[3] * f);
    }
    __syncthreads();
    if (qjl) {
        // (S q)_jo of heads 0..3 (the two-term score covers G <= 4)
        const int jo = tid;
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 *srow = reinterpret_cast<const float4 *>(a.S + (int64_t)jo * kD);
#pragma unroll 4
        for (int d4 = 0; d4 < 32; ++d4) {
            const float4 s4 = __ldg(srow + d4);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const float4 q4 = reinterpret_cast<const float4 *>(raw + hh * kD)[d4];
                acc4[hh] = fmaf(s4.x, q4.x, fmaf(s4.y, q4.y, fmaf(s4.z, q4.z, fmaf(s4.w, q4.w, acc4[hh]))));
            }
        }
        __syncthreads();   // every raw query is read before the products overwrite them
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) raw[hh * kD + jo] = acc4[hh];
        __syncthreads();
    }
    const int p = warp;
    if (p < 2 || (p == 2 && qjl)) {
        const float *buf = p == 2 ? raw : qs;
        // column g of n-tile nt: head 4 nt + g / 2, part g & 1 (hi, lo); with 5 to 8 query heads per
        // KV head, head g, part nt
        const int nt = p == 2 ? 0 : p, g = lane >> 2, t = lane & 3;
        const bool h8 = a.G > 4 && p < 2;
        const int head = h8 ? g : 4 * nt + (g >> 1);
        const bool lo_part = h8 ? nt == 1 : (g & 1) != 0;
        uint32_t w[16];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const float4 q4 = reinterpret_cast<const float4 *>(buf + head * kD + 32 * t + 4 * ks)[0];
            float e[4] = {q4.x, q4.y, q4.z, q4.w};
            if (lo_part) {
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] -= __half2float(__float2half_rn(e[i]));
            }
            w[2 * ks] = prep_half2(e[0], e[1]);
            w[2 * ks + 1] = prep_half2(e[2], e[3]);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(a.ws + plan.frag_off + j * kFragWords) + p * 128 + lane * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
}

// Merge for the tensor-core kernel's partition: the slots of segment
// j = (sequence, KV head) are the warps whose chunk ranges touch it.  One
// CTA per (sequence, query head) of 128 x ng threads: thread d of slot
// group g reduces output dim d over batches g, g + ng, ... of 32 slots.
// Reading what other SMs just wrote costs a full L2 round trip, so each
// thread issues every load of a batch at once (m and l of each slot -- the
// same address across the group -- and its dim of acc) and only then
// reduces, with the running max rescaled between batches; the groups run
// their rounds side by side and meet in shared memory.  Launched as a
// programmatic dependent of the attention kernel: its CTAs wait here until
// that grid has finished and its writes are visible.
__global__ void __launch_bounds__(kAttnThreads * kCombineMaxGroups) attn_combine_mma_kernel(
    const float *ws, MmaPlan plan, int Hq, int Hkv, int rotate_back, uint32_t s0, uint32_t s1, uint32_t s2,
    uint32_t s3, float *out) {
    constexpr int kBatch = 32;
    __shared__ float buf[kD];
    __shared__ float gacc[kCombineMaxGroups][kD];
    __shared__ float gml[kCombineMaxGroups][2];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int d = threadIdx.x & (kD - 1), grp = threadIdx.x / kD, ng = blockDim.x / kD;
    const int b = blockIdx.x / Hq, h = blockIdx.x % Hq;
    const int G = Hq / Hkv;
    const int64_t j = (int64_t)b * Hkv + h / G;
    const int64_t first = mma_worker_of_chunk(j * plan.C, plan);
    const int nslots = (int)(mma_worker_of_chunk((j + 1) * plan.C - 1, plan) - first + 1);
    const float *base = ws + (int64_t)blockIdx.x * plan.Smax * kPartialFloats;
    float M = -INFINITY, l = 0.f, acc = 0.f;
    for (int sb = grp * kBatch; sb < nslots; sb += ng * kBatch) {
        float mv[kBatch], lv[kBatch], xv[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const bool ok = sb + i < nslots;
            const float *ps = base + (int64_t)(sb + i) * kPartialFloats;
            mv[i] = ok ? __ldcg(ps) : -INFINITY;
            lv[i] = ok ? __ldcg(ps + 1) : 0.f;
            xv[i] = ok ? __ldcg(ps + 4 + d) : 0.f;
        }
        float Mb = M;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) Mb = fmaxf(Mb, mv[i]);
        if (Mb == -INFINITY) continue;   // nothing valid so far
        if (M != -INFINITY && Mb != M) {
            const float c = exp2f(M - Mb);
            l *= c;
            acc *= c;
        }
        M = Mb;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const float w = mv[i] == -INFINITY ? 0.f : exp2f(mv[i] - M);
            l = fmaf(w, lv[i], l);
            acc = fmaf(w, xv[i], acc);
        }
    }
    if (ng > 1) {
        // the groups' states, rescaled to their common max (every thread of a group holds the same
        // M and l)
        gacc[grp][d] = acc;
        if (d == 0) {
            gml[grp][0] = M;
            gml[grp][1] = l;
        }
        __syncthreads();
        if (grp == 0) {
            float Mt = -INFINITY;
            for (int g = 0; g < ng; ++g) Mt = fmaxf(Mt, gml[g][0]);
            l = 0.f;
            acc = 0.f;
            if (Mt != -INFINITY) {
                for (int g = 0; g < ng; ++g) {
                    const float mg = gml[g][0];
                    const float w = mg == -INFINITY ? 0.f : exp2f(mg - Mt);
                    l = fmaf(w, gml[g][1], l);
                    acc = fmaf(w, gacc[g][d], acc);
                }
            }
        }
    }
    const float o = (l > 0.f || l != l) ? acc / l : 0.f;   // a NaN l (failed copy) propagates
    if (!rotate_back) {
        if (grp == 0) out[(int64_t)blockIdx.x * kD + d] = o;
        return;
    }
    // inverse rotation by group 0; every thread passes the same barriers
    if (grp == 0) buf[d] = o;
    __syncthreads();
#pragma unroll
    for (int L = 1; L < kD; L <<= 1) {
        float v = 0.f, w = 0.f;
        if (grp == 0) {
            v = buf[d];
            w = buf[d ^ L];
        }
        __syncthreads();
        if (grp == 0) buf[d] = (d & L) ? (w - v) : (v + w);
        __syncthreads();
    }
    if (grp == 0) {
        const uint32_t sw[4] = {s0, s1, s2, s3};
        const float v = buf[d] * 0.08838834764831845f;
        out[(int64_t)blockIdx.x * kD + d] = ((sw[d >> 5] >> (d & 31)) & 1u) ? -v : v;
    }
}

static int attn_smem_bytes(int kb, int vb) {
    const int head = (1040 * 2 + 8 * kD + kTT * 8 + 8 * 4 + 32) * 4;
    const int kbb = 2 + 16 * kb, vbb = vb == 16 ? 256 : 2 + 16 * vb;
    const int stage = ((kTT * kbb + 15) & ~15) + ((kTT * vbb + 15) & ~15) + kTT * 16 + kTT * 2;
    return head + 2 * stage;
}

}  // namespace tq

using namespace tq;

namespace tq {

int launch_attn_mma_paged_k2(const AttnArgs &a, MmaPlan &plan, int vb, int nt, cudaStream_t st);
int launch_attn_mma_paged_k3(const AttnArgs &a, MmaPlan &plan, int vb, int nt, cudaStream_t st);
int launch_attn_mma_paged_k4(const AttnArgs &a, MmaPlan &plan, int vb, int nt, cudaStream_t st);

namespace {

// The tensor-core decode path: query prep -> attention (contiguous or paged cache) -> combine,
// chained as programmatic dependents.
int mma_path(AttnArgs &a, int kb, int vb, bool qjl, bool packed_v, tq_signs signs, float *out, bool paged,
             cudaStream_t st) {
    MmaPlan mp = mma_plan(a.B, a.Hq, a.Hkv, a.T, kb, vb, qjl, a.G);
    attn_prep_mma_kernel<<<a.B * a.Hkv, kAttnThreads, 0, st>>>(a, mp, qjl ? 1 : 0);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
    int r;
    if (paged) {
        const int nt = a.G <= 4 ? 1 : 2;
        r = kb == 2 ? launch_attn_mma_paged_k2(a, mp, vb, nt, st)
                    : kb == 3 ? launch_attn_mma_paged_k3(a, mp, vb, nt, st) : launch_attn_mma_paged_k4(a, mp, vb, nt, st);
    } else {
        r = launch_attn_mma(a, mp, kb, vb, qjl, st);
    }
    if (r != TQ_OK) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.B * a.Hq));
    cfg.blockDim = dim3(kAttnThreads * mma_combine_groups(mp));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn_combine_mma_kernel, (const float *)a.ws, mp, a.Hq, a.Hkv, packed_v ? 1 : 0,
                           signs.w[0], signs.w[1], signs.w[2], signs.w[3], out) != cudaSuccess)
        return TQ_ERR_CUDA;
    return launch_status();
}

}  // namespace
}  // namespace tq

extern "C" size_t tq_attn_workspace_bytes_sms(int B, int Hq, int Hkv, int T_cap, int sms) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || T_cap <= 0 || Hq % Hkv) return 0;
    int splits, tps;
    attn_split_plan(B, Hkv, T_cap, &splits, &tps);
    const int64_t split_floats = (int64_t)B * Hq * splits * kPartialFloats;
    const int64_t mma_floats = mma_workspace_floats(B, Hq, Hkv, T_cap, sms);
    return (size_t)(split_floats > mma_floats ? split_floats : mma_floats) * sizeof(float);
}

extern "C" size_t tq_attn_workspace_bytes(int B, int Hq, int Hkv, int T_cap) {
    return tq_attn_workspace_bytes_sms(B, Hq, Hkv, T_cap, 0);
}

extern "C" int tq_attn_decode(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                              const void *v, const tq_codebook *vcb, const int32_t *seq_lens, int B, int Hq,
                              int Hkv, int T_cap, int T, float scale, tq_signs signs, const uint8_t *qjl_bits,
                              const uint16_t *res_norm_f16, const float *S, float *out, void *workspace,
                              size_t workspace_bytes, void *stream) {
    if (kcb && (kcb->bits == 8 || (vcb && vcb->bits == 8))) {
        // turboq8 keys with 2/3/4-bit values, or 4-bit keys with turboq8 values (the fork's asymmetric
        // pairs): the split-K tensor-core path when a workspace of the usual size is given, else the
        // M = 1 case of the tensor-core causal attention, which needs none
        if (qjl_bits || res_norm_f16 || S || !vcb) return TQ_ERR_UNSUPPORTED;
        const bool pair = (kcb->bits == 8 && vcb->bits >= 2 && vcb->bits <= 4) || (kcb->bits == 4 && vcb->bits == 8);
        const bool ws_ok = workspace && aligned(workspace, 16) && B > 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0 &&
                           Hq / Hkv <= 8 && T_cap > 0 && workspace_bytes >= tq_attn_workspace_bytes(B, Hq, Hkv, T_cap);
        if (!pair || !ws_ok)
            return tq_attn_prefill(q, q_dtype, k_blocks, kcb, static_cast<const uint8_t *>(v), vcb, seq_lens, B, 1,
                                   Hq, Hkv, T_cap, T, scale, signs, out, stream);
    }
    if (!q || !k_blocks || !kcb || !v || !out || !workspace) return TQ_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T_cap <= 0 || T < 1 || T > T_cap || (T_cap & 7))
        return TQ_ERR_ARG;
    if (!std::isfinite(scale)) return TQ_ERR_ARG;
    const int G = Hq / Hkv;
    if (G > 8 || dtype_bytes(q_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    // (bits 8: the turboq8 pairs admitted above)
    if (kcb->head_dim != kD || ((kcb->bits < 2 || kcb->bits > 4) && kcb->bits != 8) ||
        kcb->levels != (1 << kcb->bits))
        return TQ_ERR_UNSUPPORTED;
    if (vcb && (vcb->head_dim != kD || ((vcb->bits < 2 || vcb->bits > 4) && vcb->bits != 8) ||
                vcb->levels != (1 << vcb->bits)))
        return TQ_ERR_UNSUPPORTED;
    const bool qjl = qjl_bits || res_norm_f16 || S;
    if (qjl && !(qjl_bits && res_norm_f16 && S)) return TQ_ERR_ARG;
    if (!aligned(q, dtype_bytes(q_dtype)) || !aligned(k_blocks, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(workspace, 16) || (qjl && (!aligned(qjl_bits, 16) || !aligned(res_norm_f16, 16) || !aligned(S, 4))))
        return TQ_ERR_ALIGN;
    if (workspace_bytes < tq_attn_workspace_bytes(B, Hq, Hkv, T_cap)) return TQ_ERR_WORKSPACE;

    AttnArgs a;
    a.drop = drop_copies();
    a.table = nullptr;
    a.max_pages = 0;
    a.page = 0;
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
    if (attn_mma_supported(kb, vb, qjl, G)) return mma_path(a, kb, vb, qjl, vcb != nullptr, signs, out, false, st);
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

extern "C" int tq_attn_decode_paged(const void *q, int q_dtype, const uint8_t *k_pool, const tq_codebook *kcb,
                                    const uint8_t *v_pool, const tq_codebook *vcb, const int32_t *block_table,
                                    int max_pages, int page_tokens, const int32_t *seq_lens, int B, int Hq, int Hkv,
                                    int T, float scale, tq_signs signs, float *out, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    if (!q || !k_pool || !kcb || !v_pool || !vcb || !out || !block_table) return TQ_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T < 1 || max_pages <= 0 || page_tokens <= 0 ||
        (page_tokens & 7) || (int64_t)max_pages * page_tokens < T)
        return TQ_ERR_ARG;
    const int G = Hq / Hkv, kb = kcb->bits, vb = vcb->bits;
    const int T8 = (T + 7) & ~7;
    // the split-K tensor-core decode kernel: packed 2/3/4-bit keys and values, pages of a multiple
    // of 32 tokens (a 32-token chunk never straddles two pages), a workspace
    if (workspace && (page_tokens & 31) == 0 && codebook_ok(kcb) && codebook_ok(vcb) &&
        attn_mma_supported(kb, vb, false, G)) {
        if (!std::isfinite(scale)) return TQ_ERR_ARG;
        if (dtype_bytes(q_dtype) == 0) return TQ_ERR_UNSUPPORTED;
        if (!aligned(q, dtype_bytes(q_dtype)) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
            !aligned(workspace, 16))
            return TQ_ERR_ALIGN;
        if (workspace_bytes < tq_attn_workspace_bytes(B, Hq, Hkv, T8)) return TQ_ERR_WORKSPACE;
        AttnArgs a;
        a.drop = drop_copies();
        a.q = q;
        a.q_dtype = q_dtype;
        a.k = k_pool;
        a.v = v_pool;
        a.seq_lens = seq_lens;
        a.qjl_bits = nullptr;
        a.rn = nullptr;
        a.S = nullptr;
        a.ws = static_cast<float *>(workspace);
        a.B = B;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.G = G;
        a.T_cap = T8;
        a.T = T;
        attn_split_plan(B, Hkv, T, &a.splits, &a.tiles_per_split);
        a.qscale = scale * 1.4426950408889634f;
        for (int i = 0; i < 16; ++i) {
            a.kc[i] = kcb->centroids[i];
            a.vc[i] = vcb->centroids[i];
        }
        for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
        a.table = block_table;
        a.max_pages = max_pages;
        a.page = page_tokens;
        return mma_path(a, kb, vb, false, true, signs, out, true, static_cast<cudaStream_t>(stream));
    }
    // otherwise the one-token case of the tensor-core causal attention (no workspace)
    return tq_attn_prefill_paged(q, q_dtype, k_pool, kcb, v_pool, vcb, block_table, max_pages, page_tokens, seq_lens,
                                 B, 1, Hq, Hkv, T, scale, signs, out, stream);
}
