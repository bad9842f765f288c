// Tensor-core decode attention: work partition and dispatch over key widths
// (the kernel template is in tq_attn_mma.cuh, instantiated in
// tq_attn_mma_k{2,3,4}.cu).
#include "tq_attn_mma.h"
#include "tq_internal.h"

namespace tq {

// CTAs per SM and warps per CTA of a configuration (0 CTAs: not covered).
void mma_shape_k2(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps);
void mma_shape_k3(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps);
void mma_shape_k4(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps);
void mma_shape_k8(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps);
int launch_attn_mma_k2(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);
int launch_attn_mma_k3(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);
int launch_attn_mma_k4(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);
int launch_attn_mma_k8(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);

// n-tiles of 4 query heads (times hi / lo parts) for G query heads per KV head
static int mma_ntiles(int G) { return G <= 4 ? 1 : 2; }

static void mma_shape(int kb, int vb, bool qjl, int G, bool wide, int *ctas_per_sm, int *warps) {
    *ctas_per_sm = 0;
    *warps = 0;
    if (G < 1 || G > 8) return;
    const int nt = mma_ntiles(G);
    switch (kb) {
        case 2: mma_shape_k2(vb, qjl, nt, wide, ctas_per_sm, warps); break;
        case 3: mma_shape_k3(vb, qjl, nt, wide, ctas_per_sm, warps); break;
        case 4: mma_shape_k4(vb, qjl, nt, wide, ctas_per_sm, warps); break;
        case 8: mma_shape_k8(vb, qjl, nt, wide, ctas_per_sm, warps); break;
        default: break;
    }
}

// Partial slots per query head: no segment of C chunks meets more than
// ceil(W / segments) + 1 worker ranges (the ranges differ in length by at
// most one chunk), nor more workers than it has chunks.
static int mma_slots(int64_t segs, int64_t C, int64_t W) {
    const int64_t s = (W + segs - 1) / segs + 1;
    return (int)(s < C ? s : C);
}

MmaPlan mma_plan(int B, int Hq, int Hkv, int T, int kb, int vb, bool qjl, int G) {
    return mma_plan_for(sm_count(), B, Hq, Hkv, T, kb, vb, qjl, G);
}

MmaPlan mma_plan_for(int sms, int B, int Hq, int Hkv, int T, int kb, int vb, bool qjl, int G) {
    MmaPlan p;
    const int64_t segs = (int64_t)B * Hkv;
    p.C = (T + kMmaChunk - 1) / kMmaChunk;
    p.Ctot = segs * p.C;
    // the 16-warp variant once every warp would get at least 32 chunks, else 12 warps per SM
    p.wide = p.Ctot >= (int64_t)32 * kMmaMaxWarpsPerSm * sms ? 1 : 0;
    int per_sm = 0, warps = 0;
    mma_shape(kb, vb, qjl, G, p.wide != 0, &per_sm, &warps);
    p.warps = warps;
    p.P = (int)min64(p.Ctot, (int64_t)(per_sm > 0 ? per_sm : 1) * sms);
    // at most one worker per chunk (every range non-empty), and on small problems no more than
    // kMmaMaxWorkersPerSeg workers per segment on average, so that a segment has at most 32
    // partials and the combine merges them in one round of loads (each further round costs ~2 us
    // of L2 latency) -- unless that would give workers more than kMmaMaxChunksCapped chunks each
    // (long ranges at low occupancy cost more than the rounds they save)
    const int64_t capped = max64(segs * kMmaMaxWorkersPerSeg, (p.Ctot + kMmaMaxChunksCapped - 1) / kMmaMaxChunksCapped);
    p.W = (int)min64(min64(p.Ctot, capped), (int64_t)p.P * (warps > 0 ? warps : 1));
    if (p.P > p.W) p.P = p.W;   // no CTA without a worker
    p.Smax = mma_slots(segs, p.C, p.W);
    p.frag_off = (int64_t)B * Hq * p.Smax * kPartialFloats;
    return p;
}

int64_t mma_workspace_floats(int B, int Hq, int Hkv, int T_cap, int sms) {
    const int64_t segs = (int64_t)B * Hkv;
    const int64_t C = (T_cap + kMmaChunk - 1) / kMmaChunk;
    const int smax = mma_slots(segs, C, (int64_t)kMmaMaxWarpsPerSm * (sms > 0 ? sms : sm_count()));
    return (int64_t)B * Hq * smax * kPartialFloats + segs * kFragWords;
}

bool attn_mma_supported(int kb, int vb, bool qjl, int G) {
    int per_sm = 0, warps = 0;
    mma_shape(kb, vb, qjl, G, true, &per_sm, &warps);
    return per_sm > 0;
}

int launch_attn_mma(const AttnArgs &a, MmaPlan &plan, int kb, int vb, bool qjl, cudaStream_t st) {
    const int nt = mma_ntiles(a.G);
    switch (kb) {
        case 2: return launch_attn_mma_k2(a, plan, vb, qjl, nt, st);
        case 3: return launch_attn_mma_k3(a, plan, vb, qjl, nt, st);
        case 4: return launch_attn_mma_k4(a, plan, vb, qjl, nt, st);
        case 8: return launch_attn_mma_k8(a, plan, vb, qjl, nt, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
