// Tensor-core decode attention: work partition and dispatch over key widths
// (the kernel template is in tq_attn_mma.cuh, instantiated in
// tq_attn_mma_k{2,3,4}.cu).
#include "tq_attn_mma.h"
#include "tq_internal.h"

namespace tq {

int mma_ctas_per_sm_k2(int vb, bool qjl, int nt);
int mma_ctas_per_sm_k3(int vb, bool qjl, int nt);
int mma_ctas_per_sm_k4(int vb, bool qjl, int nt);
int launch_attn_mma_k2(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);
int launch_attn_mma_k3(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);
int launch_attn_mma_k4(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st);

// n-tiles of 4 query heads (times hi / lo parts) for G query heads per KV head
static int mma_ntiles(int G) { return G <= 4 ? 1 : 2; }

// CTAs per SM of a configuration (its shared memory and registers decide: 1
// or 2); 0 when the tensor-core kernel does not cover it.
static int mma_ctas_per_sm(int kb, int vb, bool qjl, int G) {
    if (G < 1 || G > 8) return 0;
    const int nt = mma_ntiles(G);
    switch (kb) {
        case 2: return mma_ctas_per_sm_k2(vb, qjl, nt);
        case 3: return mma_ctas_per_sm_k3(vb, qjl, nt);
        case 4: return mma_ctas_per_sm_k4(vb, qjl, nt);
        default: return 0;
    }
}

MmaPlan mma_plan(int B, int Hkv, int T, int kb, int vb, bool qjl, int G) {
    MmaPlan p;
    p.C = (T + kMmaChunk - 1) / kMmaChunk;
    p.Ctot = (int64_t)B * Hkv * p.C;
    const int per_sm = mma_ctas_per_sm(kb, vb, qjl, G);
    p.P = (int)min64(p.Ctot, (int64_t)(per_sm > 0 ? per_sm : 1) * sm_count());
    const int64_t segs = (int64_t)B * Hkv;
    p.Smax = (int)((p.P + segs - 1) / segs) + 1;
    return p;
}

int mma_max_slots(int B, int Hkv, int T_cap) {
    // no configuration runs more than two CTAs per SM
    const int64_t segs = (int64_t)B * Hkv;
    const int64_t P = min64(segs * ((T_cap + kMmaChunk - 1) / kMmaChunk), 2 * (int64_t)sm_count());
    return (int)((P + segs - 1) / segs) + 1;
}

bool attn_mma_supported(int kb, int vb, bool qjl, int G) { return mma_ctas_per_sm(kb, vb, qjl, G) > 0; }

int launch_attn_mma(const AttnArgs &a, MmaPlan &plan, int kb, int vb, bool qjl, cudaStream_t st) {
    const int nt = mma_ntiles(a.G);
    switch (kb) {
        case 2: return launch_attn_mma_k2(a, plan, vb, qjl, nt, st);
        case 3: return launch_attn_mma_k3(a, plan, vb, qjl, nt, st);
        case 4: return launch_attn_mma_k4(a, plan, vb, qjl, nt, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
