// Tensor-core decode attention, turboq8 keys ("TurboQuant KV Cache (turboq2 /
// turboq3 / turboq4)", At a glance and the turboq8 paragraph; section 2,
// Asymmetric K/V): instantiations of the kernel template in tq_attn_mma.cuh
// for 2/3/4-bit values.
#include "tq_attn_mma.cuh"

namespace tq {

void mma_shape_k8(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps) {
    *ctas_per_sm = *warps = 0;
#define TQ_CASE(V, N) \
    if (vb == V && !qjl && nt == N) return shape_of<8, V, false, N>(wide, ctas_per_sm, warps);
    TQ_CASE(2, 1) TQ_CASE(3, 1) TQ_CASE(4, 1) TQ_CASE(2, 2) TQ_CASE(3, 2) TQ_CASE(4, 2)
#undef TQ_CASE
}

int launch_attn_mma_k8(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st) {
#define TQ_CASE(V, N) \
    if (vb == V && !qjl && nt == N) return launch_cfg<8, V, false, N>(a, plan, st);
    TQ_CASE(2, 1) TQ_CASE(3, 1) TQ_CASE(4, 1) TQ_CASE(2, 2) TQ_CASE(3, 2) TQ_CASE(4, 2)
#undef TQ_CASE
    return TQ_ERR_UNSUPPORTED;
}

int wait_failed_attn_k8(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

}  // namespace tq
