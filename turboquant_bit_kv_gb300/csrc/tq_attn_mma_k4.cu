// Tensor-core decode attention, 4-bit keys: instantiations of the kernel
// template in tq_attn_mma.cuh for every value format (2/3/4-bit codes,
// turboq8, raw fp16).
#include "tq_attn_mma.cuh"

namespace tq {

void mma_shape_k4(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps) {
    *ctas_per_sm = *warps = 0;
#define TQ_CASE(V, Q, N) \
    if (vb == V && qjl == Q && nt == N) return shape_of<4, V, Q, N>(wide, ctas_per_sm, warps);
    TQ_CASE(2, false, 1) TQ_CASE(3, false, 1) TQ_CASE(4, false, 1) TQ_CASE(16, false, 1)
    TQ_CASE(2, false, 2) TQ_CASE(3, false, 2) TQ_CASE(4, false, 2) TQ_CASE(16, false, 2)
    TQ_CASE(8, false, 1) TQ_CASE(8, false, 2)

#undef TQ_CASE
}

int launch_attn_mma_k4(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st) {
#define TQ_CASE(V, Q, N) \
    if (vb == V && qjl == Q && nt == N) return launch_cfg<4, V, Q, N>(a, plan, st);
    TQ_CASE(2, false, 1) TQ_CASE(3, false, 1) TQ_CASE(4, false, 1) TQ_CASE(16, false, 1)
    TQ_CASE(2, false, 2) TQ_CASE(3, false, 2) TQ_CASE(4, false, 2) TQ_CASE(16, false, 2)
    TQ_CASE(8, false, 1) TQ_CASE(8, false, 2)

#undef TQ_CASE
    return TQ_ERR_UNSUPPORTED;
}

// Paged caches (packed keys and values, no QJL term).
int launch_attn_mma_paged_k4(const AttnArgs &a, MmaPlan &plan, int vb, int nt, cudaStream_t st) {
#define TQ_CASE(V, N) \
    if (vb == V && nt == N) return launch_cfg<4, V, false, N, true>(a, plan, st);
    TQ_CASE(2, 1) TQ_CASE(3, 1) TQ_CASE(4, 1) TQ_CASE(2, 2) TQ_CASE(3, 2) TQ_CASE(4, 2)
#undef TQ_CASE
    return TQ_ERR_UNSUPPORTED;
}

int wait_failed_attn_k4(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

}  // namespace tq
