// Tensor-core decode attention, 3-bit keys: instantiations of the kernel
// template in tq_attn_mma.cuh for every value format (2/3/4-bit codes, raw
// fp16), and the QJL two-term score with 2-bit or raw values.
#include "tq_attn_mma.cuh"

namespace tq {

void mma_shape_k3(int vb, bool qjl, int nt, bool wide, int *ctas_per_sm, int *warps) {
    *ctas_per_sm = *warps = 0;
#define TQ_CASE(V, Q, N) \
    if (vb == V && qjl == Q && nt == N) return shape_of<3, V, Q, N>(wide, ctas_per_sm, warps);
    TQ_CASE(2, false, 1) TQ_CASE(3, false, 1) TQ_CASE(4, false, 1) TQ_CASE(16, false, 1)
    TQ_CASE(2, false, 2) TQ_CASE(3, false, 2) TQ_CASE(4, false, 2) TQ_CASE(16, false, 2)
    TQ_CASE(2, true, 1) TQ_CASE(16, true, 1)
#undef TQ_CASE
}

int launch_attn_mma_k3(const AttnArgs &a, MmaPlan &plan, int vb, bool qjl, int nt, cudaStream_t st) {
#define TQ_CASE(V, Q, N) \
    if (vb == V && qjl == Q && nt == N) return launch_cfg<3, V, Q, N>(a, plan, st);
    TQ_CASE(2, false, 1) TQ_CASE(3, false, 1) TQ_CASE(4, false, 1) TQ_CASE(16, false, 1)
    TQ_CASE(2, false, 2) TQ_CASE(3, false, 2) TQ_CASE(4, false, 2) TQ_CASE(16, false, 2)
    TQ_CASE(2, true, 1) TQ_CASE(16, true, 1)
#undef TQ_CASE
    return TQ_ERR_UNSUPPORTED;
}

// Paged caches (packed keys and values, no QJL term).
int launch_attn_mma_paged_k3(const AttnArgs &a, MmaPlan &plan, int vb, int nt, cudaStream_t st) {
#define TQ_CASE(V, N) \
    if (vb == V && nt == N) return launch_cfg<3, V, false, N, true>(a, plan, st);
    TQ_CASE(2, 1) TQ_CASE(3, 1) TQ_CASE(4, 1) TQ_CASE(2, 2) TQ_CASE(3, 2) TQ_CASE(4, 2)
#undef TQ_CASE
    return TQ_ERR_UNSUPPORTED;
}

int wait_failed_attn_k3(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

}  // namespace tq
