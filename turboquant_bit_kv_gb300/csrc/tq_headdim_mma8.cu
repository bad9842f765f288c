// Decode attention at head dims 64 .. 160 on the tensor cores: the
// instantiations of attn_dm_kernel (tq_headdim_mma.cuh) for five to eight
// query heads per KV head (one n-tile of the heads, the hi and lo parts of
// the query and of P as separate products), in a unit of their own so that
// the two sets compile in parallel.

#include "tq_headdim_mma.cuh"

namespace tq {

HmKernel hm_select_g8(int d, int kb, int vb) {
    HM_SELECT(true)
    return HmKernel{nullptr, 0, nullptr, nullptr};
}

}  // namespace tq
