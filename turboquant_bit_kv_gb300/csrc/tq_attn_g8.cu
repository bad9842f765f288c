// Split-pass instantiations of the decode-attention kernel for up to 8
// query heads per KV head (kept in their own translation unit so the
// instantiations compile in parallel).
#include "tq_attn.cuh"
#include "tq_internal.h"

namespace tq {

template <int KB, int VB>
static int launch_one(const AttnArgs &a, dim3 grid, int smem, cudaStream_t st) {
    static int done[64] = {0};
    if (set_smem_limit((const void *)attn_split_kernel<8, KB, VB>, smem, done) != TQ_OK) return TQ_ERR_CUDA;
    attn_split_kernel<8, KB, VB><<<grid, kAttnThreads, smem, st>>>(a);
    return launch_status();
}

int launch_attn_split_g8(int kb, int vb, const AttnArgs &a, dim3 grid, int smem, cudaStream_t st) {
    switch (kb * 32 + vb) {
        case 2 * 32 + 2: return launch_one<2, 2>(a, grid, smem, st);
        case 2 * 32 + 3: return launch_one<2, 3>(a, grid, smem, st);
        case 2 * 32 + 4: return launch_one<2, 4>(a, grid, smem, st);
        case 2 * 32 + 16: return launch_one<2, 16>(a, grid, smem, st);
        case 3 * 32 + 2: return launch_one<3, 2>(a, grid, smem, st);
        case 3 * 32 + 3: return launch_one<3, 3>(a, grid, smem, st);
        case 3 * 32 + 4: return launch_one<3, 4>(a, grid, smem, st);
        case 3 * 32 + 16: return launch_one<3, 16>(a, grid, smem, st);
        case 4 * 32 + 2: return launch_one<4, 2>(a, grid, smem, st);
        case 4 * 32 + 3: return launch_one<4, 3>(a, grid, smem, st);
        case 4 * 32 + 4: return launch_one<4, 4>(a, grid, smem, st);
        case 4 * 32 + 16: return launch_one<4, 16>(a, grid, smem, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
