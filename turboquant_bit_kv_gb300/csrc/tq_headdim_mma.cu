// Decode attention at head dims 64 .. 160 on the tensor cores: the
// instantiations for up to four query heads per KV head, and the plan and
// launch of the kernel (attn_dm_kernel, tq_headdim_mma.cuh) for every head
// count it covers.

#include "tq_headdim_mma.cuh"

namespace tq {

HmKernel hm_select_g4(int d, int kb, int vb) {
    HM_SELECT(false)
    return HmKernel{nullptr, 0, nullptr, nullptr};
}

static HmKernel hm_select(const HdAttnArgs &a, int d) {
    if (a.G <= 4) return hm_select_g4(d, a.kbits, a.vbits);
    if (a.G <= 8) return hm_select_g8(d, a.kbits, a.vbits);
    return HmKernel{nullptr, 0, nullptr, nullptr};
}

int hd_attn_mma_plan(HdAttnArgs &a, int d) {
    const HmKernel k = hm_select(a, d);
    if (!k.fn) return 1;
    if (set_smem_limit(k.fn, k.smem, k.done) != TQ_OK) return TQ_ERR_CUDA;
    if (*k.resident <= 0 &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(k.resident, k.fn, kHmThreads, k.smem) != cudaSuccess)
        return TQ_ERR_CUDA;
    hd_split_plan(a.B, a.Hkv, a.T, sm_count() * (*k.resident > 0 ? *k.resident : 1), kHmWarps, &a.splits, &a.tps);
    return TQ_OK;
}

int hd_attn_mma_launch(const HdAttnArgs &a, int d, cudaStream_t st) {
    const HmKernel k = hm_select(a, d);
    if (!k.fn) return TQ_ERR_UNSUPPORTED;
    const int smem = k.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kHmThreads);
    cfg.gridDim = dim3(a.splits, a.Hkv, a.B);
    cfg.dynamicSmemBytes = smem;
    void *args[] = {const_cast<HdAttnArgs *>(&a)};
    if (cudaLaunchKernelExC(&cfg, k.fn, args) != cudaSuccess) return TQ_ERR_CUDA;
    return TQ_OK;
}

}  // namespace tq
