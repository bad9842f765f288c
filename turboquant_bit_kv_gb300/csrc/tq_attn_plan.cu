// tq_attn_plan: the work partition tq_attn_decode's tensor-core path uses
// for a shape (split-K over the context of "TurboQuant KV Cache Compression
// — Spec", Optimization: Fused dequant-dot), for tests and tuning; and
// tq_attn_plan_d, the context splits of tq_attn_decode_d for a given count
// of resident CTAs.  Host only: they compute the plan and touch no device
// memory.

#include "tq.h"
#include "tq_attn_mma.h"
#include "tq_headdim.cuh"
#include "tq_internal.h"

using namespace tq;

extern "C" int tq_attn_plan(int B, int Hq, int Hkv, int T, int key_bits, int value_bits, int qjl, int sms,
                            int64_t *out) {
    if (!out || B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || Hq % Hkv) return TQ_ERR_ARG;
    if (key_bits < 2 || key_bits > 4 || (value_bits != 16 && (value_bits < 2 || value_bits > 4)))
        return TQ_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    if (!attn_mma_supported(key_bits, value_bits, qjl != 0, G)) return TQ_ERR_UNSUPPORTED;
    const MmaPlan p = mma_plan_for(sms > 0 ? sms : sm_count(), B, Hq, Hkv, T, key_bits, value_bits, qjl != 0, G);
    out[0] = p.C;
    out[1] = p.Ctot;
    out[2] = p.P;
    out[3] = p.W;
    out[4] = p.Smax;
    out[5] = mma_combine_groups(p);
    out[6] = p.warps;
    return TQ_OK;
}

extern "C" int tq_attn_plan_d(int B, int Hkv, int T, int ctas_resident, int warps_per_cta, int32_t *out) {
    if (!out || B <= 0 || Hkv <= 0 || T <= 0 || ctas_resident <= 0 || warps_per_cta <= 0) return TQ_ERR_ARG;
    int splits = 0, tps = 0;
    hd_split_plan(B, Hkv, T, ctas_resident, warps_per_cta, &splits, &tps);
    out[0] = splits;
    out[1] = tps;
    out[2] = hd_max_splits(T);
    return TQ_OK;
}
