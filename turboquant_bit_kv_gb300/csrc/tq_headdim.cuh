// Declarations shared by the head-dim decode attention units: tq_headdim.cu
// (query prep, combine, the C ABI) and tq_headdim_mma.cuh with its
// instantiation units tq_headdim_mma.cu / tq_headdim_mma8.cu (the
// tensor-core attention kernel).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int kHdThreads = 256;   // 8 warps per CTA (codec, prep and combine kernels)
constexpr int kHdWarps = kHdThreads / 32;

struct HdAttnArgs {
    const void *q;
    const uint8_t *k, *v;
    const int32_t *seq_lens;
    const float *R;
    float *ws;               // partials [B][Hq][splits][2 + d]: m (log2 units), l, acc[d]
    float *qrot;             // rotated, scaled queries [B][Hq][d] (after the partials)
    float *out;
    int q_dtype, B, Hq, Hkv, G, T_cap, T, kbits, vbits, splits, tps;
    float qscale;            // scale * log2(e)
    float kc[16], vc[16];
};

// Most context splits of T tokens, and the split plan for `slots` CTAs of `warps` warps resident
// at once.
int hd_max_splits(int T);
void hd_split_plan(int B, int Hkv, int T, int slots, int warps, int *splits, int *tps);

// The tensor-core attention kernel (tq_headdim_mma.cuh), up to 8 heads per KV head and 2-, 3- or
// 4-bit keys and values: hd_attn_mma_plan returns 1 when it does not cover the call, else sets
// a.splits / a.tps from the kernel's occupancy and returns a TQ_ status; hd_attn_mma_launch
// enqueues it as a programmatic dependent of the kernel before it.
int hd_attn_mma_plan(HdAttnArgs &a, int d);
int hd_attn_mma_launch(const HdAttnArgs &a, int d, cudaStream_t st);

}  // namespace tq
