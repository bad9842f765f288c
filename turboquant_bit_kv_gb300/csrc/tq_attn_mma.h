// Work partition of the tensor-core decode-attention kernels (shared by the
// launcher, the query-prep and combine kernels and the workspace size query).
#pragma once

#include <stdint.h>

#include "tq_attn.cuh"

namespace tq {

constexpr int kMmaChunk = 32;        // tokens per chunk
constexpr int kMmaMaxWarpsPerSm = 16;   // no configuration runs more warps per SM
constexpr int kMmaMaxWorkersPerSeg = 31;   // workers <= 31 x segments: at most 32 partial slots,
constexpr int kMmaMaxChunksCapped = 5;     // as long as that leaves each worker 5 chunks or fewer
// Query fragments per (sequence, KV head) segment, in 32-bit words: three
// parts (n-tiles 0 and 1 of the rotated query, the sketched query) x 32
// lanes x 16 words.
constexpr int kFragWords = 3 * 32 * 16;

// Chunks are ordered by (sequence, KV head, position); worker w (warp
// w / P of CTA w % P, so that small grids spread over every CTA) covers
// chunks [w * Ctot / W, (w + 1) * Ctot / W), W <= Ctot (never empty).  Smax
// bounds the number of workers that touch one (sequence, KV head) segment,
// i.e. the partial slots per query head.  Workspace: partials
// [B][Hq][Smax][132] floats | query fragments [B * Hkv][kFragWords] words.
struct MmaPlan {
    int C;              // chunks per segment, ceil(T / kMmaChunk)
    int64_t Ctot;       // B * Hkv * C
    int P;              // CTAs (all resident), at most W
    int W;              // workers: min(Ctot, P x warps per CTA, and on small problems the cap below)
    int Smax;           // partial slots per (sequence, query head)
    int64_t frag_off;   // float offset of the query fragments in the workspace
    int wide;           // 2-bit values, one n-tile: 16 warps per SM (else 12)
    int warps;          // warps per CTA of the configuration
};

// kb / vb: key / value bits (vb = 16: raw fp16 values); qjl: two-term
// score; G: query heads per KV head.  Workers are capped at
// kMmaMaxWorkersPerSeg per segment while that leaves each worker at most
// kMmaMaxChunksCapped chunks.  mma_plan_for takes the SM count explicitly
// (mma_plan uses the current device's).
MmaPlan mma_plan_for(int sms, int B, int Hq, int Hkv, int T, int kb, int vb, bool qjl, int G);
MmaPlan mma_plan(int B, int Hq, int Hkv, int T, int kb, int vb, bool qjl, int G);
// Workspace floats the tensor-core path needs for any T <= T_cap on a GPU of
// `sms` SMs (sms <= 0: the current device's).
int64_t mma_workspace_floats(int B, int Hq, int Hkv, int T_cap, int sms);
bool attn_mma_supported(int kb, int vb, bool qjl, int G);
int launch_attn_mma(const AttnArgs &a, MmaPlan &plan, int kb, int vb, bool qjl, cudaStream_t st);

// Worker that owns chunk x: the largest w with floor(w * Ctot / W) <= x.
__host__ __device__ inline int64_t mma_worker_of_chunk(int64_t x, const MmaPlan &p) {
    return ((x + 1) * p.W - 1) / p.Ctot;
}

// Slot groups of 128 threads in a combine CTA: one per 32 slots of Smax, at most kCombineMaxGroups.
inline int mma_combine_groups(const MmaPlan &p) {
    const int g = (p.Smax + 31) / 32;
    return g < 1 ? 1 : (g > kCombineMaxGroups ? kCombineMaxGroups : g);
}

}  // namespace tq
