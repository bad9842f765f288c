// Work partition of the tensor-core decode-attention kernel (shared by the
// launcher, the combine kernel and the workspace size query).
#pragma once

#include <stdint.h>

#include "tq_attn.cuh"

namespace tq {

constexpr int kMmaChunk = 32;        // tokens per chunk
constexpr int64_t kMmaCtas = 304;    // CTAs of the partition (2 per SM on 152 SMs)

// Chunks are ordered by (sequence, KV head, position); CTA i covers
// [i * Ctot / P, (i + 1) * Ctot / P).  Smax bounds the number of CTAs that
// touch one (sequence, KV head) segment, i.e. the partial slots per head.
struct MmaPlan {
    int C;          // chunks per segment, ceil(T / kMmaChunk)
    int64_t Ctot;   // B * Hkv * C
    int P;          // CTAs
    int Smax;       // partial slots per (sequence, query head)
};

MmaPlan mma_plan(int B, int Hkv, int T);
bool attn_mma_supported(int kb, int vb, bool qjl);
int launch_attn_mma(const AttnArgs &a, const MmaPlan &plan, cudaStream_t st);

// CTA that owns chunk x: the largest i with floor(i * Ctot / P) <= x.
__host__ __device__ inline int64_t mma_cta_of_chunk(int64_t x, const MmaPlan &p) {
    return ((x + 1) * p.P - 1) / p.Ctot;
}

}  // namespace tq
