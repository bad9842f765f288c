// Work partition of the tensor-core decode-attention kernel (shared by the
// launcher, the combine kernel and the workspace size query).
#pragma once

#include <stdint.h>

#include "tq_attn.cuh"

namespace tq {

constexpr int kMmaChunk = 32;        // tokens per chunk

// Chunks are ordered by (sequence, KV head, position); CTA i covers
// [i * Ctot / P, (i + 1) * Ctot / P).  Smax bounds the number of CTAs that
// touch one (sequence, KV head) segment, i.e. the partial slots per head.
struct MmaPlan {
    int C;          // chunks per segment, ceil(T / kMmaChunk)
    int64_t Ctot;   // B * Hkv * C
    int P;          // CTAs (all resident: CTAs per SM of the configuration x SMs, at most Ctot)
    int Smax;       // partial slots per (sequence, query head)
};

// kb / vb: key / value bits (vb = 16: raw fp16 values); qjl: two-term
// score; G: query heads per KV head.
MmaPlan mma_plan(int B, int Hkv, int T, int kb, int vb, bool qjl, int G);
int mma_max_slots(int B, int Hkv, int T_cap);   // Smax bound over every configuration
bool attn_mma_supported(int kb, int vb, bool qjl, int G);
int launch_attn_mma(const AttnArgs &a, MmaPlan &plan, int kb, int vb, bool qjl, cudaStream_t st);

// CTA that owns chunk x: the largest i with floor(i * Ctot / P) <= x.
__host__ __device__ inline int64_t mma_cta_of_chunk(int64_t x, const MmaPlan &p) {
    return ((x + 1) * p.P - 1) / p.Ctot;
}

}  // namespace tq
