// Fused decode attention over a packed TurboQuant cache (sm_103a).
//
// Restates "TurboQuant KV Cache Compression — Spec", Optimization: Fused
// dequant-dot (rotate the query once; score against centroid x norm in the
// rotated domain with no per-key inverse rotation; accumulate values in the
// rotated domain; one inverse rotation per output), and, for the two-term
// key score, "RotorQuant KV Cache Compression", Fused Kernel Logic
// (term2 = rn * sqrt(pi/2)/m * <S q, sign>, score = (term1 + term2) * scale).
//
// Split pass: one CTA per (context split, KV head, sequence); its G query
// heads share every staged K/V tile (grouped-query head sharing).  K/V tiles
// of 64 tokens are staged into shared memory with 16-byte cp.async copies,
// double buffered.  Scores are kept in the log2 domain (scale * log2(e)
// folded into the rotated query) and an online softmax runs per tile; each
// split writes (m, l, acc[128]) for each query head.  The combine pass merges
// the splits of one (sequence, query head) and applies the inverse rotation.
#pragma once

#include "tq_device.cuh"

namespace tq {

constexpr int kAttnThreads = 128;
constexpr int kCombineMaxGroups = 4;   // slot groups of 128 threads in one combine CTA
constexpr int kTT = 64;                  // tokens per staged tile
constexpr int kPartialFloats = 132;      // m, l, pad, pad, acc[128]
constexpr int kTargetCtas = 1216;        // split-count target (8 x 152 SMs)

struct AttnArgs {
    const void *q;
    int q_dtype;
    const uint8_t *k;        // [B][Hkv][T_cap] K blocks
    const uint8_t *v;        // [B][Hkv][T_cap] V blocks, or raw fp16 rows
    const int32_t *seq_lens;
    const uint8_t *qjl_bits; // [B][Hkv][T_cap][16]
    const uint16_t *rn;      // [B][Hkv][T_cap]
    const float *S;          // [128][128]
    float *ws;               // [B][Hq][splits][132]
    int B, Hq, Hkv, G, T_cap, T, splits, tiles_per_split;
    float qscale;            // scale * log2(e)
    float kc[16], vc[16];
    uint32_t signs[4];
    int drop;                // test hook: issue no bulk copies (the waits for them run out)
    // paged cache (the paged kernels only): token t of sequence b is slot t % page of page
    // table[b * max_pages + t / page] of pools [pages][Hkv][page]; page a multiple of 32
    const int32_t *table;
    int max_pages, page;
};

__host__ __device__ inline int attn_tiles(int T) { return (T + kTT - 1) / kTT; }

// Split count of a shape; device independent so workspace sizes are stable.
__host__ inline void attn_split_plan(int B, int Hkv, int T, int *splits, int *tiles_per_split) {
    int tiles = attn_tiles(T);
    int bh = B * Hkv;
    int s = (kTargetCtas + bh - 1) / bh;
    if (s > tiles) s = tiles;
    if (s < 1) s = 1;
    int tps = (tiles + s - 1) / s;
    *tiles_per_split = tps;
    *splits = (tiles + tps - 1) / tps;
}

// q-row element d of dtype dt.
__device__ __forceinline__ float load_q(const void *q, int dt, int64_t idx) {
    if (dt == TQ_F32) return reinterpret_cast<const float *>(q)[idx];
    if (dt == TQ_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(q)[idx]);
    return __half2float(reinterpret_cast<const __half *>(q)[idx]);
}

// Index of (dim d, head g) in the [128][8] query tables; the upper 64 dims are
// shifted by 4 floats so the two halves of a warp hit different banks.
__device__ __forceinline__ int qidx(int d, int g) { return d * 8 + g + ((d >> 6) << 2); }

// In-place unnormalised Walsh-Hadamard transform of GP rows of 128 floats in
// shared memory by 128 threads (thread d owns element d of every row).
template <int GP>
__device__ __forceinline__ void smem_fwht_rows(float *buf /* [GP][128] */) {
    const int d = threadIdx.x;
#pragma unroll
    for (int L = 1; L < kD; L <<= 1) {
        float v[GP], w[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            v[g] = buf[g * kD + d];
            w[g] = buf[g * kD + (d ^ L)];
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < GP; ++g) buf[g * kD + d] = (d & L) ? (w[g] - v[g]) : (v[g] + w[g]);
        __syncthreads();
    }
}

template <int KB, int VB>
struct AttnTile {
    static constexpr int kKB = 2 + 16 * KB;
    static constexpr int kVB = VB == 16 ? 256 : 2 + 16 * VB;
    static constexpr int kKBytes = (kTT * kKB + 15) & ~15;
    static constexpr int kVBytes = (kTT * kVB + 15) & ~15;
    static constexpr int kBits = kTT * 16;
    static constexpr int kRn = kTT * 2;
    static constexpr int kStage = kKBytes + kVBytes + kBits + kRn;
};

// Copy [t0, t0 + n) of one (b, kv head) stream of `per` bytes per token into
// shared memory; the region starts 16-byte aligned (t0 and T_cap multiples of
// 8) and may be read up to the next multiple of 16 bytes (inside T_cap).
__device__ __forceinline__ void stage_bytes(uint8_t *dst, const uint8_t *src, int nbytes) {
    const int nch = (nbytes + 15) >> 4;
    for (int c = threadIdx.x; c < nch; c += kAttnThreads) cp_async16(dst + 16 * c, src + 16 * c);
}

template <int GP, int KB, int VB>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(AttnArgs a) {
    using Tile = AttnTile<KB, VB>;
    constexpr int KBB = Tile::kKB, VBB = Tile::kVB;
    extern __shared__ __align__(16) uint8_t smem[];
    float *qr = reinterpret_cast<float *>(smem);          // [128][8] (+4 pad) rotated, scaled queries
    float *sq = qr + 1040;                                // [128][8] (+4 pad) sketched queries (QJL)
    float *buf = sq + 1040;                               // [8][128] scratch for the query transform
    float *sc = buf + 8 * kD;                             // [64][8] scores -> weights
    float *mrow = sc + kTT * 8;                           // [8] running max (log2 domain)
    float *lrow = mrow + 8;                               // [8] running sum
    float *crow = lrow + 8;                               // [8] rescale of this tile
    float *tot = crow + 8;                                // [8] sum_j sq_j (QJL)
    float *lutk = tot + 8;                                // [16]
    float *lutv = lutk + 16;                              // [16]
    uint8_t *stages = reinterpret_cast<uint8_t *>(lutv + 16);

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const bool qjl = a.qjl_bits != nullptr;
    int L = a.T;
    if (a.seq_lens) {
        int sl = a.seq_lens[b];
        L = sl < 0 ? 0 : (sl > a.T ? a.T : sl);
    }
    const int t_begin = split * a.tiles_per_split * kTT;
    const int t_end = min(L, (split + 1) * a.tiles_per_split * kTT);

    if (tid < 16) {
        lutk[tid] = a.kc[tid];
        lutv[tid] = a.vc[tid];
    }
    if (tid < 8) {
        mrow[tid] = -INFINITY;
        lrow[tid] = 0.f;
        tot[tid] = 0.f;
    }
    // ---- query prep: R q = H (D q) / sqrt(128), scaled by scale*log2(e)
    {
        const int d = tid;
        const uint32_t sbit = (a.signs[d >> 5] >> (d & 31)) & 1u;
        for (int g = 0; g < GP; ++g) {
            float v = 0.f;
            if (g < a.G) v = load_q(a.q, a.q_dtype, ((int64_t)b * a.Hq + kvh * a.G + g) * kD + d);
            buf[g * kD + d] = sbit ? -v : v;
        }
        __syncthreads();
        if (qjl) {
            // (S q)_d for each head, from the unrotated query (undo the sign).
            float accs[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) accs[g] = 0.f;
            for (int j = 0; j < kD; ++j) {
                const float s = a.S[d * kD + j];
                const float sj = ((a.signs[j >> 5] >> (j & 31)) & 1u) ? -1.f : 1.f;
#pragma unroll
                for (int g = 0; g < GP; ++g) accs[g] = fmaf(s, sj * buf[g * kD + j], accs[g]);
            }
            const float c2 = 1.2533141373155003f / 128.f * a.qscale;  // sqrt(pi/2)/m
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                sq[qidx(d, g)] = accs[g] * c2;
                float r = accs[g] * c2;
                for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
                if ((tid & 31) == 0) atomicAdd(&tot[g], r);
            }
        }
        __syncthreads();
        smem_fwht_rows<GP>(buf);
        const float f = a.qscale * 0.08838834764831845f;
#pragma unroll
        for (int g = 0; g < GP; ++g) qr[qidx(d, g)] = buf[g * kD + d] * f;
    }

    const int64_t bh = (int64_t)b * a.Hkv + kvh;
    const uint8_t *kbase = a.k + bh * a.T_cap * KBB;
    const uint8_t *vbase = a.v + bh * a.T_cap * VBB;
    const uint8_t *bbase = qjl ? a.qjl_bits + bh * a.T_cap * 16 : nullptr;
    const uint8_t *rbase = qjl ? reinterpret_cast<const uint8_t *>(a.rn + bh * a.T_cap) : nullptr;

    auto issue = [&](int stage, int t0) {
        uint8_t *st = stages + stage * Tile::kStage;
        const int n = min(kTT, t_end - t0);
        stage_bytes(st, kbase + (int64_t)t0 * KBB, n * KBB);
        stage_bytes(st + Tile::kKBytes, vbase + (int64_t)t0 * VBB, n * VBB);
        if (qjl) {
            stage_bytes(st + Tile::kKBytes + Tile::kVBytes, bbase + (int64_t)t0 * 16, n * 16);
            stage_bytes(st + Tile::kKBytes + Tile::kVBytes + Tile::kBits, rbase + (int64_t)t0 * 2, n * 2);
        }
    };

    float acc[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) acc[g] = 0.f;

    if (t_begin < t_end) issue(0, t_begin);
    cp_async_commit();
    int it = 0;
    for (int t0 = t_begin; t0 < t_end; t0 += kTT, ++it) {
        if (t0 + kTT < t_end) issue((it + 1) & 1, t0 + kTT);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint8_t *st = stages + (it & 1) * Tile::kStage;
        const uint8_t *kt = st, *vt = st + Tile::kKBytes;
        const uint8_t *bt = st + Tile::kKBytes + Tile::kVBytes;
        const uint16_t *rt = reinterpret_cast<const uint16_t *>(bt + Tile::kBits);
        const int nvalid = min(kTT, t_end - t0);

        // ---- scores: thread = (token, half of the dims)
        {
            const int tt = tid >> 1, h = tid & 1;
            float s[GP], s2[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                s[g] = 0.f;
                s2[g] = 0.f;
            }
            const uint8_t *blk = kt + tt * KBB;
            const float *qb = qr + qidx(64 * h, 0);
            if constexpr (KB == 4) {
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const uint32_t word = lds_u32_a2(blk + 2 + 32 * h + 4 * w);
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float c = lutk[(word >> (4 * m)) & 15u];
                        const float *qd = qb + (8 * w + m) * 8;
#pragma unroll
                        for (int g = 0; g < GP; ++g) s[g] = fmaf(c, qd[g], s[g]);
                    }
                }
            } else if constexpr (KB == 2) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t word = lds_u32_a2(blk + 2 + 16 * h + 4 * w);
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const float c = lutk[(word >> (2 * m)) & 3u];
                        const float *qd = qb + (16 * w + m) * 8;
#pragma unroll
                        for (int g = 0; g < GP; ++g) s[g] = fmaf(c, qd[g], s[g]);
                    }
                }
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t lo = lds_u32_a2(blk + 2 + 16 * h + 4 * w);
                    const uint32_t hiw = lds_u32_a2(blk + 34 + 8 * h + 4 * (w >> 1));
                    const uint32_t hi = hiw >> (16 * (w & 1));
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const uint32_t code = ((lo >> (2 * m)) & 3u) | (((hi >> m) & 1u) << 2);
                        const float c = lutk[code];
                        const float *qd = qb + (16 * w + m) * 8;
#pragma unroll
                        for (int g = 0; g < GP; ++g) s[g] = fmaf(c, qd[g], s[g]);
                    }
                }
            }
            if (qjl) {
                const uint32_t *bw = reinterpret_cast<const uint32_t *>(bt + tt * 16 + 8 * h);
                const float *sb = sq + qidx(64 * h, 0);
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const uint32_t word = bw[w];
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const float bit = (float)((word >> m) & 1u);
                        const float *qd = sb + (32 * w + m) * 8;
#pragma unroll
                        for (int g = 0; g < GP; ++g) s2[g] = fmaf(bit, qd[g], s2[g]);
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                s[g] += __shfl_xor_sync(0xffffffffu, s[g], 1);
                s2[g] += __shfl_xor_sync(0xffffffffu, s2[g], 1);
            }
            if (h == 0) {
                const float nk = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(blk)));
                const float rn = qjl ? __half2float(__ushort_as_half(rt[tt])) : 0.f;
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    float v = nk * s[g];
                    if (qjl) v = fmaf(rn, 2.f * s2[g] - tot[g], v);
                    sc[tt * 8 + g] = (tt < nvalid) ? v : -INFINITY;
                }
            }
        }
        __syncthreads();
        // ---- online softmax per head (warp w handles heads w, w + 4)
        {
            const int warp = tid >> 5, lane = tid & 31;
            for (int g = warp; g < GP; g += 4) {
                float s0 = sc[lane * 8 + g], s1 = sc[(lane + 32) * 8 + g];
                float mx = fmaxf(s0, s1);
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mold = mrow[g];
                const float mnew = fmaxf(mold, mx);
                float p0 = 0.f, p1 = 0.f, corr = 1.f;
                if (mnew != -INFINITY) {
                    p0 = exp2f(s0 - mnew);
                    p1 = exp2f(s1 - mnew);
                    corr = exp2f(mold - mnew);
                }
                float sum = p0 + p1;
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                float nv0 = 1.f, nv1 = 1.f;
                if constexpr (VB != 16) {
                    nv0 = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(vt + lane * VBB)));
                    nv1 = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(vt + (lane + 32) * VBB)));
                }
                sc[lane * 8 + g] = lane < nvalid ? p0 * nv0 : 0.f;
                sc[(lane + 32) * 8 + g] = lane + 32 < nvalid ? p1 * nv1 : 0.f;
                if (lane == 0) {
                    mrow[g] = mnew;
                    lrow[g] = lrow[g] * corr + sum;
                    crow[g] = corr;
                }
            }
        }
        __syncthreads();
        // ---- P V in the rotated domain: thread = dim
        {
            const int d = tid;
#pragma unroll
            for (int g = 0; g < GP; ++g) acc[g] *= crow[g];
            for (int tt = 0; tt < nvalid; ++tt) {
                float v;
                if constexpr (VB == 16) {
                    v = __half2float(reinterpret_cast<const __half *>(vt + tt * VBB)[d]);
                } else if constexpr (VB == 4) {
                    v = lutv[(vt[tt * VBB + 2 + (d >> 1)] >> (4 * (d & 1))) & 15u];
                } else if constexpr (VB == 2) {
                    v = lutv[(vt[tt * VBB + 2 + (d >> 2)] >> (2 * (d & 3))) & 3u];
                } else {
                    const uint32_t lo = (vt[tt * VBB + 2 + (d >> 2)] >> (2 * (d & 3))) & 3u;
                    const uint32_t hi = (vt[tt * VBB + 34 + (d >> 3)] >> (d & 7)) & 1u;
                    v = lutv[lo | (hi << 2)];
                }
                const float *pw = sc + tt * 8;
#pragma unroll
                for (int g = 0; g < GP; ++g) acc[g] = fmaf(pw[g], v, acc[g]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    // ---- partials
    for (int g = 0; g < a.G; ++g) {
        float *pr = a.ws + (((int64_t)b * a.Hq + kvh * a.G + g) * a.splits + split) * kPartialFloats;
        float accg = 0.f;
#pragma unroll
        for (int gg = 0; gg < GP; ++gg)
            if (gg == g) accg = acc[gg];
        pr[4 + tid] = accg;
        if (tid == 0) {
            pr[0] = mrow[g];
            pr[1] = lrow[g];
        }
    }
}

}  // namespace tq
