// QJL residual sketch of bf16 / fp16 keys on the 5th-generation tensor cores
// (sm_103a): "RotorQuant KV Cache Compression", The QJL Estimator Formula
// and Implementation Requirements 1-2 (residual r = k - k_mse after the MSE
// stage, fp16 ||r||, sign bits of S r with a Gaussian S, m = 128).
//
// The residual is formed in the rotated domain.  With R = H D / sqrt(128)
// (orthogonal) and k_mse = n16 R^T c[code] (the dequantiser of "TurboQuant
// KV Cache Compression — Spec", Quantize / Dequantize):
//   R r   = R k - n16 c[code] = u / sqrt(128) - n16 c[code],   u = H D k,
//   ||r|| = ||R r||,
//   S r   = S' (R r)  with  S' = S R^T = S D H / sqrt(128).
// So per tile of 128 keys two dense contractions do all the arithmetic:
//   U = X (H D)^T        (bf16 / fp16 keys times +-1: exact products)
//   P = (R r) S'^T       (fp16 hi / lo splits of R r and S': float32-grade)
// and the per-element work in between is one centroid lookup and one FMA.
//
// One CTA per SM (the operands take ~205 KB of shared memory): a producer
// warp issues the TMA loads of key tiles and all MMAs; eight epilogue warps
// (two per 32-row group of tensor-memory lanes, one 64-column half each)
// read U, form R r from the staged blocks, write its hi / lo fp16 tiles for
// the second product, add the two halves' sums of squares in a fixed order
// for ||r||, then read P and pack its signs.  R r is scaled by a power of two
// chosen from the block norm before the fp16 split (signs and, after
// undoing the scale, the norm are unchanged; the scale only keeps the split
// inside fp16's normal range).  Every mbarrier wait is bounded.

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {
namespace {

constexpr int kQRows = 128;                          // keys per tile = MMA M = tensor-memory lanes
constexpr int kQEpiWarps = 8;
constexpr int kQThreads = 32 * (kQEpiWarps + 1);     // + one producer warp
constexpr int kQTile = kQRows * 256;                 // one 128 x 128 16-bit operand tile
constexpr uint32_t kQCols = 512;                     // U (two stages) at 0 / 128, P at 256
constexpr unsigned kQFull = 0xffffffffu;

struct QjlTcArgs {
    const uint8_t *blocks;
    int64_t block_stride;   // bytes
    int64_t n_vec;
    const float *S;         // [128][128] row-major
    uint8_t *bits;          // [n_vec][16]
    uint16_t *rn;           // [n_vec]
    float c[16];            // centroids
    uint32_t signs[4];
};

template <int BITS>
struct QjlSmem {
    static constexpr int BB = 2 + 16 * BITS;
    static constexpr int kHW = BB / 2;                          // 16-bit words per block
    static constexpr int kPitch = BB + 2;                       // staged row: 2 pad bytes, norm, codes (4-aligned)
    static constexpr int kPre = (32 * kHW + 63) / 64;           // block words a thread prefetches per tile
    static constexpr int kHD = 0;                               // H D (key dtype)
    static constexpr int kSh = kHD + kQTile;                    // S' hi (fp16)
    static constexpr int kSl = kSh + kQTile;                    // S' lo (fp16)
    static constexpr int kX = kSl + kQTile;                     // key tile (TMA)
    static constexpr int kA2 = kX + kQTile;                     // R r hi tile, then lo tile
    static constexpr int kBlk = kA2 + 2 * kQTile;               // the tile's blocks
    static constexpr int kCtab = kBlk + ((kQRows * kPitch + 15) & ~15);   // centroids, lane-replicated
    static constexpr int kPart = kCtab + 16 * 32 * 4;           // per-row partial sums of squares [2][128]
    static constexpr int kBars = kPart + 2 * kQRows * 4;        // 8 mbarriers
    static constexpr int kSlot = kBars + 8 * 8;                 // tensor-memory base address
    static constexpr int kTotal = kSlot + 16 + 1024;            // + alignment slack of the base
};

// mbarriers: key tile landed, key tile consumed, U ready [2], U released [2], R r staged, P ready
enum { kBarFull = 0, kBarXFree = 1, kBarURdy = 2, kBarUFree = 4, kBarA2 = 6, kBarP = 7 };

__device__ __forceinline__ void sts128_q(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// fp16 (hi, lo) split of a pair: x = hi + lo to about 2^-22 of x.
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 f = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_h2(x0 - f.x, x1 - f.y);
}

// Code of element e (0..63) of one half of a block row, from that half's
// code words (4-bit: 8 words; 2-bit: 4 words; 3-bit: 4 low-plane words,
// then 2 high-plane words).
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int e) {
    if constexpr (BITS == 4) {
        return (w[e >> 3] >> (4 * (e & 7))) & 15u;
    } else if constexpr (BITS == 2) {
        return (w[e >> 4] >> (2 * (e & 15))) & 3u;
    } else {
        return ((w[e >> 4] >> (2 * (e & 15))) & 3u) | (((w[4 + (e >> 5)] >> (e & 31)) & 1u) << 2);
    }
}

template <int BITS, int DT>
__global__ void __launch_bounds__(kQThreads, 1)
    qjl_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ QjlTcArgs a) {
    using Q = QjlSmem<BITS>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // 1024-byte aligned base: the 128-byte swizzle is a function of address bits 4..9
    const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_s - raw_s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = base_s + Q::kBars;

    // ---- setup: H D, S' (hi / lo), centroid table, barriers, tensor memory
    for (int q = threadIdx.x; q < kQRows * 16; q += kQThreads) {
        const int n = q >> 4, kc = q & 15;   // row n of H D, 8-column chunk kc
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t pair = 0;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int k = 8 * kc + 2 * j + e;
                const uint32_t neg = ((uint32_t)__popc(n & k) & 1u) ^ ((a.signs[k >> 5] >> (k & 31)) & 1u);
                const uint32_t one = DT == TQ_BF16 ? (neg ? 0xBF80u : 0x3F80u) : (neg ? 0xBC00u : 0x3C00u);
                pair |= one << (16 * e);
            }
            w[j] = pair;
        }
        const int off = Q::kHD + (kc >> 3) * 16384 + n * 128 + (((kc & 7) ^ (n & 7)) << 4);
        *reinterpret_cast<uint4 *>(smem + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    // row j of S' = H (D S_j) / sqrt(128): lane holds elements 4 lane .. 4 lane + 3
    for (int j = warp; j < 128; j += kQThreads / 32) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int l = 4 * lane + k;
            const float s = a.S[j * 128 + l];
            v[k] = ((a.signs[l >> 5] >> (l & 31)) & 1u) ? -s : s;
        }
        const float x0 = v[0] + v[1], x1 = v[0] - v[1], x2 = v[2] + v[3], x3 = v[2] - v[3];
        v[0] = x0 + x2;
        v[2] = x0 - x2;
        v[1] = x1 + x3;
        v[3] = x1 - x3;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float o = __shfl_xor_sync(kQFull, v[k], m);
                v[k] = (lane & m) ? (o - v[k]) : (v[k] + o);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] *= 0.08838834764831845f;
        uint32_t h0, l0, h1, l1;
        split_pair(v[0], v[1], h0, l0);
        split_pair(v[2], v[3], h1, l1);
        const int kc = lane >> 1;   // 8-element chunk of elements 4 lane .. + 3
        const int off = (kc >> 3) * 16384 + j * 128 + (((kc & 7) ^ (j & 7)) << 4) + (lane & 1) * 8;
        *reinterpret_cast<uint2 *>(smem + Q::kSh + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2 *>(smem + Q::kSl + off) = make_uint2(l0, l1);
    }
    float *ctab = reinterpret_cast<float *>(smem + Q::kCtab);
    for (int q = threadIdx.x; q < 16 * 32; q += kQThreads) ctab[q] = a.c[q >> 5];
    if (threadIdx.x == 0) {
        tc_mbar_init(bars + 8 * kBarFull, 1);
        tc_mbar_init(bars + 8 * kBarXFree, 1);
        tc_mbar_init(bars + 8 * kBarURdy, 1);
        tc_mbar_init(bars + 8 * (kBarURdy + 1), 1);
        tc_mbar_init(bars + 8 * kBarUFree, kQEpiWarps);
        tc_mbar_init(bars + 8 * (kBarUFree + 1), kQEpiWarps);
        tc_mbar_init(bars + 8 * kBarA2, kQEpiWarps);
        tc_mbar_init(bars + 8 * kBarP, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base_s + Q::kSlot),
                     "r"(kQCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // H D and S' were written by ordinary stores and are read by the tensor cores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + Q::kSlot);
    const int64_t ntiles = (a.n_vec + kQRows - 1) / kQRows;

    if (warp == kQEpiWarps) {
        // ---- producer: key tiles by TMA, U = X (H D)^T, and after each tile's R r is staged
        // P = Rr_hi S'_hi^T + Rr_hi S'_lo^T + Rr_lo S'_hi^T.  The next tile's load and U are
        // issued around P so that U is ready when the epilogue reaches that tile.
        if (lane == 0) {
            const uint32_t hd_s = base_s + Q::kHD, x_s = base_s + Q::kX, a2_s = base_s + Q::kA2;
            const uint32_t sh_s = base_s + Q::kSh, sl_s = base_s + Q::kSl;
            auto load_x = [&](int64_t tile) {
                tc_mbar_expect_tx(bars + 8 * kBarFull, kQTile);
                tc_tma_load_2d(x_s, &tmap, 0, (int)(tile * kQRows), bars + 8 * kBarFull);
                tc_tma_load_2d(x_s + 16384, &tmap, 64, (int)(tile * kQRows), bars + 8 * kBarFull);
            };
            // a wait that gives up marks the CTA's work failed and is skipped from then on: the
            // loops still run to the end (no thread is left waiting at a barrier)
            bool ok = true;
            auto wait = [&](int b, uint32_t parity) {
                if (ok) ok = tc_mbar_wait(bars + 8 * b, parity);
            };
            int64_t tile = blockIdx.x;
            if (tile < ntiles) {
                load_x(tile);
                wait(kBarFull, 0u);
                tc_fence_after();
                tc_mma_tile<DT>(tmem, x_s, hd_s, false);
                tc_commit(bars + 8 * kBarURdy);
                tc_commit(bars + 8 * kBarXFree);
            }
            for (int i = 0; tile < ntiles; ++i, tile += gridDim.x) {
                const int64_t next = tile + gridDim.x;
                if (next < ntiles) {
                    wait(kBarXFree, (uint32_t)i & 1u);   // U of tile i has read X
                    load_x(next);
                }
                wait(kBarA2, (uint32_t)i & 1u);          // R r of tile i staged
                tc_fence_after();
                const uint32_t p_t = tmem + 256u;
                tc_mma_tile<TQ_F16>(p_t, a2_s, sh_s, false);
                tc_mma_tile<TQ_F16>(p_t, a2_s, sl_s, true);
                tc_mma_tile<TQ_F16>(p_t, a2_s + kQTile, sh_s, true);
                tc_commit(bars + 8 * kBarP);
                if (next < ntiles) {
                    const int n1 = i + 1, st = n1 & 1;
                    wait(kBarFull, (uint32_t)n1 & 1u);
                    if (n1 >= 2) wait(kBarUFree + st, (uint32_t)((n1 >> 1) - 1) & 1u);
                    tc_fence_after();
                    tc_mma_tile<DT>(tmem + (uint32_t)(st * 128), x_s, hd_s, false);
                    tc_commit(bars + 8 * (kBarURdy + st));
                    tc_commit(bars + 8 * kBarXFree);
                }
            }
        }
    } else {
        // ---- epilogue: warp w owns tensor-memory lanes (= tile rows) 32 (w & 3) .. + 31 and columns
        // 64 hf .. + 63 (hf = w >> 2); the two warps of a row group meet on named barrier 1 + (w & 3)
        const int grp = warp & 3, hf = warp >> 2;
        const int r = 32 * grp + lane, tid64 = 32 * hf + lane;
        const uint32_t pair_bar = 1u + (uint32_t)grp;
        float *part = reinterpret_cast<float *>(smem + Q::kPart);
        uint8_t *blk = smem + Q::kBlk;
        const uint32_t ctab_s = base_s + Q::kCtab + 4u * lane;
        const uint32_t a2_row = base_s + Q::kA2 + hf * 16384 + r * 128;
        // the row group's 32 blocks, as 16-bit words, loaded one tile ahead
        uint32_t pre[Q::kPre];
        auto prefetch = [&](int64_t tile) {
            const int64_t v0 = tile * kQRows + 32 * grp;
#pragma unroll
            for (int k = 0; k < Q::kPre; ++k) {
                const int q = tid64 + 64 * k, row = q / Q::kHW, h = q - row * Q::kHW;
                pre[k] = (q < 32 * Q::kHW && tile < ntiles && v0 + row < a.n_vec)
                             ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(
                                   a.blocks + (v0 + row) * a.block_stride + 2 * h))
                             : 0u;
            }
        };
        auto stage = [&]() {
#pragma unroll
            for (int k = 0; k < Q::kPre; ++k) {
                const int q = tid64 + 64 * k, row = q / Q::kHW, h = q - row * Q::kHW;
                if (q < 32 * Q::kHW)
                    *reinterpret_cast<uint16_t *>(blk + (32 * grp + row) * Q::kPitch + 2 + 2 * h) = (uint16_t)pre[k];
            }
        };
        prefetch(blockIdx.x);
        bool ok = true;   // as in the producer: a wait that gave up is not repeated, the loop runs on
        auto wait = [&](int b, uint32_t parity) {
            if (ok) ok = tc_mbar_wait(bars + 8 * b, parity);
        };
        int i = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
            const int st = i & 1;
            const int64_t v0 = tile * kQRows;
            const int nv = (int)min64(kQRows, a.n_vec - v0);
            stage();
            prefetch(tile + gridDim.x);
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");   // the group's blocks are staged

            // ---- U of this row half
            wait(kBarURdy + st, (uint32_t)(i >> 1) & 1u);
            tc_fence_after();
            float x[2][32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * grp) << 16) + (uint32_t)(st * 128 + 64 * hf);
            tc_ld32(taddr, x[0]);
            tc_ld32(taddr + 32, x[1]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bars + 8 * (kBarUFree + st));

            // ---- R r = u / sqrt(128) - n16 c[code], scaled by 2^(7 - E) with n16 in [2^(E-1), 2^E)
            const uint8_t *rb = blk + r * Q::kPitch;
            const float nf = r < nv ? __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(rb + 2))) : 0.f;
            float scale = 1.f;   // inf / NaN norms: left unscaled
            if (nf == 0.f) {
                scale = 1073741824.f;   // 2^30
            } else if (nf < 65536.f) {
                const int E = (int)((__float_as_uint(nf) >> 23) & 0xFF) - 126;
                scale = __uint_as_float((uint32_t)(127 + 7 - E) << 23);
            }
            const float inv_rs = 0.08838834764831845f * scale, nn = -(nf * scale);
            uint32_t cw[BITS == 4 ? 8 : BITS == 3 ? 6 : 4];
            if constexpr (BITS == 4) {
#pragma unroll
                for (int q = 0; q < 8; ++q) cw[q] = *reinterpret_cast<const uint32_t *>(rb + 4 + 32 * hf + 4 * q);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) cw[q] = *reinterpret_cast<const uint32_t *>(rb + 4 + 16 * hf + 4 * q);
                if constexpr (BITS == 3) {
                    cw[4] = *reinterpret_cast<const uint32_t *>(rb + 36 + 8 * hf);
                    cw[5] = *reinterpret_cast<const uint32_t *>(rb + 40 + 8 * hf);
                }
            }
            float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float c0 = lds_f32(ctab_s + code_at<BITS>(cw, e) * 128u);
                const float c1 = lds_f32(ctab_s + code_at<BITS>(cw, e + 1) * 128u);
                const float2 u2 = __fmul2_rn(make_float2(x[e >> 5][e & 31], x[e >> 5][(e & 31) + 1]),
                                             make_float2(inv_rs, inv_rs));
                const float2 r2 = __ffma2_rn(make_float2(c0, c1), make_float2(nn, nn), u2);
                x[e >> 5][e & 31] = r2.x;
                x[e >> 5][(e & 31) + 1] = r2.y;
                q2 = __ffma2_rn(r2, r2, q2);
            }
            part[hf * kQRows + r] = q2.x + q2.y;
            // fp16 hi / lo tiles of R r (K-major, 128-byte swizzle), then hand them to the tensor cores
#pragma unroll
            for (int kc = 0; kc < 8; ++kc) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int e = 8 * kc + 2 * p;
                    split_pair(x[e >> 5][e & 31], x[e >> 5][(e & 31) + 1], h[p], l[p]);
                }
                const uint32_t addr = a2_row + (uint32_t)(((kc ^ (r & 7)) << 4));
                sts128_q(addr, h[0], h[1], h[2], h[3]);
                sts128_q(addr + kQTile, l[0], l[1], l[2], l[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bars + 8 * kBarA2);
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");   // both halves' sums of squares
            const float ss = part[r] + part[kQRows + r];
            const unsigned short rn16 = __half_as_ushort(__float2half_rn(sqrtf(ss) * (1.f / scale)));

            // ---- signs of P = S r for this row half: bit j of the row's 128 = [(S r)_j >= 0]
            wait(kBarP, (uint32_t)i & 1u);
            tc_fence_after();
            const uint32_t paddr = tmem + ((uint32_t)(32 * grp) << 16) + (uint32_t)(256 + 64 * hf);
            tc_ld32(paddr, x[0]);
            tc_ld32(paddr + 32, x[1]);
            tc_wait_ld();
            tc_fence_before();
            uint32_t wb[2] = {0u, 0u};
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int k = 0; k < 32; ++k) wb[c] |= (x[c][k] >= 0.f ? 1u : 0u) << k;
            if (r < nv) {
                *reinterpret_cast<uint2 *>(a.bits + (v0 + r) * 16 + 8 * hf) = make_uint2(wb[0], wb[1]);
                if (hf == 0) a.rn[v0 + r] = rn16;
            }
        }
    }

    // ---- teardown: every MMA was waited for and every tensor-memory load completed
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kQCols) : "memory");
}

template <int BITS, int DT>
int launch_qjl_tc(const CUtensorMap &map, const QjlTcArgs &a, cudaStream_t st) {
    static int done[64] = {0};
    if (set_smem_limit((const void *)qjl_tc_kernel<BITS, DT>, QjlSmem<BITS>::kTotal, done) != TQ_OK)
        return TQ_ERR_CUDA;
    const int64_t ntiles = (a.n_vec + kQRows - 1) / kQRows;
    const int grid = (int)std::min<int64_t>(ntiles, (int64_t)sm_count());
    qjl_tc_kernel<BITS, DT><<<grid, kQThreads, QjlSmem<BITS>::kTotal, st>>>(map, a);
    return launch_status();
}

}  // namespace

int qjl_encode_tc(const void *k, int k_dtype, int64_t n_vec, int64_t k_stride_bytes, const uint8_t *blocks,
                  int64_t block_stride, int bits, const float *centroids, const uint32_t *signs, const float *S,
                  uint8_t *qjl_bits, uint16_t *res_norm_f16, cudaStream_t st) {
    if (k_dtype != TQ_BF16 && k_dtype != TQ_F16) return 1;
    CUtensorMap map;
    if (!make_row_tile_map(&map, k, k_dtype, n_vec, k_stride_bytes)) return 1;
    QjlTcArgs a;
    a.blocks = blocks;
    a.block_stride = block_stride;
    a.n_vec = n_vec;
    a.S = S;
    a.bits = qjl_bits;
    a.rn = res_norm_f16;
    for (int i = 0; i < 16; ++i) a.c[i] = centroids[i];
    for (int i = 0; i < 4; ++i) a.signs[i] = signs[i];
    const bool bf = k_dtype == TQ_BF16;
    switch (bits) {
        case 2: return bf ? launch_qjl_tc<2, TQ_BF16>(map, a, st) : launch_qjl_tc<2, TQ_F16>(map, a, st);
        case 3: return bf ? launch_qjl_tc<3, TQ_BF16>(map, a, st) : launch_qjl_tc<3, TQ_F16>(map, a, st);
        case 4: return bf ? launch_qjl_tc<4, TQ_BF16>(map, a, st) : launch_qjl_tc<4, TQ_F16>(map, a, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
