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
// One CTA per SM (the operands take ~219 KB of shared memory): a producer
// warp issues the TMA loads of key tiles and all MMAs; sixteen epilogue warps
// (four per 32-row group of tensor-memory lanes, one 32-column slice each)
// read U, form R r from the staged blocks, write its hi / lo fp16 tiles for
// the second product, add the slices' sums of squares in a fixed order for
// ||r||, then read P and pack its signs.  R r is scaled by a power of two
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
constexpr int kQEpiWarps = 16;                       // four per 32-row group of lanes
constexpr int kQSlices = kQEpiWarps / 4;             // column slices of a row
constexpr int kQNC = 128 / kQSlices;                 // columns (elements) per epilogue thread
constexpr int kQThreads = 32 * (kQEpiWarps + 1);     // + one producer warp
constexpr int kQTile = kQRows * 256;                 // one 128 x 128 16-bit operand tile
constexpr uint32_t kQCols = 512;                     // U (two stages) at 0 / 128, P (two) at 256 / 384
constexpr unsigned kQFull = 0xffffffffu;

struct QjlTcArgs {
    const uint8_t *blocks;
    int64_t block_stride;   // bytes
    int dense;              // blocks back to back (stride = block bytes) from a 16-byte aligned start
    int64_t n_vec;
    const float *S;         // [128][128] row-major
    uint8_t *bits;          // [n_vec][16]
    uint16_t *rn;           // [n_vec]
    float c[16];            // centroids
    uint32_t signs[4];
    int drop;               // test hook: issue no TMA loads (the waits for them run out)
};

template <int BITS>
struct QjlSmem {
    static constexpr int BB = 2 + 16 * BITS;
    static constexpr int kHW = BB / 2;                          // 16-bit words per block
    static constexpr int kPitch = BB;                           // staged rows back to back, as in memory
    static constexpr int kPre = (32 * kHW + 32 * kQSlices - 1) / (32 * kQSlices);   // block words a thread prefetches
    static constexpr int kVec = 2 * BB;                         // 16-byte pieces of a row group's 32 blocks
    static constexpr int kPreV = (kVec + 32 * kQSlices - 1) / (32 * kQSlices);       // pieces a thread prefetches
    // centroid lookups: 2/3-bit codes by pairs (float2 of both centroids, 2^(2 BITS) entries), 4-bit
    // codes one at a time (16 floats); each entry replicated once per lane, so that lanes never
    // collide on a bank
    static constexpr bool kPairs = BITS < 4;
    static constexpr int kTabBytes = kPairs ? (1 << (2 * BITS)) * 256 : 16 * 32 * 4;
    static constexpr int kHD = 0;                               // H D (key dtype)
    static constexpr int kSh = kHD + kQTile;                    // S' hi (fp16)
    static constexpr int kSl = kSh + kQTile;                    // S' lo (fp16)
    static constexpr int kX = kSl + kQTile;                     // key tile (TMA)
    static constexpr int kA2 = kX + kQTile;                     // R r hi tile, then lo tile
    static constexpr int kBlk = kA2 + 2 * kQTile;               // the tile's blocks
    static constexpr int kCtab = kBlk + ((kQRows * kPitch + 16 + 15) & ~15);   // (+ slack read by the last row)
    static constexpr int kPart = kCtab + kTabBytes;             // per-row partial sums of squares [2][slice][128]
    static constexpr int kBars = kPart + 2 * kQSlices * kQRows * 4;   // 9 mbarriers
    static constexpr int kSlot = kBars + 9 * 8;                 // tensor-memory base address
    static constexpr int kTotal = kSlot + 16 + 1024;            // + alignment slack of the base
    static_assert(kTotal <= 232448, "shared memory of one CTA");
};

// mbarriers: key tile landed, key tile consumed, U ready [2], U released [2], R r staged, P ready,
// and the producer's last commit before teardown
enum { kBarFull = 0, kBarXFree = 1, kBarURdy = 2, kBarUFree = 4, kBarA2 = 6, kBarP = 7, kBarDrain = 8 };

__device__ __forceinline__ void sts128_q(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float2 lds_f2_q(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// N 32-bit words starting at byte offset off (even) of a shared buffer: aligned loads, and a funnel
// shift by 16 bits when off is 2 mod 4
template <int N>
__device__ __forceinline__ void words_at(const uint8_t *buf, int off, uint32_t *out) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(buf + (off & ~3));
    const uint32_t sh = (uint32_t)(off & 2) * 8u;
    uint32_t v[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) v[i] = w[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(v[i], v[i + 1], sh);
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

// Code of element e of a slice of a block row, from the slice's code words
// (4-bit: NC / 8 words; 2-bit: NC / 16 words; 3-bit: NC / 16 low-plane
// words, then NC / 32 high-plane words).
template <int BITS, int NC>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int e) {
    if constexpr (BITS == 4) {
        return (w[e >> 3] >> (4 * (e & 7))) & 15u;
    } else if constexpr (BITS == 2) {
        return (w[e >> 4] >> (2 * (e & 15))) & 3u;
    } else {
        return ((w[e >> 4] >> (2 * (e & 15))) & 3u) | (((w[NC / 16 + (e >> 5)] >> (e & 31)) & 1u) << 2);
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
    if constexpr (Q::kPairs) {
        // entry p (256 bytes: 32 copies): the centroids of codes (p_lo, p_hi) of two consecutive
        // elements; 3-bit: p = (low-plane bits of both) | (high-plane bits of both) << 4
        float2 *ptab = reinterpret_cast<float2 *>(smem + Q::kCtab);
        for (int q = threadIdx.x; q < (1 << (2 * BITS)) * 32; q += kQThreads) {
            const int p = q >> 5;
            int c0, c1;
            if constexpr (BITS == 2) {
                c0 = p & 3;
                c1 = p >> 2;
            } else {
                c0 = (p & 3) | ((p >> 2) & 4);
                c1 = ((p >> 2) & 3) | ((p >> 3) & 4);
            }
            ptab[q] = make_float2(a.c[c0], a.c[c1]);
        }
    } else {
        float *ctab = reinterpret_cast<float *>(smem + Q::kCtab);
        for (int q = threadIdx.x; q < 16 * 32; q += kQThreads) ctab[q] = a.c[q >> 5];
    }
    if (threadIdx.x == 0) {
        tc_mbar_init(bars + 8 * kBarFull, 1);
        tc_mbar_init(bars + 8 * kBarXFree, 1);
        tc_mbar_init(bars + 8 * kBarURdy, 1);
        tc_mbar_init(bars + 8 * (kBarURdy + 1), 1);
        tc_mbar_init(bars + 8 * kBarUFree, kQEpiWarps);
        tc_mbar_init(bars + 8 * (kBarUFree + 1), kQEpiWarps);
        tc_mbar_init(bars + 8 * kBarA2, kQEpiWarps);
        tc_mbar_init(bars + 8 * kBarP, 1);
        tc_mbar_init(bars + 8 * kBarDrain, 1);
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
            // the key-tile load of parity `pend_par` not yet seen complete (-1: none)
            int pend = -1;
            uint32_t pend_par = 0;
            auto load_x = [&](int64_t tile, uint32_t parity) {
                if (a.drop) return;   // (test hook: no load, so the wait for it runs out)
                tc_mbar_expect_tx(bars + 8 * kBarFull, kQTile);
                tc_tma_load_2d(x_s, &tmap, 0, (int)(tile * kQRows), bars + 8 * kBarFull);
                tc_tma_load_2d(x_s + 16384, &tmap, 64, (int)(tile * kQRows), bars + 8 * kBarFull);
                pend = 1;
                pend_par = parity;
            };
            // a wait that gives up is recorded and ends the producer's loop: no further load or
            // product is issued (the epilogue's waits then give up too, or are skipped)
            bool ok = true;
            auto wait = [&](int b, uint32_t parity) {
                if (ok && !tc_mbar_wait(bars + 8 * b, parity)) {
                    ok = false;
                    note_wait_failed();
                }
                if (ok && b == kBarFull) pend = -1;
            };
            int64_t tile = blockIdx.x;
            if (tile < ntiles) {
                load_x(tile, 0u);
                wait(kBarFull, 0u);
                if (ok) {
                    tc_fence_after();
                    tc_mma_tile<DT>(tmem, x_s, hd_s, false);
                    tc_commit(bars + 8 * kBarURdy);
                    tc_commit(bars + 8 * kBarXFree);
                }
            }
            for (int i = 0; ok && tile < ntiles; ++i, tile += gridDim.x) {
                const int64_t next = tile + gridDim.x;
                // U of the next tile is issued as soon as its keys have landed (while the epilogue
                // still forms R r of tile i), so that the epilogue finds it ready; P of tile i
                // follows and runs while the epilogue packs signs and starts the next tile
                if (next < ntiles) {
                    wait(kBarXFree, (uint32_t)i & 1u);   // U of tile i has read X
                    if (!ok) break;
                    const int n1 = i + 1, st = n1 & 1;
                    load_x(next, (uint32_t)n1 & 1u);
                    wait(kBarFull, (uint32_t)n1 & 1u);
                    if (n1 >= 2) wait(kBarUFree + st, (uint32_t)((n1 >> 1) - 1) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    tc_mma_tile<DT>(tmem + (uint32_t)(st * 128), x_s, hd_s, false);
                    tc_commit(bars + 8 * (kBarURdy + st));
                    tc_commit(bars + 8 * kBarXFree);
                }
                wait(kBarA2, (uint32_t)i & 1u);          // R r of tile i staged
                if (!ok) break;
                tc_fence_after();
                const uint32_t p_t = tmem + 256u + 128u * (uint32_t)(i & 1);   // P double-buffered
                tc_mma_tile<TQ_F16>(p_t, a2_s, sh_s, false);
                tc_mma_tile<TQ_F16>(p_t, a2_s, sl_s, true);
                tc_mma_tile<TQ_F16>(p_t, a2_s + kQTile, sh_s, true);
                tc_commit(bars + 8 * kBarP);
            }
            // before teardown: every product issued here has completed (one more commit, on a barrier
            // of its own), and a load whose wait gave up has landed (bounded waits)
            tc_commit(bars + 8 * kBarDrain);
            tc_mbar_wait(bars + 8 * kBarDrain, 0u);
            if (pend >= 0) tc_mbar_wait(bars + 8 * kBarFull, pend_par);
        }
    } else {
        // ---- epilogue: warp w owns tensor-memory lanes (= tile rows) 32 (w & 3) .. + 31 and columns
        // kQNC sl .. + kQNC - 1 (slice sl = w >> 2); a row group's warps meet on named barrier 1 + (w & 3)
        const int grp = warp & 3, sl = warp >> 2;
        const int r = 32 * grp + lane, tidg = 32 * sl + lane, c0 = kQNC * sl;
        const uint32_t grp_bar = 1u + (uint32_t)grp;
        float *part = reinterpret_cast<float *>(smem + Q::kPart);
        uint8_t *blk = smem + Q::kBlk;
        const uint32_t ctab_s = base_s + Q::kCtab + 4u * lane;
        const uint32_t a2_row = base_s + Q::kA2 + (c0 >> 6) * 16384 + r * 128;
        // the row group's 32 blocks, loaded one tile ahead: sixteen bytes at a time when the blocks are
        // back to back (a group of 32 starts 32 * BB bytes apart, a multiple of 16) and the group is
        // whole, else as 16-bit words; staged back to back, as in memory
        uint32_t pre[Q::kPre];
        uint4 prev[Q::kPreV];
        bool pvec = false;
        auto prefetch = [&](int64_t tile) {
            const int64_t v0 = tile * kQRows + 32 * grp;
            pvec = a.dense != 0 && tile < ntiles && v0 + 32 <= a.n_vec;
            if (pvec) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.blocks + v0 * Q::BB);
#pragma unroll
                for (int k = 0; k < Q::kPreV; ++k) {
                    const int q = tidg + 32 * kQSlices * k;
                    if (q < Q::kVec) prev[k] = __ldg(src + q);
                }
            } else {
#pragma unroll
                for (int k = 0; k < Q::kPre; ++k) {
                    const int q = tidg + 32 * kQSlices * k, row = q / Q::kHW, h = q - row * Q::kHW;
                    pre[k] = (q < 32 * Q::kHW && tile < ntiles && v0 + row < a.n_vec)
                                 ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(
                                       a.blocks + (v0 + row) * a.block_stride + 2 * h))
                                 : 0u;
                }
            }
        };
        auto stage = [&]() {
            uint8_t *g = blk + 32 * grp * Q::kPitch;
            if (pvec) {
#pragma unroll
                for (int k = 0; k < Q::kPreV; ++k) {
                    const int q = tidg + 32 * kQSlices * k;
                    if (q < Q::kVec) *reinterpret_cast<uint4 *>(g + 16 * q) = prev[k];
                }
            } else {
#pragma unroll
                for (int k = 0; k < Q::kPre; ++k) {
                    const int q = tidg + 32 * kQSlices * k;
                    if (q < 32 * Q::kHW) *reinterpret_cast<uint16_t *>(g + 2 * q) = (uint16_t)pre[k];
                }
            }
        };
        auto grp_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(grp_bar), "n"(32 * kQSlices) : "memory"); };
        prefetch(blockIdx.x);
        // a wait that gives up is recorded and not repeated: the loop still runs to its end (every
        // named barrier is met), on products that are then not valid
        bool ok = true;
        auto wait = [&](int b, uint32_t parity) {
            if (ok && !tc_mbar_wait(bars + 8 * b, parity)) {
                ok = false;
                note_wait_failed();
            }
        };
        // signs of P = S r for tile j (this slice): bit k of the row's 128 = [(S r)_k >= 0]; run one
        // tile late, so that the tensor cores compute P of tile j + 1 meanwhile
        // signs of P = S r for tile j (this slice): bit k of the row's 128 = [(S r)_k >= 0]; run one
        // tile late, so that the tensor cores compute P of tile j + 1 meanwhile
        auto signs_out = [&](int j, int64_t pv0, int pnv, unsigned short prn) {
            float y[kQNC / 32][32];
            const uint32_t paddr = tmem + ((uint32_t)(32 * grp) << 16) + (uint32_t)(256 + 128 * (j & 1) + c0);
#pragma unroll
            for (int c = 0; c < kQNC / 32; ++c) tc_ld32(paddr + 32 * c, y[c]);
            tc_wait_ld();
            tc_fence_before();
            uint32_t wb[kQNC / 32];
#pragma unroll
            for (int c = 0; c < kQNC / 32; ++c) {
                wb[c] = 0u;
#pragma unroll
                for (int k = 0; k < 32; ++k) wb[c] |= (y[c][k] >= 0.f ? 1u : 0u) << k;
            }
            if (r < pnv) {
                uint8_t *dst = a.bits + (pv0 + r) * 16 + c0 / 8;
                if constexpr (kQNC == 64) *reinterpret_cast<uint2 *>(dst) = make_uint2(wb[0], wb[1]);
                else *reinterpret_cast<uint32_t *>(dst) = wb[0];
                if (sl == 0) a.rn[pv0 + r] = prn;
            }
        };
        // fp16 ||r|| of tile j from the slices' partial sums (double-buffered by tile parity: the
        // sums of tile j are complete at the group barrier that opens tile j + 1)
        auto norm_of = [&](int j, float jscale) -> unsigned short {
            const float *pp = part + (j & 1) * (kQSlices * kQRows);
            float ss = 0.f;
#pragma unroll
            for (int q = 0; q < kQSlices; ++q) ss += pp[q * kQRows + r];
            return __half_as_ushort(__float2half_rn(sqrtf(ss) * (1.f / jscale)));
        };
        int64_t pv0 = 0;
        int pnv = 0;
        float pscale = 1.f;
        int i = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
            const int st = i & 1;
            const int64_t v0 = tile * kQRows;
            const int nv = (int)min64(kQRows, a.n_vec - v0);
            stage();
            prefetch(tile + gridDim.x);
            grp_sync();   // the group's blocks are staged, the previous tile's partial sums complete
            const unsigned short prn = i >= 1 ? norm_of(i - 1, pscale) : (unsigned short)0;

            // ---- U of this row slice
            wait(kBarURdy + st, (uint32_t)(i >> 1) & 1u);
            tc_fence_after();
            float x[kQNC / 32][32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * grp) << 16) + (uint32_t)(st * 128 + c0);
#pragma unroll
            for (int c = 0; c < kQNC / 32; ++c) tc_ld32(taddr + 32 * c, x[c]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bars + 8 * (kBarUFree + st));

            // ---- R r = u / sqrt(128) - n16 c[code], scaled by 2^(7 - E) with n16 in [2^(E-1), 2^E)
            const int rb = r * Q::kPitch;   // the row's block in the staging buffer (2-byte aligned)
            const float nf = r < nv ? __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(blk + rb))) : 0.f;
            float scale = 1.f;   // inf / NaN norms: left unscaled
            if (nf == 0.f) {
                scale = 1073741824.f;   // 2^30
            } else if (nf < 65536.f) {
                const int E = (int)((__float_as_uint(nf) >> 23) & 0xFF) - 126;
                scale = __uint_as_float((uint32_t)(127 + 7 - E) << 23);
            }
            const float inv_rs = 0.08838834764831845f * scale, nn = -(nf * scale);
            float2 q2 = make_float2(0.f, 0.f);
            auto element_pair = [&](int e, float cv0, float cv1) {
                const float2 u2 = __fmul2_rn(make_float2(x[e >> 5][e & 31], x[e >> 5][(e & 31) + 1]),
                                             make_float2(inv_rs, inv_rs));
                const float2 r2 = __ffma2_rn(make_float2(cv0, cv1), make_float2(nn, nn), u2);
                x[e >> 5][e & 31] = r2.x;
                x[e >> 5][(e & 31) + 1] = r2.y;
                q2 = __ffma2_rn(r2, r2, q2);
            };
            if constexpr (Q::kPairs) {
                // one lookup per two elements: both low-plane code pairs sit in 4 adjacent bits, both
                // high-plane bits (3-bit codes) in 2
                uint32_t lw[kQNC / 16], hw[1] = {0u};
                words_at<kQNC / 16>(blk, rb + 2 + c0 / 4, lw);
                if constexpr (BITS == 3) words_at<1>(blk, rb + 34 + c0 / 8, hw);
                const uint32_t ptab_s = base_s + Q::kCtab + 8u * (uint32_t)lane;
#pragma unroll
                for (int e = 0; e < kQNC; e += 2) {
                    uint32_t pidx = (lw[e >> 4] >> (2 * (e & 15))) & 15u;
                    if constexpr (BITS == 3) pidx |= ((hw[0] >> (e & 31)) & 3u) << 4;
                    const float2 cv = lds_f2_q(ptab_s + pidx * 256u);
                    element_pair(e, cv.x, cv.y);
                }
            } else {
                uint32_t cw[kQNC / 8];
                words_at<kQNC / 8>(blk, rb + 2 + c0 / 2, cw);
#pragma unroll
                for (int e = 0; e < kQNC; e += 2) {
                    const float cv0 = lds_f32(ctab_s + code_at<BITS, kQNC>(cw, e) * 128u);
                    const float cv1 = lds_f32(ctab_s + code_at<BITS, kQNC>(cw, e + 1) * 128u);
                    element_pair(e, cv0, cv1);
                }
            }
            part[(i & 1) * (kQSlices * kQRows) + sl * kQRows + r] = q2.x + q2.y;
            // the previous tile's P is complete: its MMAs have read the R r tiles rewritten below
            if (i >= 1) wait(kBarP, (uint32_t)(i - 1) & 1u);
            tc_fence_after();
            // fp16 hi / lo tiles of R r (K-major, 128-byte swizzle), then hand them to the tensor cores
#pragma unroll
            for (int kc = 0; kc < kQNC / 8; ++kc) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int e = 8 * kc + 2 * p;
                    split_pair(x[e >> 5][e & 31], x[e >> 5][(e & 31) + 1], h[p], l[p]);
                }
                const int chunk = ((c0 & 63) >> 3) + kc;
                const uint32_t addr = a2_row + (uint32_t)(((chunk ^ (r & 7)) << 4));
                sts128_q(addr, h[0], h[1], h[2], h[3]);
                sts128_q(addr + kQTile, l[0], l[1], l[2], l[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bars + 8 * kBarA2);
            if (i >= 1) signs_out(i - 1, pv0, pnv, prn);
            pv0 = v0;
            pnv = nv;
            pscale = scale;
        }
        if (i >= 1) {
            grp_sync();   // the last tile's partial sums
            const unsigned short prn = norm_of(i - 1, pscale);
            wait(kBarP, (uint32_t)(i - 1) & 1u);
            tc_fence_after();
            signs_out(i - 1, pv0, pnv, prn);
        }
    }

    // ---- teardown: every MMA has completed (the producer waited for its last commit) and every
    // tensor-memory load completed
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

int wait_failed_qjl(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

int qjl_encode_tc(const void *k, int k_dtype, int64_t n_vec, int64_t k_stride_bytes, const uint8_t *blocks,
                  int64_t block_stride, int bits, const float *centroids, const uint32_t *signs, const float *S,
                  uint8_t *qjl_bits, uint16_t *res_norm_f16, cudaStream_t st) {
    if (k_dtype != TQ_BF16 && k_dtype != TQ_F16) return 1;
    CUtensorMap map;
    if (!make_row_tile_map(&map, k, k_dtype, n_vec, k_stride_bytes)) return 1;
    QjlTcArgs a;
    a.drop = drop_copies();
    a.blocks = blocks;
    a.block_stride = block_stride;
    a.dense = block_stride == 2 + 16 * bits && (reinterpret_cast<uintptr_t>(blocks) & 15) == 0 ? 1 : 0;
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
