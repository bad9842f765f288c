// Decode attention at head dims 64, 96, 128 and 160 on the tensor cores
// (mma.sync m16n8k16, fp16 operands, float32 accumulation), for up to eight
// query heads per KV head and 2-, 3- or 4-bit keys and values.
//
// "TurboQuant KV Cache Compression — Spec", Optimization: Fused dequant-dot
// (scores of the rotated query against centroid lookups, no per-key inverse
// rotation), with the head-dim codec of Types / Codebook Generation.  The
// call's query prep and combine (R q, and the merge of the splits with R^T)
// are those of tq_headdim.cu; this header holds the attention kernel,
// tq_headdim_mma.cu instantiates it for up to four heads per KV head (and
// plans and launches), tq_headdim_mma8.cu for five to eight.
//
// One CTA of 4 warps per (sequence, KV head, context split); a warp takes
// 32-token chunks t0 + 32 (warp + 4 i), staged in shared memory by
// double-buffered 16-byte cp.async copies.
//   * Scores: S[32 tokens x 8] = K Q^T over the d dims as d / 16 k-steps.
//     The contraction order is free as long as both operands follow it:
//     lane t of a quad takes the contiguous dims [t d/4, (t + 1) d/4) of
//     every token, four per k-step, so it reads its codes as one contiguous
//     slice of the block.  A-fragment words come from a table of code pairs
//     (hi and lo fp16 parts of the two centroids, 16 copies so that a half
//     warp never meets a bank conflict); the B operand holds the 4 heads x
//     (hi, lo) parts of the rotated query in registers, so each product sums
//     all four cross terms and score = column hi + column lo.  With five to
//     eight heads the n-tile's columns are the heads, and the hi and lo
//     parts go through separate products into the same accumulators
//     (K_hi Q_hi, K_lo Q_hi, K_hi Q_lo).
//   * Online softmax per head on the accumulators (a lane's four tokens of
//     head t -- with five to eight heads, of heads 2t and 2t + 1 -- then the
//     8 lanes of that head), probabilities times value norms written as fp16
//     hi / lo into a small per-warp tile.
//   * Values: O^T[d x 8] += V^T P^T over the chunk's tokens: the m-tile rows
//     are dims (lane group g takes the contiguous dims [g d/8, (g + 1) d/8)),
//     the k-slots tokens in order; A-fragment words come from a table of
//     (token 2j, token 2j + 1) code pairs at one dim, their indices built by
//     interleaving the two tokens' code slices (3-bit: the 2-bit planes as
//     for 2-bit codes, the two high bits in index bits 4 and 5); B from the
//     probability tile (five to eight heads: a hi tile and a lo tile, two
//     products).
// The warps' states are merged in shared memory into one partial per head
// and split, in the layout the combine kernel reads.

#pragma once

#include <cmath>
#include <cstring>

#include "tq_device.cuh"
#include "tq_headdim.cuh"
#include "tq_internal.h"

namespace tq {

// One instantiation: the kernel, its shared memory, and (per instantiation) the devices whose
// shared-memory limit has been raised for it and its CTAs per SM.
struct HmKernel {
    const void *fn;
    int smem;
    int *done;       // [64], see set_smem_limit
    int *resident;   // CTAs per SM (0: not yet asked)
};

// The kernel for (d, key bits, value bits) with up to four (g4) or five to eight (g8) heads per KV
// head; fn = nullptr when not covered.
HmKernel hm_select_g4(int d, int kb, int vb);
HmKernel hm_select_g8(int d, int kb, int vb);

namespace {

constexpr unsigned kHmFull = 0xffffffffu;
constexpr int kHmWarps = 4;   // per CTA: small CTAs fill the SMs' slots in whole waves
constexpr int kHmThreads = 32 * kHmWarps;
constexpr int kHmPsRow = 68;   // bytes per column of the probability tile (32 fp16 + padding)

template <int ND, int KB, int VB, bool H8>
struct HmCfg {
    static constexpr int D = 32 * ND;
    static constexpr int KBB = 2 + D * KB / 8, VBB = 2 + D * VB / 8;
    static constexpr int NK = 1 << (2 * KB), NV = 1 << (2 * VB);   // pair-table entries
    static constexpr int kHeads = H8 ? 8 : 4;                      // heads per warp in the merge area
    static constexpr int kKT = 0;                                  // [NK][16] (hi, lo) words
    static constexpr int kVT = kKT + NK * 128;                     // [NV][32] words
    static constexpr int kPs = kVT + NV * 128;                     // [warp][1 or 2][8 columns][kHmPsRow]
    static constexpr int kStage = 32 * (KBB + VBB);                // one chunk's K then V blocks
    static constexpr int kSt = kPs + kHmWarps * (H8 ? 2 : 1) * 8 * kHmPsRow;   // [warp][2][kStage], then the merge
    static constexpr int kStages = kHmWarps * 2 * kStage, kPart = kHmWarps * kHeads * (2 + D) * 4;
    static constexpr int kTotal = kSt + (kStages > kPart ? kStages : kPart) + 16;   // (+ 16: see hm_bytes)
    static_assert(kSt % 16 == 0 && kStage % 16 == 0, "16-byte aligned stages");
};

__device__ __forceinline__ void hm_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 hm_lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t hm_lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t hm_h2(float lo_elem, float hi_elem) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo_elem)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(hi_elem)) << 16);
}

// fp16 hi part and the fp16 of the remainder.
__device__ __forceinline__ void hm_split(float v, float &hi, float &lo) {
    hi = __half2float(__float2half_rn(v));
    lo = v - hi;
}

// The two codes of pair-table entry e (3-bit: e = low bits of both | high bits of both << 4).
template <int KB>
__device__ __forceinline__ void hm_key_pair(int e, int &c0, int &c1) {
    if constexpr (KB == 3) {
        c0 = (e & 3) | (((e >> 4) & 1) << 2);
        c1 = ((e >> 2) & 3) | (((e >> 5) & 1) << 2);
    } else {
        c0 = e & ((1 << KB) - 1);
        c1 = e >> KB;
    }
}

// The 4 (N + 3) / 4 bytes from any shared address p on, as little-endian 32-bit words: aligned
// 32-bit loads from the word at or below p, joined by funnel shifts (may read up to 7 bytes past the
// last word: the shared-memory layout leaves 16 bytes after the stages).
template <int N>
__device__ __forceinline__ void hm_bytes(const uint8_t *p, uint32_t (&w)[(N + 3) / 4]) {
    constexpr int NW = (N + 3) / 4;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    const uint32_t base = a & ~3u, sh = (a & 3u) * 8u;
    uint32_t raw[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) raw[i] = hm_lds32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

__device__ __forceinline__ uint32_t hm_byte(const uint32_t *w, int i) { return (w[i >> 2] >> (8 * (i & 3))) & 0xFFu; }

// Key slice of one token for this lane (dims [t d/4, (t + 1) d/4)): its code bytes (4-bit: 4 ND
// bytes; 2- and 3-bit: the 2 ND bytes of the 2-bit plane, and for 3-bit the ND bytes of high bits).
template <int ND, int KB>
struct HmKeySlice {
    static constexpr int NW = KB == 4 ? ND : (2 * ND + 3) / 4;
    uint32_t w[NW];
    uint32_t h[KB == 3 ? (ND + 3) / 4 : 1];

    __device__ __forceinline__ void load(const uint8_t *blk, int t) {
        constexpr int D = 32 * ND;
        if constexpr (KB == 4) {
            hm_bytes<4 * ND>(blk + 2 + t * 4 * ND, w);
        } else {
            hm_bytes<2 * ND>(blk + 2 + t * 2 * ND, w);
            if constexpr (KB == 3) hm_bytes<ND>(blk + 2 + D / 4 + t * ND, h);
        }
    }
    // pair-table byte offsets (index << 7) of k-step ks: x = dims 4 ks, 4 ks + 1 of the slice,
    // y = dims 4 ks + 2, 4 ks + 3
    __device__ __forceinline__ void pick(int ks, uint32_t &x, uint32_t &y) const {
        if constexpr (KB == 4) {
            const uint32_t b2 = (w[ks >> 1] >> (16 * (ks & 1))) & 0xFFFFu;
            x = (b2 & 0xFFu) << 7;
            y = (b2 >> 8) << 7;
        } else {
            const uint32_t b = hm_byte(w, ks);
            uint32_t i0 = b & 15u, i1 = b >> 4;
            if constexpr (KB == 3) {
                const uint32_t hn = (hm_byte(h, ks >> 1) >> (4 * (ks & 1))) & 15u;
                i0 |= (hn & 3u) << 4;
                i1 |= (hn >> 2) << 4;
            }
            x = i0 << 7;
            y = i1 << 7;
        }
    }
};

// Value slice of one token for this lane (dims [g d/8, (g + 1) d/8)) as 32-bit words: word w holds
// slice dims 16 w .. (2-bit codes and the 2-bit plane of 3-bit codes) or 8 w .. (4-bit codes); for
// 3-bit codes h holds the slice's 4 ND high bits (bit i: slice dim i).
template <int ND, int VB>
struct HmValueSlice {
    static constexpr int NB = ND * (VB == 3 ? 2 : VB) / 2;   // bytes of the slice (of the 2-bit plane)
    static constexpr int NW = (NB + 3) / 4;
    uint32_t w[NW];
    uint32_t h;
    __device__ __forceinline__ void load(const uint8_t *blk, int g) {
        hm_bytes<NB>(blk + 2 + g * NB, w);
        if constexpr (VB == 3) {
            // the slice starts at bit 4 ND g of the high plane: a byte, plus a nibble when ND g is odd
            constexpr int D = 32 * ND;
            const uint32_t a = (uint32_t)__cvta_generic_to_shared(blk + 2 + D / 4 + ((g * ND) >> 1));
            const uint32_t base = a & ~3u, sh = (a & 3u) * 8u + 4u * ((g * ND) & 1);   // < 32
            h = __funnelshift_r(hm_lds32(base), hm_lds32(base + 4), sh);
        }
    }
};

// ((x >> (B k)) & (2^B - 1)) << 7 for a constant field k of width B (4 or 8): a pair-table byte
// offset, in two operations.
template <int B, int K>
__device__ __forceinline__ uint32_t hm_field7(uint32_t x) {
    constexpr uint32_t mask = ((1u << B) - 1u) << 7;
    if constexpr (B * K >= 32) return 0u;   // (a field past the word: not reached)
    else if constexpr (B * K >= 7) return (x >> (B * K - 7)) & mask;
    else return (x << (7 - B * K)) & mask;
}

// ((x >> 2 k) & 3) << 11: the two high bits of a 3-bit value pair as pair-table index bits 4 and 5
// (byte offset bits 11 and 12); k is a constant once the m-tile loop is unrolled.
__device__ __forceinline__ uint32_t hm_hfield(uint32_t x, int k) {
    return 2 * k >= 11 ? (x >> (2 * k - 11)) & (3u << 11) : (x << (11 - 2 * k)) & (3u << 11);
}

template <int ND, int KB, int VB, bool H8>
__global__ void __launch_bounds__(kHmThreads, H8 ? 2 : 3) attn_dm_kernel(const __grid_constant__ HdAttnArgs a) {
    using C = HmCfg<ND, KB, VB, H8>;
    constexpr int D = C::D, KBB = C::KBB, VBB = C::VBB, NKS = D / 16;
    constexpr int NQ = H8 ? 2 : 1;   // query operand sets: (hi | lo columns) or hi, lo
    constexpr int NH = H8 ? 2 : 1;   // heads per lane: t, or 2 t and 2 t + 1
    extern __shared__ __align__(16) uint8_t hm_smem[];
    const uint32_t smem_s = (uint32_t)__cvta_generic_to_shared(hm_smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int b = blockIdx.z, kvh = blockIdx.y, sp = blockIdx.x;
    int L = a.T;
    if (a.seq_lens) {
        const int sl = a.seq_lens[b];
        L = sl < 0 ? 0 : (sl > a.T ? a.T : sl);
    }
    const int t0 = sp * a.tps, t1 = min(L, t0 + a.tps);
    const int64_t seg = ((int64_t)b * a.Hkv + kvh) * a.T_cap;
    const uint8_t *kseg = a.k + seg * KBB, *vseg = a.v + seg * VBB;
    uint8_t *wst = hm_smem + C::kSt + warp * 2 * C::kStage;
    // the K then V blocks of tokens [base, base + n) into stage buf, in whole 16-byte pieces (the last
    // piece may run up to 15 bytes past the n-th block, still inside the segment's T_cap blocks)
    auto issue = [&](int base, int buf) {
        const int n = min(32, t1 - base);
        const int nk = (n * KBB + 15) >> 4, nv = (n * VBB + 15) >> 4;
        const uint8_t *sk = kseg + (int64_t)base * KBB, *sv = vseg + (int64_t)base * VBB;
        uint8_t *dk = wst + buf * C::kStage, *dv = dk + 32 * KBB;
        for (int q = lane; q < nk; q += 32) cp_async16(dk + 16 * q, sk + 16 * q);
        for (int q = lane; q < nv; q += 32) cp_async16(dv + 16 * q, sv + 16 * q);
        cp_async_commit();
    };
    int base = t0 + 32 * warp;
    if (base < t1) issue(base, 0);   // the first chunk is on its way while the tables are built

    // ---- pair tables: keys (hi, lo) words, 16 copies; values one word, 32 copies
    {
        uint2 *kt = reinterpret_cast<uint2 *>(hm_smem + C::kKT);
        for (int i = threadIdx.x; i < C::NK * 16; i += kHmThreads) {
            int c0, c1;
            hm_key_pair<KB>(i >> 4, c0, c1);
            float h0, l0, h1, l1;
            hm_split(a.kc[c0], h0, l0);
            hm_split(a.kc[c1], h1, l1);
            kt[i] = make_uint2(hm_h2(h0, h1), hm_h2(l0, l1));
        }
        uint32_t *vt = reinterpret_cast<uint32_t *>(hm_smem + C::kVT);
        for (int i = threadIdx.x; i < C::NV * 32; i += kHmThreads) {
            int c0, c1;
            hm_key_pair<VB>(i >> 5, c0, c1);   // (the same pair-index layout as the keys)
            vt[i] = hm_h2(a.vc[c0], a.vc[c1]);
        }
    }
    // the rotated queries come from the prep kernel this one depends on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // B fragments of the scores; k-step ks holds this lane's slice dims 4 ks .. 4 ks + 3, i.e. dims
    // t d/4 + 4 ks + e.  Up to 4 heads: column g = head g / 2, part g % 2 (hi, lo), one set; 5 to 8
    // heads: column g = head g, set 0 the hi parts and set 1 the lo parts.
    uint32_t qb[NQ][NKS][2];
    {
        const int hd = H8 ? g : g >> 1;
        const float *qr = a.qrot + ((int64_t)b * a.Hq + kvh * a.G + hd) * D + t * (D / 4);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (hd < a.G) {
                const float2 p0 = *reinterpret_cast<const float2 *>(qr + 4 * ks);
                const float2 p1 = *reinterpret_cast<const float2 *>(qr + 4 * ks + 2);
                v[0] = p0.x;
                v[1] = p0.y;
                v[2] = p1.x;
                v[3] = p1.y;
            }
            float h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) hm_split(v[e], h[e], l[e]);
            if constexpr (H8) {
                qb[0][ks][0] = hm_h2(h[0], h[1]);
                qb[0][ks][1] = hm_h2(h[2], h[3]);
                qb[NQ - 1][ks][0] = hm_h2(l[0], l[1]);
                qb[NQ - 1][ks][1] = hm_h2(l[2], l[3]);
            } else {
                const bool part = g & 1;
                qb[0][ks][0] = part ? hm_h2(l[0], l[1]) : hm_h2(h[0], h[1]);
                qb[0][ks][1] = part ? hm_h2(l[2], l[3]) : hm_h2(h[2], h[3]);
            }
        }
    }
    __syncthreads();

    const uint32_t kt_s = smem_s + C::kKT + (lane & 15) * 8, vt_s = smem_s + C::kVT + lane * 4;
    // probability tile(s) of this warp: [NQ][8 columns][kHmPsRow]
    uint8_t *ps = hm_smem + C::kPs + warp * NQ * 8 * kHmPsRow;
    const uint32_t ps_s = smem_s + C::kPs + warp * NQ * 8 * kHmPsRow;
    // running state of the lane's heads (uniform over the 8 lanes with the same t), this lane's share
    // of l, and the value sums O^T: up to 4 heads, o[mt][0 / 1] = dim g d/8 + 2 mt, columns (hi, lo)
    // of head t, [2 / 3] = dim + 1; 5 to 8 heads, o[mt][e] = that dim, head 2 t + e, [2 + e] = dim + 1
    float m_run[NH], l_run[NH];
#pragma unroll
    for (int e = 0; e < NH; ++e) {
        m_run[e] = -INFINITY;
        l_run[e] = 0.f;
    }
    float o[NKS][4];
#pragma unroll
    for (int mt = 0; mt < NKS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    int buf = 0;
    for (; base < t1; base += 32 * kHmWarps) {
        const int nb = base + 32 * kHmWarps;
        if (nb < t1) issue(nb, buf ^ 1);
        else cp_async_commit();   // (an empty group: the wait below always leaves one group)
        cp_async_wait<1>();
        __syncwarp();
        const uint8_t *sk = wst + buf * C::kStage, *sv = sk + 32 * KBB;
        const int n = min(32, t1 - base);

        // ---- scores of this lane's tokens 16 mt + g + 8 r against its heads
        float sc[2][2][NH];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int tok0 = 16 * mt + g, tok1 = tok0 + 8;
            HmKeySlice<ND, KB> k0, k1;
            k0.load(sk + tok0 * KBB, t);
            k1.load(sk + tok1 * KBB, t);
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
                uint32_t x0, y0, x1, y1;
                k0.pick(ks, x0, y0);
                k1.pick(ks, x1, y1);
                const uint2 e0 = hm_lds64(kt_s + x0), e1 = hm_lds64(kt_s + x1);
                const uint2 e2 = hm_lds64(kt_s + y0), e3 = hm_lds64(kt_s + y1);
                hm_mma(s, e0.x, e1.x, e2.x, e3.x, qb[0][ks][0], qb[0][ks][1]);
                hm_mma(s, e0.y, e1.y, e2.y, e3.y, qb[0][ks][0], qb[0][ks][1]);
                if constexpr (H8) hm_mma(s, e0.x, e1.x, e2.x, e3.x, qb[NQ - 1][ks][0], qb[NQ - 1][ks][1]);
            }
            const float kn0 = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(sk + tok0 * KBB)));
            const float kn1 = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(sk + tok1 * KBB)));
            // (a stage holds stale bytes past the n-th token: every use below is selected away)
            if constexpr (H8) {
#pragma unroll
                for (int e = 0; e < NH; ++e) {
                    sc[mt][0][e] = tok0 < n ? s[e] * kn0 : -INFINITY;
                    sc[mt][1][e] = tok1 < n ? s[2 + e] * kn1 : -INFINITY;
                }
            } else {
                sc[mt][0][0] = tok0 < n ? (s[0] + s[1]) * kn0 : -INFINITY;
                sc[mt][1][0] = tok1 < n ? (s[2] + s[3]) * kn1 : -INFINITY;
            }
        }
        // ---- online softmax per head: the lane's four tokens, then the head's 8 lanes
        float corr[NH], pv[2][2][NH];
#pragma unroll
        for (int e = 0; e < NH; ++e) {
            float mx = fmaxf(fmaxf(sc[0][0][e], sc[0][1][e]), fmaxf(sc[1][0][e], sc[1][1][e]));
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kHmFull, mx, off));
            const float mn = fmaxf(m_run[e], mx);   // finite: the chunk holds at least one token
            corr[e] = exp2f(m_run[e] - mn);
            m_run[e] = mn;
            float psum = 0.f;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float p = exp2f(sc[mt][r][e] - mn);   // 0 past the n-th token
                    psum += p;
                    pv[mt][r][e] = p;
                }
            l_run[e] = fmaf(l_run[e], corr[e], psum);
        }
        // probabilities times the value norms, as fp16 hi / lo
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int tok = 16 * mt + g + 8 * r;
                const float vn = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(sv + tok * VBB)));
#pragma unroll
                for (int e = 0; e < NH; ++e) {
                    const float x = tok < n ? pv[mt][r][e] * vn : 0.f;
                    float h, l;
                    hm_split(x, h, l);
                    // up to 4 heads: columns 2 t (hi) and 2 t + 1 (lo) of one tile; 5 to 8: column
                    // 2 t + e of the hi tile and of the lo tile
                    const int ch = H8 ? 2 * t + e : 2 * t, cl = H8 ? 8 + 2 * t + e : 2 * t + 1;
                    reinterpret_cast<__half *>(ps + ch * kHmPsRow)[tok] = __float2half_rn(h);
                    reinterpret_cast<__half *>(ps + cl * kHmPsRow)[tok] = __float2half_rn(l);
                }
            }
#pragma unroll
        for (int mt = 0; mt < NKS; ++mt) {
            o[mt][0] *= corr[0];
            o[mt][1] *= corr[NH - 1];
            o[mt][2] *= corr[0];
            o[mt][3] *= corr[NH - 1];
        }
        __syncwarp();

        // ---- O^T += V^T P^T over the chunk's two 16-token k-steps
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int ta = 16 * kk + 2 * t;   // tokens ta, ta + 1 (k-slots 2t, 2t + 1) and ta + 8, ta + 9
            HmValueSlice<ND, VB> xa, xb, xc, xd;
            xa.load(sv + ta * VBB, g);
            xb.load(sv + (ta + 1) * VBB, g);
            xc.load(sv + (ta + 8) * VBB, g);
            xd.load(sv + (ta + 9) * VBB, g);
            uint32_t pb[NQ][2];
#pragma unroll
            for (int s = 0; s < NQ; ++s) {
                pb[s][0] = hm_lds32(ps_s + (8 * s + g) * kHmPsRow + 2 * ta);
                pb[s][1] = hm_lds32(ps_s + (8 * s + g) * kHmPsRow + 2 * (ta + 8));
            }
            // per slice word: e* field k = (code of the first token, of the second) at an even slice dim,
            // o* field k at the odd dim after it (nibbles for 2-bit codes and 3-bit low planes, bytes
            // for 4-bit)
            constexpr int NW = HmValueSlice<ND, VB>::NW;
            constexpr uint32_t M = VB == 4 ? 0x0F0F0F0Fu : 0x33333333u;
            constexpr int SH = VB == 4 ? 4 : 2;
            uint32_t eab[NW], oab[NW], ecd[NW], ocd[NW];
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                eab[w] = (xa.w[w] & M) | ((xb.w[w] & M) << SH);
                oab[w] = ((xa.w[w] >> SH) & M) | (xb.w[w] & (M << SH));
                ecd[w] = (xc.w[w] & M) | ((xd.w[w] & M) << SH);
                ocd[w] = ((xc.w[w] >> SH) & M) | (xd.w[w] & (M << SH));
            }
            // 3-bit high bits, 2-bit fields in the same pattern: field k = (high bit of the first token,
            // of the second) at slice dim 2 k (eh*) or 2 k + 1 (oh*)
            uint32_t ehab = 0u, ohab = 0u, ehcd = 0u, ohcd = 0u;
            if constexpr (VB == 3) {
                ehab = (xa.h & 0x55555555u) | ((xb.h & 0x55555555u) << 1);
                ohab = ((xa.h >> 1) & 0x55555555u) | (xb.h & 0xAAAAAAAAu);
                ehcd = (xc.h & 0x55555555u) | ((xd.h & 0x55555555u) << 1);
                ohcd = ((xc.h >> 1) & 0x55555555u) | (xd.h & 0xAAAAAAAAu);
            }
            // m-tile mt: slice dims 2 mt (row g) and 2 mt + 1 (row g + 8)
            constexpr int FPW = VB == 4 ? 4 : 8;   // fields per word
            constexpr int FB = VB == 4 ? 8 : 4;    // field width
#pragma unroll
            for (int mt = 0; mt < NKS; ++mt) {
                const int w = mt / FPW;
                uint32_t f0, f1, f2, f3;
                switch (mt % FPW) {
#define HM_FIELDS(K)                                                                        \
    case K:                                                                                 \
        f0 = hm_field7<FB, K>(eab[w]);                                                      \
        f1 = hm_field7<FB, K>(oab[w]);                                                      \
        f2 = hm_field7<FB, K>(ecd[w]);                                                      \
        f3 = hm_field7<FB, K>(ocd[w]);                                                      \
        break;
                    HM_FIELDS(0) HM_FIELDS(1) HM_FIELDS(2) HM_FIELDS(3)
                    HM_FIELDS(4) HM_FIELDS(5) HM_FIELDS(6)
                    default: HM_FIELDS(7)
#undef HM_FIELDS
                }
                if constexpr (VB == 3) {
                    f0 |= hm_hfield(ehab, mt);
                    f1 |= hm_hfield(ohab, mt);
                    f2 |= hm_hfield(ehcd, mt);
                    f3 |= hm_hfield(ohcd, mt);
                }
                const uint32_t a0 = hm_lds32(vt_s + f0), a1 = hm_lds32(vt_s + f1);
                const uint32_t a2 = hm_lds32(vt_s + f2), a3 = hm_lds32(vt_s + f3);
#pragma unroll
                for (int s = 0; s < NQ; ++s) hm_mma(o[mt], a0, a1, a2, a3, pb[s][0], pb[s][1]);
            }
        }
        __syncwarp();   // the stage and the probability tile are free for the next chunk
        buf ^= 1;
    }
    cp_async_wait<0>();
    // the combine kernel may take its place on the SMs now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    __syncthreads();   // every warp is done with its stages: the merge area takes their place

    // ---- the warps' states per head into shared memory; then each head is merged by one warp
    constexpr int HP = C::kHeads;   // heads per warp in the merge area
    float *part = reinterpret_cast<float *>(hm_smem + C::kSt);   // [warp][HP][2 + D]
#pragma unroll
    for (int e = 0; e < NH; ++e) {
        float lw = l_run[e];
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) lw += __shfl_xor_sync(kHmFull, lw, off);
        const int hd = H8 ? 2 * t + e : t;
        if (hd < a.G) {
            float *pp = part + (warp * HP + hd) * (2 + D);
            if (g == 0) {
                pp[0] = m_run[e];
                pp[1] = lw;
            }
#pragma unroll
            for (int mt = 0; mt < NKS; ++mt) {
                if constexpr (H8) {
                    pp[2 + g * (D / 8) + 2 * mt] = o[mt][e];
                    pp[2 + g * (D / 8) + 2 * mt + 1] = o[mt][2 + e];
                } else {
                    pp[2 + g * (D / 8) + 2 * mt] = o[mt][0] + o[mt][1];
                    pp[2 + g * (D / 8) + 2 * mt + 1] = o[mt][2] + o[mt][3];
                }
            }
        }
    }
    __syncthreads();
    for (int h = warp; h < a.G; h += kHmWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kHmWarps; ++w) M = fmaxf(M, part[(w * HP + h) * (2 + D)]);
        float lt = 0.f, acc[ND];
#pragma unroll
        for (int k = 0; k < ND; ++k) acc[k] = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kHmWarps; ++w) {
                const float *pp = part + (w * HP + h) * (2 + D);
                const float f = pp[0] == -INFINITY ? 0.f : exp2f(pp[0] - M);
                lt = fmaf(pp[1], f, lt);
#pragma unroll
                for (int k = 0; k < ND; ++k) acc[k] = fmaf(pp[2 + lane + 32 * k], f, acc[k]);
            }
        }
        float *dst = a.ws + (((int64_t)b * a.Hq + kvh * a.G + h) * a.splits + sp) * (2 + D);
        if (lane == 0) {
            dst[0] = M;
            dst[1] = lt;
        }
#pragma unroll
        for (int k = 0; k < ND; ++k) dst[2 + lane + 32 * k] = acc[k];
    }
}

template <int ND, int KB, int VB, bool H8>
HmKernel hm_kernel() {
    static int done[64] = {0};
    static int resident = 0;
    return HmKernel{(const void *)attn_dm_kernel<ND, KB, VB, H8>, HmCfg<ND, KB, VB, H8>::kTotal, done, &resident};
}

// (d, key bits, value bits) -> hm_kernel<ND, KB, VB, H8>, for every covered combination
#define HM_CASE(ND, KBv, VBv, H8) \
    if (d == 32 * ND && kb == KBv && vb == VBv) return hm_kernel<ND, KBv, VBv, H8>();
#define HM_VB(ND, VBv, H8) HM_CASE(ND, 2, VBv, H8) HM_CASE(ND, 3, VBv, H8) HM_CASE(ND, 4, VBv, H8)
#define HM_DIM(ND, H8) HM_VB(ND, 2, H8) HM_VB(ND, 3, H8) HM_VB(ND, 4, H8)
#define HM_SELECT(H8) HM_DIM(2, H8) HM_DIM(3, H8) HM_DIM(4, H8) HM_DIM(5, H8)

}  // namespace
}  // namespace tq
