// Tensor-core decode attention for the 4-bit-key / 2-bit-value cache (sm_103a).
//
// Same computation as attn_split_kernel ("TurboQuant KV Cache Compression —
// Spec", Optimization: Fused dequant-dot): rotated query, scores against
// dequantised rotated keys, online softmax, values accumulated in the
// rotated domain, one inverse rotation per output (in the combine kernel).
//
// Once a tile of codes is looked up, both products are dense contractions:
//   scores  S[16 tokens x 8 heads]  = Khat[16 x 128] * Qrot^T[128 x 8]
//   values  O[128 dims x 8 heads]  += Vhat^T[128 x 16] * P[16 tokens x 8]
// and run as mma.sync m16n8k16 (fp16 operands, float32 accumulate; the G
// query heads sharing a KV head fill N = 8, zero-padded).
//   * Keys: a thread reads one 16-byte code slice per token (its dims
//     32t..32t+31, the MMA's k-columns permuted to match) and turns each code
//     byte (two 4-bit codes) into a half2 fragment register with one lookup
//     in a lane-replicated 256-entry table (word e * 32 + lane: every lane
//     reads its own bank, conflict-free).
//   * Values: a thread owns dims 16g..16g+15 (the MMA's m-rows permuted), i.e.
//     one 32-bit code word per token; a fragment register holds one dim of two
//     tokens, built by one byte permute from an 8-byte register table of the
//     four fp16 centroids.
//   * Softmax runs on the score accumulators per 32-token chunk; the value
//     norm is folded into P, which is transposed into the PV operand layout
//     with movmatrix.
//
// Work partition: the B * Hkv * ceil(T / 32) chunks, ordered by (sequence,
// KV head, position), are cut into kMmaCtas equal contiguous ranges, one per
// CTA (two CTAs per SM), so every CTA does the same work and there is no
// wave tail.  A CTA walks the (sequence, KV head) segments its range
// touches; its eight warps take the segment's chunks round-robin, each with
// its own cp.async double buffer and softmax state, merge in a three-round
// tree, and write one partial per query head into slot (CTA - first CTA of
// the segment).  tq_attn_mma_combine merges each segment's slots.

#include <cmath>

#include "tq_attn.cuh"
#include "tq_attn_mma.h"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kW = 8;                          // warps per CTA
constexpr int kThreadsMma = kW * 32;
constexpr int kKB4 = 66, kVB2 = 34;
constexpr int kKStage = kMmaChunk * kKB4;      // 2112 (16-byte multiple)
constexpr int kVStage = kMmaChunk * kVB2;      // 1088 (16-byte multiple)
constexpr int kWarpStage = kKStage + kVStage + 16;  // +16: word reads past a 2-aligned slice stay inside
constexpr int kLutBytes = 256 * 32 * 4;        // replicated key table
constexpr int kMergeSlot = 8 * 132;            // floats per warp slot in the merge buffer
constexpr unsigned kFull = 0xffffffffu;

constexpr int kSmemLut = 0;
constexpr int kSmemStages = kSmemLut + kLutBytes;
constexpr int kSmemQ = kSmemStages + kW * 2 * kWarpStage;
constexpr int kSmemMerge = kSmemQ + 8 * 128 * 4;
constexpr int kSmemTotal = kSmemMerge + 4 * kMergeSlot * 4;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// NW 32-bit words starting at a 2-byte aligned shared address: the aligned
// words around it, funnel-shifted by the misalignment.
template <int NW>
__device__ __forceinline__ void lds_words_a2(uint32_t addr, uint32_t (&w)[NW]) {
    const uint32_t base = addr & ~3u, sh = (addr & 3u) * 8u;
    uint32_t raw[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) raw[i] = lds32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void cp16_zfill(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__global__ void __launch_bounds__(kThreadsMma, 2) attn_mma_k4v2_kernel(const __grid_constant__ AttnArgs a,
                                                                       MmaPlan plan) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const uint32_t smem_s = (uint32_t)__cvta_generic_to_shared(smem);
    float *qbuf = reinterpret_cast<float *>(smem + kSmemQ);
    float *merge = reinterpret_cast<float *>(smem + kSmemMerge);

    // ---- key table: word e * 32 + l = half2(c[e & 15], c[e >> 4]); rotated stores are conflict-free
    {
        const int e = tid;  // 256 threads, 256 entries
        const uint32_t val = pack_half2(a.kc[e & 15], a.kc[e >> 4]);
        uint32_t *lut = reinterpret_cast<uint32_t *>(smem + kSmemLut);
#pragma unroll 8
        for (int j = 0; j < 32; ++j) lut[e * 32 + ((j + e) & 31)] = val;
    }
    // value table for prmt: bytes 0-3 = low bytes, 4-7 = high bytes of the four fp16 centroids
    uint32_t vlo = 0, vhi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t hb = __half_as_ushort(__float2half_rn(a.vc[i]));
        vlo |= (hb & 0xFFu) << (8 * i);
        vhi |= (hb >> 8) << (8 * i);
    }
    const uint32_t lut_s = smem_s + kSmemLut + lane * 4;
    const uint32_t stage_s = smem_s + kSmemStages + warp * 2 * kWarpStage;

    const int64_t lo = (int64_t)blockIdx.x * plan.Ctot / plan.P;
    const int64_t hi = (int64_t)(blockIdx.x + 1) * plan.Ctot / plan.P;
    for (int64_t x = lo; x < hi;) {
        const int64_t j = x / plan.C;                       // segment = (sequence, KV head)
        const int64_t seg_lo = j * plan.C;
        const int64_t xe = min64(hi, seg_lo + plan.C);
        const int b = (int)(j / a.Hkv), kvh = (int)(j % a.Hkv);
        int L = a.T;
        if (a.seq_lens) {
            const int sl = a.seq_lens[b];
            L = sl < 0 ? 0 : (sl > a.T ? a.T : sl);
        }
        const int slot = (int)(blockIdx.x - mma_cta_of_chunk(seg_lo, plan));

        // ---- rotated, scaled query of head `warp` (zero for padded heads), warp-local transform
        __syncthreads();   // previous segment's readers of qbuf / merge are done
        {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (warp < a.G) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int d = 4 * lane + k;
                    const float qv = load_q(a.q, a.q_dtype, ((int64_t)b * a.Hq + kvh * a.G + warp) * kD + d);
                    v[k] = ((a.signs[d >> 5] >> (d & 31)) & 1u) ? -qv : qv;
                }
            }
            float x0 = v[0] + v[1], x1 = v[0] - v[1], x2 = v[2] + v[3], x3 = v[2] - v[3];
            v[0] = x0 + x2;
            v[2] = x0 - x2;
            v[1] = x1 + x3;
            v[3] = x1 - x3;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float o = __shfl_xor_sync(kFull, v[k], m);
                    v[k] = (lane & m) ? (o - v[k]) : (v[k] + o);
                }
            }
            const float f = a.qscale * 0.08838834764831845f;
            reinterpret_cast<float4 *>(qbuf + warp * 128)[lane] = make_float4(v[0] * f, v[1] * f, v[2] * f, v[3] * f);
        }
        __syncthreads();
        // B fragments of Q^T: k-step ks, columns {2t, 2t+1, 2t+8, 2t+9} <-> dims 32t + 4ks + {0, 1, 2, 3}
        uint32_t qb[8][2];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const float4 q4 = reinterpret_cast<const float4 *>(qbuf + g * 128 + 32 * t + 4 * ks)[0];
            qb[ks][0] = pack_half2(q4.x, q4.y);
            qb[ks][1] = pack_half2(q4.z, q4.w);
        }

        const int64_t bh = (int64_t)b * a.Hkv + kvh;
        const uint8_t *kbase = a.k + bh * a.T_cap * kKB4;
        const uint8_t *vbase = a.v + bh * a.T_cap * kVB2;
        auto tok0 = [&](int64_t c) { return (int)((c - seg_lo) * kMmaChunk); };
        auto issue = [&](int buf, int64_t c) {
            const int t0 = tok0(c);
            const int n = min(kMmaChunk, L - t0);
            const uint32_t dk = stage_s + buf * kWarpStage, dv = dk + kKStage;
            const int nk = (n * kKB4 + 15) >> 4, nvb = (n * kVB2 + 15) >> 4;
            const uint8_t *sk = kbase + (int64_t)t0 * kKB4, *sv = vbase + (int64_t)t0 * kVB2;
            for (int q = lane; q < kKStage / 16; q += 32) cp16_zfill(dk + 16 * q, q < nk ? sk + 16 * q : kbase, q < nk);
            for (int q = lane; q < kVStage / 16; q += 32) cp16_zfill(dv + 16 * q, q < nvb ? sv + 16 * q : vbase, q < nvb);
        };

        float o[8][4];
#pragma unroll
        for (int m = 0; m < 8; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
        float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};

        // this warp's chunks: x + warp, x + warp + 8, ... below xe and with tokens left (t0 < L)
        int64_t c = x + warp;
        auto live = [&](int64_t cc) { return cc < xe && tok0(cc) < L; };
        if (live(c)) issue(0, c);
        cp_async_commit();
        for (int it = 0; live(c); ++it, c += kW) {
            if (live(c + kW)) issue((it + 1) & 1, c + kW);
            cp_async_commit();
            cp_async_wait<1>();
            __syncwarp();
            const int nvalid = min(kMmaChunk, L - tok0(c));
            const uint32_t ks_s = stage_s + (it & 1) * kWarpStage, vs_s = ks_s + kKStage;

            // ---- scores for 2 tiles of 16 tokens (rows g, g + 8); four independent MMA chains
            uint32_t cw[2][2][4];                 // [tile][row half][word]
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) lds_words_a2<4>(ks_s + (16 * mt + g + 8 * rh) * kKB4 + 2 + 16 * t, cw[mt][rh]);
            float acc[2][2][4];                   // [tile][k-step parity][fragment]
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int par = 0; par < 2; ++par) acc[mt][par][0] = acc[mt][par][1] = acc[mt][par][2] = acc[mt][par][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t s0 = 0x4440u + 2 * (ks & 1), s1 = s0 + 1;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const uint32_t wa = cw[mt][0][ks >> 1], wb = cw[mt][1][ks >> 1];
                    const uint32_t a0 = lds32(lut_s + prmt(wa, 0, s0) * 128u);
                    const uint32_t a2 = lds32(lut_s + prmt(wa, 0, s1) * 128u);
                    const uint32_t a1 = lds32(lut_s + prmt(wb, 0, s0) * 128u);
                    const uint32_t a3 = lds32(lut_s + prmt(wb, 0, s1) * 128u);
                    mma16816(acc[mt][ks & 1], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
            }
            float s[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int ta = 16 * mt + g, tb = ta + 8;
                const float na = __half2float(__ushort_as_half((unsigned short)lds_u16(ks_s + ta * kKB4)));
                const float nb = __half2float(__ushort_as_half((unsigned short)lds_u16(ks_s + tb * kKB4)));
                s[mt][0] = ta < nvalid ? (acc[mt][0][0] + acc[mt][1][0]) * na : -INFINITY;
                s[mt][1] = ta < nvalid ? (acc[mt][0][1] + acc[mt][1][1]) * na : -INFINITY;
                s[mt][2] = tb < nvalid ? (acc[mt][0][2] + acc[mt][1][2]) * nb : -INFINITY;
                s[mt][3] = tb < nvalid ? (acc[mt][0][3] + acc[mt][1][3]) * nb : -INFINITY;
            }
            // ---- online softmax for heads 2t (cols 0, 2) and 2t + 1 (cols 1, 3)
            float mx[2] = {fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2])),
                           fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]))};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], off));
            float corr[2];
            bool moved = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float mn = fmaxf(mrun[h], mx[h]);
                moved |= mn != mrun[h];
                corr[h] = mn == -INFINITY ? 1.f : exp2f(mrun[h] - mn);
                mrun[h] = mn;
                lrun[h] *= corr[h];
            }
            if (__any_sync(kFull, moved)) {   // the running max rarely moves once it has settled
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    o[m][0] *= corr[0];
                    o[m][1] *= corr[1];
                    o[m][2] *= corr[0];
                    o[m][3] *= corr[1];
                }
            }
            // ---- P (times the value norm) and P V for each 16-token tile
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                float p[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float mm = mrun[jj & 1];
                    p[jj] = mm == -INFINITY ? 0.f : exp2f(s[mt][jj] - mm);
                }
                lrun[0] += p[0] + p[2];
                lrun[1] += p[1] + p[3];
                const int ta = 16 * mt + g, tb = ta + 8;
                const float nva = __half2float(__ushort_as_half((unsigned short)lds_u16(vs_s + ta * kVB2)));
                const float nvb = __half2float(__ushort_as_half((unsigned short)lds_u16(vs_s + tb * kVB2)));
                const uint32_t b0 = movmatrix_trans(pack_half2(p[0] * nva, p[1] * nva));
                const uint32_t b1 = movmatrix_trans(pack_half2(p[2] * nvb, p[3] * nvb));
                // value codes of tokens 2t, 2t+1, 2t+8, 2t+9 of the tile: dims 16g..16g+15
                uint32_t w0[1], w1[1], w2[1], w3[1];
                lds_words_a2<1>(vs_s + (16 * mt + 2 * t) * kVB2 + 2 + 4 * g, w0);
                lds_words_a2<1>(vs_s + (16 * mt + 2 * t + 1) * kVB2 + 2 + 4 * g, w1);
                lds_words_a2<1>(vs_s + (16 * mt + 2 * t + 8) * kVB2 + 2 + 4 * g, w2);
                lds_words_a2<1>(vs_s + (16 * mt + 2 * t + 9) * kVB2 + 2 + 4 * g, w3);
                // interleave the two tokens of each register: bytes [A0, B0, A1, B1] / [A2, B2, A3, B3]
                const uint32_t x01 = prmt(w0[0], w1[0], 0x5140u), x23 = prmt(w0[0], w1[0], 0x7362u);
                const uint32_t y01 = prmt(w2[0], w3[0], 0x5140u), y23 = prmt(w2[0], w3[0], 0x7362u);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    // m-tile m: row g <-> dim 16g + 2m, row g + 8 <-> dim 16g + 2m + 1
                    const int j0 = 2 * m, j1 = 2 * m + 1;
                    const uint32_t xs = (j0 < 8) ? x01 : x23, ys = (j0 < 8) ? y01 : y23;
                    const int sh0 = 16 * ((j0 >> 2) & 1) + 2 * (j0 & 3), sh1 = 16 * ((j1 >> 2) & 1) + 2 * (j1 & 3);
                    const uint32_t a0 = prmt(vlo, vhi, ((xs >> sh0) & 0x0303u) * 0x11u + 0x4040u);
                    const uint32_t a1 = prmt(vlo, vhi, ((xs >> sh1) & 0x0303u) * 0x11u + 0x4040u);
                    const uint32_t a2 = prmt(vlo, vhi, ((ys >> sh0) & 0x0303u) * 0x11u + 0x4040u);
                    const uint32_t a3 = prmt(vlo, vhi, ((ys >> sh1) & 0x0303u) * 0x11u + 0x4040u);
                    mma16816(o[m], a0, a1, a2, a3, b0, b1);
                }
            }
            __syncwarp();
        }
        cp_async_wait<0>();

        // ---- merge the eight warps (rounds: 4 -> 2 -> 1), then warp 0 writes the partials
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) lrun[h] += __shfl_xor_sync(kFull, lrun[h], off);
#pragma unroll
        for (int half = kW / 2; half >= 1; half >>= 1) {
            __syncthreads();
            if (warp >= half && warp < 2 * half) {
                float *mw = merge + (warp - half) * kMergeSlot;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int d0 = 16 * g + 2 * m;
                    mw[(2 * t) * 132 + 4 + d0] = o[m][0];
                    mw[(2 * t + 1) * 132 + 4 + d0] = o[m][1];
                    mw[(2 * t) * 132 + 4 + d0 + 1] = o[m][2];
                    mw[(2 * t + 1) * 132 + 4 + d0 + 1] = o[m][3];
                }
                if (g == 0) {
                    mw[(2 * t) * 132] = mrun[0];
                    mw[(2 * t) * 132 + 1] = lrun[0];
                    mw[(2 * t + 1) * 132] = mrun[1];
                    mw[(2 * t + 1) * 132 + 1] = lrun[1];
                }
            }
            __syncthreads();
            if (warp < half) {
                const float *mw = merge + warp * kMergeSlot;
                float fs[2], fo[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float mo = mw[(2 * t + h) * 132], lo2 = mw[(2 * t + h) * 132 + 1];
                    const float M = fmaxf(mrun[h], mo);
                    fs[h] = mrun[h] == -INFINITY ? 0.f : exp2f(mrun[h] - M);
                    fo[h] = mo == -INFINITY ? 0.f : exp2f(mo - M);
                    lrun[h] = lrun[h] * fs[h] + lo2 * fo[h];
                    mrun[h] = M;
                }
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int d0 = 16 * g + 2 * m;
                    o[m][0] = o[m][0] * fs[0] + mw[(2 * t) * 132 + 4 + d0] * fo[0];
                    o[m][1] = o[m][1] * fs[1] + mw[(2 * t + 1) * 132 + 4 + d0] * fo[1];
                    o[m][2] = o[m][2] * fs[0] + mw[(2 * t) * 132 + 4 + d0 + 1] * fo[0];
                    o[m][3] = o[m][3] * fs[1] + mw[(2 * t + 1) * 132 + 4 + d0 + 1] * fo[1];
                }
            }
        }
        if (warp == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int head = 2 * t + h;
                if (head < a.G) {
                    float *pr = a.ws + (((int64_t)b * a.Hq + kvh * a.G + head) * plan.Smax + slot) * kPartialFloats;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int d0 = 16 * g + 2 * m;
                        pr[4 + d0] = o[m][h];
                        pr[4 + d0 + 1] = o[m][2 + h];
                    }
                    if (g == 0) {
                        pr[0] = mrun[h];
                        pr[1] = lrun[h];
                    }
                }
            }
        }
        x = xe;
    }
}

}  // namespace

MmaPlan mma_plan(int B, int Hkv, int T) {
    MmaPlan p;
    p.C = (T + kMmaChunk - 1) / kMmaChunk;
    p.Ctot = (int64_t)B * Hkv * p.C;
    p.P = (int)min64(p.Ctot, kMmaCtas);
    const int64_t segs = (int64_t)B * Hkv;
    p.Smax = (int)((p.P + segs - 1) / segs) + 1;
    return p;
}

bool attn_mma_supported(int kb, int vb, bool qjl) { return kb == 4 && vb == 2 && !qjl; }

int launch_attn_mma(const AttnArgs &a, const MmaPlan &plan, cudaStream_t st) {
    static int done[64] = {0};
    if (set_smem_limit((const void *)attn_mma_k4v2_kernel, kSmemTotal, done) != TQ_OK) return TQ_ERR_CUDA;
    attn_mma_k4v2_kernel<<<plan.P, kThreadsMma, kSmemTotal, st>>>(a, plan);
    return launch_status();
}

}  // namespace tq
