// Quantise-on-insert (tq_encode_kv) for sm_103a.
//
// Restates "TurboQuant KV Cache Compression — Spec": As-Built Notes (random
// signs before the Walsh-Hadamard transform, H (D x); normalise by the L2
// norm), Algorithm Detail Step 2 (level index from the boundaries) and
// Step 3 (bit packing); and "TurboQuant KV Cache (turboq2 / turboq3 /
// turboq4)" section 4 (block = fp16 norm + packed codes).
//
// Work split: two threads own one 128-element vector, 64 elements each.
// Thread h of a pair reads the 16-byte chunks 2c + h (c = 0..7) of its row
// straight into registers (each 32-byte sector is consumed by one pair in
// one instruction); it therefore holds elements e = 16c + 8h + k, k = 0..7.
// The next tile's rows are loaded while the current tile is processed.
//   * Six of the seven butterfly stages (element-index bits 0-2 and 4-6) run
//     in registers on packed float2 pairs; the stage on bit 3 is one full
//     exchange with the partner thread (shfl.xor 1) and one packed FMA with a
//     per-thread sign, which leaves both threads with exact butterfly
//     outputs (no role-dependent selects).
//   * The norm comes from a float32 sum of squares; when it falls within
//     2^-20 of an fp16 rounding boundary it is recomputed exactly
//     (double-float), and tiny/huge vectors (sum of squares outside
//     [2^-100, 2^100]) are rescaled by an exact power of two first.
//   * Quantisation never divides by the norm: u (u = H D x) is scaled once
//     to G y (y = u / (sqrt(128) n)), G chosen so that no cell of width 1
//     holds two boundaries; adding 64 + 1.5 * 2^20 rounds G y + 64 to a
//     multiple of 1/8 whose integer part (the cell index, cells
//     [j - 1/16, j + 15/16)) times 8 is bits 3..9 of the float, i.e. the byte
//     offset of the cell's 8-byte entry after one AND.  The 128-entry table
//     gives the cell's count of boundaries below it and the boundary inside
//     it, and one comparison finishes #{i : b_i <= y} (3- and 4-bit).  The
//     2-bit code is three comparisons against -b, 0, +b (scaled by
//     sqrt(128) n) in the float32 kernel.
//   * Codes are packed per 8 elements and written into a shared-memory block
//     tile, which the CTA stores with coalesced 16-byte stores (or block by
//     block for strided / scattered destinations).

#include <algorithm>
#include <cmath>
#include <cstring>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {
namespace {

constexpr int kEncThreads = 128;
constexpr int kEncVecs = kEncThreads / 2;  // vectors per tile
constexpr int kBuckets = 128;
constexpr unsigned kFull = 0xffffffffu;

struct EncArgs {
    const uint8_t *x;
    const uint8_t *x2;  // paired encode: the rows whose blocks fill the second half of each slot
    int64_t n_vec;
    int64_t x_stride;   // bytes
    uint8_t *out;
    int64_t out_stride; // bytes
    const int64_t *dst_index;
    int contiguous;
    int idx_bulk;       // destination indices into contiguous, 16-byte aligned slots: runs may leave in bulk
    float b0;           // 2-bit: the positive boundary
    float grid;         // 3/4-bit: cells per unit of y
    float2 table[kBuckets];  // cell j: (boundary inside it in G*y units | +inf, bits of #boundaries below it)
    uint32_t signs[4];
    int drop;           // test hook: the tensor-core kernel issues no TMA loads (its waits run out)
};

// Raw 64-element share of a row, as loaded (16-bit inputs: 8 chunks;
// float32: 16 chunks).
template <int DT>
struct Raw {
    uint4 r[DT == TQ_F32 ? 16 : 8];
};

template <int DT>
__device__ __forceinline__ void load_raw(Raw<DT> &raw, const uint8_t *row, bool valid, int h) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        if constexpr (DT == TQ_F32) {
            const uint4 *p = reinterpret_cast<const uint4 *>(row + (2 * c + h) * 32);
            raw.r[2 * c] = valid ? __ldcs(p) : make_uint4(0, 0, 0, 0);
            raw.r[2 * c + 1] = valid ? __ldcs(p + 1) : make_uint4(0, 0, 0, 0);
        } else {
            const uint4 *p = reinterpret_cast<const uint4 *>(row + (2 * c + h) * 16);
            raw.r[c] = valid ? __ldcs(p) : make_uint4(0, 0, 0, 0);
        }
    }
}

// Sign-flipped values as pairs p[c'][k] = (e(c', k), e(c' + 4, k)) with
// e(c, k) = element 16c + 8h + k.
template <int DT>
__device__ __forceinline__ void to_pairs(const Raw<DT> &raw, const uint32_t *sg16, const uint32_t *sg32, int h,
                                         float2 (&p)[4][8]) {
    float v[8][8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        if constexpr (DT == TQ_F32) {
            const uint4 s0 = reinterpret_cast<const uint4 *>(sg32 + 16 * c + 8 * h)[0];
            const uint4 s1 = reinterpret_cast<const uint4 *>(sg32 + 16 * c + 8 * h)[1];
            const uint4 a = raw.r[2 * c], b = raw.r[2 * c + 1];
            v[c][0] = __uint_as_float(a.x ^ s0.x);
            v[c][1] = __uint_as_float(a.y ^ s0.y);
            v[c][2] = __uint_as_float(a.z ^ s0.z);
            v[c][3] = __uint_as_float(a.w ^ s0.w);
            v[c][4] = __uint_as_float(b.x ^ s1.x);
            v[c][5] = __uint_as_float(b.y ^ s1.y);
            v[c][6] = __uint_as_float(b.z ^ s1.z);
            v[c][7] = __uint_as_float(b.w ^ s1.w);
        } else {
            const uint4 s = reinterpret_cast<const uint4 *>(sg16 + 8 * c + 4 * h)[0];
            const uint32_t w[4] = {raw.r[c].x ^ s.x, raw.r[c].y ^ s.y, raw.r[c].z ^ s.z, raw.r[c].w ^ s.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if constexpr (DT == TQ_BF16) {
                    v[c][2 * m] = bf16_bits_lo(w[m]);
                    v[c][2 * m + 1] = bf16_bits_hi(w[m]);
                } else {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[m]));
                    v[c][2 * m] = f.x;
                    v[c][2 * m + 1] = f.y;
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < 8; ++k) p[c][k] = make_float2(v[c][k], v[c + 4][k]);
}

// 0xFFFFFFFF when a >= b, else 0 (one set instruction).
__device__ __forceinline__ uint32_t set_ge(float a, float b) {
    uint32_t r;
    asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

// 8-byte shared-memory load at a 32-bit shared address.
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ float sumsq_pairs(const float2 (&p)[4][8]) {
    float2 acc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = __fmul2_rn(p[c][0], p[c][0]);
#pragma unroll
    for (int k = 1; k < 8; ++k)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = __ffma2_rn(p[c][k], p[c][k], acc[c]);
    acc[0] = __fadd2_rn(acc[0], acc[1]);
    acc[2] = __fadd2_rn(acc[2], acc[3]);
    acc[0] = __fadd2_rn(acc[0], acc[2]);
    return acc[0].x + acc[0].y;
}

template <int BITS, int DT>
__global__ void __launch_bounds__(kEncThreads, 3) encode_kernel(const __grid_constant__ EncArgs a) {
    constexpr int L = 1 << BITS, H = L / 2, BB = BlockFmt<BITS>::kBytes;
    __shared__ __align__(16) uint32_t sg16[64];
    __shared__ __align__(16) uint32_t sg32[128];
    __shared__ __align__(16) float2 tab[kBuckets];
    __shared__ __align__(16) uint8_t sm_out[(kEncVecs * BB + 15) & ~15];

    for (int j = threadIdx.x; j < kD; j += kEncThreads) sg32[j] = ((a.signs[j >> 5] >> (j & 31)) & 1u) << 31;
    for (int w = threadIdx.x; w < 64; w += kEncThreads) {
        const int j = 2 * w;
        sg16[w] = (((a.signs[j >> 5] >> (j & 31)) & 1u) << 15) | (((a.signs[j >> 5] >> ((j + 1) & 31)) & 1u) << 31);
    }
    for (int j = threadIdx.x; j < kBuckets; j += kEncThreads) tab[j] = a.table[j];
    __syncthreads();

    const int pv = threadIdx.x >> 1, h = threadIdx.x & 1;
    const float sgn = h ? -1.f : 1.f;
    const int64_t ntiles = (a.n_vec + kEncVecs - 1) / kEncVecs;
    int64_t tile = blockIdx.x;
    Raw<DT> raw;
    if (tile < ntiles) {
        const int64_t row = tile * kEncVecs + pv;
        load_raw<DT>(raw, a.x + row * a.x_stride, row < a.n_vec, h);
    }
    for (; tile < ntiles; tile += gridDim.x) {
        const int64_t v0 = tile * kEncVecs;
        const int nv = (int)min64(kEncVecs, a.n_vec - v0);
        float2 p[4][8];
        to_pairs<DT>(raw, sg16, sg32, h, p);
        const int64_t next = tile + gridDim.x;
        if (next < ntiles) {
            const int64_t row = next * kEncVecs + pv;
            load_raw<DT>(raw, a.x + row * a.x_stride, row < a.n_vec, h);
        }

        // ---- norm
        float ss = sumsq_pairs(p);
        ss += __shfl_xor_sync(kFull, ss, 1);
        const bool out_of_range = !(ss >= 7.888609052210118e-31f && ss <= 1.2676506002282294e30f);
        float n = sqrtf(ss);
        unsigned short n16 = __half_as_ushort(__float2half_rn(n));
        const bool near = !out_of_range && near_fp16_tie(n, 9.5367431640625e-07f /* 2^-20 */);
        if (__any_sync(kFull, near)) {
            // exact: double-float sums of squares of both halves, one rounding
            SumSq2 acc;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    acc.add(p[c][k].x);
                    acc.add(p[c][k].y);
                }
            const float os = __shfl_xor_sync(kFull, acc.s, 1), oc = __shfl_xor_sync(kFull, acc.c, 1);
            SumSq2 tot;
            two_sum(acc.s, os, tot.s, tot.c);
            tot.c += acc.c + oc;
            if (near) n16 = tot.sqrt_fp16();
        }
        if (__any_sync(kFull, out_of_range)) {
            // tiny, huge or zero vector: norm in double, values rescaled by 2^-e
            double sd = 0.0;
            float amax = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    sd = fma((double)p[c][k].x, (double)p[c][k].x, sd);
                    sd = fma((double)p[c][k].y, (double)p[c][k].y, sd);
                    amax = fmaxf(amax, fmaxf(fabsf(p[c][k].x), fabsf(p[c][k].y)));
                }
            sd += __shfl_xor_sync(kFull, sd, 1);
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            if (out_of_range) {
                n16 = __half_as_ushort(__double2half(sqrt(sd)));
                if (amax > 0.f) {
                    int e;
                    frexpf(amax, &e);
                    const int e1 = -e / 2, e2 = -e - e1;
                    const float2 f1 = make_float2(ldexpf(1.f, e1), ldexpf(1.f, e1));
                    const float2 f2 = make_float2(ldexpf(1.f, e2), ldexpf(1.f, e2));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int k = 0; k < 8; ++k) p[c][k] = __fmul2_rn(__fmul2_rn(p[c][k], f1), f2);
                }
            }
            float s2 = sumsq_pairs(p);
            s2 += __shfl_xor_sync(kFull, s2, 1);
            if (out_of_range) n = sqrtf(s2);
        }

        // ---- transform and quantise
        fwht_pair128(p, sgn);
        const float sc = n > 0.f ? n * 11.313708498984761f : 1.f;  // sqrt(128) n
        uint8_t *blk = sm_out + pv * BB;
        if constexpr (BITS == 2) {
            const float t = a.b0 * sc;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t w = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float u = cc < 4 ? p[cc][k].x : p[cc - 4][k].y;
                    // code = [u >= -t] + [u >= 0] + [u >= t]; set.ge gives -1 / 0
                    const uint32_t m = set_ge(u, -t) + set_ge(u, 0.f) + set_ge(u, t);
                    w -= m << (2 * k);
                }
                *reinterpret_cast<uint16_t *>(blk + 2 + 4 * cc + 2 * h) = (uint16_t)w;
            }
        } else {
            const float cs = a.grid / sc;
            const float2 cs2 = make_float2(cs, cs);
            const float2 off2 = make_float2(1572928.f, 1572928.f);  // 64 + 1.5 * 2^20
            const uint32_t tab_base = (uint32_t)__cvta_generic_to_shared(tab);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t wx = 0, wy = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 yp = __fmul2_rn(p[cc][k], cs2);
                    const float2 t = __fadd2_rn(yp, off2);
                    const float2 ex = lds_f2(tab_base + (__float_as_uint(t.x) & 0x3F8u));
                    const float2 ey = lds_f2(tab_base + (__float_as_uint(t.y) & 0x3F8u));
                    const uint32_t cx = __float_as_uint(ex.y) - set_ge(yp.x, ex.x);
                    const uint32_t cy = __float_as_uint(ey.y) - set_ge(yp.y, ey.x);
                    wx += cx << (4 * k);
                    wy += cy << (4 * k);
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c8 = cc + 4 * half;
                    const uint32_t w = half ? wy : wx;
                    if constexpr (BITS == 4) {
                        uint16_t *d = reinterpret_cast<uint16_t *>(blk + 2 + 8 * c8 + 4 * h);
                        d[0] = (uint16_t)w;
                        d[1] = (uint16_t)(w >> 16);
                    } else {
                        // split the 8 nibble-held 3-bit codes into the 2-bit and 1-bit planes
                        uint32_t lo = w & 0x33333333u;
                        lo = (lo | (lo >> 2)) & 0x0F0F0F0Fu;
                        lo = (lo | (lo >> 4)) & 0x00FF00FFu;
                        lo = (lo | (lo >> 8)) & 0x0000FFFFu;
                        uint32_t hi = (w >> 2) & 0x11111111u;
                        hi = (hi | (hi >> 3)) & 0x03030303u;
                        hi = (hi | (hi >> 6)) & 0x000F000Fu;
                        hi = (hi | (hi >> 12)) & 0x000000FFu;
                        *reinterpret_cast<uint16_t *>(blk + 2 + 4 * c8 + 2 * h) = (uint16_t)lo;
                        blk[34 + 2 * c8 + h] = (uint8_t)hi;
                    }
                }
            }
        }
        if (h == 0) *reinterpret_cast<uint16_t *>(blk) = n16;
        __syncthreads();

        // ---- store the tile
        if (a.contiguous) {
            uint8_t *dst = a.out + v0 * BB;
            const int nbytes = nv * BB, nch = nbytes >> 4;
            for (int c = threadIdx.x; c < nch; c += kEncThreads)
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(sm_out)[c];
            for (int q = (nch << 3) + threadIdx.x; q < (nbytes >> 1); q += kEncThreads)
                reinterpret_cast<uint16_t *>(dst)[q] = reinterpret_cast<const uint16_t *>(sm_out)[q];
        } else {
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            for (int r = warp * 16; r < min(nv, warp * 16 + 16); ++r) {
                const int64_t di = a.dst_index ? a.dst_index[v0 + r] : (v0 + r);
                uint16_t *d = reinterpret_cast<uint16_t *>(a.out + di * a.out_stride);
                const uint16_t *s = reinterpret_cast<const uint16_t *>(sm_out + r * BB);
                for (int q = lane; q < BB / 2; q += 32) d[q] = s[q];
            }
        }
        __syncthreads();
    }
}


// ---------------------------------------------------------------------------
// Tensor-core variant for bf16 / fp16 inputs.
//
// H_128 = H_8 (x) H_16 in Sylvester order (element e = 16 i + j), so
// u = H (D x) splits into a 16-point transform of each 16-element chunk c
// (with the chunk's signs folded in) followed by an 8-point transform across
// the chunks.  The first is a dense contraction: for 16 vectors at a time,
// [16 vectors x 16 dims] x [16 dims x 16 outputs] per chunk, exact in one
// mma.sync m16n8k16 (bf16/fp16 inputs times +-1, float32 accumulate).  The
// A operand comes straight from the staged bf16 rows with ldmatrix (rows
// padded to 272 bytes, conflict-free); the B operand (+-1 = H_16 D_c with
// its output columns permuted so that thread t of a quad ends with outputs
// 4t..4t+3) lives in registers.  The 8-point stage runs on the accumulator
// registers, which already come in float2 pairs.
// ---------------------------------------------------------------------------

constexpr int kPlainPitch = 272;           // 256-byte bf16 row + 16-byte pad
constexpr int kRowPitch = kPlainPitch;
constexpr int kWarpRows = 16;               // vectors per warp tile
constexpr int kWarpStage = kWarpRows * kRowPitch;

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d = a * b (fresh accumulator: the C operand is a zero register).
template <int DT>
__device__ __forceinline__ void mma_16816_zero(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    if constexpr (DT == TQ_BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
    }
}

template <int DT>
__device__ __forceinline__ float elem_smem(const uint8_t *row, int j) {
    const uint16_t b = reinterpret_cast<const uint16_t *>(row)[j];
    if constexpr (DT == TQ_BF16) return __uint_as_float((uint32_t)b << 16);
    else return __half2float(__ushort_as_half(b));
}

// Element j of row r of a staged tile: SW = false: rows of kPlainPitch bytes;
// SW = true: the tensor-core layout of a 128-row tile (two 64-column blocks
// of 16 KB, 128-byte rows whose 16-byte chunks are XOR-swizzled by the row's
// position in its 8-row group).
template <int DT, bool SW>
__device__ __forceinline__ float elem_at(const uint8_t *base, int r, int j) {
    if constexpr (SW) {
        const int off = (j >> 6) * 16384 + r * 128 + ((((j & 63) >> 3) ^ (r & 7)) << 4) + (j & 7) * 2;
        const uint16_t b = *reinterpret_cast<const uint16_t *>(base + off);
        if constexpr (DT == TQ_BF16) return __uint_as_float((uint32_t)b << 16);
        else return __half2float(__ushort_as_half(b));
    } else {
        return elem_smem<DT>(base + r * kPlainPitch, j);
    }
}

// fp16 of the L2 norm of row `row` (128 values of dtype DT in shared memory):
// double-float sum of squares over the quad (lane t sums 32t..32t+31), one
// rounding.  Every lane of the warp calls it (shuffles inside); out of line
// because the fast float32 norm needs it only near an fp16 rounding boundary.
template <int DT>
__device__ __noinline__ unsigned short exact_norm_quad(const uint8_t *row, int t) {
    SumSq2 part;
    for (int j = 32 * t; j < 32 * t + 32; ++j) part.add(elem_smem<DT>(row, j));
    float s1 = part.s, c1 = part.c;
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        const float os = __shfl_xor_sync(kFull, s1, o), oc = __shfl_xor_sync(kFull, c1, o);
        float ns, ne;
        two_sum(s1, os, ns, ne);
        s1 = ns;
        c1 = c1 + oc + ne;
    }
    SumSq2 tot;
    tot.s = s1;
    tot.c = c1;
    return tot.sqrt_fp16();
}

// Block of one row whose sum of squares leaves float32's safe range (tiny,
// huge or zero vectors), by one thread: norm from a double sum of the exact
// squares; the row scaled by an exact power of two (2^-e, e the exponent of
// its largest magnitude) so the float32 transform and the cell quantiser work
// in range (codes do not depend on the scale); a zero row gets code L/2
// everywhere.  Out of line: such rows essentially never occur.
template <int BITS, int DT, bool SW>
__device__ __noinline__ void encode_row_slow(const uint8_t *base, int r, const float2 *tab, float grid,
                                             const uint32_t (&signs)[4], uint8_t *blk) {
    constexpr int BB = BlockFmt<BITS>::kBytes;
    float v[kD];
    double sd = 0.0;
    float amax = 0.f;
    for (int j = 0; j < kD; ++j) {
        v[j] = elem_at<DT, SW>(base, r, j);
        sd = fma((double)v[j], (double)v[j], sd);
        amax = fmaxf(amax, fabsf(v[j]));
    }
    for (int j = 2; j < BB; ++j) blk[j] = 0;
    *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(__double2half(sqrt(sd)));
    uint32_t code[kD];
    if (!(amax > 0.f && amax < INFINITY)) {
        for (int j = 0; j < kD; ++j) code[j] = (1u << BITS) / 2;
    } else {
        int e;
        frexpf(amax, &e);
        for (int j = 0; j < kD; ++j) {
            const float x = ldexpf(v[j], -e);
            v[j] = ((signs[j >> 5] >> (j & 31)) & 1u) ? -x : x;
        }
        for (int L = 1; L < kD; L <<= 1)
            for (int j = 0; j < kD; ++j)
                if (!(j & L)) {
                    const float x = v[j], y = v[j + L];
                    v[j] = x + y;
                    v[j + L] = x - y;
                }
        float ss = 0.f;
        for (int j = 0; j < kD; ++j) ss = fmaf(v[j], v[j], ss);
        const float cs = grid / sqrtf(ss);
        for (int j = 0; j < kD; ++j) {
            const float yp = v[j] * cs;
            const float tt = yp + 1572928.f;   // 64 + 1.5 * 2^20
            const float2 ent = tab[(__float_as_uint(tt) & 0x3F8u) >> 3];
            code[j] = __float_as_uint(ent.y) + (yp >= ent.x ? 1u : 0u);
        }
    }
    for (int j = 0; j < kD; ++j) {
        if constexpr (BITS == 4) {
            blk[2 + j / 2] |= (uint8_t)(code[j] << (4 * (j & 1)));
        } else if constexpr (BITS == 2) {
            blk[2 + j / 4] |= (uint8_t)(code[j] << (2 * (j & 3)));
        } else {
            blk[2 + j / 4] |= (uint8_t)((code[j] & 3u) << (2 * (j & 3)));
            blk[34 + j / 8] |= (uint8_t)((code[j] >> 2) << (j & 7));
        }
    }
}

// Each warp is independent: it stages its own 16 rows (double buffered,
// cp.async with zero fill past the end), transforms and quantises them, and
// stores its own 16 blocks; warps never wait for each other.
template <int BITS, int DT>
__global__ void __launch_bounds__(kEncThreads, 4) encode_mma_kernel(const __grid_constant__ EncArgs a) {
    constexpr int BB = BlockFmt<BITS>::kBytes;
    constexpr int OUTB = (kWarpRows * BB + 15) & ~15;
    constexpr int WARP_SMEM = 2 * kWarpStage + OUTB;
    extern __shared__ __align__(16) uint8_t smem[];
    float2 *tab = reinterpret_cast<float2 *>(smem);                               // kBuckets entries
    uint4 *bfrag = reinterpret_cast<uint4 *>(smem + kBuckets * sizeof(float2));    // [8][32]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint8_t *wsm = smem + kBuckets * sizeof(float2) + 8 * 32 * sizeof(uint4) + warp * WARP_SMEM;
    uint8_t *sm_out = wsm + 2 * kWarpStage;

    for (int j = threadIdx.x; j < kBuckets; j += kEncThreads) tab[j] = a.table[j];
    // B fragments of lane l for chunk c: {nt0 k0-7, nt0 k8-15, nt1 k0-7, nt1 k8-15}; entry
    // (k, n) = H16[o][k] * D[16c + k] with output column o = 4 (n >> 1) + 2 nt + (n & 1).
    for (int q = threadIdx.x; q < 8 * 32; q += kEncThreads) {
        const int c = q >> 5, l = q & 31, lg = l >> 2, lt = l & 3;
        uint32_t w[4];
        for (int nt = 0; nt < 2; ++nt)
            for (int r = 0; r < 2; ++r) {
                const int o = 4 * (lg >> 1) + 2 * nt + (lg & 1);
                uint32_t pair = 0;
                for (int e = 0; e < 2; ++e) {
                    const int k = 2 * lt + 8 * r + e, dim = 16 * c + k;
                    const uint32_t neg = ((uint32_t)__popc(o & k) & 1u) ^ ((a.signs[dim >> 5] >> (dim & 31)) & 1u);
                    const uint32_t one = DT == TQ_BF16 ? (neg ? 0xBF80u : 0x3F80u) : (neg ? 0xBC00u : 0x3C00u);
                    pair |= one << (16 * e);
                }
                w[2 * nt + r] = pair;
            }
        bfrag[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();

    const int64_t ntiles = (a.n_vec + kWarpRows - 1) / kWarpRows;
    const int64_t nwarps = (int64_t)gridDim.x * (kEncThreads / 32);
    const uint32_t stage_s = (uint32_t)__cvta_generic_to_shared(wsm);
    auto issue = [&](int buf, int64_t tl) {
        const int64_t r0 = tl * kWarpRows;
        const uint32_t d0 = stage_s + buf * kWarpStage + (lane >> 4) * kRowPitch + (lane & 15) * 16;
        if (r0 + kWarpRows <= a.n_vec) {
            const uint8_t *s0 = a.x + (r0 + (lane >> 4)) * a.x_stride + (lane & 15) * 16;
            const int64_t step = 2 * a.x_stride;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d0 + i * 2 * kRowPitch),
                             "l"(s0 + i * step) : "memory");
        } else {
#pragma unroll
            for (int q = lane; q < kWarpRows * 16; q += 32) {
                const int r = q >> 4, col = q & 15;
                const bool valid = r0 + r < a.n_vec;
                const uint8_t *src = valid ? a.x + (r0 + r) * a.x_stride + col * 16 : a.x;
                cp_async16_zfill(stage_s + buf * kWarpStage + r * kRowPitch + col * 16, src, valid);
            }
        }
    };
    int64_t tile = (int64_t)blockIdx.x * (kEncThreads / 32) + warp;
    if (tile < ntiles) issue(0, tile);
    cp_async_commit();
    const float2 off2 = make_float2(1572928.f, 1572928.f);  // 64 + 1.5 * 2^20
    const uint32_t tab_s = (uint32_t)__cvta_generic_to_shared(tab);
    for (int it = 0; tile < ntiles; ++it, tile += nwarps) {
        const int64_t next = tile + nwarps;
        if (next < ntiles) issue((it + 1) & 1, next);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const int64_t v0 = tile * kWarpRows;
        const int nv = (int)min64(kWarpRows, a.n_vec - v0);
        const uint8_t *rows = wsm + (it & 1) * kWarpStage;
        const uint32_t lrow = stage_s + (it & 1) * kWarpStage + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kRowPitch +
                              (lane >> 4) * 16;

        // ---- 16-point stage on the tensor cores
        float acc[8][2][4];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t af[4];
            ldsm_x4(lrow + c * 32, af);
            const uint4 b = bfrag[c * 32 + lane];
            mma_16816_zero<DT>(acc[c][0], af, b.x, b.y);
            mma_16816_zero<DT>(acc[c][1], af, b.z, b.w);
        }
        // ---- 8-point stage across chunks, on the accumulator pairs
        float2 u[8][2][2];
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                u[c][nt][0] = make_float2(acc[c][nt][0], acc[c][nt][1]);
                u[c][nt][1] = make_float2(acc[c][nt][2], acc[c][nt][3]);
            }
#pragma unroll
        for (int L = 1; L < 8; L <<= 1)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                if ((c & L) == 0)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int vh = 0; vh < 2; ++vh) {
                            const float2 x = u[c][nt][vh], y = u[c + L][nt][vh];
                            u[c][nt][vh] = __fadd2_rn(x, y);
                            u[c + L][nt][vh] = sub2(x, y);
                        }
        // u[i][nt][vh] = (u_e, u_{e+1}), e = 16 i + 4 t + 2 nt, of row g + 8 vh.

        // ---- norms (sum of squares of u = 128 ||x||^2), one per row half
        float ss[2];
#pragma unroll
        for (int vh = 0; vh < 2; ++vh) {
            float2 q2 = __fmul2_rn(u[0][0][vh], u[0][0][vh]);
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    if (c | nt) q2 = __ffma2_rn(u[c][nt][vh], u[c][nt][vh], q2);
            float v = q2.x + q2.y;
            v += __shfl_xor_sync(kFull, v, 1);
            v += __shfl_xor_sync(kFull, v, 2);
            ss[vh] = v;
        }
        unsigned short n16[2];
        float sc[2];
        bool near[2], oor[2];
#pragma unroll
        for (int vh = 0; vh < 2; ++vh) {
            oor[vh] = !(ss[vh] >= 1.0097419586828951e-28f /* 128 * 2^-100 */ && ss[vh] <= 1.2676506002282294e30f);
            sc[vh] = sqrtf(ss[vh]);
            const float n = sc[vh] * 0.08838834764831845f;
            n16[vh] = __half_as_ushort(__float2half_rn(n));
            near[vh] = near_fp16_tie_fast(n);
        }
        if (__any_sync(kFull, near[0] || near[1])) {
            // exact norms (double-float sums of the staged rows, one rounding to fp16);
            // lane t of the quad sums elements 32t..32t+31
#pragma unroll
            for (int vh = 0; vh < 2; ++vh) {
                if (!__any_sync(kFull, near[vh])) continue;
                const unsigned short ex = exact_norm_quad<DT>(rows + (g + 8 * vh) * kRowPitch, t);
                if (near[vh]) n16[vh] = ex;
            }
        }
        // ---- quantise and pack (four consecutive elements per thread and 16-block)
#pragma unroll
        for (int vh = 0; vh < 2; ++vh) {
            const float cs = a.grid / sc[vh];
            const float2 cs2 = make_float2(cs, cs);
            uint8_t *blk = sm_out + (g + 8 * vh) * BB;
            uint32_t hnib[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t code4[4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float2 yp = __fmul2_rn(u[i][nt][vh], cs2);
                    const float2 tt = __fadd2_rn(yp, off2);
                    const float2 ex = lds_f2(tab_s + (__float_as_uint(tt.x) & 0x3F8u));
                    const float2 ey = lds_f2(tab_s + (__float_as_uint(tt.y) & 0x3F8u));
                    code4[2 * nt] = __float_as_uint(ex.y) + (yp.x >= ex.x ? 1u : 0u);
                    code4[2 * nt + 1] = __float_as_uint(ey.y) + (yp.y >= ey.x ? 1u : 0u);
                }
                if constexpr (BITS == 4) {
                    const uint32_t w = code4[0] + code4[1] * 16u + code4[2] * 256u + code4[3] * 4096u;
                    *reinterpret_cast<uint16_t *>(blk + 2 + 8 * i + 2 * t) = (uint16_t)w;
                } else if constexpr (BITS == 2) {
                    blk[2 + 4 * i + t] = (uint8_t)(code4[0] + code4[1] * 4u + code4[2] * 16u + code4[3] * 64u);
                } else {
                    blk[2 + 4 * i + t] = (uint8_t)((code4[0] & 3u) | ((code4[1] & 3u) << 2) | ((code4[2] & 3u) << 4) |
                                                   ((code4[3] & 3u) << 6));
                    hnib[i] = (code4[0] >> 2) | ((code4[1] >> 2) << 1) | ((code4[2] >> 2) << 2) | ((code4[3] >> 2) << 3);
                }
            }
            if constexpr (BITS == 3) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t other = __shfl_xor_sync(kFull, hnib[i], 1);
                    if ((t & 1) == 0) blk[34 + 2 * i + (t >> 1)] = (uint8_t)(hnib[i] | (other << 4));
                }
            }
            if (t == 0) *reinterpret_cast<uint16_t *>(blk) = n16[vh];
        }
        __syncwarp();
        if (__any_sync(kFull, oor[0] || oor[1])) {
            // rows outside float32's safe range: lane r (< 16) redoes row r on its own
            const bool o0 = __shfl_sync(kFull, oor[0], (lane & 7) * 4);   // row lane & 7
            const bool o1 = __shfl_sync(kFull, oor[1], (lane & 7) * 4);   // row 8 + (lane & 7)
            if (lane < kWarpRows && ((lane >> 3) ? o1 : o0))
                encode_row_slow<BITS, DT, false>(rows, lane, tab, a.grid, a.signs, sm_out + lane * BB);
            __syncwarp();
        }

        // ---- store this warp's 16 blocks (16 * BB bytes, 16-byte aligned when contiguous)
        if (a.contiguous) {
            uint8_t *dst = a.out + v0 * BB;
            const int nbytes = nv * BB, nch = nbytes >> 4;
            for (int c = lane; c < nch; c += 32)
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(sm_out)[c];
            for (int q = (nch << 3) + lane; q < (nbytes >> 1); q += 32)
                reinterpret_cast<uint16_t *>(dst)[q] = reinterpret_cast<const uint16_t *>(sm_out)[q];
        } else {
            for (int r = 0; r < nv; ++r) {
                const int64_t di = a.dst_index ? a.dst_index[v0 + r] : (v0 + r);
                uint16_t *d = reinterpret_cast<uint16_t *>(a.out + di * a.out_stride);
                const uint16_t *s2p = reinterpret_cast<const uint16_t *>(sm_out + r * BB);
                for (int q = lane; q < BB / 2; q += 32) d[q] = s2p[q];
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
}

template <int BITS, int DT>
int launch_mma(const EncArgs &a, cudaStream_t st) {
    static int per_sm[64] = {0};
    static int smem_set[64] = {0};
    const int smem = kBuckets * (int)sizeof(float2) + 8 * 32 * 16 +
                     (kEncThreads / 32) * (2 * kWarpStage + ((kWarpRows * BlockFmt<BITS>::kBytes + 15) & ~15));
    if (set_smem_limit((const void *)encode_mma_kernel<BITS, DT>, smem, smem_set) != TQ_OK) return TQ_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    int occ = dev < 64 ? per_sm[dev] : 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, encode_mma_kernel<BITS, DT>, kEncThreads, smem) !=
                cudaSuccess ||
            occ < 1)
            occ = 1;
        if (dev < 64) per_sm[dev] = occ;
    }
    const int64_t ntiles = (a.n_vec + kWarpRows - 1) / kWarpRows;
    const int64_t cta_tiles = (ntiles + (kEncThreads / 32) - 1) / (kEncThreads / 32);
    const int grid = (int)std::min<int64_t>(cta_tiles, (int64_t)occ * sm_count());
    encode_mma_kernel<BITS, DT><<<grid, kEncThreads, smem, st>>>(a);
    return launch_status();
}

template <int BITS, int DT>
int launch(const EncArgs &a, cudaStream_t st) {
    static int per_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    int occ = dev < 64 ? per_sm[dev] : 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, encode_kernel<BITS, DT>, kEncThreads, 0) !=
                cudaSuccess ||
            occ < 1)
            occ = 1;
        if (dev < 64) per_sm[dev] = occ;
    }
    const int64_t ntiles = (a.n_vec + kEncVecs - 1) / kEncVecs;
    const int grid = (int)std::min<int64_t>(ntiles, (int64_t)occ * sm_count());
    encode_kernel<BITS, DT><<<grid, kEncThreads, 0, st>>>(a);
    return launch_status();
}

// ---------------------------------------------------------------------------
// tcgen05 variant for bf16 / fp16 rows (the default path for them).
//
// The whole rotation u = H (D x) of 128 rows at a time is one dense
// contraction U[128 rows x 128] = X[128 x 128] * (H D)^T, exact on the 5th-
// generation tensor cores (bf16/fp16 inputs times +-1, float32 accumulate):
// the row tile arrives by TMA (two 64-column boxes, 128-byte swizzle) into
// shared memory, H D sits in shared memory in the same layout, eight
// tcgen05.mma (M 128, N 128, K 16) accumulate into tensor memory, and each
// of the 128 rows is read from tensor memory (tcgen05.ld) by two epilogue
// threads, one per 64-column half, and quantised: norm from the sum of
// squares (Parseval), then the cell-table quantiser of the mma.sync kernel
// over 16-column chunks re-read from tensor memory, codes packed straight
// into the row's block.  A full group of 32 blocks leaves by one bulk async
// copy.  Rows whose norm lies within 2^-20 of an fp16 rounding boundary, or
// whose sum of squares leaves float32's safe range, are listed and finished
// after the CTA's last tile from the rows in memory (correctly rounded norm;
// exact power-of-two rescaled path), which keeps calls out of the hot loop.
// One producer warp issues the TMA loads and the MMAs; two stages of row
// tiles and accumulators let the loads and MMAs of tile i + 1 run under the
// epilogue of tile i.  Every mbarrier wait is bounded.
// ---------------------------------------------------------------------------

constexpr int kTcRows = 128;                          // rows per tile = MMA M = tensor-memory lanes
constexpr int kTcEpiWarps = 8;                      // two per 32-row group: column halves
constexpr int kTcThreads = 32 * (kTcEpiWarps + 1);    // + one producer warp
constexpr int kTcTileBytes = kTcRows * 256;           // one row tile (two 16 KB column blocks)
constexpr uint32_t kTcCols = 256;                     // tensor-memory columns: two 128-column accumulators
constexpr int kTcFixCap = 240;                        // rows a CTA can list for finishing after its main loop

// PAIR: two row sets encoded into the two halves of 2 BB-byte slots (K then V
// block of a storage slot), tile i of both by the same CTA; one row-tile
// buffer (freed when the tile's MMAs complete) keeps two CTAs per SM.
template <int BITS, bool PAIR = false>
struct TcSmem {
    static constexpr int BB = 2 + 16 * BITS;
    static constexpr int kSlotB = PAIR ? 2 * BB : BB;                // bytes per output slot
    static constexpr int kABufs = PAIR ? 1 : 2;                       // row-tile buffers
    static constexpr int kB = 0;                                     // H D, 32 KB (1024-byte aligned)
    static constexpr int kA = kB + kTcTileBytes;                     // row tiles
    static constexpr int kOut = kA + kABufs * kTcTileBytes;          // 128 slots
    static constexpr int kTab = kOut + ((kTcRows * kSlotB + 15) & ~15);  // cell table, 128 x 8 B
    static constexpr int kPart = kTab + kBuckets * 8;                // per-row partial sums of squares, [2][128]
    static constexpr int kFix = kPart + 2 * kTcRows * 4;             // rows finished after the main loop
    static constexpr int kBars = kFix + (4 + kTcFixCap) * 4;          // full[2], mma[2], empty[2], drain
    static constexpr int kSlot = kBars + 7 * 8;                      // tensor-memory base address
    static constexpr int kTotal = kSlot + 16 + 1024;                 // + alignment slack of the base
};


// 16 consecutive float32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Wait for this thread's tensor-memory loads; v (their destination) is tied to
// the wait so no use of it is scheduled before it.
__device__ __forceinline__ void tc_wait_ld16(float (&v)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                   "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15])
                 :
                 : "memory");
}

// fp16 of the L2 norm of row r of a tensor-core row tile: double-float sum of
// the exact squares, one rounding (near an fp16 rounding boundary only).
template <int DT>
__device__ __noinline__ unsigned short exact_norm_row(const uint8_t *tile, int r) {
    SumSq2 acc;
    for (int j = 0; j < kD; ++j) acc.add(elem_at<DT, true>(tile, r, j));
    return acc.sqrt_fp16();
}

// Finish one listed row, by a whole warp, from its values in memory (the
// row tile is gone by then); lane j reads elements 4j .. 4j + 3 (16-bit
// rows).  A zero row gets the constant block (norm 0, code L/2 everywhere);
// a row outside float32's safe range (listed so, or, with `check`, 128
// ||x||^2 outside [2^-92, 2^99], a superset of the rows the main loop sends
// to the exact path) gets its whole block from the exact path; any other row
// gets the correctly rounded norm (double-float sum of squares).
template <int BITS, int DT>
__device__ __forceinline__ void finish_row_warp(const EncArgs &a, const float2 *tab, int64_t v, bool whole, bool check,
                                                int lane, int half = 0) {
    static_assert(DT != TQ_F32, "16-bit rows");
    constexpr int BB = BlockFmt<BITS>::kBytes;
    const uint8_t *xrow = (half ? a.x2 : a.x) + v * a.x_stride;
    const uint2 raw = *reinterpret_cast<const uint2 *>(xrow + 8 * lane);
    const uint32_t h[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
    SumSq2 acc;
    bool nz = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float f = DT == TQ_BF16 ? __uint_as_float(h[k] << 16) : __half2float(__ushort_as_half((unsigned short)h[k]));
        acc.add(f);
        nz |= f != 0.f;   // true for NaN as well
    }
    float s1 = acc.s, c1 = acc.c;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float os = __shfl_xor_sync(kFull, s1, o), oc = __shfl_xor_sync(kFull, c1, o);
        float ns, ne;
        two_sum(s1, os, ns, ne);
        s1 = ns;
        c1 = c1 + oc + ne;
    }
    const int64_t di = a.dst_index ? a.dst_index[v] : v;
    uint8_t *dst = a.out + di * a.out_stride + half * BB;
    if (!__any_sync(kFull, nz)) {
        const uint8_t fill = BITS == 4 ? 0x88 : BITS == 2 ? 0xAA : 0x00;   // code L/2 in every field
        for (int j = lane; j < BB; j += 32) dst[j] = j < 2 ? 0 : (BITS == 3 && j >= 34) ? 0xFF : fill;
        return;
    }
    if (check) {
        const float s128 = (s1 + c1) * 128.f;
        whole = !(s128 >= 2.0194839173657902e-28f /* 2^-92 */ && s128 <= 6.338253001141147e29f /* 2^99 */);
    }
    if (lane == 0) {
        if (whole) {
            encode_row_slow<BITS, DT, false>(xrow, 0, tab, a.grid, a.signs, dst);
        } else {
            SumSq2 tot;
            tot.s = s1;
            tot.c = c1;
            *reinterpret_cast<uint16_t *>(dst) = tot.sqrt_fp16();
        }
    }
}

template <int BITS, int DT, bool PAIR = false>
// two CTAs (2 x 288 threads) per SM; tmap2: the second row set (PAIR only)
__global__ void __launch_bounds__(kTcThreads, 2)
    encode_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap2,
                     const __grid_constant__ EncArgs a) {
    using S = TcSmem<BITS, PAIR>;
    constexpr int NH = PAIR ? 2 : 1;   // row sets per tile
    constexpr int BB = S::BB;
    __shared__ __align__(16) float2 s_tab[kBuckets];   // cell table at a fixed shared address
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // 1024-byte aligned base: the 128-byte swizzle is a function of address bits 4..9
    const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_s - raw_s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = base_s + S::kBars;   // full[s] at 8s, mma[s] at 16 + 8s, empty[s] at 32 + 8s

    // ---- setup: (H D) in the swizzled K-major layout, cell table, barriers, tensor memory
    for (int q = threadIdx.x; q < kTcRows * 16; q += kTcThreads) {
        const int n = q >> 4, kc = q & 15;   // row n of H D (an output of u), 8-column chunk kc
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
        const int off = S::kB + (kc >> 3) * 16384 + n * 128 + (((kc & 7) ^ (n & 7)) << 4);
        *reinterpret_cast<uint4 *>(smem + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    float2 *tab = s_tab;
    for (int j = threadIdx.x; j < kBuckets; j += kTcThreads) tab[j] = a.table[j];
    if (threadIdx.x == 0) {
#pragma unroll
        reinterpret_cast<int *>(smem + S::kFix)[0] = 0;   // listed rows
        reinterpret_cast<int *>(smem + S::kFix)[1] = 0;   // list overflowed
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(bars + 8 * i, 1);                 // full: the producer's arrival + the TMA bytes
            tc_mbar_init(bars + 16 + 8 * i, 1);            // mma: tcgen05.commit
            tc_mbar_init(bars + 32 + 8 * i, kTcEpiWarps);  // empty: one arrival per epilogue warp
        }
        tc_mbar_init(bars + 48, 1);                        // drain: the producer's last tcgen05.commit
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base_s + S::kSlot),
                     "r"(kTcCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // (H D) was written by ordinary stores and is read by the tensor cores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S::kSlot);

    const int64_t ntiles = (a.n_vec + kTcRows - 1) / kTcRows;
    if (warp == kTcEpiWarps) {
        // ---- producer: row tiles by TMA, then eight MMAs into the stage's accumulator
        if (lane == 0) {
            const uint32_t idesc = tc_idesc<DT>();
            // a wait that gives up is recorded and ends the producer's loop: no further load or
            // product is issued (the epilogue's waits then give up too, or are skipped)
            bool ok = true;
            auto wait = [&](uint32_t bar, uint32_t parity) {
                if (ok && !tc_mbar_wait(bar, parity)) {
                    ok = false;
                    note_wait_failed();
                }
            };
            int pend_bar = -1;   // full barrier of a load not yet seen complete, and its parity
            uint32_t pend_par = 0;
            int i = 0;
            for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x)
            for (int half = 0; ok && half < NH; ++half, ++i) {
                const int st = i & 1;
                const uint32_t use = (uint32_t)(i >> 1);
                if (i >= 2) wait(bars + 32 + 8 * st, (use - 1u) & 1u);   // stage released
                // PAIR: one row-tile buffer, free once the previous tile's MMAs have completed
                if (PAIR && i >= 1) wait(bars + 16 + 8 * (st ^ 1), (uint32_t)((i - 1) >> 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                const int ab = PAIR ? 0 : st;   // row-tile buffer and its full barrier
                const uint32_t a_s = base_s + S::kA + ab * kTcTileBytes, full = bars + 8 * ab;
                const CUtensorMap *map = (PAIR && half) ? &tmap2 : &tmap;
                const uint32_t fpar = PAIR ? ((uint32_t)i & 1u) : (use & 1u);
                if (!a.drop) {   // (test hook: no load, so the wait below runs out)
                    tc_mbar_expect_tx(full, kTcTileBytes);
                    tc_tma_load_2d(a_s, map, 0, (int)(tile * kTcRows), full);
                    tc_tma_load_2d(a_s + 16384, map, 64, (int)(tile * kTcRows), full);
                    pend_bar = ab;
                    pend_par = fpar;
                }
                wait(full, fpar);
                if (!ok) break;   // no product on a tile that did not land
                pend_bar = -1;
                const uint32_t d = tmem + (uint32_t)(st * 128);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32);
                    tc_mma(d, tc_desc_sw128(a_s + off), tc_desc_sw128(base_s + S::kB + off), idesc, ks > 0 ? 1u : 0u);
                }
                tc_commit(bars + 16 + 8 * st);
            }
            // before teardown: every product issued here has completed (one more commit, on a barrier
            // of its own), and a load whose wait gave up has landed (bounded waits)
            tc_commit(bars + 48);
            tc_mbar_wait(bars + 48, 0u);
            if (pend_bar >= 0) tc_mbar_wait(bars + 8 * pend_bar, pend_par);
        }
    } else {
        // ---- epilogue: warp w reads tensor-memory lanes (= tile rows) 32 (w & 3) .. + 31, columns
        // 64 hf .. + 63 (hf = w >> 2); the two warps of a row group meet on named barrier 1 + (w & 3)
        const int grp = warp & 3, hf = warp >> 2;
        const int r = 32 * grp + lane;
        const uint32_t pair_bar = 1u + (uint32_t)grp;
        float *part = reinterpret_cast<float *>(smem + S::kPart);
        int *fix = reinterpret_cast<int *>(smem + S::kFix);   // [0] count, [1] overflow, [4 ..] rows
        uint8_t *sm_out = smem + S::kOut;
        const uint32_t tab_s = (uint32_t)__cvta_generic_to_shared(s_tab);
        // full 32-block groups of a contiguous destination (or whose destination indices form one
        // aligned run) leave by one bulk copy each
        const bool bulk_out = a.contiguous != 0 || a.idx_bulk != 0;
        const float2 off2 = make_float2(1572928.f, 1572928.f);   // 64 + 1.5 * 2^20
        // a wait that gives up is recorded and not repeated: the loop still runs to its end (every
        // named barrier is met), on an accumulator that is then not valid
        bool ok = true;
        int i = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x)
        for (int half = 0; half < NH; ++half, ++i) {
            const int st = i & 1;
            if (ok && !tc_mbar_wait(bars + 16 + 8 * st, (uint32_t)(i >> 1) & 1u)) {
                ok = false;
                note_wait_failed();
            }
            tc_fence_after();
            const int64_t v0 = tile * kTcRows;
            const int nv = (int)min64(kTcRows, a.n_vec - v0);
            const int rows = max(0, min(32, nv - 32 * grp));
            // destination rows of this warp's group, requested now (one coalesced load) so that
            // the load is in flight during the quantiser
            int64_t my_di = 0;
            if (!a.contiguous)
                my_di = lane < rows ? (a.dst_index ? __ldg(a.dst_index + v0 + 32 * grp + lane) : v0 + 32 * grp + lane) : 0;
            const uint32_t taddr = tmem + ((uint32_t)(32 * grp) << 16) + (uint32_t)(st * 128 + 64 * hf);
            // ---- norm: sum of squares of u (= 128 ||x||^2), the two halves added in a fixed order
            float2 q2 = make_float2(0.f, 0.f);
            {
                float uu[2][32];
                tc_ld32(taddr, uu[0]);
                tc_ld32(taddr + 32, uu[1]);
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const float2 p2 = make_float2(uu[c][k], uu[c][k + 1]);
                        q2 = __ffma2_rn(p2, p2, q2);
                    }
            }
            part[hf * kTcRows + r] = q2.x + q2.y;
            // the previous tile's bulk store has read the group's blocks before they are rewritten
            if (bulk_out && hf == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            const float ss = part[r] + part[kTcRows + r];
            // ss == 0 is a zero row or one whose squares underflow: the accumulator (still held)
            // tells them apart; both warps of the pair see the same ss, so both take this branch
            bool zero_row = false;
            if (__any_sync(kFull, ss == 0.f)) {
                float z[2][32];
                tc_ld32(taddr, z[0]);
                tc_ld32(taddr + 32, z[1]);
                tc_wait_ld();
                bool nz = false;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) nz |= z[c][k] != 0.f;
                asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");   // partial sums read
                reinterpret_cast<int *>(part)[hf * kTcRows + r] = nz ? 1 : 0;
                asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
                zero_row = ss == 0.f && reinterpret_cast<int *>(part)[r] == 0 &&
                           reinterpret_cast<int *>(part)[kTcRows + r] == 0;
            }
            const bool oor = !zero_row && !(ss >= 1.0097419586828951e-28f /* 128 * 2^-100 */ && ss <= 1.2676506002282294e30f);
            const float sc = sqrtf(ss);
            const float nrm = sc * 0.08838834764831845f;
            uint8_t *blk = sm_out + r * S::kSlotB + half * BB;
            if (hf == 0) {
                *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(__float2half_rn(nrm));
                // rows whose norm lies within 2^-20 of an fp16 rounding boundary, or whose sum of
                // squares leaves float32's safe range, are listed and finished after the main loop
                const bool need = (oor || near_fp16_tie_fast(nrm)) && !zero_row && r < nv;
                const uint32_t m = __ballot_sync(kFull, need);
                if (m) {
                    const int leader = __ffs(m) - 1;
                    int base = 0;
                    if (lane == leader) base = atomicAdd(&fix[0], __popc(m));
                    base = __shfl_sync(kFull, base, leader);
                    if (need) {
                        const int slot = base + __popc(m & ((1u << lane) - 1u));
                        if (slot < kTcFixCap)
                            fix[4 + slot] = (int)(v0 + r) | (half ? 0x40000000 : 0) | (oor ? (int)0x80000000 : 0);
                        else fix[1] = 1;
                    }
                }
            }

            // ---- quantise and pack this half of the row's codes: code = base - [y >= boundary]
            // (set.ge gives 0 / -1), accumulated straight into the packed words
            const float cs = zero_row ? 0.f : a.grid / sc;   // a zero row: y = 0, code L/2
            const float2 cs2 = make_float2(cs, cs);
            uint16_t *b16 = reinterpret_cast<uint16_t *>(blk + 2);
            // codes per 16-bit word of the (low) plane; 3-bit codes are first gathered as nibbles, eight
            // to a word, and the word is then split into its 2-bit and 1-bit planes
            constexpr int PER = BITS == 4 ? 4 : 8;
            constexpr int B = BITS == 3 ? 4 : BITS;   // accumulation width of a code
            // 16 columns at a time, re-read from tensor memory (the next chunk's load in flight)
            float ub[2][16];
            tc_ld16(taddr, ub[0]);
            tc_wait_ld16(ub[0]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c < 3) tc_ld16(taddr + 16 * (c + 1), ub[(c + 1) & 1]);
                const float *u = ub[c & 1];
                const int cq = 4 * hf + c;   // 16-column chunk of the row
                uint32_t hi = 0;             // 3-bit: the 16 high bits of the chunk
#pragma unroll
                for (int g = 0; g < 16 / PER; ++g) {
                    uint32_t w = 0;
#pragma unroll
                    for (int e = 0; e < PER; e += 2) {
                        const int k = PER * g + e;
                        const float2 yp = __fmul2_rn(make_float2(u[k], u[k + 1]), cs2);
                        const float2 tt = __fadd2_rn(yp, off2);
                        const float2 ex = lds_f2(tab_s + (__float_as_uint(tt.x) & 0x3F8u));
                        const float2 ey = lds_f2(tab_s + (__float_as_uint(tt.y) & 0x3F8u));
                        w += __float_as_uint(ex.y) << (B * e);
                        w -= set_ge(yp.x, ex.x) << (B * e);
                        w += __float_as_uint(ey.y) << (B * e + B);
                        w -= set_ge(yp.y, ey.x) << (B * e + B);
                    }
                    if constexpr (BITS == 3) {
                        // low plane: bits 0-1 of nibble e to bits 2e, 2e + 1; high plane: bit 2 of nibble e to bit e
                        uint32_t lo = w & 0x33333333u;
                        lo = (lo | (lo >> 2)) & 0x0F0F0F0Fu;
                        lo = (lo | (lo >> 4)) & 0x00FF00FFu;
                        lo = (lo | (lo >> 8)) & 0x0000FFFFu;
                        uint32_t hb = (w >> 2) & 0x11111111u;
                        hb = (hb | (hb >> 3)) & 0x03030303u;
                        hb = (hb | (hb >> 6)) & 0x000F000Fu;
                        hb = (hb | (hb >> 12)) & 0x000000FFu;
                        b16[2 * cq + g] = (uint16_t)lo;
                        hi |= hb << (8 * g);
                    } else {
                        b16[(16 / PER) * cq + g] = (uint16_t)w;
                    }
                }
                if constexpr (BITS == 3) reinterpret_cast<uint16_t *>(blk + 34)[cq] = (uint16_t)hi;
                if (c < 3) tc_wait_ld16(ub[(c + 1) & 1]);
            }
            if (bulk_out) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // blocks -> bulk copy
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");   // both halves of the 32 blocks written

            // ---- release the stage (accumulator and row tile), then store the group's 32 blocks
            tc_fence_before();
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bars + 32 + 8 * st);
            // a run of 32 consecutive, 16-byte aligned destination slots goes out like a contiguous group
            int64_t di0 = v0 + 32 * grp;
            bool run = a.contiguous != 0;
            if (!a.contiguous) {
                di0 = __shfl_sync(kFull, my_di, 0);
                run = __all_sync(kFull, a.idx_bulk && rows == 32 && my_di == di0 + lane && ((di0 * BB) & 15) == 0);
            }
            if (bulk_out && rows == 32 && run) {
                // 32 slots (32 * kSlotB bytes, a multiple of 16) at a 16-byte aligned offset; paired:
                // once both halves of the slots are written
                if ((!PAIR || half == NH - 1) && hf == 0 && lane == 0) {
                    uint8_t *dst = a.out + di0 * S::kSlotB;
                    const uint32_t src = (uint32_t)__cvta_generic_to_shared(sm_out + 32 * grp * S::kSlotB);
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                                 "r"(32 * S::kSlotB)
                                 : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                }
            } else if (PAIR) {
                // not reached: paired calls cover whole 128-row tiles of contiguous slots
            } else if (a.contiguous) {
                uint8_t *dst = a.out + (v0 + 32 * grp) * BB;
                const uint8_t *src = sm_out + 32 * grp * BB;
                const int nbytes = rows * BB, nch = nbytes >> 4;
                for (int q = lane + 32 * hf; q < nch; q += 64)
                    reinterpret_cast<uint4 *>(dst)[q] = reinterpret_cast<const uint4 *>(src)[q];
                for (int q = (nch << 3) + lane + 32 * hf; q < (nbytes >> 1); q += 64)
                    reinterpret_cast<uint16_t *>(dst)[q] = reinterpret_cast<const uint16_t *>(src)[q];
            } else {
                // to the destination rows (2-byte aligned slots) in pieces shared by both warps of the
                // group: a block is (BB - 2) / 4 four-byte words and one 2-byte piece, the piece last
                // when the block starts 4-byte aligned, else first
                constexpr int NW = (BB - 2) / 4, NP = NW + 1;
                for (int p0 = 32 * hf; p0 < rows * NP; p0 += 64) {
                    const int p = p0 + lane;
                    const bool valid = p < rows * NP;
                    const int j = valid ? p / NP : 0, k = p - j * NP;
                    const int64_t di = __shfl_sync(kFull, my_di, j);
                    if (valid) {
                        uint8_t *d = a.out + di * a.out_stride;
                        const uint8_t *sp = sm_out + (32 * grp + j) * BB;
                        const int lead = ((uint32_t)(uintptr_t)d & 2u) ? 1 : 0;   // 2-byte piece first
                        if (k == (lead ? 0 : NW)) {
                            const int o = lead ? 0 : 4 * NW;
                            *reinterpret_cast<uint16_t *>(d + o) = *reinterpret_cast<const uint16_t *>(sp + o);
                        } else {
                            const int o = 4 * (k - lead) + 2 * lead;
                            const uint32_t w = (uint32_t)*reinterpret_cast<const uint16_t *>(sp + o) |
                                               ((uint32_t)*reinterpret_cast<const uint16_t *>(sp + o + 2) << 16);
                            *reinterpret_cast<uint32_t *>(d + o) = w;
                        }
                    }
                }
            }

            // ---- paired calls cover twice the rows per CTA: keep the list of rows to finish from
            // overflowing (an overflowing CTA rechecks every row it encoded) -- once the next tile could
            // fill it, finish the listed rows now, from memory (every block of the CTA has left: the
            // bulk stores are waited for), and empty it.  The count is read between two barriers, so
            // every epilogue warp takes the same decision.  (Unpaired calls keep their warps free of
            // CTA-wide barriers: about one row in 250 is listed, so a list covers ~60 k rows per CTA.)
            if constexpr (PAIR) {
            asm volatile("bar.sync 5, %0;" ::"n"(32 * kTcEpiWarps) : "memory");
            const int listed = fix[0], overflowed = fix[1];
            asm volatile("bar.sync 5, %0;" ::"n"(32 * kTcEpiWarps) : "memory");
            if (listed > kTcFixCap - kTcRows && overflowed == 0) {
                if (bulk_out && hf == 0 && lane == 0) {
                    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                asm volatile("bar.sync 5, %0;" ::"n"(32 * kTcEpiWarps) : "memory");
                for (int q = warp; q < listed; q += kTcEpiWarps) {
                    const uint32_t e = (uint32_t)fix[4 + q];
                    finish_row_warp<BITS, DT>(a, s_tab, (int64_t)(e & 0x3FFFFFFFu), (e >> 31) != 0, false, lane,
                                              (int)((e >> 30) & 1u));
                }
                asm volatile("bar.sync 5, %0;" ::"n"(32 * kTcEpiWarps) : "memory");
                if (threadIdx.x == 0) fix[0] = 0;
                asm volatile("bar.sync 5, %0;" ::"n"(32 * kTcEpiWarps) : "memory");
            }
            }
        }

        // ---- finish the listed rows once every block of this CTA is in memory
        if (bulk_out && hf == 0 && lane == 0) {
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        asm volatile("bar.sync 5, %0;" ::"n"(32 * kTcEpiWarps) : "memory");
        if (fix[1] == 0) {
            const int nfix = min(fix[0], kTcFixCap);
            for (int q = warp; q < nfix; q += kTcEpiWarps) {
                const uint32_t e = (uint32_t)fix[4 + q];
                finish_row_warp<BITS, DT>(a, s_tab, (int64_t)(e & 0x3FFFFFFFu), (e >> 31) != 0, false, lane,
                                          (int)((e >> 30) & 1u));
            }
        } else {
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x)
                for (int half = 0; half < NH; ++half)
                    for (int rr = warp; rr < kTcRows; rr += kTcEpiWarps)
                        if (tile * kTcRows + rr < a.n_vec)
                            finish_row_warp<BITS, DT>(a, s_tab, tile * kTcRows + rr, false, true, lane, half);
        }
    }

    // ---- teardown: every MMA has completed (the producer waited for its last commit) and every
    // tensor-memory load completed
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols) : "memory");
}

// Launch the tcgen05 kernel; returns 1 when the rows cannot be described by a
// tensor map (the caller then uses the mma.sync kernel).
template <int BITS, int DT>
int launch_tc(const EncArgs &a, cudaStream_t st) {
    CUtensorMap map;
    if (!make_row_tile_map(&map, a.x, DT, a.n_vec, a.x_stride)) return 1;
    static int done[64] = {0};
    if (set_smem_limit((const void *)encode_tc_kernel<BITS, DT, false>, TcSmem<BITS>::kTotal, done) != TQ_OK)
        return TQ_ERR_CUDA;
    const int64_t ntiles = (a.n_vec + kTcRows - 1) / kTcRows;
    const int grid = (int)std::min<int64_t>(ntiles, 2 * (int64_t)sm_count());
    encode_tc_kernel<BITS, DT, false><<<grid, kTcThreads, TcSmem<BITS>::kTotal, st>>>(map, map, a);
    return launch_status();
}

// Paired launch: rows of a.x into the first and rows of a.x2 into the second
// half of each 2 BB-byte slot; 1 when the rows cannot be described by tensor
// maps.
template <int BITS, int DT>
int launch_tc_pair(const EncArgs &a, cudaStream_t st) {
    CUtensorMap map, map2;
    if (!make_row_tile_map(&map, a.x, DT, a.n_vec, a.x_stride) || !make_row_tile_map(&map2, a.x2, DT, a.n_vec, a.x_stride))
        return 1;
    static int done[64] = {0};
    if (set_smem_limit((const void *)encode_tc_kernel<BITS, DT, true>, TcSmem<BITS, true>::kTotal, done) != TQ_OK)
        return TQ_ERR_CUDA;
    const int64_t ntiles = a.n_vec / kTcRows;
    const int grid = (int)std::min<int64_t>(ntiles, 2 * (int64_t)sm_count());
    encode_tc_kernel<BITS, DT, true><<<grid, kTcThreads, TcSmem<BITS, true>::kTotal, st>>>(map, map2, a);
    return launch_status();
}

// Up to this many rows (eight 128-row tiles) the tensor-core kernel's
// per-CTA setup (H D in shared memory, tensor-memory allocation, barriers)
// outweighs the work: the warp-independent mma.sync kernel serves such
// calls (the append of one token per sequence and KV head).
constexpr int64_t kTcMaxSmallRows = 1024;

template <int BITS, int DT>
int launch_16bit(const EncArgs &a, cudaStream_t st) {
    if (a.n_vec <= kTcMaxSmallRows) return launch_mma<BITS, DT>(a, st);
    const int r = launch_tc<BITS, DT>(a, st);
    return r == 1 ? launch_mma<BITS, DT>(a, st) : r;
}

// Cell table of a codebook.  With z = G y, cell j holds
// z + 64 in [j - 1/16, j + 15/16) (the cells of rounding z + 64 to 1/8 and
// taking the integer part); G is the smallest integer above
// 1 / (smallest gap between adjacent boundaries), so no cell holds two
// boundaries, and G <= 62 keeps |z| <= G (|y| <= 1) inside the table.
void build_table(const tq_codebook *cb, EncArgs *a) {
    const int L = 1 << cb->bits;
    double gap = 1.0;
    for (int i = 0; i + 1 < L - 1; ++i)
        gap = std::min(gap, (double)cb->boundaries[i + 1] - (double)cb->boundaries[i]);
    const float G = (float)std::min(62.0, std::floor(1.0 / gap) + 1.0);
    a->grid = G;
    for (int j = 0; j < kBuckets; ++j) {
        int below = 0;
        float inner = INFINITY;
        for (int i = 0; i < L - 1; ++i) {
            const float z = G * cb->boundaries[i];
            if (z + 64.f < j - 0.0625f) ++below;
            else if (z + 64.f < j + 0.9375f) inner = z;
        }
        const uint32_t code = (uint32_t)below;
        float codef;
        memcpy(&codef, &code, 4);
        a->table[j] = make_float2(inner, codef);
    }
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" int tq_encode_kv(const void *x, int x_dtype, int64_t n_vec, int64_t x_stride_elems,
                            const tq_codebook *cb, tq_signs signs, uint8_t *blocks,
                            int64_t block_stride_bytes, const int64_t *dst_index, void *stream) {
    if (n_vec < 0 || !cb) return TQ_ERR_ARG;
    if (cb->bits == 8)   // turboq8 (tq_ext.cu)
        return tq_encode_kv_ex(x, x_dtype, n_vec, x_stride_elems, cb, signs, blocks, block_stride_bytes, dst_index, 0,
                               stream);
    if (!codebook_ok(cb) || dtype_bytes(x_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    const int es = dtype_bytes(x_dtype);
    const int64_t bb = (int64_t)tq_block_bytes(cb->bits);
    if (!x || !blocks || x_stride_elems < kD || block_stride_bytes < bb) return TQ_ERR_ARG;
    if (!aligned(x, 16) || (x_stride_elems * es) % 16 || !aligned(blocks, 2) || (block_stride_bytes & 1))
        return TQ_ERR_ALIGN;
    EncArgs a;
    memset(&a, 0, sizeof(a));
    a.drop = drop_copies();
    a.x = static_cast<const uint8_t *>(x);
    a.n_vec = n_vec;
    a.x_stride = x_stride_elems * es;
    a.out = blocks;
    a.out_stride = block_stride_bytes;
    a.dst_index = dst_index;
    a.contiguous = (!dst_index && block_stride_bytes == bb && aligned(blocks, 16)) ? 1 : 0;
    a.idx_bulk = (dst_index && block_stride_bytes == bb && aligned(blocks, 16)) ? 1 : 0;
    a.b0 = cb->boundaries[(1 << cb->bits) / 2];
    build_table(cb, &a);
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    cudaStream_t st = (cudaStream_t)stream;
    switch (cb->bits * 8 + x_dtype) {
        case 2 * 8 + TQ_F32: return launch<2, TQ_F32>(a, st);
        case 2 * 8 + TQ_BF16: return launch_16bit<2, TQ_BF16>(a, st);
        case 2 * 8 + TQ_F16: return launch_16bit<2, TQ_F16>(a, st);
        case 3 * 8 + TQ_F32: return launch<3, TQ_F32>(a, st);
        case 3 * 8 + TQ_BF16: return launch_16bit<3, TQ_BF16>(a, st);
        case 3 * 8 + TQ_F16: return launch_16bit<3, TQ_F16>(a, st);
        case 4 * 8 + TQ_F32: return launch<4, TQ_F32>(a, st);
        case 4 * 8 + TQ_BF16: return launch_16bit<4, TQ_BF16>(a, st);
        case 4 * 8 + TQ_F16: return launch_16bit<4, TQ_F16>(a, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

namespace tq {

int wait_failed_encode(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

// Paired encode for the storage layout: row i of k into bytes [0, BB) and row
// i of v into bytes [BB, 2 BB) of slot i (slot = 2 BB bytes, contiguous), both
// with codebook cb, so that every 32 slots leave as one bulk copy instead of
// two launches each writing half of every slot.  Returns 1 (nothing
// enqueued) when the call is not of that form: 16-bit rows, a whole number
// of 128-row tiles (fewer than 2^30 rows), 16-byte aligned rows and slots.
int encode_kv_pair(const void *k, const void *v, int x_dtype, int64_t n_vec, int64_t x_stride_elems,
                   const tq_codebook *cb, tq_signs signs, uint8_t *slots, cudaStream_t st) {
    if (!cb || !codebook_ok(cb) || (x_dtype != TQ_BF16 && x_dtype != TQ_F16)) return 1;
    if (n_vec <= 0 || n_vec % kTcRows || n_vec >= (int64_t(1) << 30)) return 1;
    const int64_t bb = (int64_t)tq_block_bytes(cb->bits);
    if (!k || !v || !slots || x_stride_elems < kD || (x_stride_elems * 2) % 16 || !aligned(k, 16) ||
        !aligned(v, 16) || !aligned(slots, 16))
        return 1;
    EncArgs a;
    memset(&a, 0, sizeof(a));
    a.drop = drop_copies();
    a.x = static_cast<const uint8_t *>(k);
    a.x2 = static_cast<const uint8_t *>(v);
    a.n_vec = n_vec;
    a.x_stride = x_stride_elems * 2;
    a.out = slots;
    a.out_stride = 2 * bb;
    a.dst_index = nullptr;
    a.contiguous = 1;
    a.idx_bulk = 0;
    a.b0 = cb->boundaries[(1 << cb->bits) / 2];
    build_table(cb, &a);
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    switch (cb->bits * 8 + x_dtype) {
        case 2 * 8 + TQ_BF16: return launch_tc_pair<2, TQ_BF16>(a, st);
        case 2 * 8 + TQ_F16: return launch_tc_pair<2, TQ_F16>(a, st);
        case 3 * 8 + TQ_BF16: return launch_tc_pair<3, TQ_BF16>(a, st);
        case 3 * 8 + TQ_F16: return launch_tc_pair<3, TQ_F16>(a, st);
        case 4 * 8 + TQ_BF16: return launch_tc_pair<4, TQ_BF16>(a, st);
        case 4 * 8 + TQ_F16: return launch_tc_pair<4, TQ_F16>(a, st);
        default: return 1;
    }
}

}  // namespace tq
