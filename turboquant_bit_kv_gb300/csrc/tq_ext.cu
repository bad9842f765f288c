// Further block formats of the TurboQuant family: the norm-corrected encode,
// the dense 8-in-3 packing of 3-bit codes, and the 8-bit turboq8 codec.
//
// * "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", section 4, Encode
//   pipeline step 4: the block norm is grp_norm / recon_norm, recon_norm the
//   L2 norm of the reconstructed centroids ("lmcache.v1.distributed.serde.
//   turboquant", Configuration: the `_nc` presets).
// * "TurboQuant KV Cache Compression — Spec", Algorithm Detail Step 3: eight
//   3-bit values packed into three bytes.
// * "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", At a glance and the
//   turboq8 paragraph: FWHT rotation, uniform 256-level grid
//   (i - 127.5) / 127.5, per-block absmax scale; 130-byte blocks.
//
// Layouts: norm-corrected blocks are the plain ones (only the stored norm
// differs); a dense 3-bit block is [fp16 norm][16 groups of 3 bytes], the
// codes of elements 8g .. 8g + 7 in the 24-bit little-endian word of group g,
// element 8g + p in bits 3p .. 3p + 2; a turboq8 block is [fp16 scale][128
// code bytes].
//
// bf16 / fp16 rows (1024 or more, blocks back to back) go to the tensor-core
// encode of tq_headdim_tc.cu (the rotation H D as one exact contraction);
// the kernels here take the rest.
//
// Kernels: two threads per row, each holding 64 of its elements in registers
// (six butterfly stages of the 128-point transform in registers, the seventh
// across the pair); a warp takes 16 rows at a time and stages and stores its
// own blocks (no CTA-wide barrier in the loop); codes by binary search of the boundaries (Lloyd-Max
// codebooks) or by rounding to the uniform grid (turboq8), decided in
// float32; stored norms and scales rounded once to fp16, recomputed in
// double precision when the float32 value lies within 2^-20 of an fp16
// rounding boundary.

#include <algorithm>
#include <cmath>
#include <cstring>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kExtThreads = 256;   // 128 rows per CTA pass, two threads per row

struct ExtArgs {
    const uint8_t *x;        // encode: rows
    uint8_t *blocks;         // encode: destination; decode: source
    uint8_t *out;            // decode: rows
    const int64_t *dst_index;
    int64_t n_vec;
    int64_t x_stride;        // bytes (encode input / decode output rows)
    int64_t block_stride;    // bytes
    int nc, dense;           // norm correction, 8-in-3 packing of 3-bit codes
    float c[16];             // centroids
    float b[16];             // boundaries (ascending; unused entries +inf)
    uint32_t signs[4];
    float grid;              // cells per unit of y of the table below
    float2 cells[128];       // cell j = floor(grid y + 64): (boundary inside it | +inf, #boundaries below as bits)
    int contiguous;          // blocks back to back from a 16-byte aligned start, no destination index
};

__device__ __forceinline__ float sign_of(const uint32_t (&s)[4], int d) {
    return ((s[d >> 5] >> (d & 31)) & 1u) ? -1.f : 1.f;
}

// Elements 64 h .. 64 h + 63 of a row of dtype DT as float.
template <int DT>
__device__ __forceinline__ void load_half_row(const uint8_t *row, int h, float (&v)[64]) {
    if constexpr (DT == TQ_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(row + 256 * h);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 f = __ldg(p + i);
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(row + 128 * h);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 w = __ldg(p + i);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float lo, hi;
                if constexpr (DT == TQ_BF16) {
                    lo = __uint_as_float(ww[k] << 16);
                    hi = __uint_as_float(ww[k] & 0xFFFF0000u);
                } else {
                    lo = __half2float(__ushort_as_half((unsigned short)(ww[k] & 0xFFFFu)));
                    hi = __half2float(__ushort_as_half((unsigned short)(ww[k] >> 16)));
                }
                v[8 * i + 2 * k] = lo;
                v[8 * i + 2 * k + 1] = hi;
            }
        }
    }
}

// The 128-point Hadamard transform of the pair's row: stages over bits 0..5 of
// the element index in registers, bit 6 across the two threads (lane ^ 1).
// Bits 0..4 run on packed pairs (v[i], v[i + 32]) (one paired add and one
// paired fused multiply-add by -1, exact like the subtraction, per two
// butterflies); bit 5 pairs the two halves of each packed pair.
__device__ __forceinline__ void fwht_pair(float (&v)[64], int h) {
    float2 p[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i] = make_float2(v[i], v[i + 32]);
    const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if ((i & m) == 0) {
                const float2 x = p[i], y = p[i + m];
                p[i] = __fadd2_rn(x, y);
                p[i + m] = __ffma2_rn(y, neg1, x);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = p[i].x + p[i].y;
        v[i + 32] = p[i].x - p[i].y;
    }
#pragma unroll
    for (int e = 0; e < 64; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[e], 1);
        v[e] = h ? (o - v[e]) : (v[e] + o);
    }
}

// True when f lies within 2^-20 (relative) of an fp16 rounding boundary (a
// midpoint between adjacent fp16 values), so float32 error could flip it.
__device__ __forceinline__ bool near_half_tie(float f) {
    if (!(f > 0.f) || !(f < 65504.f)) return false;
    const __half h = __float2half_rn(f);
    const float hv = __half2float(h);
    const float up = __half2float(__ushort_as_half((unsigned short)(__half_as_ushort(h) + 1)));
    const float dn = __half2float(__ushort_as_half((unsigned short)(__half_as_ushort(h) - 1)));
    const float t = f * 9.5367431640625e-07f;   // 2^-20
    return fabsf(f - 0.5f * (hv + up)) <= t || fabsf(f - 0.5f * (hv + dn)) <= t;
}

// Binary search: #{i : b_i <= y} over the 2^BITS - 1 boundaries.
template <int BITS>
__device__ __forceinline__ uint32_t level_of(float y, const float *b) {
    uint32_t i = 0;
#pragma unroll
    for (int step = 1 << (BITS - 1); step >= 1; step >>= 1)
        if (y >= b[i + step - 1]) i += step;
    return i;
}

__device__ __forceinline__ void st16(uint8_t *p, uint32_t v) { *reinterpret_cast<uint16_t *>(p) = (uint16_t)v; }

// Staged output blocks: per warp, the 16 rows of its pass, up to the largest (130-byte) block, back to
// back.  Warps work on their own (their own rows, staging and stores): no CTA-wide barrier in the loop.
constexpr int kExtWarpRows = 16;
constexpr int kExtWarpStage = kExtWarpRows * 130;
constexpr int kExtStage = (kExtThreads / 32) * kExtWarpStage;

template <int BITS, int DT>
__global__ void __launch_bounds__(kExtThreads, 2) encode_ext_kernel(const __grid_constant__ ExtArgs a) {
    __shared__ float s_c[16];
    __shared__ float2 s_cell[128];
    __shared__ __align__(16) uint8_t s_out[kExtStage];
    if (threadIdx.x < 16) s_c[threadIdx.x] = a.c[threadIdx.x];
    if (threadIdx.x < 128) s_cell[threadIdx.x] = a.cells[threadIdx.x];
    __syncthreads();
    constexpr int BB = BITS == 8 ? 130 : 2 + 16 * BITS;
    const int h = threadIdx.x & 1, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *w_out = s_out + warp * kExtWarpStage;
    const int64_t gw = (int64_t)blockIdx.x * (kExtThreads / 32) + warp;
    const int64_t wstride = (int64_t)gridDim.x * (kExtThreads / 32) * kExtWarpRows;
    for (int64_t base = gw * kExtWarpRows; base < a.n_vec; base += wstride) {
        const int64_t row = base + (lane >> 1);
        const bool valid = row < a.n_vec;           // both threads of a pair agree
        const uint8_t *xr = a.x + (valid ? row : 0) * a.x_stride;
        float v[64];
        load_half_row<DT>(xr, h, v);
        if (!valid) {
#pragma unroll
            for (int e = 0; e < 64; ++e) v[e] = 0.f;
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 64; ++e) ss = fmaf(v[e], v[e], ss);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        {
            // D x: the sign bits of elements 64 h .. 64 h + 63 flip the float sign bits
            const uint32_t s0 = a.signs[2 * h], s1 = a.signs[2 * h + 1];
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const uint32_t w = e < 32 ? s0 : s1;
                const uint32_t m = (w << (31 - (e & 31))) & 0x80000000u;
                v[e] = __uint_as_float(__float_as_uint(v[e]) ^ m);
            }
        }
        fwht_pair(v, h);
        const float rs = 0.08838834764831845f;   // 1 / sqrt(128)
        uint8_t code[64];
        uint32_t n16 = 0;
        if constexpr (BITS == 8) {
            // turboq8: a = max |u|, codes on the uniform grid of u / a, scale fp16(a)
            float amax = 0.f;
            int arg = 0;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const float m = fabsf(v[e]);
                if (m > amax) {
                    amax = m;
                    arg = 64 * h + e;
                }
            }
            const float om = __shfl_xor_sync(0xffffffffu, amax, 1);
            const int oa = __shfl_xor_sync(0xffffffffu, arg, 1);
            if (om > amax || (om == amax && oa < arg)) {
                amax = om;
                arg = oa;
            }
            const float a32 = amax * rs;
            const float inv = amax > 0.f ? 1.f / amax : 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                // u / a (the 1 / sqrt(128) cancels), in [-1, 1]: 127.5 y + 128 lies in [0.5, 255.5]
                const float y = v[e] * inv;
                code[e] = (uint8_t)(uint32_t)floorf(fmaf(127.5f, y, 128.f));
            }
            n16 = __half_as_ushort(__float2half_rn(a32));
            if (__any_sync(0xffffffffu, near_half_tie(a32))) {
                // the largest coordinate again in double precision: u_j = sum_d H_jd D_d x_d / sqrt(128)
                float xr2[64];
                load_half_row<DT>(xr, h, xr2);
                double part = 0.0;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const int d = 64 * h + e;
                    const double hd = (__popc(arg & d) & 1) ? -1.0 : 1.0;
                    part += hd * (double)sign_of(a.signs, d) * (double)xr2[e];
                }
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                if (near_half_tie(a32)) n16 = __half_as_ushort(__double2half(fabs(part) / sqrt(128.0)));
            }
            if (amax == 0.f) n16 = 0;
        } else {
            const float n = sqrtf(ss);
            const float inv = n > 0.f ? rs / n : 0.f;
            float csq = 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                // #{i : b_i <= y}: the cell's count below plus its one inner boundary
                const float y = v[e] * inv;
                const int j = min(127, max(0, (int)fmaf(a.grid, y, 64.f)));
                const float2 cell = s_cell[j];
                const uint32_t c = __float_as_uint(cell.y) + (y >= cell.x ? 1u : 0u);
                code[e] = (uint8_t)c;
                csq = fmaf(s_c[c], s_c[c], csq);
            }
            csq += __shfl_xor_sync(0xffffffffu, csq, 1);
            const float stored = a.nc ? (n > 0.f ? n / sqrtf(csq) : 0.f) : n;
            n16 = __half_as_ushort(__float2half_rn(stored));
            if (__any_sync(0xffffffffu, near_half_tie(stored))) {
                // norm (and recon norm) in double precision, one rounding to fp16
                float xr2[64];
                load_half_row<DT>(xr, h, xr2);
                double sx = 0.0, sc = 0.0;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    sx += (double)xr2[e] * (double)xr2[e];
                    sc += (double)s_c[code[e]] * (double)s_c[code[e]];
                }
                sx += __shfl_xor_sync(0xffffffffu, sx, 1);
                sc += __shfl_xor_sync(0xffffffffu, sc, 1);
                const double nd = sqrt(sx);
                if (near_half_tie(stored)) n16 = __half_as_ushort(__double2half(a.nc ? nd / sqrt(sc) : nd));
            }
            if (!(n > 0.f)) n16 = 0;
        }
        uint8_t *blk = w_out + (lane >> 1) * BB;   // staged back to back, then stored by the warp
        if (h == 0) st16(blk, n16);
        if constexpr (BITS == 8) {
#pragma unroll
            for (int k = 0; k < 32; ++k) st16(blk + 2 + 64 * h + 2 * k, code[2 * k] | ((uint32_t)code[2 * k + 1] << 8));
        } else if constexpr (BITS == 4) {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                st16(blk + 2 + 32 * h + 2 * k, code[4 * k] | (code[4 * k + 1] << 4) | (code[4 * k + 2] << 8) |
                                                   ((uint32_t)code[4 * k + 3] << 12));
        } else if constexpr (BITS == 2) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t w = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) w |= (uint32_t)code[8 * k + i] << (2 * i);
                st16(blk + 2 + 16 * h + 2 * k, w);
            }
        } else if (a.dense) {
            // 3-bit, eight codes per three bytes: this thread's groups 8 h .. 8 h + 7 = bytes 2 + 24 h ..
            uint8_t by[24];
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                uint32_t w = 0;
#pragma unroll
                for (int p = 0; p < 8; ++p) w |= (uint32_t)code[8 * g + p] << (3 * p);
                by[3 * g] = (uint8_t)w;
                by[3 * g + 1] = (uint8_t)(w >> 8);
                by[3 * g + 2] = (uint8_t)(w >> 16);
            }
#pragma unroll
            for (int k = 0; k < 12; ++k) st16(blk + 2 + 24 * h + 2 * k, by[2 * k] | ((uint32_t)by[2 * k + 1] << 8));
        } else {
            // 3-bit split planes: low 2 bits four per byte, high bit eight per byte
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t w = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) w |= (uint32_t)(code[8 * k + i] & 3u) << (2 * i);
                st16(blk + 2 + 16 * h + 2 * k, w);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t w = 0;
#pragma unroll
                for (int i = 0; i < 16; ++i) w |= (uint32_t)(code[16 * k + i] >> 2) << i;
                st16(blk + 34 + 8 * h + 2 * k, w);
            }
        }
        __syncwarp();
        // the warp's blocks: contiguous ones as 16-byte pieces, others row by row in 2-byte pieces
        const int nrows = (int)min64(kExtWarpRows, a.n_vec - base);
        if (a.contiguous) {
            // the pass's blocks form one run starting 16-byte aligned (16 x BB is a multiple of 16)
            uint4 *dst = reinterpret_cast<uint4 *>(a.blocks + base * BB);
            const uint4 *src = reinterpret_cast<const uint4 *>(w_out);
            const int n16 = nrows * BB / 16;
            for (int q = lane; q < n16; q += 32) dst[q] = src[q];
            for (int q = 16 * n16 + lane; q < nrows * BB; q += 32) a.blocks[base * BB + q] = w_out[q];
        } else {
            constexpr int NH = BB / 2;
            for (int q = lane; q < nrows * NH; q += 32) {
                const int r = q / NH, o = 2 * (q - r * NH);
                const int64_t di = a.dst_index ? a.dst_index[base + r] : base + r;
                *reinterpret_cast<uint16_t *>(a.blocks + di * a.block_stride + o) =
                    *reinterpret_cast<const uint16_t *>(w_out + r * BB + o);
            }
        }
        __syncwarp();
    }
}

__device__ __forceinline__ uint32_t ld16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

template <int BITS, int DT>
__global__ void __launch_bounds__(kExtThreads, 2) decode_ext_kernel(const __grid_constant__ ExtArgs a) {
    __shared__ float s_c[16];
    if (threadIdx.x < 16) s_c[threadIdx.x] = a.c[threadIdx.x];
    __syncthreads();
    const int h = threadIdx.x & 1;
    for (int64_t base = (int64_t)blockIdx.x * (kExtThreads / 2); base < a.n_vec;
         base += (int64_t)gridDim.x * (kExtThreads / 2)) {
        const int64_t row = base + (threadIdx.x >> 1);
        const bool valid = row < a.n_vec;
        const uint8_t *blk = a.blocks + (valid ? row : 0) * a.block_stride;
        const float scale = __half2float(__ushort_as_half((unsigned short)ld16(blk)));
        float v[64];
        if constexpr (BITS == 8) {
            const float f = scale * (1.f / 127.5f);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const uint32_t w = ld16(blk + 2 + 64 * h + 2 * k);
                v[2 * k] = ((float)(w & 0xFFu) - 127.5f) * f;
                v[2 * k + 1] = ((float)(w >> 8) - 127.5f) * f;
            }
        } else if constexpr (BITS == 4) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t w = ld16(blk + 2 + 32 * h + 2 * k);
#pragma unroll
                for (int i = 0; i < 4; ++i) v[4 * k + i] = s_c[(w >> (4 * i)) & 15u] * scale;
            }
        } else if constexpr (BITS == 2) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t w = ld16(blk + 2 + 16 * h + 2 * k);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[8 * k + i] = s_c[(w >> (2 * i)) & 3u] * scale;
            }
        } else if (a.dense) {
            uint8_t by[24];
#pragma unroll
            for (int k = 0; k < 12; ++k) {
                const uint32_t w = ld16(blk + 2 + 24 * h + 2 * k);
                by[2 * k] = (uint8_t)w;
                by[2 * k + 1] = (uint8_t)(w >> 8);
            }
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint32_t w = by[3 * g] | ((uint32_t)by[3 * g + 1] << 8) | ((uint32_t)by[3 * g + 2] << 16);
#pragma unroll
                for (int p = 0; p < 8; ++p) v[8 * g + p] = s_c[(w >> (3 * p)) & 7u] * scale;
            }
        } else {
            uint32_t hb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) hb[k] = ld16(blk + 34 + 8 * h + 2 * k);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t w = ld16(blk + 2 + 16 * h + 2 * k);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = 8 * k + i;
                    const uint32_t c = ((w >> (2 * i)) & 3u) | (((hb[e >> 4] >> (e & 15)) & 1u) << 2);
                    v[e] = s_c[c] * scale;
                }
            }
        }
        // x_hat = D H v / sqrt(128)
        fwht_pair(v, h);
        const float rs = 0.08838834764831845f;
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] *= rs * sign_of(a.signs, 64 * h + e);
        if (!valid) continue;
        uint8_t *o = a.out + row * a.x_stride;
        if constexpr (DT == TQ_F32) {
            float4 *p = reinterpret_cast<float4 *>(o + 256 * h);
#pragma unroll
            for (int i = 0; i < 16; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
            uint4 *p = reinterpret_cast<uint4 *>(o + 128 * h);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = v[8 * i + 2 * k], hi = v[8 * i + 2 * k + 1];
                    if constexpr (DT == TQ_BF16) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                        w[k] = *reinterpret_cast<const uint32_t *>(&b2);
                    } else {
                        const __half2 h2 = __floats2half2_rn(lo, hi);
                        w[k] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                }
                p[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
}

template <class K>
int launch_ext(K kernel, const ExtArgs &a, cudaStream_t st) {
    static int per_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    int occ = dev < 64 ? per_sm[dev] : 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kExtThreads, 0) != cudaSuccess || occ < 1)
            occ = 1;
        if (dev < 64) per_sm[dev] = occ;
    }
    const int64_t ctas = (a.n_vec + kExtThreads / 2 - 1) / (kExtThreads / 2);   // (16 rows per warp)
    const int grid = (int)std::min<int64_t>(ctas, (int64_t)occ * sm_count());
    kernel<<<grid, kExtThreads, 0, st>>>(a);
    return launch_status();
}

template <int BITS>
int encode_ext_bits(const ExtArgs &a, int dt, cudaStream_t st) {
    switch (dt) {
        case TQ_F32: return launch_ext(encode_ext_kernel<BITS, TQ_F32>, a, st);
        case TQ_BF16: return launch_ext(encode_ext_kernel<BITS, TQ_BF16>, a, st);
        case TQ_F16: return launch_ext(encode_ext_kernel<BITS, TQ_F16>, a, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

template <int BITS>
int decode_ext_bits(const ExtArgs &a, int dt, cudaStream_t st) {
    switch (dt) {
        case TQ_F32: return launch_ext(decode_ext_kernel<BITS, TQ_F32>, a, st);
        case TQ_BF16: return launch_ext(decode_ext_kernel<BITS, TQ_BF16>, a, st);
        case TQ_F16: return launch_ext(decode_ext_kernel<BITS, TQ_F16>, a, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

// Codebook and flags of an extended call: bits 2..4 with a Lloyd-Max
// codebook (TQ_FMT_NORM_CORRECT; TQ_FMT_DENSE3 for 3 bits), or bits 8
// (turboq8, no flags).
int ext_check(const tq_codebook *cb, int flags) {
    if (!cb) return TQ_ERR_ARG;
    if (flags & ~(TQ_FMT_NORM_CORRECT | TQ_FMT_DENSE3)) return TQ_ERR_ARG;
    if (cb->head_dim != kD) return TQ_ERR_UNSUPPORTED;
    if (cb->bits == 8) return (cb->levels == 256 && flags == 0) ? TQ_OK : TQ_ERR_UNSUPPORTED;
    if (!codebook_ok(cb)) return TQ_ERR_UNSUPPORTED;
    if ((flags & TQ_FMT_DENSE3) && cb->bits != 3) return TQ_ERR_UNSUPPORTED;
    return TQ_OK;
}

void ext_tables(const tq_codebook *cb, ExtArgs *a) {
    for (int i = 0; i < 16; ++i) {
        a->c[i] = (cb->bits != 8 && i < cb->levels) ? cb->centroids[i] : 0.f;
        a->b[i] = (cb->bits != 8 && i + 1 < cb->levels) ? cb->boundaries[i] : INFINITY;
    }
    // cells of width 1 / grid over y in [-1, 1], each holding at most one boundary: cell j covers
    // grid y + 64 in [j, j + 1); it lists the boundaries at or below its start and the one inside it
    a->grid = 1.f;
    for (int j = 0; j < 128; ++j) a->cells[j] = make_float2(INFINITY, 0.f);
    if (cb->bits == 8) return;
    const int L = cb->levels;
    double gap = 2.0;
    for (int i = 0; i + 2 < L; ++i) gap = std::min(gap, (double)cb->boundaries[i + 1] - (double)cb->boundaries[i]);
    const float G = (float)std::min(62.0, std::floor(1.0 / gap) + 1.0);
    a->grid = G;
    for (int j = 0; j < 128; ++j) {
        uint32_t below = 0;
        float inner = INFINITY;
        for (int i = 0; i + 1 < L; ++i) {
            const double z = (double)G * (double)cb->boundaries[i] + 64.0;
            if (z <= (double)j) ++below;
            else if (z < (double)j + 1.0) inner = cb->boundaries[i];
        }
        float bf;
        std::memcpy(&bf, &below, 4);
        a->cells[j] = make_float2(inner, bf);
    }
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" size_t tq_block_bytes_ex(int bits, int flags) {
    if (flags & ~(TQ_FMT_NORM_CORRECT | TQ_FMT_DENSE3)) return 0;
    if (bits == 8) return flags == 0 ? 130 : 0;
    if ((flags & TQ_FMT_DENSE3) && bits != 3) return 0;
    return tq_block_bytes(bits);
}

extern "C" int tq_encode_kv_ex(const void *x, int x_dtype, int64_t n_vec, int64_t x_stride_elems,
                               const tq_codebook *cb, tq_signs signs, uint8_t *blocks, int64_t block_stride_bytes,
                               const int64_t *dst_index, int flags, void *stream) {
    if (n_vec < 0) return TQ_ERR_ARG;
    const int r = ext_check(cb, flags);
    if (r != TQ_OK) return r;
    if (dtype_bytes(x_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    const int es = dtype_bytes(x_dtype);
    const int64_t bb = (int64_t)tq_block_bytes_ex(cb->bits, flags);
    if (!x || !blocks || x_stride_elems < kD || block_stride_bytes < bb) return TQ_ERR_ARG;
    if (!aligned(x, 16) || (x_stride_elems * es) % 16 || !aligned(blocks, 2) || (block_stride_bytes & 1))
        return TQ_ERR_ALIGN;
    ExtArgs a;
    a.x = static_cast<const uint8_t *>(x);
    a.blocks = blocks;
    a.out = nullptr;
    a.dst_index = dst_index;
    a.n_vec = n_vec;
    a.x_stride = x_stride_elems * es;
    a.block_stride = block_stride_bytes;
    a.nc = (flags & TQ_FMT_NORM_CORRECT) ? 1 : 0;
    a.dense = (flags & TQ_FMT_DENSE3) ? 1 : 0;
    a.contiguous = (!dst_index && block_stride_bytes == bb && aligned(blocks, 16)) ? 1 : 0;
    ext_tables(cb, &a);
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // bf16 / fp16 rows into blocks back to back: the tensor-core encode (1: not its form)
    if (!dst_index && block_stride_bytes == bb) {
        const int t = ext_encode_tc(x, x_dtype, n_vec, a.x_stride, cb, signs.w, a.nc, a.dense, blocks, st);
        if (t != 1) return t;
    }
    switch (cb->bits) {
        case 2: return encode_ext_bits<2>(a, x_dtype, st);
        case 3: return encode_ext_bits<3>(a, x_dtype, st);
        case 4: return encode_ext_bits<4>(a, x_dtype, st);
        case 8: return encode_ext_bits<8>(a, x_dtype, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

extern "C" int tq_decode_kv_ex(const uint8_t *blocks, int64_t block_stride_bytes, int64_t n_vec,
                               const tq_codebook *cb, tq_signs signs, void *out, int out_dtype,
                               int64_t out_stride_elems, int flags, void *stream) {
    if (n_vec < 0) return TQ_ERR_ARG;
    const int r = ext_check(cb, flags);
    if (r != TQ_OK) return r;
    if (dtype_bytes(out_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    const int es = dtype_bytes(out_dtype);
    const int64_t bb = (int64_t)tq_block_bytes_ex(cb->bits, flags);
    if (!blocks || !out || out_stride_elems < kD || block_stride_bytes < bb) return TQ_ERR_ARG;
    if (!aligned(out, 16) || (out_stride_elems * es) % 16 || !aligned(blocks, 2) || (block_stride_bytes & 1))
        return TQ_ERR_ALIGN;
    ExtArgs a;
    a.x = nullptr;
    a.blocks = const_cast<uint8_t *>(blocks);
    a.out = static_cast<uint8_t *>(out);
    a.dst_index = nullptr;
    a.n_vec = n_vec;
    a.x_stride = out_stride_elems * es;
    a.block_stride = block_stride_bytes;
    a.nc = 0;
    a.dense = (flags & TQ_FMT_DENSE3) ? 1 : 0;
    a.contiguous = 0;
    ext_tables(cb, &a);
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (cb->bits) {
        case 2: return decode_ext_bits<2>(a, out_dtype, st);
        case 3: return decode_ext_bits<3>(a, out_dtype, st);
        case 4: return decode_ext_bits<4>(a, out_dtype, st);
        case 8: return decode_ext_bits<8>(a, out_dtype, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}
