// The codec and decode attention at head dims 64, 96, 128 and 160.
//
// "TurboQuant KV Cache Compression — Spec", Types / Codebook Generation
// (target dimensions 64, 96, 128, 160; the Lloyd-Max codebook of
// Beta(d/2, d/2) per dimension), Hadamard Transform Detail (for a head dim
// that is not a power of two, "a dense random orthogonal matrix"),
// Algorithm Detail steps 1-3 and Optimization: Fused dequant-dot.  The
// rotation is the caller's orthogonal matrix R (d x d, float32): y =
// R x / ||x||, x_hat = n16 R^T c[code]; for a power-of-two d,
// tq_rotation_hadamard builds R = H D / sqrt(d).  Blocks generalise the
// 128-element layout: [fp16 norm][codes], 2-bit four per byte, 4-bit two per
// byte, 3-bit a 2-bit low plane of d / 4 bytes then a 1-bit high plane of
// d / 8 bytes.
//
// Kernels (CUDA cores, float32; d = 32 ND): a warp per row, lane l holds
// elements l + 32 k.  R sits in shared memory with rows padded to d + 1
// floats, so that the 32 lanes reading one column (encode: outputs
// l + 32 k, input j) hit 32 different banks.  The rotation of a row is d
// shuffles of its inputs and d ND fused multiply-adds per lane.  Codes are
// the count of float32 boundaries <= y; norms are rounded once to fp16 and
// recomputed in double precision when the float32 norm lies within 2^-20 of
// an fp16 rounding boundary.  The codec kernels rotate four rows per warp at
// once, so every element of R read from shared memory serves four rows.
// Decode attention: a prep kernel rotates every query once (R q, scale
// log2(e) folded in); one CTA of 8 warps per (sequence, KV head, context
// split) then takes 32 tokens per warp step: lane t scores its token
// against n_t c[code_t] for every head (no cross-lane sums), the warp keeps
// an online softmax per head, and the value sums run with lanes over dims,
// each token's probabilities broadcast by shuffles; the warps merge in shared
// memory, and a combine kernel merges the splits and rotates back (R^T).

#include <cmath>
#include <cstring>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kHdThreads = 256;     // 8 warps
constexpr int kHdWarps = kHdThreads / 32;
constexpr unsigned kHdFull = 0xffffffffu;

bool hd_dim_ok(int d) { return d == 64 || d == 96 || d == 128 || d == 160; }

int hd_block_bytes(int d, int bits) { return (bits < 2 || bits > 4 || !hd_dim_ok(d)) ? 0 : 2 + d * bits / 8; }

bool hd_codebook_ok(const tq_codebook *cb, int d) {
    return cb && cb->head_dim == d && cb->bits >= 2 && cb->bits <= 4 && cb->levels == (1 << cb->bits);
}

struct HdArgs {
    const void *x;           // encode: rows
    uint8_t *blocks;         // encode: destination; decode: source
    void *out;               // decode: rows
    const float *R;          // [d][d] row-major
    int64_t n_vec;
    int bits, dt;
    float c[16];             // centroids
    float b[16];             // boundaries (ascending; unused entries +inf)
};

__device__ __forceinline__ float hd_load(const void *p, int dt, int64_t i) {
    if (dt == TQ_F32) return reinterpret_cast<const float *>(p)[i];
    if (dt == TQ_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return __half2float(reinterpret_cast<const __half *>(p)[i]);
}

__device__ __forceinline__ void hd_store(void *p, int dt, int64_t i, float v) {
    if (dt == TQ_F32) reinterpret_cast<float *>(p)[i] = v;
    else if (dt == TQ_BF16) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<__half *>(p)[i] = __float2half_rn(v);
}

// Code of element j of a block (layout above).
template <int D>
__device__ __forceinline__ uint32_t hd_code(const uint8_t *blk, int bits, int j) {
    if (bits == 2) return (blk[2 + (j >> 2)] >> (2 * (j & 3))) & 3u;
    if (bits == 4) return (blk[2 + (j >> 1)] >> (4 * (j & 1))) & 15u;
    return ((blk[2 + (j >> 2)] >> (2 * (j & 3))) & 3u) | (((blk[2 + D / 4 + (j >> 3)] >> (j & 7)) & 1u) << 2);
}

// Byte q of a block's code area from the codes of its D elements (layout above).
template <int D>
__device__ __forceinline__ uint32_t hd_code_byte(const uint8_t *codes, int bits, int q) {
    uint32_t v = 0;
    if (bits == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v |= (uint32_t)(codes[4 * q + i] & 3u) << (2 * i);
    } else if (bits == 4) {
        v = (codes[2 * q] & 15u) | ((uint32_t)(codes[2 * q + 1] & 15u) << 4);
    } else if (q < D / 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v |= (uint32_t)(codes[4 * q + i] & 3u) << (2 * i);
    } else {
        const int p = q - D / 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) v |= (uint32_t)((codes[8 * p + i] >> 2) & 1u) << i;
    }
    return v;
}

__device__ __forceinline__ float hd_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kHdFull, v, o);
    return v;
}

__device__ __forceinline__ double hd_warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kHdFull, v, o);
    return v;
}

// R into shared memory, rows padded to D + 1 floats.
template <int D>
__device__ __forceinline__ void hd_load_R(float *Rs, const float *R) {
    for (int i = threadIdx.x; i < D * D; i += blockDim.x) Rs[(i / D) * (D + 1) + i % D] = R[i];
}

// out[k] += sum_j M(lane + 32 k, j) v_j over the warp's D inputs v (element j in lane j % 32,
// register j / 32): the rows of M are those of R (TRANSPOSE false: y = R v) or its columns
// (TRANSPOSE true: y = R^T v).
template <int ND, bool TRANSPOSE>
__device__ __forceinline__ void hd_rotate(const float *Rs, const float (&v)[ND], float (&out)[ND], int lane) {
    constexpr int D = 32 * ND, P = D + 1;
#pragma unroll
    for (int k = 0; k < ND; ++k) out[k] = 0.f;
#pragma unroll
    for (int jj = 0; jj < ND; ++jj) {
#pragma unroll 8
        for (int src = 0; src < 32; ++src) {
            const float vj = __shfl_sync(kHdFull, v[jj], src);
            const int j = 32 * jj + src;
#pragma unroll
            for (int k = 0; k < ND; ++k) {
                const float r = TRANSPOSE ? Rs[j * P + lane + 32 * k] : Rs[(lane + 32 * k) * P + j];
                out[k] = fmaf(r, vj, out[k]);
            }
        }
    }
}

// The same for NR rows at once: every element of R read from shared memory serves NR rows.
template <int ND, bool TRANSPOSE, int NR>
__device__ __forceinline__ void hd_rotate_rows(const float *Rs, const float (&v)[NR][ND], float (&out)[NR][ND],
                                               int lane) {
    constexpr int D = 32 * ND, P = D + 1;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int k = 0; k < ND; ++k) out[r][k] = 0.f;
#pragma unroll
    for (int jj = 0; jj < ND; ++jj) {
#pragma unroll 4
        for (int src = 0; src < 32; ++src) {
            float vj[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) vj[r] = __shfl_sync(kHdFull, v[r][jj], src);
            const int j = 32 * jj + src;
#pragma unroll
            for (int k = 0; k < ND; ++k) {
                const float m = TRANSPOSE ? Rs[j * P + lane + 32 * k] : Rs[(lane + 32 * k) * P + j];
#pragma unroll
                for (int r = 0; r < NR; ++r) out[r][k] = fmaf(m, vj[r], out[r][k]);
            }
        }
    }
}

constexpr int kHdRows = 4;   // rows a warp rotates at once in the codec kernels

template <int ND>
__global__ void __launch_bounds__(kHdThreads) encode_d_kernel(const __grid_constant__ HdArgs a) {
    constexpr int D = 32 * ND;
    extern __shared__ __align__(16) float hd_smem[];
    float *Rs = hd_smem;
    uint8_t *codes = reinterpret_cast<uint8_t *>(Rs + D * (D + 1));   // [8 warps][D]
    hd_load_R<D>(Rs, a.R);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *wc = codes + warp * D;
    const int L = 1 << a.bits, BB = 2 + D * a.bits / 8;
    for (int64_t r0 = ((int64_t)blockIdx.x * kHdWarps + warp) * kHdRows; r0 < a.n_vec;
         r0 += (int64_t)gridDim.x * kHdWarps * kHdRows) {
        float x[kHdRows][ND], y[kHdRows][ND], ss[kHdRows];
#pragma unroll
        for (int r = 0; r < kHdRows; ++r) {
            const bool valid = r0 + r < a.n_vec;
            ss[r] = 0.f;
#pragma unroll
            for (int k = 0; k < ND; ++k) {
                x[r][k] = valid ? hd_load(a.x, a.dt, (r0 + r) * D + lane + 32 * k) : 0.f;
                ss[r] = fmaf(x[r][k], x[r][k], ss[r]);
            }
            ss[r] = hd_warp_sum(ss[r]);
        }
        hd_rotate_rows<ND, false, kHdRows>(Rs, x, y, lane);
#pragma unroll
        for (int r = 0; r < kHdRows; ++r) {
            if (r0 + r >= a.n_vec) break;   // (warp-uniform)
            const int64_t row = r0 + r;
            const float n = sqrtf(ss[r]);
            const float inv = n > 0.f ? 1.f / n : 0.f;
#pragma unroll
            for (int k = 0; k < ND; ++k) {
                const float yk = y[r][k] * inv;   // a zero row: y = 0, code L / 2
                uint32_t code = 0;
                for (int i = 0; i + 1 < L; ++i) code += (yk >= a.b[i]) ? 1u : 0u;
                wc[lane + 32 * k] = (uint8_t)code;
            }
            uint32_t n16 = __half_as_ushort(__float2half_rn(n));
            if (__any_sync(kHdFull, n > 0.f && near_fp16_tie_fast(n))) {
                double sd = 0.0;
#pragma unroll
                for (int k = 0; k < ND; ++k) sd += (double)x[r][k] * (double)x[r][k];
                sd = hd_warp_sum_d(sd);
                n16 = __half_as_ushort(__double2half(sqrt(sd)));
            }
            if (!(n > 0.f)) n16 = 0;
            __syncwarp();
            uint8_t *blk = a.blocks + row * BB;
            if (lane == 0) {
                blk[0] = (uint8_t)(n16 & 0xFFu);
                blk[1] = (uint8_t)(n16 >> 8);
            }
            for (int q = lane; q < BB - 2; q += 32) blk[2 + q] = (uint8_t)hd_code_byte<D>(wc, a.bits, q);
            __syncwarp();
        }
    }
}

template <int ND>
__global__ void __launch_bounds__(kHdThreads) decode_d_kernel(const __grid_constant__ HdArgs a) {
    constexpr int D = 32 * ND;
    extern __shared__ __align__(16) float hd_smem[];
    float *Rs = hd_smem;
    hd_load_R<D>(Rs, a.R);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BB = 2 + D * a.bits / 8;
    for (int64_t r0 = ((int64_t)blockIdx.x * kHdWarps + warp) * kHdRows; r0 < a.n_vec;
         r0 += (int64_t)gridDim.x * kHdWarps * kHdRows) {
        float v[kHdRows][ND], x[kHdRows][ND];
#pragma unroll
        for (int r = 0; r < kHdRows; ++r) {
            const bool valid = r0 + r < a.n_vec;
            const uint8_t *blk = a.blocks + (valid ? r0 + r : 0) * BB;
            const float n = valid ? __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8)))) : 0.f;
#pragma unroll
            for (int k = 0; k < ND; ++k) v[r][k] = a.c[hd_code<D>(blk, a.bits, lane + 32 * k)] * n;
        }
        hd_rotate_rows<ND, true, kHdRows>(Rs, v, x, lane);
#pragma unroll
        for (int r = 0; r < kHdRows; ++r) {
            if (r0 + r >= a.n_vec) break;
#pragma unroll
            for (int k = 0; k < ND; ++k) hd_store(a.out, a.dt, (r0 + r) * D + lane + 32 * k, x[r][k]);
        }
    }
}

int hd_smem_bytes(int d, bool codes) { return d * (d + 1) * 4 + (codes ? kHdWarps * d : 0); }

template <int ND>
int hd_launch_codec(const HdArgs &a, bool encode, cudaStream_t st) {
    constexpr int D = 32 * ND;
    static int done_e[64] = {0}, done_d[64] = {0};
    const int smem = hd_smem_bytes(D, encode);
    const void *k = encode ? (const void *)encode_d_kernel<ND> : (const void *)decode_d_kernel<ND>;
    if (set_smem_limit(k, smem, encode ? done_e : done_d) != TQ_OK) return TQ_ERR_CUDA;
    const int64_t ctas = (a.n_vec + kHdWarps * kHdRows - 1) / (kHdWarps * kHdRows);
    const int grid = (int)(ctas < (int64_t)sm_count() * 2 ? ctas : (int64_t)sm_count() * 2);
    if (encode) encode_d_kernel<ND><<<grid, kHdThreads, smem, st>>>(a);
    else decode_d_kernel<ND><<<grid, kHdThreads, smem, st>>>(a);
    return launch_status();
}

int hd_codec(const HdArgs &a, int d, bool encode, cudaStream_t st) {
    switch (d) {
        case 64: return hd_launch_codec<2>(a, encode, st);
        case 96: return hd_launch_codec<3>(a, encode, st);
        case 128: return hd_launch_codec<4>(a, encode, st);
        case 160: return hd_launch_codec<5>(a, encode, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

// ---------------------------------------------------------------- decode attention

struct HdAttnArgs {
    const void *q;
    const uint8_t *k, *v;
    const int32_t *seq_lens;
    const float *R;
    float *ws;               // partials [B][Hq][splits][2 + d]: m (log2 units), l, acc[d]
    float *qrot;             // rotated, scaled queries [B][Hq][d] (after the partials)
    float *out;
    int q_dtype, B, Hq, Hkv, G, T_cap, T, kbits, vbits, splits, tps;
    float qscale;            // scale * log2(e)
    float kc[16], vc[16];
};

// Context splits: enough CTAs for about two per SM, at least 64 tokens each.
void hd_split_plan(int B, int Hkv, int T, int *splits, int *tps) {
    const int segs = B * Hkv;
    const int want = (2 * sm_count() + segs - 1) / segs;
    const int most = (T + 63) / 64;
    int s = want < most ? want : most;
    if (s < 1) s = 1;
    *tps = (T + s - 1) / s;
    *splits = (T + *tps - 1) / *tps;
}

// R q times scale log2(e) for every (sequence, query head), kHdRows per warp.
template <int ND>
__global__ void __launch_bounds__(kHdThreads) attn_d_prep_kernel(const __grid_constant__ HdAttnArgs a) {
    constexpr int D = 32 * ND;
    extern __shared__ __align__(16) float hd_smem[];
    float *Rs = hd_smem;
    hd_load_R<D>(Rs, a.R);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)a.B * a.Hq;
    const int64_t r0 = ((int64_t)blockIdx.x * kHdWarps + warp) * kHdRows;
    if (r0 >= rows) return;
    float x[kHdRows][ND], y[kHdRows][ND];
#pragma unroll
    for (int r = 0; r < kHdRows; ++r)
#pragma unroll
        for (int k = 0; k < ND; ++k) x[r][k] = r0 + r < rows ? hd_load(a.q, a.q_dtype, (r0 + r) * D + lane + 32 * k) : 0.f;
    hd_rotate_rows<ND, false, kHdRows>(Rs, x, y, lane);
#pragma unroll
    for (int r = 0; r < kHdRows; ++r)
        if (r0 + r < rows)
#pragma unroll
            for (int k = 0; k < ND; ++k) a.qrot[(r0 + r) * D + lane + 32 * k] = y[r][k] * a.qscale;
}

template <int ND>
__global__ void __launch_bounds__(kHdThreads) attn_d_kernel(const __grid_constant__ HdAttnArgs a) {
    constexpr int D = 32 * ND;
    extern __shared__ __align__(16) float hd_smem[];
    float *qs = hd_smem;                              // [8 heads][D] this KV head's rotated queries
    float *ctab = qs + 8 * D;                         // key centroids [16] | value centroids [16]
    float *part = ctab + 32;                          // [8 warps][8 heads][2 + D]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y, sp = blockIdx.x;
    const float *qg = a.qrot + ((int64_t)b * a.Hq + kvh * a.G) * D;
    for (int i = threadIdx.x; i < a.G * D; i += blockDim.x) qs[i] = qg[i];
    if (threadIdx.x < 16) {
        ctab[threadIdx.x] = a.kc[threadIdx.x];
        ctab[16 + threadIdx.x] = a.vc[threadIdx.x];
    }
    __syncthreads();
    int L = a.T;
    if (a.seq_lens) {
        const int sl = a.seq_lens[b];
        L = sl < 0 ? 0 : (sl > a.T ? a.T : sl);
    }
    const int t0 = sp * a.tps, t1 = min(L, t0 + a.tps);
    const int KB = 2 + D * a.kbits / 8, VB = 2 + D * a.vbits / 8;
    const int64_t seg = ((int64_t)b * a.Hkv + kvh) * a.T_cap;
    // per head: the warp's running maximum (uniform), this lane's share of l, and the value sums of
    // dims lane + 32 k
    float m[8], l[8], acc[8][ND];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int k = 0; k < ND; ++k) acc[h][k] = 0.f;
    }
    // 32 tokens per warp step: lane = token for the scores, lane = dims for the value sums
    for (int base = t0 + 32 * warp; base < t1; base += 32 * kHdWarps) {
        const int t = base + lane;
        const bool valid = t < t1;
        const uint8_t *kb = a.k + (seg + (valid ? t : base)) * KB;
        float s[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) s[h] = 0.f;
        // the token's D codes, 16 bits at a time (blocks are 2-byte aligned)
        const uint16_t *kw = reinterpret_cast<const uint16_t *>(kb);
        if (a.kbits == 3) {
            for (int w = 0; w < D / 8; ++w) {   // 2-bit plane word w: dims 8w .. 8w + 7
                const uint32_t lo = kw[1 + w];
                const uint32_t hb = (kw[1 + D / 8 + (w >> 1)] >> (8 * (w & 1))) & 0xFFu;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float c = ctab[((lo >> (2 * e)) & 3u) | (((hb >> e) & 1u) << 2)];
                    const int j = 8 * w + e;
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        if (h < a.G) s[h] = fmaf(qs[h * D + j], c, s[h]);
                }
            }
        } else {
            const int per = 16 / a.kbits;        // codes per 16-bit word
            const uint32_t mask = (1u << a.kbits) - 1u;
            for (int w = 0; w < D / per; ++w) {
                const uint32_t word = kw[1 + w];
                for (int e = 0; e < per; ++e) {
                    const float c = ctab[(word >> (a.kbits * e)) & mask];
                    const int j = per * w + e;
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        if (h < a.G) s[h] = fmaf(qs[h * D + j], c, s[h]);
                }
            }
        }
        const float kn = __half2float(__ushort_as_half(kw[0]));
        float p[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            if (h >= a.G) break;
            const float sh = valid ? s[h] * kn : -INFINITY;
            float mx = sh;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kHdFull, mx, o));
            const float mn = fmaxf(m[h], mx);   // finite: the step holds at least one valid token
            const float corr = exp2f(m[h] - mn);
            p[h] = valid ? exp2f(sh - mn) : 0.f;
            l[h] = fmaf(l[h], corr, p[h]);
#pragma unroll
            for (int k = 0; k < ND; ++k) acc[h][k] *= corr;
            m[h] = mn;
        }
        // value sums: token base + tt broadcast to the warp, lanes over dims
        const int nt = min(32, t1 - base);
        for (int tt = 0; tt < nt; ++tt) {
            const uint8_t *vb = a.v + (seg + base + tt) * VB;
            const float vn = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(vb)));
            float vv[ND];
#pragma unroll
            for (int k = 0; k < ND; ++k) vv[k] = ctab[16 + hd_code<D>(vb, a.vbits, lane + 32 * k)] * vn;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                if (h >= a.G) break;
                const float ph = __shfl_sync(kHdFull, p[h], tt);
#pragma unroll
                for (int k = 0; k < ND; ++k) acc[h][k] = fmaf(ph, vv[k], acc[h][k]);
            }
        }
    }
    // l over the warp's lanes, then the warps' states into shared memory; warp h merges head h
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        if (h >= a.G) break;
        const float lw = hd_warp_sum(l[h]);
        float *pw = part + (warp * 8 + h) * (2 + D);
        if (lane == 0) {
            pw[0] = m[h];
            pw[1] = lw;
        }
#pragma unroll
        for (int k = 0; k < ND; ++k) pw[2 + lane + 32 * k] = acc[h][k];
    }
    __syncthreads();
    if (warp < a.G) {
        const int h = warp;
        float M = -INFINITY;
        for (int w = 0; w < kHdWarps; ++w) M = fmaxf(M, part[(w * 8 + h) * (2 + D)]);
        float lt = 0.f, o[ND];
#pragma unroll
        for (int k = 0; k < ND; ++k) o[k] = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kHdWarps; ++w) {
                const float *pw = part + (w * 8 + h) * (2 + D);
                const float f = pw[0] == -INFINITY ? 0.f : exp2f(pw[0] - M);
                lt = fmaf(pw[1], f, lt);
#pragma unroll
                for (int k = 0; k < ND; ++k) o[k] = fmaf(pw[2 + lane + 32 * k], f, o[k]);
            }
        }
        float *dst = a.ws + (((int64_t)b * a.Hq + kvh * a.G + h) * a.splits + sp) * (2 + D);
        if (lane == 0) {
            dst[0] = M;
            dst[1] = lt;
        }
#pragma unroll
        for (int k = 0; k < ND; ++k) dst[2 + lane + 32 * k] = o[k];
    }
}

// One warp per (sequence, query head): merge the splits, o = R^T (acc / l).
template <int ND>
__global__ void __launch_bounds__(kHdThreads) attn_d_combine_kernel(const __grid_constant__ HdAttnArgs a) {
    constexpr int D = 32 * ND;
    extern __shared__ __align__(16) float hd_smem[];
    float *Rs = hd_smem;
    hd_load_R<D>(Rs, a.R);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kHdWarps + warp;   // b * Hq + head
    if (row >= (int64_t)a.B * a.Hq) return;
    const float *src = a.ws + row * a.splits * (2 + D);
    float M = -INFINITY;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, src[s * (2 + D)]);
    float lt = 0.f, o[ND], x[ND];
#pragma unroll
    for (int k = 0; k < ND; ++k) o[k] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < a.splits; ++s) {
            const float *ps = src + s * (2 + D);
            const float f = ps[0] == -INFINITY ? 0.f : exp2f(ps[0] - M);
            lt = fmaf(ps[1], f, lt);
#pragma unroll
            for (int k = 0; k < ND; ++k) o[k] = fmaf(ps[2 + lane + 32 * k], f, o[k]);
        }
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;   // an empty sequence gives a zero row
#pragma unroll
    for (int k = 0; k < ND; ++k) o[k] *= inv;
    hd_rotate<ND, true>(Rs, o, x, lane);
#pragma unroll
    for (int k = 0; k < ND; ++k) a.out[row * D + lane + 32 * k] = x[k];
}

template <int ND>
int hd_launch_attn(const HdAttnArgs &a, cudaStream_t st) {
    constexpr int D = 32 * ND;
    static int done_p[64] = {0}, done_a[64] = {0}, done_c[64] = {0};
    const int smem_a = (8 * D + 32 + kHdWarps * 8 * (2 + D)) * 4;
    const int smem_r = D * (D + 1) * 4;
    if (set_smem_limit((const void *)attn_d_prep_kernel<ND>, smem_r, done_p) != TQ_OK) return TQ_ERR_CUDA;
    if (set_smem_limit((const void *)attn_d_kernel<ND>, smem_a, done_a) != TQ_OK) return TQ_ERR_CUDA;
    if (set_smem_limit((const void *)attn_d_combine_kernel<ND>, smem_r, done_c) != TQ_OK) return TQ_ERR_CUDA;
    const int64_t rows = (int64_t)a.B * a.Hq;
    attn_d_prep_kernel<ND><<<(int)((rows + kHdWarps * kHdRows - 1) / (kHdWarps * kHdRows)), kHdThreads, smem_r, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
    attn_d_kernel<ND><<<dim3(a.splits, a.Hkv, a.B), kHdThreads, smem_a, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
    attn_d_combine_kernel<ND><<<(int)((rows + kHdWarps - 1) / kHdWarps), kHdThreads, smem_r, st>>>(a);
    return launch_status();
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" size_t tq_block_bytes_d(int head_dim, int bits) { return (size_t)hd_block_bytes(head_dim, bits); }

extern "C" int tq_rotation_hadamard(int head_dim, tq_signs signs, float *R_host) {
    if (!R_host) return TQ_ERR_ARG;
    if (head_dim != 64 && head_dim != 128) return TQ_ERR_UNSUPPORTED;
    const float r = 1.f / std::sqrt((float)head_dim);
    for (int i = 0; i < head_dim; ++i)
        for (int j = 0; j < head_dim; ++j) {
            const float h = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1.f : 1.f;
            const float s = ((signs.w[j >> 5] >> (j & 31)) & 1u) ? -1.f : 1.f;
            R_host[i * head_dim + j] = h * s * r;
        }
    return TQ_OK;
}

static int hd_fill(HdArgs &a, const tq_codebook *cb) {
    for (int i = 0; i < 16; ++i) {
        a.c[i] = i < cb->levels ? cb->centroids[i] : 0.f;
        a.b[i] = i + 1 < cb->levels ? cb->boundaries[i] : INFINITY;
    }
    return TQ_OK;
}

extern "C" int tq_encode_kv_d(const void *x, int x_dtype, int64_t n_vec, int head_dim, const tq_codebook *cb,
                              const float *R, uint8_t *blocks, void *stream) {
    if (n_vec < 0 || !cb || !R || (n_vec > 0 && (!x || !blocks))) return TQ_ERR_ARG;
    if (!hd_dim_ok(head_dim) || !hd_codebook_ok(cb, head_dim) || dtype_bytes(x_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    if (!aligned(x, 4) || !aligned(R, 16)) return TQ_ERR_ALIGN;
    HdArgs a;
    std::memset(&a, 0, sizeof(a));
    a.x = x;
    a.blocks = blocks;
    a.R = R;
    a.n_vec = n_vec;
    a.bits = cb->bits;
    a.dt = x_dtype;
    hd_fill(a, cb);
    return hd_codec(a, head_dim, true, static_cast<cudaStream_t>(stream));
}

extern "C" int tq_decode_kv_d(const uint8_t *blocks, int64_t n_vec, int head_dim, const tq_codebook *cb,
                              const float *R, void *out, int out_dtype, void *stream) {
    if (n_vec < 0 || !cb || !R || (n_vec > 0 && (!blocks || !out))) return TQ_ERR_ARG;
    if (!hd_dim_ok(head_dim) || !hd_codebook_ok(cb, head_dim) || dtype_bytes(out_dtype) == 0)
        return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    if (!aligned(out, 4) || !aligned(R, 16)) return TQ_ERR_ALIGN;
    HdArgs a;
    std::memset(&a, 0, sizeof(a));
    a.blocks = const_cast<uint8_t *>(blocks);
    a.out = out;
    a.R = R;
    a.n_vec = n_vec;
    a.bits = cb->bits;
    a.dt = out_dtype;
    hd_fill(a, cb);
    return hd_codec(a, head_dim, false, static_cast<cudaStream_t>(stream));
}

extern "C" size_t tq_attn_workspace_bytes_d(int B, int Hq, int Hkv, int T_cap, int head_dim) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || T_cap <= 0 || Hq % Hkv || !hd_dim_ok(head_dim)) return 0;
    int splits, tps;
    hd_split_plan(B, Hkv, T_cap, &splits, &tps);
    return ((size_t)B * Hq * splits * (2 + head_dim) + (size_t)B * Hq * head_dim) * sizeof(float);
}

extern "C" int tq_attn_decode_d(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                                const uint8_t *v_blocks, const tq_codebook *vcb, const int32_t *seq_lens, int B,
                                int Hq, int Hkv, int T_cap, int T, int head_dim, float scale, const float *R,
                                float *out, void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k_blocks || !kcb || !v_blocks || !vcb || !R || !out || !workspace) return TQ_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T_cap <= 0 || T < 1 || T > T_cap || !std::isfinite(scale))
        return TQ_ERR_ARG;
    const int G = Hq / Hkv;
    if (G > 8 || !hd_dim_ok(head_dim) || !hd_codebook_ok(kcb, head_dim) || !hd_codebook_ok(vcb, head_dim) ||
        dtype_bytes(q_dtype) == 0)
        return TQ_ERR_UNSUPPORTED;
    if (!aligned(q, dtype_bytes(q_dtype)) || !aligned(out, 4) || !aligned(R, 16) || !aligned(workspace, 16))
        return TQ_ERR_ALIGN;
    if (workspace_bytes < tq_attn_workspace_bytes_d(B, Hq, Hkv, T_cap, head_dim)) return TQ_ERR_WORKSPACE;
    HdAttnArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k_blocks;
    a.v = v_blocks;
    a.seq_lens = seq_lens;
    a.R = R;
    a.ws = static_cast<float *>(workspace);
    a.out = out;
    a.q_dtype = q_dtype;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.T_cap = T_cap;
    a.T = T;
    a.kbits = kcb->bits;
    a.vbits = vcb->bits;
    hd_split_plan(B, Hkv, T, &a.splits, &a.tps);
    // the rotated queries after the partials of the plan for T_cap (the workspace's size)
    {
        int sc, tc;
        hd_split_plan(B, Hkv, T_cap, &sc, &tc);
        a.qrot = a.ws + (int64_t)B * Hq * sc * (2 + head_dim);
    }
    a.qscale = scale * 1.4426950408889634f;
    for (int i = 0; i < 16; ++i) {
        a.kc[i] = i < kcb->levels ? kcb->centroids[i] : 0.f;
        a.vc[i] = i < vcb->levels ? vcb->centroids[i] : 0.f;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (head_dim) {
        case 64: return hd_launch_attn<2>(a, st);
        case 96: return hd_launch_attn<3>(a, st);
        case 128: return hd_launch_attn<4>(a, st);
        case 160: return hd_launch_attn<5>(a, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}
