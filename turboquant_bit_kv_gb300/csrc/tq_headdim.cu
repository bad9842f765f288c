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
// This unit holds the CUDA-core codec kernels, the decode attention's query
// prep and combine kernels and the C ABI; bf16 / fp16 encodes of 1024 rows or
// more run on the tensor cores (tq_headdim_tc.cu), and so does the attention
// kernel itself (tq_headdim_mma.cuh).
//
// Codec kernels (CUDA cores, float32; d = 32 ND): a warp per row, lane l
// holds elements l + 32 k.  R sits in shared memory with rows padded to
// d + 1 floats, so that the 32 lanes reading one column (encode: outputs
// l + 32 k, input j) hit 32 different banks.  The rotation of a row is d
// shuffles of its inputs and d ND fused multiply-adds per lane.  Codes are
// the count of float32 boundaries <= y; norms are rounded once to fp16 and
// recomputed in double precision when the float32 norm lies within 2^-20 of
// an fp16 rounding boundary.  The codec kernels rotate four rows per warp at
// once, so every element of R read from shared memory serves four rows.
// Decode attention: a prep kernel rotates every query once (R q, scale
// log2(e) folded in; a small tiled product); the attention kernel (one CTA
// of 4 warps per (sequence, KV head, context split) on the tensor cores)
// writes one partial per head and split; a combine kernel merges the splits
// and rotates back (R^T, a small tiled product).  The three are chained as
// programmatic dependents; the split count is chosen from the attention
// kernel's occupancy so that the CTAs fill whole waves.

#include <cmath>
#include <cstring>

#include "tq_device.cuh"
#include "tq_headdim.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

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

// R into shared memory, rows padded to D + 1 floats: 16-byte loads (R is 16-byte aligned and a
// row holds D / 4 of them), all of a thread's loads issued before its stores.
template <int D>
__device__ __forceinline__ void hd_load_R(float *Rs, const float *R) {
    constexpr int N4 = D * D / 4;
    const float4 *R4 = reinterpret_cast<const float4 *>(R);
    for (int q0 = threadIdx.x; q0 < N4; q0 += 8 * blockDim.x) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int q = q0 + u * blockDim.x;
            if (q < N4) v[u] = __ldg(R4 + q);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int q = q0 + u * blockDim.x;
            if (q < N4) {
                float *d = Rs + (4 * q / D) * (D + 1) + (4 * q) % D;
                d[0] = v[u].x;
                d[1] = v[u].y;
                d[2] = v[u].z;
                d[3] = v[u].w;
            }
        }
    }
}

// out[r][k] = sum_j M(lane + 32 k, j) v[r]_j for NR rows of D inputs v (element j in lane j % 32,
// register j / 32): the rows of M are those of R (TRANSPOSE false: y = R v) or its columns
// (TRANSPOSE true: y = R^T v); every element of R read from shared memory serves NR rows.
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

}  // namespace

// Context splits of a (sequence, KV head).  A split is a whole number of 32-token chunks, at least
// kHdMinChunks of them (two warp steps per warp), so the most splits a context of T tokens takes is
// hd_max_splits(T); the workspace holds that many partials per (sequence, query head).
constexpr int kHdMinChunks = 16;

int hd_max_splits(int T) {
    const int s = ((T + 31) / 32) / kHdMinChunks;
    return s < 1 ? 1 : s;
}

// Of those split counts, the one with the shortest makespan for `slots` CTAs of `warps` warps
// resident at once: waves of CTAs times warp steps per CTA (plus one for the CTA's start and merge).
void hd_split_plan(int B, int Hkv, int T, int slots, int warps, int *splits, int *tps) {
    const int64_t segs = (int64_t)B * Hkv;
    const int C = (T + 31) / 32, smax = hd_max_splits(T);
    if (slots < 1) slots = 1;
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= smax; ++s) {
        const int64_t waves = (segs * s + slots - 1) / slots;
        const int64_t steps = ((C + s - 1) / s + warps - 1) / warps + 1;
        if (best_cost < 0 || waves * steps < best_cost) {
            best_cost = waves * steps;
            best = s;
        }
    }
    *tps = (C + best - 1) / best * 32;
    *splits = (T + *tps - 1) / *tps;
}

namespace {

// R q times scale log2(e) for every (sequence, query head): a small tiled product, one CTA per
// 32 rows x 32 outputs (R's 32 output rows and the 32 query rows staged in shared memory, rows padded
// to D + 1 floats); thread (tx, ty) forms outputs 32 c + tx of rows ty + 8 m, m < 4.
constexpr int kHdTile = 32;

template <int ND>
__global__ void __launch_bounds__(kHdThreads) attn_d_prep_kernel(const __grid_constant__ HdAttnArgs a) {
    constexpr int D = 32 * ND, P = D + 1;
    // the attention kernel may start now: its first copies do not depend on this grid
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(16) float hd_smem[];
    float *Rs = hd_smem;                  // [32 outputs][P]
    float *Qs = Rs + kHdTile * P;         // [32 rows][P]
    const int c0 = blockIdx.x * kHdTile;
    const int64_t rows = (int64_t)a.B * a.Hq, r0 = (int64_t)blockIdx.y * kHdTile;
    // R's 32 output rows: 16-byte loads, all of a thread's issued before its stores
    constexpr int N4 = kHdTile * D / 4;
    constexpr int U = (N4 + kHdThreads - 1) / kHdThreads;
    float4 rv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int q = threadIdx.x + u * kHdThreads;
        if (q < N4) rv[u] = __ldg(reinterpret_cast<const float4 *>(a.R + (int64_t)c0 * D) + q);
    }
    float qv[(kHdTile * D + kHdThreads - 1) / kHdThreads];
#pragma unroll
    for (int u = 0; u < (kHdTile * D + kHdThreads - 1) / kHdThreads; ++u) {
        const int i = threadIdx.x + u * kHdThreads, r = i / D;
        qv[u] = (i < kHdTile * D && r0 + r < rows) ? hd_load(a.q, a.q_dtype, r0 * D + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int q = threadIdx.x + u * kHdThreads;
        if (q < N4) {
            float *d = Rs + (4 * q / D) * P + (4 * q) % D;
            d[0] = rv[u].x;
            d[1] = rv[u].y;
            d[2] = rv[u].z;
            d[3] = rv[u].w;
        }
    }
#pragma unroll
    for (int u = 0; u < (kHdTile * D + kHdThreads - 1) / kHdThreads; ++u) {
        const int i = threadIdx.x + u * kHdThreads;
        if (i < kHdTile * D) Qs[(i / D) * P + i % D] = qv[u];
    }
    __syncthreads();
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int i = 0; i < D; ++i) {
        const float r = Rs[tx * P + i];
#pragma unroll
        for (int m = 0; m < 4; ++m) y[m] = fmaf(r, Qs[(ty + 8 * m) * P + i], y[m]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int64_t row = r0 + ty + 8 * m;
        if (row < rows) a.qrot[row * D + c0 + tx] = y[m] * a.qscale;
    }
}

// The merged, normalised value sums of one (sequence, query head) row, lanes over dims
// lane + 32 k: up to eight splits at a time, all their loads issued before any is used, folded
// into a running maximum.
template <int ND>
__device__ __forceinline__ void hd_merge_row(const HdAttnArgs &a, int64_t row, int lane, float (&o)[ND]) {
    constexpr int D = 32 * ND;
    const float *src = a.ws + row * a.splits * (2 + D);
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int k = 0; k < ND; ++k) o[k] = 0.f;
    for (int s0 = 0; s0 < a.splits; s0 += 8) {
        const int ns = min(8, a.splits - s0);
        float ms[8], ls[8], av[8][ND];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            ms[t] = -INFINITY;
            ls[t] = 0.f;
#pragma unroll
            for (int k = 0; k < ND; ++k) av[t][k] = 0.f;
            if (t < ns) {
                const float *ps = src + (s0 + t) * (2 + D);
                ms[t] = ps[0];
                ls[t] = ps[1];
#pragma unroll
                for (int k = 0; k < ND; ++k) av[t][k] = ps[2 + lane + 32 * k];
            }
        }
        float mn = M;
#pragma unroll
        for (int t = 0; t < 8; ++t) mn = fmaxf(mn, ms[t]);
        if (mn == -INFINITY) continue;   // no tokens so far
        const float cr = exp2f(M - mn);  // 0 while M is -inf
        L *= cr;
#pragma unroll
        for (int k = 0; k < ND; ++k) o[k] *= cr;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float f = ms[t] == -INFINITY ? 0.f : exp2f(ms[t] - mn);
            L = fmaf(ls[t], f, L);
#pragma unroll
            for (int k = 0; k < ND; ++k) o[k] = fmaf(av[t][k], f, o[k]);
        }
        M = mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;   // an empty sequence gives a zero row
#pragma unroll
    for (int k = 0; k < ND; ++k) o[k] *= inv;
}

// Merge the splits and rotate back, x = R^T (acc / l): one CTA per 16 rows x 32 outputs.  Warp w
// merges rows w and w + 8 into shared memory; R's 32 output columns are staged beside them (before
// the wait: R does not depend on the attention kernel); thread (tx, ty) forms outputs 32 c + tx of
// rows ty and ty + 8.
constexpr int kHdCRows = 16;

template <int ND>
__global__ void __launch_bounds__(kHdThreads) attn_d_combine_kernel(const __grid_constant__ HdAttnArgs a) {
    constexpr int D = 32 * ND, P = D + 1;
    extern __shared__ __align__(16) float hd_smem[];
    float *Os = hd_smem;                  // [16 rows][P]: merged, normalised value sums
    float *Rc = Os + kHdCRows * P;        // [D][33]: R[j][32 c + t]
    const int c0 = blockIdx.x * kHdTile;
    const int64_t rows = (int64_t)a.B * a.Hq, r0 = (int64_t)blockIdx.y * kHdCRows;
    for (int i = threadIdx.x; i < D * kHdTile; i += blockDim.x) {
        const int j = i / kHdTile, t = i % kHdTile;
        Rc[j * (kHdTile + 1) + t] = a.R[(int64_t)j * D + c0 + t];
    }
    // the partials come from the attention kernel this one depends on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < kHdCRows / kHdWarps; ++m) {
        const int rr = warp + kHdWarps * m;
        float o[ND];
        if (r0 + rr < rows) hd_merge_row<ND>(a, r0 + rr, lane, o);
        else
#pragma unroll
            for (int k = 0; k < ND; ++k) o[k] = 0.f;
#pragma unroll
        for (int k = 0; k < ND; ++k) Os[rr * P + lane + 32 * k] = o[k];
    }
    __syncthreads();
    const int tx = lane, ty = warp;
    float x[kHdCRows / kHdWarps] = {};
#pragma unroll 8
    for (int j = 0; j < D; ++j) {
        const float r = Rc[j * (kHdTile + 1) + tx];
#pragma unroll
        for (int m = 0; m < kHdCRows / kHdWarps; ++m) x[m] = fmaf(r, Os[(ty + kHdWarps * m) * P + j], x[m]);
    }
#pragma unroll
    for (int m = 0; m < kHdCRows / kHdWarps; ++m) {
        const int64_t row = r0 + ty + kHdWarps * m;
        if (row < rows) a.out[row * D + c0 + tx] = x[m];
    }
}

template <int ND>
int hd_launch_attn(HdAttnArgs &a, cudaStream_t st) {
    constexpr int D = 32 * ND;
    static int done_p[64] = {0}, done_c[64] = {0};
    const int smem_p = 2 * kHdTile * (D + 1) * 4, smem_c = (kHdCRows * (D + 1) + D * (kHdTile + 1)) * 4;
    if (set_smem_limit((const void *)attn_d_prep_kernel<ND>, smem_p, done_p) != TQ_OK) return TQ_ERR_CUDA;
    if (set_smem_limit((const void *)attn_d_combine_kernel<ND>, smem_c, done_c) != TQ_OK) return TQ_ERR_CUDA;
    // the attention kernel (tq_headdim_mma.cu) covers every width and up to eight heads per KV head
    // (the only shapes the entry point accepts); its plan sets the split count from its occupancy
    const int plan = hd_attn_mma_plan(a, D);
    if (plan == 1) return TQ_ERR_UNSUPPORTED;
    if (plan != TQ_OK) return plan;
    const int64_t rows = (int64_t)a.B * a.Hq;
    const dim3 tiles(D / kHdTile, (unsigned)((rows + kHdTile - 1) / kHdTile));
    attn_d_prep_kernel<ND><<<tiles, kHdThreads, smem_p, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
    // the attention and combine kernels are programmatic dependents of the kernel before them: each
    // starts its independent part (first copies; R) while its predecessor finishes
    const int r = hd_attn_mma_launch(a, D, st);
    if (r != TQ_OK) return r;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kHdThreads);
    cfg.gridDim = dim3(D / kHdTile, (unsigned)((rows + kHdCRows - 1) / kHdCRows));
    cfg.dynamicSmemBytes = smem_c;
    if (cudaLaunchKernelEx(&cfg, attn_d_combine_kernel<ND>, a) != cudaSuccess) return TQ_ERR_CUDA;
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
    // bf16 / fp16 rows: the tensor-core kernel (1: not its form, e.g. few rows)
    const int r = hd_encode_tc(x, x_dtype, n_vec, head_dim, cb, R, blocks, static_cast<cudaStream_t>(stream));
    if (r != 1) return r;
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
    return ((size_t)B * Hq * hd_max_splits(T_cap) * (2 + head_dim) + (size_t)B * Hq * head_dim) * sizeof(float);
}

extern "C" int tq_attn_decode_d(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                                const uint8_t *v_blocks, const tq_codebook *vcb, const int32_t *seq_lens, int B,
                                int Hq, int Hkv, int T_cap, int T, int head_dim, float scale, const float *R,
                                float *out, void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k_blocks || !kcb || !v_blocks || !vcb || !R || !out || !workspace) return TQ_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T_cap <= 0 || T < 1 || T > T_cap || (T_cap & 7) ||
        !std::isfinite(scale))
        return TQ_ERR_ARG;
    const int G = Hq / Hkv;
    // (grid limits: the attention grid is [splits][Hkv][B], the prep and combine grids take 32 and 16
    // (sequence, query head) rows per CTA row)
    if (G > 8 || !hd_dim_ok(head_dim) || !hd_codebook_ok(kcb, head_dim) || !hd_codebook_ok(vcb, head_dim) ||
        dtype_bytes(q_dtype) == 0 || B > 65535 || Hkv > 65535 || (int64_t)B * Hq > 65535LL * 16)
        return TQ_ERR_UNSUPPORTED;
    if (!aligned(q, dtype_bytes(q_dtype)) || !aligned(k_blocks, 16) || !aligned(v_blocks, 16) || !aligned(out, 4) ||
        !aligned(R, 16) || !aligned(workspace, 16))
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
    // the rotated queries after room for the most partials a context of T_cap tokens takes (the
    // split plan itself is made at launch, from the kernel's occupancy)
    a.qrot = a.ws + (int64_t)B * Hq * hd_max_splits(T_cap) * (2 + head_dim);
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
