// Quantise-on-insert, dequantise and QJL residual sketch kernels (sm_103a),
// with their C-ABI entry points and the storage serialise / deserialise
// driver built on them.
//
// Pages restated:
//  * "TurboQuant KV Cache Compression — Spec": As-Built Notes (H (D x) order,
//    L2-norm normalisation), Algorithm Detail Steps 1-3, Hadamard Transform
//    Detail, Overview (dequantise = centroid lookup + rotate back).
//  * "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)" section 4: block
//    structures (fp16 norm, 2-bit codes 4 per byte, 3-bit split planes, 4-bit
//    nibbles).
//  * "RotorQuant KV Cache Compression": Key Compression Workflow (residual,
//    its norm, sign of the sketched residual).
//  * "lmcache.v1.distributed.serde.turboquant": Configuration and Tensor
//    Layout (raw first | compressed middle | raw last layers).
//
// Design (QJL): one thread owns one 128-element vector.  A CTA of
// 128 threads stages a tile of 128 rows into shared memory with 16-byte
// cp.async copies (double buffered across a persistent grid), each thread
// holds its vector in registers as 64 packed float2 pairs and runs the whole
// Walsh-Hadamard transform there with packed adds, and the CTA stores its
// tile to HBM with coalesced 16-byte stores.  The quantise-on-insert kernel
// lives in tq_encode.cu, the dequantise kernel in tq_decode.cu.

#include <algorithm>
#include <cmath>
#include <cstring>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kThreads = 128;  // vectors per tile, one per thread

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

int set_smem_limit(const void *kernel, int bytes, int *done_for_device) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev < 64 && done_for_device[dev] >= bytes) return TQ_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return TQ_ERR_CUDA;
    if (dev < 64) done_for_device[dev] = bytes;
    return TQ_OK;
}

// Sign table in shared memory.  For 16-bit inputs/outputs: word w holds the
// sign bits of elements 2w (bit 15) and 2w+1 (bit 31).  For float32: word j
// holds element j's sign in bit 31.
__device__ __forceinline__ void build_sign_tables(uint32_t *sg16, uint32_t *sg32, const uint32_t (&s)[4]) {
    for (int j = threadIdx.x; j < kD; j += blockDim.x) {
        uint32_t bit = (s[j >> 5] >> (j & 31)) & 1u;
        sg32[j] = bit << 31;
    }
    for (int w = threadIdx.x; w < kD / 2; w += blockDim.x) {
        int j = 2 * w;
        uint32_t b0 = (s[j >> 5] >> (j & 31)) & 1u;
        uint32_t b1 = (s[(j + 1) >> 5] >> ((j + 1) & 31)) & 1u;
        sg16[w] = (b0 << 15) | (b1 << 31);
    }
}

// Row of 128 inputs (dtype DT) in shared memory -> sign-flipped pairs.
template <int DT>
__device__ __forceinline__ void load_signed_pairs(const uint8_t *row, const uint32_t *sg16,
                                                  const uint32_t *sg32, float2 (&p)[64]) {
    if constexpr (DT == TQ_F32) {
        const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
        const uint4 *s4 = reinterpret_cast<const uint4 *>(sg32);
        float v[128];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            uint4 w = r4[k], s = s4[k];
            v[4 * k + 0] = __uint_as_float(w.x ^ s.x);
            v[4 * k + 1] = __uint_as_float(w.y ^ s.y);
            v[4 * k + 2] = __uint_as_float(w.z ^ s.z);
            v[4 * k + 3] = __uint_as_float(w.w ^ s.w);
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) p[i] = make_float2(v[i], v[i + 64]);
    } else {
        const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
        const uint4 *s4 = reinterpret_cast<const uint4 *>(sg16);
        uint32_t w[64];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            uint4 a = r4[k], s = s4[k];
            w[4 * k + 0] = a.x ^ s.x;
            w[4 * k + 1] = a.y ^ s.y;
            w[4 * k + 2] = a.z ^ s.z;
            w[4 * k + 3] = a.w ^ s.w;
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            uint32_t a = w[i >> 1], b = w[32 + (i >> 1)];
            if constexpr (DT == TQ_BF16) {
                p[i] = (i & 1) ? make_float2(bf16_bits_hi(a), bf16_bits_hi(b))
                               : make_float2(bf16_bits_lo(a), bf16_bits_lo(b));
            } else {
                float2 fa = __half22float2(*reinterpret_cast<__half2 *>(&a));
                float2 fb = __half22float2(*reinterpret_cast<__half2 *>(&b));
                p[i] = (i & 1) ? make_float2(fa.y, fb.y) : make_float2(fa.x, fb.x);
            }
        }
    }
}

// Read a block (norm + code words) from a 2-byte aligned shared address.
template <int BITS>
__device__ __forceinline__ unsigned short load_block_smem(const uint8_t *base,
                                                          uint32_t (&cw)[BlockFmt<BITS>::kWords]) {
#pragma unroll
    for (int k = 0; k < BlockFmt<BITS>::kWords; ++k) cw[k] = lds_u32_a2(base + 2 + 4 * k);
    return *reinterpret_cast<const uint16_t *>(base);
}

// Code j of a packed block.
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&cw)[BlockFmt<BITS>::kWords], int j) {
    if constexpr (BITS == 4) return (cw[j >> 3] >> (4 * (j & 7))) & 15u;
    else if constexpr (BITS == 2) return (cw[j >> 4] >> (2 * (j & 15))) & 3u;
    else return ((cw[j >> 4] >> (2 * (j & 15))) & 3u) | (((cw[8 + (j >> 5)] >> (j & 31)) & 1u) << 2);
}

// Rotated-domain reconstruction c[code] as pairs.
template <int BITS>
__device__ __forceinline__ void lut_pairs(const uint32_t (&cw)[BlockFmt<BITS>::kWords], const float *lut,
                                          float2 (&p)[64]) {
#pragma unroll
    for (int i = 0; i < 64; ++i) p[i] = make_float2(lut[code_at<BITS>(cw, i)], lut[code_at<BITS>(cw, i + 64)]);
}

template <int DT>
__device__ __forceinline__ void stage_rows(uint8_t *st, const uint8_t *x, int64_t stride, int nv) {
    constexpr int cpr = InFmt<DT>::kRowBytes / 16;
    for (int c = threadIdx.x; c < nv * cpr; c += kThreads) {
        int r = c / cpr, col = c - r * cpr;
        cp_async16(st + r * InFmt<DT>::kPitch + col * 16, x + r * stride + col * 16);
    }
}


template <int BITS>
__device__ __forceinline__ void stage_blocks(uint8_t *st, const uint8_t *src, int64_t stride, int nv,
                                             int contiguous) {
    constexpr int BB = BlockFmt<BITS>::kBytes;
    if (contiguous) {
        int nbytes = nv * BB, nch = nbytes >> 4;
        for (int c = threadIdx.x; c < nch; c += kThreads) cp_async16(st + 16 * c, src + 16 * c);
        for (int h = (nch << 3) + threadIdx.x; h < (nbytes >> 1); h += kThreads)
            reinterpret_cast<uint16_t *>(st)[h] = reinterpret_cast<const uint16_t *>(src)[h];
    } else {
        int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int r = warp * 32; r < min(nv, warp * 32 + 32); ++r) {
            const uint16_t *s = reinterpret_cast<const uint16_t *>(src + r * stride);
            uint16_t *d = reinterpret_cast<uint16_t *>(st + r * BB);
            for (int h = lane; h < BB / 2; h += 32) d[h] = s[h];
        }
    }
}

struct QjlArgs {
    const uint8_t *k;
    int64_t k_stride;  // bytes
    const uint8_t *blocks;
    int64_t block_stride;
    int64_t n_vec;
    const float *S;
    uint8_t *bits;
    uint16_t *rn;
    DevCodebook cb;
    uint32_t signs[4];
};

// One thread per key: k_mse by the dequantiser, residual in registers,
// sketch S r against S held in shared memory in pair layout
// (S[i][j], S[i][j+64]) so that each product is one packed FMA.
template <int BITS, int DT>
__global__ void __launch_bounds__(kThreads) qjl_encode_kernel(QjlArgs a) {
    constexpr int BB = BlockFmt<BITS>::kBytes;
    constexpr int PITCH = InFmt<DT>::kPitch;
    extern __shared__ __align__(16) uint8_t smem[];
    float2 *Sp = reinterpret_cast<float2 *>(smem);                 // [128][64] pairs = 64 KB
    uint8_t *krows = smem + 128 * 64 * 8;                          // kThreads * PITCH
    uint8_t *kblk = krows + kThreads * PITCH;                      // kThreads * BB (padded)
    uint32_t *sg16 = reinterpret_cast<uint32_t *>(kblk + ((kThreads * BB + 15) & ~15));
    uint32_t *sg32 = sg16 + 64;
    float *lut = reinterpret_cast<float *>(sg32 + 128);
    build_sign_tables(sg16, sg32, a.signs);
    for (int i = threadIdx.x; i < 16; i += kThreads) lut[i] = a.cb.c[i];
    for (int e = threadIdx.x; e < 128 * 64; e += kThreads) {
        int i = e >> 6, j = e & 63;
        Sp[e] = make_float2(a.S[i * 128 + j], a.S[i * 128 + j + 64]);
    }
    const float inv_rs = 0.08838834764831845f;
    const int64_t ntiles = (a.n_vec + kThreads - 1) / kThreads;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t v0 = tile * kThreads;
        const int nv = (int)min64(kThreads, a.n_vec - v0);
        __syncthreads();
        stage_rows<DT>(krows, a.k + v0 * a.k_stride, a.k_stride, nv);
        cp_async_commit();
        stage_blocks<BITS>(kblk, a.blocks + v0 * a.block_stride, a.block_stride, nv, 0);
        cp_async_wait<0>();
        __syncthreads();
        const int t = threadIdx.x;
        if (t < nv) {
            uint32_t cw[BlockFmt<BITS>::kWords];
            unsigned short n16 = load_block_smem<BITS>(kblk + t * BB, cw);
            float2 r[64];
            lut_pairs<BITS>(cw, lut, r);
            fwht128(r);
            const float f = __half2float(__ushort_as_half(n16)) * inv_rs;
            // k_mse_j = s_j * f * (H c)_j; residual r = k - k_mse, with the
            // signs applied to k first so both terms share them: s_j * (s_j k_j - f (H c)_j).
            float2 ks[64];
            load_signed_pairs<DT>(krows + t * PITCH, sg16, sg32, ks);
            const float2 mf = make_float2(-f, -f);
#pragma unroll
            for (int i = 0; i < 64; ++i) r[i] = __ffma2_rn(r[i], mf, ks[i]);
            // r now holds D * residual; norms are sign-blind.  The residual is
            // itself a float32 quantity, so its norm is rounded from float32.
            unsigned short rn16 = __half_as_ushort(__float2half_rn(sqrtf(sumsq128(r))));
            // Undo D so r is the residual itself.
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                uint32_t sx = sg32[i], sy = sg32[i + 64];
                r[i] = make_float2(__uint_as_float(__float_as_uint(r[i].x) ^ sx),
                                   __uint_as_float(__float_as_uint(r[i].y) ^ sy));
            }
            uint32_t bw[4] = {0u, 0u, 0u, 0u};
            for (int i = 0; i < 128; ++i) {
                const float4 *row = reinterpret_cast<const float4 *>(Sp + i * 64);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float4 s4 = row[j];
                    acc0 = __ffma2_rn(make_float2(s4.x, s4.y), r[2 * j], acc0);
                    acc1 = __ffma2_rn(make_float2(s4.z, s4.w), r[2 * j + 1], acc1);
                }
                float2 acc = add2(acc0, acc1);
                float proj = acc.x + acc.y;
                bw[i >> 5] |= (proj >= 0.f ? 1u : 0u) << (i & 31);
            }
            *reinterpret_cast<uint4 *>(a.bits + (v0 + t) * 16) = make_uint4(bw[0], bw[1], bw[2], bw[3]);
            a.rn[v0 + t] = rn16;
        }
    }
}

DevCodebook to_dev(const tq_codebook *cb) {
    DevCodebook d;
    for (int i = 0; i < 16; ++i) d.c[i] = cb->centroids[i];
    for (int i = 0; i < 15; ++i) d.b[i] = cb->boundaries[i];
    d.bits = cb->bits;
    return d;
}

bool codebook_ok(const tq_codebook *cb) {
    return cb && cb->head_dim == kD && cb->bits >= 2 && cb->bits <= 4 && cb->levels == (1 << cb->bits);
}

template <int BITS, int DT>
int launch_qjl(const QjlArgs &a, cudaStream_t st) {
    static int done[64] = {0};
    const int smem = 128 * 64 * 8 + kThreads * InFmt<DT>::kPitch + ((kThreads * BlockFmt<BITS>::kBytes + 15) & ~15) +
                     (64 + 128 + 16) * 4;
    if (set_smem_limit((const void *)qjl_encode_kernel<BITS, DT>, smem, done) != TQ_OK) return TQ_ERR_CUDA;
    const int64_t ntiles = (a.n_vec + kThreads - 1) / kThreads;
    int grid = (int)min64(ntiles, (int64_t)sm_count());
    qjl_encode_kernel<BITS, DT><<<grid, kThreads, smem, st>>>(a);
    return launch_status();
}

}  // namespace tq

using namespace tq;

#define TQ_DISPATCH(LAUNCH, BITS, DT, ARGS, STREAM)                                    \
    do {                                                                               \
        int _r = TQ_ERR_UNSUPPORTED;                                                   \
        switch ((BITS) * 8 + (DT)) {                                                   \
            case 2 * 8 + TQ_F32: _r = LAUNCH<2, TQ_F32>(ARGS, STREAM); break;          \
            case 2 * 8 + TQ_BF16: _r = LAUNCH<2, TQ_BF16>(ARGS, STREAM); break;        \
            case 2 * 8 + TQ_F16: _r = LAUNCH<2, TQ_F16>(ARGS, STREAM); break;          \
            case 3 * 8 + TQ_F32: _r = LAUNCH<3, TQ_F32>(ARGS, STREAM); break;          \
            case 3 * 8 + TQ_BF16: _r = LAUNCH<3, TQ_BF16>(ARGS, STREAM); break;        \
            case 3 * 8 + TQ_F16: _r = LAUNCH<3, TQ_F16>(ARGS, STREAM); break;          \
            case 4 * 8 + TQ_F32: _r = LAUNCH<4, TQ_F32>(ARGS, STREAM); break;          \
            case 4 * 8 + TQ_BF16: _r = LAUNCH<4, TQ_BF16>(ARGS, STREAM); break;        \
            case 4 * 8 + TQ_F16: _r = LAUNCH<4, TQ_F16>(ARGS, STREAM); break;          \
            default: break;                                                            \
        }                                                                              \
        return _r;                                                                     \
    } while (0)

extern "C" int tq_qjl_encode(const void *k, int k_dtype, int64_t n_vec, int64_t k_stride_elems,
                             const uint8_t *k_blocks, int64_t block_stride_bytes, const tq_codebook *cb,
                             tq_signs signs, const float *S, uint8_t *qjl_bits, uint16_t *res_norm_f16,
                             void *stream) {
    if (n_vec < 0 || !cb) return TQ_ERR_ARG;
    if (!codebook_ok(cb) || dtype_bytes(k_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    const int es = dtype_bytes(k_dtype);
    const int64_t bb = (int64_t)tq_block_bytes(cb->bits);
    if (!k || !k_blocks || !S || !qjl_bits || !res_norm_f16 || k_stride_elems < kD || block_stride_bytes < bb)
        return TQ_ERR_ARG;
    if (!aligned(k, 16) || (k_stride_elems * es) % 16 || !aligned(k_blocks, 2) || (block_stride_bytes & 1) ||
        !aligned(qjl_bits, 16) || !aligned(res_norm_f16, 2) || !aligned(S, 4))
        return TQ_ERR_ALIGN;
    const int tc = qjl_encode_tc(k, k_dtype, n_vec, k_stride_elems * es, k_blocks, block_stride_bytes, cb->bits,
                                 cb->centroids, signs.w, S, qjl_bits, res_norm_f16, (cudaStream_t)stream);
    if (tc != 1) return tc;
    QjlArgs a;
    a.k = static_cast<const uint8_t *>(k);
    a.k_stride = k_stride_elems * es;
    a.blocks = k_blocks;
    a.block_stride = block_stride_bytes;
    a.n_vec = n_vec;
    a.S = S;
    a.bits = qjl_bits;
    a.rn = res_norm_f16;
    a.cb = to_dev(cb);
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    TQ_DISPATCH(launch_qjl, cb->bits, k_dtype, a, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- serde

namespace {

struct SerdeGeom {
    int64_t L, T, hidden, H, nblk, bs, qs, qe, kbb, vbb, slot, es;
    int64_t raw_first, comp;  // bytes
};

int serde_geom(int elem_dtype, int num_layers, int num_tokens, int hidden_dim, int head_dim, int block_size,
               int skip_first, int skip_last, const tq_codebook *kcb, const tq_codebook *vcb, SerdeGeom *g) {
    if (!kcb || !vcb || num_layers < 0 || num_tokens < 0 || hidden_dim <= 0 || block_size <= 0 ||
        skip_first < 0 || skip_last < 0)
        return TQ_ERR_ARG;
    if (head_dim != kD || hidden_dim % kD || !codebook_ok(kcb) || !codebook_ok(vcb) ||
        (elem_dtype != TQ_BF16 && elem_dtype != TQ_F16))
        return TQ_ERR_UNSUPPORTED;
    g->L = num_layers;
    g->T = num_tokens;
    g->hidden = hidden_dim;
    g->H = hidden_dim / kD;
    g->bs = block_size;
    g->nblk = (num_tokens + block_size - 1) / block_size;
    g->qs = std::min(skip_first, num_layers);
    g->qe = std::max<int64_t>(g->qs, num_layers - skip_last);
    g->kbb = (int64_t)tq_block_bytes(kcb->bits);
    g->vbb = (int64_t)tq_block_bytes(vcb->bits);
    g->slot = g->kbb + g->vbb;
    g->es = 2;
    g->raw_first = 2 * g->qs * g->T * g->hidden * g->es;
    g->comp = (g->qe - g->qs) * g->nblk * g->bs * g->H * g->slot;
    return TQ_OK;
}

}  // namespace

extern "C" int tq_serde_serialize(const void *src, int elem_dtype, int num_layers, int num_tokens,
                                  int hidden_dim, int head_dim, int block_size, int skip_first, int skip_last,
                                  const tq_codebook *kcb, const tq_codebook *vcb, tq_signs signs, uint8_t *dst,
                                  void *stream) {
    SerdeGeom g;
    int r = serde_geom(elem_dtype, num_layers, num_tokens, hidden_dim, head_dim, block_size, skip_first, skip_last,
                       kcb, vcb, &g);
    if (r != TQ_OK) return r;
    if (!src || !dst) return TQ_ERR_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16)) return TQ_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    const uint8_t *s = static_cast<const uint8_t *>(src);
    const int64_t layer_bytes = g.T * g.hidden * g.es;  // one [T, hidden] plane
    const int64_t layer_elems = g.T * g.hidden;
    // raw first layers: keys [0, qs) then values [0, qs)
    if (g.qs > 0) {
        if (cudaMemcpyAsync(dst, s, g.qs * layer_bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(dst + g.qs * layer_bytes, s + g.L * layer_bytes, g.qs * layer_bytes,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return TQ_ERR_CUDA;
    }
    uint8_t *comp = dst + g.raw_first;
    const int64_t Lc = g.qe - g.qs;
    const int64_t layer_slots = g.nblk * g.bs * g.H;
    if (Lc > 0) {
        const int es = g.es;
        if (g.T % g.bs == 0) {
            // one paired launch fills whole slots (K block then V block) when both halves use the
            // same codebook; otherwise one launch per half
            const bool same = kcb->bits == vcb->bits && g.slot == 2 * g.kbb &&
                              memcmp(kcb->centroids, vcb->centroids, sizeof(kcb->centroids)) == 0 &&
                              memcmp(kcb->boundaries, vcb->boundaries, sizeof(kcb->boundaries)) == 0;
            r = same ? encode_kv_pair(s + g.qs * layer_bytes, s + (g.L + g.qs) * layer_bytes, elem_dtype,
                                      Lc * g.T * g.H, kD, kcb, signs, comp, st)
                     : 1;
            if (r == 1) {
                r = tq_encode_kv(s + g.qs * layer_bytes, elem_dtype, Lc * g.T * g.H, kD, kcb, signs, comp, g.slot,
                                 nullptr, stream);
                if (r != TQ_OK) return r;
                r = tq_encode_kv(s + (g.L + g.qs) * layer_bytes, elem_dtype, Lc * g.T * g.H, kD, vcb, signs,
                                 comp + g.kbb, g.slot, nullptr, stream);
            }
            if (r != TQ_OK) return r;
        } else {
            for (int64_t li = 0; li < Lc; ++li) {
                const int64_t l = g.qs + li;
                uint8_t *lay = comp + li * layer_slots * g.slot;
                r = tq_encode_kv(s + l * layer_elems * es, elem_dtype, g.T * g.H, kD, kcb, signs, lay, g.slot,
                                 nullptr, stream);
                if (r != TQ_OK) return r;
                r = tq_encode_kv(s + (g.L + l) * layer_elems * es, elem_dtype, g.T * g.H, kD, vcb, signs,
                                 lay + g.kbb, g.slot, nullptr, stream);
                if (r != TQ_OK) return r;
                const int64_t pad = (g.nblk * g.bs - g.T) * g.H * g.slot;
                if (cudaMemsetAsync(lay + g.T * g.H * g.slot, 0, pad, st) != cudaSuccess) return TQ_ERR_CUDA;
            }
        }
    }
    // raw last layers: keys [qe, L) then values [qe, L)
    const int64_t nl = g.L - g.qe;
    if (nl > 0) {
        uint8_t *last = comp + g.comp;
        if (cudaMemcpyAsync(last, s + g.qe * layer_bytes, nl * layer_bytes, cudaMemcpyDeviceToDevice, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(last + nl * layer_bytes, s + (g.L + g.qe) * layer_bytes, nl * layer_bytes,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return TQ_ERR_CUDA;
    }
    return TQ_OK;
}

extern "C" int tq_serde_deserialize(const uint8_t *src, int elem_dtype, int num_layers, int num_tokens,
                                    int hidden_dim, int head_dim, int block_size, int skip_first, int skip_last,
                                    const tq_codebook *kcb, const tq_codebook *vcb, tq_signs signs, void *dst,
                                    void *stream) {
    SerdeGeom g;
    int r = serde_geom(elem_dtype, num_layers, num_tokens, hidden_dim, head_dim, block_size, skip_first, skip_last,
                       kcb, vcb, &g);
    if (r != TQ_OK) return r;
    if (!src || !dst) return TQ_ERR_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16)) return TQ_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *d = static_cast<uint8_t *>(dst);
    const int64_t layer_bytes = g.T * g.hidden * g.es;
    if (g.qs > 0) {
        if (cudaMemcpyAsync(d, src, g.qs * layer_bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(d + g.L * layer_bytes, src + g.qs * layer_bytes, g.qs * layer_bytes,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return TQ_ERR_CUDA;
    }
    const uint8_t *comp = src + g.raw_first;
    const int64_t Lc = g.qe - g.qs;
    const int64_t layer_slots = g.nblk * g.bs * g.H;
    if (Lc > 0 && g.T % g.bs == 0) {
        // no padding slots: the compressed keys (values) of all middle layers are one run of
        // slots and one run of rows
        r = tq_decode_kv(comp, g.slot, Lc * g.T * g.H, kcb, signs, d + g.qs * layer_bytes, elem_dtype, kD, stream);
        if (r != TQ_OK) return r;
        r = tq_decode_kv(comp + g.kbb, g.slot, Lc * g.T * g.H, vcb, signs, d + (g.L + g.qs) * layer_bytes,
                         elem_dtype, kD, stream);
        if (r != TQ_OK) return r;
    }
    for (int64_t li = 0; li < Lc && g.T % g.bs != 0; ++li) {
        const int64_t l = g.qs + li;
        const uint8_t *lay = comp + li * layer_slots * g.slot;
        r = tq_decode_kv(lay, g.slot, g.T * g.H, kcb, signs, d + l * layer_bytes, elem_dtype, kD, stream);
        if (r != TQ_OK) return r;
        r = tq_decode_kv(lay + g.kbb, g.slot, g.T * g.H, vcb, signs, d + (g.L + l) * layer_bytes, elem_dtype, kD,
                         stream);
        if (r != TQ_OK) return r;
    }
    const int64_t nl = g.L - g.qe;
    if (nl > 0) {
        const uint8_t *last = comp + g.comp;
        if (cudaMemcpyAsync(d + g.qe * layer_bytes, last, nl * layer_bytes, cudaMemcpyDeviceToDevice, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(d + (g.L + g.qe) * layer_bytes, last + nl * layer_bytes, nl * layer_bytes,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return TQ_ERR_CUDA;
    }
    return TQ_OK;
}
