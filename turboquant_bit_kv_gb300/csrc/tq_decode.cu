// Dequantise (tq_decode_kv) for sm_103a.
//
// Restates "TurboQuant KV Cache Compression — Spec", Overview and Hadamard
// Transform Detail (dequantise: centroid lookup, scale by the stored norm,
// rotate back; H is symmetric with H H = 128 I, so x = n D H c / sqrt(128)),
// and "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)" section 4 (block =
// fp16 norm + packed codes; 3-bit codes in a 2-bit plane and a 1-bit plane).
//
// Work split: two threads own one vector, 64 elements each, in the pair
// layout of fwht_pair128 (thread h holds elements 16c + 8h + k).  A warp
// decodes 16 vectors per tile with no CTA-wide synchronisation: it stages
// its 16 blocks with cp.async (double buffered over a persistent grid), turns
// each pair of codes into two float32 centroids with one 8-byte lookup in a
// lane-replicated table (entry * 256 + lane * 8: conflict-free), runs the
// transform in registers, scales by n / sqrt(128), converts, applies the
// signs and stores each thread's 8-element runs with 16-byte streaming
// stores straight into the output rows.

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kDecRows = 16;               // vectors per warp tile
constexpr int kStridedPitch = 72;          // staged block of a strided input: 18 words
constexpr int kSpanMaxStride = 144;        // strides up to this stage the 16 blocks' whole byte span

template <int BITS>
struct DecGeo {
    static constexpr int BB = 2 + 16 * BITS;
    static constexpr int kLutEntries = BITS == 4 ? 256 : BITS == 3 ? 64 : 16;
    static constexpr int kLutBytes = kLutEntries * 256;
    static constexpr int kStage = kDecRows * kSpanMaxStride + 32;   // >= 16 * 72 and >= 16 * BB
    static constexpr int kSmem = kLutBytes + (64 + 128) * 4 + kDecWarps * 2 * kStage;
    static_assert(kStage >= kDecRows * BB, "stage");
};

struct DecArgs {
    const uint8_t *blocks;
    int64_t block_stride;
    int64_t n_vec;
    uint8_t *out;
    int64_t out_stride;   // bytes
    int contiguous;       // block_stride == block bytes and 16-byte aligned base
    int span;             // otherwise, block_stride <= kSpanMaxStride: stage the tile's whole byte span
    float c[16];
    uint32_t signs[4];
};

// Codes of the two elements of a pair-table entry (4-bit: the code byte, low
// nibble first; 2-bit: a nibble; 3-bit: the 2-bit-plane nibble | the two
// high-plane bits << 4).
template <int BITS>
__device__ __forceinline__ void entry_codes(int e, int &c0, int &c1) {
    if constexpr (BITS == 4) {
        c0 = e & 15;
        c1 = e >> 4;
    } else if constexpr (BITS == 2) {
        c0 = e & 3;
        c1 = (e >> 2) & 3;
    } else {
        c0 = (e & 3) | ((e >> 2) & 4);
        c1 = ((e >> 2) & 3) | ((e >> 3) & 4);
    }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// 32-bit word at a 2-byte aligned shared address.
__device__ __forceinline__ uint32_t lds32_a2(uint32_t addr) {
    const uint32_t base = addr & ~3u;
    return __funnelshift_r(lds32(base), lds32(base + 4), (addr & 3u) * 8u);
}

__device__ __forceinline__ void cp_async_zfill(uint32_t dst, const void *src, int bytes, int valid_bytes) {
    if (bytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid_bytes)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(valid_bytes)
                     : "memory");
}

__device__ __forceinline__ void stg_cs(uint8_t *p, uint4 v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Stage the warp's blocks [v0, v0 + nv) into `st`.  Contiguous input: one
// copy of nv * BB bytes (block r at r * BB).  Short strides (e.g. the halves
// of 132-byte storage slots): the byte span from the 16-byte boundary at or
// below block v0 to the end of block v0 + nv - 1, in 16-byte copies (block r
// at (address of block v0 & 15) + r * stride; the first copy may start up to
// 15 bytes before block v0, inside the same aligned 16 bytes, and the last
// copies only bytes of the span).  Other strides: block r's enclosing 32-bit
// words at r * 72 (block at r * 72 + (address & 3)); the last word copies
// only the bytes that belong to the block.
template <int BITS>
__device__ __forceinline__ void stage_tile(const DecArgs &a, uint32_t st, int64_t v0, int nv, int lane) {
    constexpr int BB = DecGeo<BITS>::BB;
    if (a.contiguous) {
        const uint8_t *src = a.blocks + v0 * BB;
        const int nbytes = nv * BB;
        for (int q = lane; q < (nbytes + 15) >> 4; q += 32)
            cp_async_zfill(st + 16 * q, src + 16 * q, 16, min(16, nbytes - 16 * q));
    } else if (a.span) {
        const uintptr_t first = reinterpret_cast<uintptr_t>(a.blocks + v0 * a.block_stride);
        const uintptr_t start = first & ~(uintptr_t)15;
        const int nbytes = (int)(first - start) + (nv - 1) * (int)a.block_stride + BB;
        for (int q = lane; q < (nbytes + 15) >> 4; q += 32)
            cp_async_zfill(st + 16 * q, reinterpret_cast<const void *>(start + 16 * q), 16, min(16, nbytes - 16 * q));
    } else {
        for (int q = lane; q < nv * 18; q += 32) {
            const int r = q / 18, w = q - 18 * r;
            const uint8_t *blk = a.blocks + (v0 + r) * a.block_stride;
            const uintptr_t start = reinterpret_cast<uintptr_t>(blk) & ~(uintptr_t)3;
            const int span = (int)(reinterpret_cast<uintptr_t>(blk) & 3) + BB;   // bytes from `start`
            if (4 * w < span)
                cp_async_zfill(st + r * kStridedPitch + 4 * w, reinterpret_cast<const void *>(start + 4 * w), 4,
                               min(4, span - 4 * w));
        }
    }
}

template <int BITS, int DT>
__global__ void __launch_bounds__(kDecThreads, 2) decode_pair_kernel(const __grid_constant__ DecArgs a) {
    using Geo = DecGeo<BITS>;
    constexpr int BB = Geo::BB;
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, pv = lane >> 1, h = lane & 1;
    uint32_t *sg16 = reinterpret_cast<uint32_t *>(smem + Geo::kLutBytes);
    uint32_t *sg32 = sg16 + 64;
    const uint32_t smem_s = (uint32_t)__cvta_generic_to_shared(smem);
    const uint32_t stage_s = smem_s + Geo::kLutBytes + (64 + 128) * 4 + warp * 2 * Geo::kStage;

    // pair table: float2 entry e at e * 256 + l * 8 for every lane l
    for (int q = threadIdx.x; q < Geo::kLutEntries * 32; q += kDecThreads) {
        const int e = q >> 5, l = q & 31;
        int c0, c1;
        entry_codes<BITS>(e, c0, c1);
        reinterpret_cast<float2 *>(smem)[e * 32 + l] = make_float2(a.c[c0], a.c[c1]);
    }
    for (int j = threadIdx.x; j < kD; j += kDecThreads) sg32[j] = ((a.signs[j >> 5] >> (j & 31)) & 1u) << 31;
    for (int w = threadIdx.x; w < 64; w += kDecThreads) {
        const int j = 2 * w;
        sg16[w] = (((a.signs[j >> 5] >> (j & 31)) & 1u) << 15) | (((a.signs[j >> 5] >> ((j + 1) & 31)) & 1u) << 31);
    }
    __syncthreads();

    const int64_t ntiles = (a.n_vec + kDecRows - 1) / kDecRows;
    const int64_t nwarps = (int64_t)gridDim.x * kDecWarps;
    int64_t tile = (int64_t)blockIdx.x * kDecWarps + warp;
    if (tile < ntiles) stage_tile<BITS>(a, stage_s, tile * kDecRows, (int)min64(kDecRows, a.n_vec - tile * kDecRows), lane);
    cp_async_commit();
    const float sgn = h ? -1.f : 1.f;
    const uint32_t lane8 = (uint32_t)lane * 8u;   // byte 0 of the table offsets below
    for (int it = 0; tile < ntiles; ++it, tile += nwarps) {
        const int64_t next = tile + nwarps;
        if (next < ntiles)
            stage_tile<BITS>(a, stage_s + ((it + 1) & 1) * Geo::kStage, next * kDecRows,
                             (int)min64(kDecRows, a.n_vec - next * kDecRows), lane);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const int64_t v0 = tile * kDecRows;
        const int64_t row = v0 + pv;
        uint32_t blk_s = stage_s + (it & 1) * Geo::kStage;
        if (a.contiguous) blk_s += pv * BB;
        else if (a.span)
            blk_s += (uint32_t)(reinterpret_cast<uintptr_t>(a.blocks + v0 * a.block_stride) & 15) +
                     (uint32_t)pv * (uint32_t)a.block_stride;
        else blk_s += pv * kStridedPitch + (row < a.n_vec ? (uint32_t)(reinterpret_cast<uintptr_t>(a.blocks + row * a.block_stride) & 3) : 0u);

        // ---- centroids of this thread's 64 elements, as pairs p[c'][k] = (e(c', k), e(c' + 4, k))
        float2 p[4][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float2 v[4];   // v[j] = centroids of elements k = 2j, 2j + 1 of chunk c
            if constexpr (BITS == 4) {
                const uint32_t w = lds32_a2(blk_s + 2 + 8 * c + 4 * h);    // byte j: elements 2j, 2j + 1
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = lds_f2(smem_s + prmt(w, lane8, 0x5504u + (j << 4)));
            } else {
                // table indices of the pairs (0,1), (4,5) in bytes 0, 1 of ev and (2,3), (6,7) of od
                uint32_t ev, od;
                const uint32_t lo = lds32_a2(blk_s + 2 + 4 * c) >> (16 * h);     // 2-bit plane, 8 codes
                if constexpr (BITS == 2) {
                    ev = lo & 0x0F0Fu;
                    od = (lo >> 4) & 0x0F0Fu;
                } else {
                    const uint32_t hb = lds32_a2(blk_s + 34 + (2 * c & ~3)) >> (8 * ((2 * c + h) & 3));
                    const uint32_t v2 = prmt(hb, 0, 0x1100u);                       // high bits, bytes 0 and 1
                    ev = (lo & 0x0F0Fu) | ((v2 << 4) & 0x0030u) | (v2 & 0x3000u);
                    od = ((lo >> 4) & 0x0F0Fu) | ((v2 << 2) & 0x0030u) | ((v2 >> 2) & 0x3000u);
                }
                // offset = index * 256 + lane * 8: byte 0 <- lane8, byte 1 <- the index byte, bytes 2-3 <- 0
                v[0] = lds_f2(smem_s + prmt(ev, lane8, 0x5504u));
                v[1] = lds_f2(smem_s + prmt(od, lane8, 0x5504u));
                v[2] = lds_f2(smem_s + prmt(ev, lane8, 0x5514u));
                v[3] = lds_f2(smem_s + prmt(od, lane8, 0x5514u));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (c < 4) {
                    p[c][2 * j].x = v[j].x;
                    p[c][2 * j + 1].x = v[j].y;
                } else {
                    p[c - 4][2 * j].y = v[j].x;
                    p[c - 4][2 * j + 1].y = v[j].y;
                }
            }
        }
        const float n = __half2float(__ushort_as_half((unsigned short)(lds32_a2(blk_s) & 0xFFFFu)));

        // ---- x = n D H c / sqrt(128)
        fwht_pair128(p, sgn);
        const float f = n * 0.08838834764831845f;
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < 8; ++k) p[c][k] = __fmul2_rn(p[c][k], f2);

        if (row < a.n_vec) {
            uint8_t *orow = a.out + row * a.out_stride;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                auto val = [&](int k) { return c < 4 ? p[c][k].x : p[c - 4][k].y; };
                if constexpr (DT == TQ_F32) {
                    const uint4 s0 = reinterpret_cast<const uint4 *>(sg32 + 16 * c + 8 * h)[0];
                    const uint4 s1 = reinterpret_cast<const uint4 *>(sg32 + 16 * c + 8 * h)[1];
                    stg_cs(orow + 4 * (16 * c + 8 * h),
                           make_uint4(__float_as_uint(val(0)) ^ s0.x, __float_as_uint(val(1)) ^ s0.y,
                                      __float_as_uint(val(2)) ^ s0.z, __float_as_uint(val(3)) ^ s0.w));
                    stg_cs(orow + 4 * (16 * c + 8 * h) + 16,
                           make_uint4(__float_as_uint(val(4)) ^ s1.x, __float_as_uint(val(5)) ^ s1.y,
                                      __float_as_uint(val(6)) ^ s1.z, __float_as_uint(val(7)) ^ s1.w));
                } else {
                    const uint4 s = reinterpret_cast<const uint4 *>(sg16 + 8 * c + 4 * h)[0];
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if constexpr (DT == TQ_BF16) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(val(2 * j), val(2 * j + 1));
                            w[j] = *reinterpret_cast<uint32_t *>(&b2);
                        } else {
                            __half2 h2 = __floats2half2_rn(val(2 * j), val(2 * j + 1));
                            w[j] = *reinterpret_cast<uint32_t *>(&h2);
                        }
                    }
                    stg_cs(orow + 2 * (16 * c + 8 * h), make_uint4(w[0] ^ s.x, w[1] ^ s.y, w[2] ^ s.z, w[3] ^ s.w));
                }
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
}

template <int BITS, int DT>
int launch_decode_pair(const DecArgs &a, cudaStream_t st) {
    using Geo = DecGeo<BITS>;
    static int done[64] = {0};
    static int per_sm[64] = {0};
    if (set_smem_limit((const void *)decode_pair_kernel<BITS, DT>, Geo::kSmem, done) != TQ_OK) return TQ_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    int occ = dev < 64 ? per_sm[dev] : 0;
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_pair_kernel<BITS, DT>, kDecThreads,
                                                          Geo::kSmem) != cudaSuccess ||
            occ < 1)
            occ = 1;
        if (dev < 64) per_sm[dev] = occ;
    }
    const int64_t ntiles = (a.n_vec + kDecRows - 1) / kDecRows;
    const int64_t ctas = (ntiles + kDecWarps - 1) / kDecWarps;
    const int grid = (int)std::min<int64_t>(ctas, (int64_t)occ * sm_count());
    decode_pair_kernel<BITS, DT><<<grid, kDecThreads, Geo::kSmem, st>>>(a);
    return launch_status();
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" int tq_decode_kv(const uint8_t *blocks, int64_t block_stride_bytes, int64_t n_vec,
                            const tq_codebook *cb, tq_signs signs, void *out, int out_dtype,
                            int64_t out_stride_elems, void *stream) {
    if (n_vec < 0 || !cb) return TQ_ERR_ARG;
    if (cb->bits == 8)   // turboq8 (tq_ext.cu)
        return tq_decode_kv_ex(blocks, block_stride_bytes, n_vec, cb, signs, out, out_dtype, out_stride_elems, 0,
                               stream);
    if (!codebook_ok(cb) || dtype_bytes(out_dtype) == 0) return TQ_ERR_UNSUPPORTED;
    if (n_vec == 0) return TQ_OK;
    const int es = dtype_bytes(out_dtype);
    const int64_t bb = (int64_t)tq_block_bytes(cb->bits);
    if (!blocks || !out || out_stride_elems < kD || block_stride_bytes < bb) return TQ_ERR_ARG;
    if (!aligned(out, 16) || (out_stride_elems * es) % 16 || !aligned(blocks, 2) || (block_stride_bytes & 1))
        return TQ_ERR_ALIGN;
    DecArgs a;
    a.blocks = blocks;
    a.block_stride = block_stride_bytes;
    a.n_vec = n_vec;
    a.out = static_cast<uint8_t *>(out);
    a.out_stride = out_stride_elems * es;
    a.contiguous = (block_stride_bytes == bb && aligned(blocks, 16)) ? 1 : 0;
    a.span = (!a.contiguous && block_stride_bytes <= kSpanMaxStride) ? 1 : 0;
    for (int i = 0; i < 16; ++i) a.c[i] = i < cb->levels ? cb->centroids[i] : 0.f;
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    cudaStream_t st = (cudaStream_t)stream;
    switch (cb->bits * 8 + out_dtype) {
        case 2 * 8 + TQ_F32: return launch_decode_pair<2, TQ_F32>(a, st);
        case 2 * 8 + TQ_BF16: return launch_decode_pair<2, TQ_BF16>(a, st);
        case 2 * 8 + TQ_F16: return launch_decode_pair<2, TQ_F16>(a, st);
        case 3 * 8 + TQ_F32: return launch_decode_pair<3, TQ_F32>(a, st);
        case 3 * 8 + TQ_BF16: return launch_decode_pair<3, TQ_BF16>(a, st);
        case 3 * 8 + TQ_F16: return launch_decode_pair<3, TQ_F16>(a, st);
        case 4 * 8 + TQ_F32: return launch_decode_pair<4, TQ_F32>(a, st);
        case 4 * 8 + TQ_BF16: return launch_decode_pair<4, TQ_BF16>(a, st);
        case 4 * 8 + TQ_F16: return launch_decode_pair<4, TQ_F16>(a, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}
