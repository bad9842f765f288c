// Encode on the tensor cores (bf16 / fp16 rows): the codec at head dims 64,
// 96, 128 and 160 with the caller's rotation, and, at d = 128, the further
// block formats (norm-corrected, dense 3-bit, turboq8) with the H D rotation.
//
// "TurboQuant KV Cache Compression — Spec", Types / Codebook Generation (the
// Lloyd-Max codebook of Beta(d/2, d/2) per dimension), Hadamard Transform
// Detail (for a head dim that is not a power of two, a dense orthogonal
// matrix), Algorithm Detail steps 1-3 (normalise by the L2 norm, rotate,
// level index from the boundaries, bit packing; eight 3-bit values in three
// bytes); "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", section 4
// Encode pipeline step 4 (block norm grp_norm / recon_norm) and the turboq8
// paragraph (uniform 256-level grid, per-block absmax scale).
//
// For 128 rows at a time, the rotation is the dense contraction
// [128 x d] x [d x d]^T: the rows come by TMA (32-column boxes, 64-byte
// swizzle, so every head dim is a whole number of boxes) as the A operand.
// The B operand is resident in shared memory for the CTA's life: the
// caller's R split into two 16-bit terms of the rows' type (R = R_hi + R_lo,
// each product exact, float32 accumulation; the error against R x is below
// 2^-18 |x| for bf16 rows and 2^-22 |x| for fp16, far inside the codec's
// 1e-5 boundary tolerance), or H D itself (+-1, one exact term; 1/sqrt(128)
// applied in the epilogue).  The products go to tensor memory (two
// accumulator stages), so the next tile's loads and products run while 16
// epilogue warps (four lane quarters x four column groups) finish this one:
//   * codec (Lloyd-Max): the norm from the staged rows (a float32 sum of
//     squares; a row whose sum leaves float32's safe range is redone in
//     double precision at once), the level index by a 128-cell table of the
//     scaled boundaries plus one comparison; norm-corrected blocks divide
//     the norm by the L2 norm of the row's centroids (a float32 sum over
//     the four column groups);
//   * turboq8: the largest |u| of the row over the four column groups (the
//     first of equal ones), codes floor(127.5 u / max + 128), the scale
//     fp16(max / sqrt(128));
// a stored norm or scale within 2^-20 of an fp16 rounding boundary is listed
// and rewritten after the main loop by a whole warp (double-float sums of
// the row in memory, or the largest coordinate in double precision).  The
// codes are packed into a shared-memory copy of the 128 blocks, which leaves
// by one bulk copy per 32 rows.  One CTA per SM, a persistent grid.

#include <cmath>
#include <cstring>

#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {
namespace {

constexpr int kHtRows = 128;       // rows per tile (tensor-memory lanes)
constexpr int kHtEpiWarps = 16;    // lane quarter (warp & 3) x column group (warp >> 2)
constexpr int kHtThreads = 32 * (kHtEpiWarps + 1);
constexpr int kHtBuckets = 128;
constexpr int kHtBox = 128 * 64;   // one 32-column box of 128 rows: 8 KB
constexpr int kHtFixCap = 512;     // rows listed for an exact norm or scale, per CTA
constexpr float kHtRs = 0.08838834764831845f;   // 1 / sqrt(128)

struct HtArgs {
    const void *x;       // rows (the listed rows' norms and scales are redone from them)
    uint8_t *blocks;
    const float *R;      // [d][d] row-major, float32 (the head-dim codec)
    int64_t n_vec;
    int64_t x_stride;    // bytes between rows
    float grid;          // cells per unit of y
    int drop;            // test hook: no TMA load is issued
    int nc, dense;       // norm-corrected blocks; 3-bit codes eight per three bytes
    uint32_t signs[4];   // D (the H D rotation)
    float c[16];         // centroids (norm correction)
    float2 table[kHtBuckets];   // cell j: (the boundary inside it in grid units | +inf, bits of #boundaries below)
};

// HAD: the rotation is H D (d = 128, +-1 entries, one exact term); else the caller's R in two terms.
template <int D, int BITS, bool HAD>
struct HtSmem {
    static constexpr int BB = BITS == 8 ? 130 : 2 + D * BITS / 8;
    static constexpr int NT = HAD ? 1 : 2;                      // B operand terms
    static constexpr int kStage = D / 32 * kHtBox;             // a row tile: D / 32 boxes
    static constexpr int kA = 0;                               // two row-tile stages
    static constexpr int kTerm = D / 32 * D * 64;              // one term: D / 32 blocks of D rows x 64 bytes
    static constexpr int kB = kA + 2 * kStage;
    static constexpr int kOut = kB + NT * kTerm;               // the tile's 128 blocks
    static constexpr int kPart = (kOut + kHtRows * BB + 15) / 16 * 16;   // [2][4 column groups][128]
    static constexpr int kFix = kPart + 2 * 4 * kHtRows * 4;   // [0] count, [1] overflow, [4 ..] (row, arg)
    static constexpr int kTab = kFix + (4 + 2 * kHtFixCap) * 4;
    static constexpr int kCb = kTab + kHtBuckets * 8;          // 16 centroids
    // full[2] at 0, mma[2] at 16, row tile free[2] at 32, drain at 48, accumulator free[2] at 56
    static constexpr int kBars = kCb + 64;
    static constexpr int kSlot = kBars + 72;
    static constexpr int kUsed = kSlot + 8;
    // at least 116 KB, so one CTA per SM: each holds a tensor-memory allocation of its own
    static constexpr int kTotal = kUsed + 1024 > 118784 ? kUsed + 1024 : 118784;
    // accumulator stage stride in tensor-memory columns (a power of two >= D) and the allocation
    static constexpr int kTS = D <= 64 ? 64 : D <= 128 ? 128 : 256;
    static constexpr int kCols = 2 * kTS;
    static_assert(kTotal <= 232448, "shared memory");
    static_assert(!HAD || D == 128, "the H D rotation is the 128-element one");
};

// Shared-memory descriptor of a K-major operand in the 64-byte swizzle layout
// (rows of 64 bytes, 16-byte chunk c of row m at ((c ^ ((m >> 1) & 3)) << 4),
// 8-row groups 512 bytes apart): start >> 4, leading byte offset 1 (unused
// with a swizzle), stride byte offset 512 >> 4, descriptor version 1, layout
// type 4 (64-byte swizzle).
__device__ __forceinline__ uint64_t ht_desc_sw64(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(512 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)4 << 61);
}

// Instruction descriptor of kind::f16: float32 accumulator, A and B of dtype DT, both K-major,
// N = D, M = 128.
template <int DT, int D>
__device__ __forceinline__ constexpr uint32_t ht_idesc() {
    return (1u << 4) | ((DT == TQ_BF16 ? 1u : 0u) << 7) | ((DT == TQ_BF16 ? 1u : 0u) << 10) | ((uint32_t)(D >> 3) << 17) |
           ((128u >> 4) << 24);
}

// Byte offset of element j of row r in a tile of 32-column boxes (64-byte swizzle).
__device__ __forceinline__ int ht_off(int r, int j) {
    return (j >> 5) * kHtBox + r * 64 + ((((j & 31) >> 3) ^ ((r >> 1) & 3)) << 4) + (j & 7) * 2;
}

template <int DT>
__device__ __forceinline__ float ht_val(uint32_t h) {
    return DT == TQ_BF16 ? __uint_as_float(h << 16) : __half2float(__ushort_as_half((unsigned short)h));
}

// 8 consecutive float32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void ht_ld8(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Wait for this thread's tensor-memory loads; v (their destination) is tied to the wait.
template <int N>
__device__ __forceinline__ void ht_wait_ld(float (&v)[N]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}

__device__ __forceinline__ uint32_t ht_set_ge(float a, float b) {
    uint32_t r;
    asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float2 ht_lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// Double-float sum of squares of a row in memory by a whole warp (lane l takes elements l + 32 k),
// reduced over the warp; every lane gets (s, c).
template <int DT, int D>
__device__ __forceinline__ void ht_warp_sumsq(const HtArgs &a, int64_t row, int lane, float &s1, float &c1) {
    const uint16_t *xr = reinterpret_cast<const uint16_t *>(static_cast<const uint8_t *>(a.x) + row * a.x_stride);
    SumSq2 acc;
    for (int j = lane; j < D; j += 32) acc.add(ht_val<DT>(xr[j]));
    s1 = acc.s;
    c1 = acc.c;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, s1, o), oc = __shfl_xor_sync(0xffffffffu, c1, o);
        float ns, ne;
        two_sum(s1, os, ns, ne);
        s1 = ns;
        c1 = c1 + oc + ne;
    }
}

// Code of element j of a written block (the layouts of the codec; dense: 3-bit, eight per 3 bytes).
template <int D, int BITS>
__device__ __forceinline__ uint32_t ht_code_at(const uint8_t *blk, int dense, int j) {
    const uint8_t *c = blk + 2;
    if constexpr (BITS == 2) return (c[j >> 2] >> (2 * (j & 3))) & 3u;
    if constexpr (BITS == 4) return (c[j >> 1] >> (4 * (j & 1))) & 15u;
    if (dense) {
        const int g = j >> 3, p = j & 7;
        const uint32_t w = c[3 * g] | ((uint32_t)c[3 * g + 1] << 8) | ((uint32_t)c[3 * g + 2] << 16);
        return (w >> (3 * p)) & 7u;
    }
    return ((c[j >> 2] >> (2 * (j & 3))) & 3u) | (((c[D / 4 + (j >> 3)] >> (j & 7)) & 1u) << 2);
}

// The exact stored norm of a listed row, by a whole warp: the norm from a double-float sum of the
// row's squares (norm-corrected: divided by the L2 norm of the centroids of the block's own codes,
// in double precision), one rounding to fp16.  A row whose sum lies outside float32's safe range
// keeps what the main loop stored (there from a double sum).  Out of line: about one row in 250.
template <int DT, int D, int BITS, int BB>
__device__ __noinline__ void ht_fix_norm(const HtArgs &a, int64_t row, int lane) {
    float s1, c1;
    ht_warp_sumsq<DT, D>(a, row, lane, s1, c1);
    uint8_t *blk = a.blocks + row * BB;
    double sc = 0.0;
    if (a.nc) {
        for (int j = lane; j < D; j += 32) {
            const double cj = a.c[ht_code_at<D, BITS>(blk, a.dense, j)];
            sc += cj * cj;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
    }
    if (lane == 0 && s1 >= 7.888609052210118e-31f /* 2^-100 */ && s1 <= 1.2676506002282294e30f) {
        uint16_t n16;
        if (a.nc) {
            const double nd = sqrt((double)s1 + (double)c1);
            n16 = __half_as_ushort(__double2half(sc > 0.0 ? nd / sqrt(sc) : 0.0));
        } else {
            SumSq2 tot;
            tot.s = s1;
            tot.c = c1;
            n16 = tot.sqrt_fp16();
        }
        *reinterpret_cast<uint16_t *>(blk) = n16;
    }
}

// The exact turboq8 scale of a listed row, by a whole warp: u_arg = sum_d H(arg, d) D_d x_d in
// double precision, fp16(|u_arg| / sqrt(128)); arg < 0: the largest |u_j| over all 128
// coordinates, each in double precision (an overflowed list).
template <int DT>
__device__ __noinline__ void ht_fix_scale(const HtArgs &a, int64_t row, int arg, int lane) {
    const uint16_t *xr = reinterpret_cast<const uint16_t *>(static_cast<const uint8_t *>(a.x) + row * a.x_stride);
    double best = 0.0;
    for (int j = (arg < 0 ? 0 : arg); j < (arg < 0 ? 128 : arg + 1); ++j) {
        double u = 0.0;
        for (int d = lane; d < 128; d += 32) {
            const double sg = ((__popc(j & d) & 1) ^ ((a.signs[d >> 5] >> (d & 31)) & 1u)) ? -1.0 : 1.0;
            u += sg * (double)ht_val<DT>(xr[d]);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
        best = fmax(best, fabs(u));
    }
    if (lane == 0) *reinterpret_cast<uint16_t *>(a.blocks + row * 130) = __half_as_ushort(__double2half(best / sqrt(128.0)));
}

// Sum of squares of row r of a staged tile in double precision (rows outside float32's safe
// range: essentially never; out of line).
template <int DT, int D>
__device__ __noinline__ double ht_row_sumsq_d(const uint8_t *tile, int r) {
    double s = 0.0;
    for (int j = 0; j < D; ++j) {
        const double e = ht_val<DT>(*reinterpret_cast<const uint16_t *>(tile + ht_off(r, j)));
        s += e * e;
    }
    return s;
}

template <int ND, int DT, int BITS, bool HAD>
__global__ void __launch_bounds__(kHtThreads, 1)
    encode_d_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ HtArgs a) {
    constexpr int D = 32 * ND;
    using S = HtSmem<D, BITS, HAD>;
    constexpr int BB = S::BB, CW = D / 4, NB = D / 32, NT = S::NT;
    extern __shared__ __align__(16) uint8_t ht_smem_raw[];
    // 1024-byte aligned base: the swizzle is a function of the address bits
    const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(ht_smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = ht_smem_raw + (base_s - raw_s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = base_s + S::kBars;

    // ---- setup: the B operand in the swizzled K-major layout (row n = output n, its D inputs along
    // K): R_hi and R_lo, or H D; the cell table and centroids, barriers, tensor memory
    for (int q = threadIdx.x; q < D * (D / 8); q += kHtThreads) {
        const int n = q / (D / 8), c = q % (D / 8);   // output row n, 8-input chunk c
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint32_t h2 = 0, l2 = 0;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int k = 8 * c + 2 * p + e;
                uint32_t hb, lb = 0;
                if constexpr (HAD) {
                    const uint32_t neg = ((uint32_t)__popc(n & k) & 1u) ^ ((a.signs[k >> 5] >> (k & 31)) & 1u);
                    hb = DT == TQ_BF16 ? (neg ? 0xBF80u : 0x3F80u) : (neg ? 0xBC00u : 0x3C00u);
                } else if constexpr (DT == TQ_BF16) {
                    const float r = a.R[n * D + k];
                    const __nv_bfloat16 h = __float2bfloat16_rn(r);
                    hb = __bfloat16_as_ushort(h);
                    lb = __bfloat16_as_ushort(__float2bfloat16_rn(r - __bfloat162float(h)));
                } else {
                    const float r = a.R[n * D + k];
                    const __half h = __float2half_rn(r);
                    hb = __half_as_ushort(h);
                    lb = __half_as_ushort(__float2half_rn(r - __half2float(h)));
                }
                h2 |= hb << (16 * e);
                l2 |= lb << (16 * e);
            }
            hi[p] = h2;
            lo[p] = l2;
        }
        const int off = (c >> 2) * (D * 64) + n * 64 + (((c & 3) ^ ((n >> 1) & 3)) << 4);
        *reinterpret_cast<uint4 *>(smem + S::kB + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if constexpr (NT == 2) *reinterpret_cast<uint4 *>(smem + S::kB + S::kTerm + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    float2 *tab = reinterpret_cast<float2 *>(smem + S::kTab);
    for (int j = threadIdx.x; j < kHtBuckets; j += kHtThreads) tab[j] = a.table[j];
    float *cbs = reinterpret_cast<float *>(smem + S::kCb);
    if (threadIdx.x < 16) cbs[threadIdx.x] = a.c[threadIdx.x];
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(bars + 8 * i, 1);                  // full: the producer's arrival + the TMA bytes
            tc_mbar_init(bars + 16 + 8 * i, 1);             // mma: tcgen05.commit
            tc_mbar_init(bars + 32 + 8 * i, kHtEpiWarps);   // row tile free: each epilogue warp, after the norms
            tc_mbar_init(bars + 56 + 8 * i, kHtEpiWarps);   // accumulator free: each epilogue warp, after its loads
        }
        tc_mbar_init(bars + 48, 1);                         // drain: the producer's last commit
        reinterpret_cast<int *>(smem + S::kFix)[0] = 0;     // listed rows
        reinterpret_cast<int *>(smem + S::kFix)[1] = 0;     // list overflowed
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base_s + S::kSlot),
                     "r"(S::kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the B operand was written by ordinary stores and is read by the tensor cores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S::kSlot);
    const int64_t ntiles = (a.n_vec + kHtRows - 1) / kHtRows;

    if (warp == kHtEpiWarps) {
        // ---- producer: a row tile by TMA, then the NT x D / 16 products into the stage's accumulator
        if (lane == 0) {
            constexpr uint32_t idesc = ht_idesc<DT, D>();
            // a wait that gives up is recorded and ends the loop: no further load or product
            bool ok = true;
            auto wait = [&](uint32_t bar, uint32_t parity) {
                if (ok && !tc_mbar_wait(bar, parity)) {
                    ok = false;
                    note_wait_failed();
                }
            };
            int pend = -1;   // stage of a load not yet seen complete, and its parity
            uint32_t pend_par = 0;
            int i = 0;
            for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++i) {
                const int st = i & 1;
                const uint32_t use = (uint32_t)(i >> 1);
                if (i >= 2) wait(bars + 32 + 8 * st, (use - 1u) & 1u);   // row tile read by the epilogue
                if (!ok) break;
                const uint32_t a_s = base_s + S::kA + st * S::kStage, full = bars + 8 * st;
                if (!a.drop) {   // (test hook: no load, so the wait below runs out)
                    tc_mbar_expect_tx(full, S::kStage);
#pragma unroll
                    for (int kb = 0; kb < NB; ++kb) tc_tma_load_2d(a_s + kb * kHtBox, &tmap, 32 * kb, (int)(tile * kHtRows), full);
                    pend = st;
                    pend_par = use & 1u;
                }
                wait(full, use & 1u);
                if (!ok) break;   // no product on a tile that did not land
                pend = -1;
                if (i >= 2) wait(bars + 56 + 8 * st, (use - 1u) & 1u);   // accumulator read by the epilogue
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(st * S::kTS);
                const uint32_t b_s = base_s + S::kB;
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int kb = 0; kb < NB; ++kb)
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            tc_mma(d, ht_desc_sw64(a_s + kb * kHtBox + 32 * ks),
                                   ht_desc_sw64(b_s + t * S::kTerm + kb * (D * 64) + 32 * ks), idesc,
                                   (t | kb | ks) ? 1u : 0u);
                tc_commit(bars + 16 + 8 * st);
            }
            // before teardown: every product issued here has completed, and a load whose wait gave
            // up has landed (bounded waits)
            tc_commit(bars + 48);
            tc_mbar_wait(bars + 48, 0u);
            if (pend >= 0) tc_mbar_wait(bars + 8 * pend, pend_par);
        }
    } else {
        // ---- epilogue: warp w reads tensor-memory lanes (= tile rows) 32 (w & 3) .. + 31, columns
        // CW (w >> 2) .. + CW - 1; the four warps of a lane quarter meet on named barrier 1 + (w & 3)
        const int grp = warp & 3, cg = warp >> 2;
        const int r = 32 * grp + lane;
        const uint32_t qbar = 1u + (uint32_t)grp;
        float *part = reinterpret_cast<float *>(smem + S::kPart);   // [2][4][128]
        float *part2 = part + 4 * kHtRows;
        int *fix = reinterpret_cast<int *>(smem + S::kFix);
        uint8_t *sm_out = smem + S::kOut;
        const uint32_t tab_s = base_s + S::kTab;
        const bool bulk_out = ((uintptr_t)a.blocks & 15u) == 0;
        const float2 off2 = make_float2(1572928.f, 1572928.f);   // 64 + 1.5 * 2^20: z + 64 to 1/8, the cell in bits 3..9
        // list row v for an exact norm / scale (arg: turboq8's coordinate); cg == 0 warps only
        auto list = [&](bool need, int64_t v, int arg) {
            const uint32_t m = __ballot_sync(0xffffffffu, need);
            if (m) {
                const int leader = __ffs(m) - 1;
                int base = 0;
                if (lane == leader) base = atomicAdd(&fix[0], __popc(m));
                base = __shfl_sync(0xffffffffu, base, leader);
                if (need) {
                    const int slot = base + __popc(m & ((1u << lane) - 1u));
                    if (slot < kHtFixCap) {
                        fix[4 + 2 * slot] = (int)v;
                        fix[5 + 2 * slot] = arg;
                    } else {
                        fix[1] = 1;
                    }
                }
            }
        };
        bool ok = true;
        int i = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
            const int st = i & 1;
            if (ok && !tc_mbar_wait(bars + 16 + 8 * st, (uint32_t)(i >> 1) & 1u)) {
                ok = false;
                note_wait_failed();
            }
            tc_fence_after();
            const int64_t v0 = tile * kHtRows;
            const int nv = (int)min64(kHtRows, a.n_vec - v0);
            const int rows = max(0, min(32, nv - 32 * grp));
            const uint8_t *at = smem + S::kA + st * S::kStage;
            // this row's accumulators of the warp's columns, requested now
            float u[CW];
            const uint32_t taddr = tmem + ((uint32_t)(32 * grp) << 16) + (uint32_t)(st * S::kTS + cg * CW);
#pragma unroll
            for (int p = 0; p < CW / 8; ++p) ht_ld8(taddr + 8 * p, u + 8 * p);
            uint8_t *blk = sm_out + r * BB;
            uint32_t n16 = 0;
            if constexpr (BITS == 8) {
                // ---- turboq8: the largest |u| of the row (the first of equal ones) over the four groups
                if (bulk_out && cg == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                __syncwarp();
                if (lane == 0) tc_mbar_arrive(bars + 32 + 8 * st);   // the row tile is not read here
                ht_wait_ld(u);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) tc_mbar_arrive(bars + 56 + 8 * st);
                float amax = 0.f;
                int arg = cg * CW;
#pragma unroll
                for (int k = 0; k < CW; ++k) {
                    const float m = fabsf(u[k]);
                    if (m > amax) {
                        amax = m;
                        arg = cg * CW + k;
                    }
                }
                part[cg * kHtRows + r] = amax;
                part2[cg * kHtRows + r] = __int_as_float(arg);
                asm volatile("bar.sync %0, 128;" ::"r"(qbar) : "memory");
                amax = part[r];
                arg = __float_as_int(part2[r]);
#pragma unroll
                for (int c = 1; c < 4; ++c) {
                    const float m = part[c * kHtRows + r];
                    if (m > amax) {   // ties keep the lower group, whose coordinates come first
                        amax = m;
                        arg = __float_as_int(part2[c * kHtRows + r]);
                    }
                }
                const float inv = amax > 0.f ? 1.f / amax : 0.f;   // a zero row: code 128 everywhere
                uint16_t *o16 = reinterpret_cast<uint16_t *>(blk + 2 + cg * CW);
#pragma unroll
                for (int k = 0; k < CW; k += 2) {
                    // u / a in [-1, 1]: 127.5 y + 128 lies in [0.5, 255.5]
                    const uint32_t c0 = (uint32_t)floorf(fmaf(127.5f, u[k] * inv, 128.f));
                    const uint32_t c1 = (uint32_t)floorf(fmaf(127.5f, u[k + 1] * inv, 128.f));
                    o16[k / 2] = (uint16_t)(c0 | (c1 << 8));
                }
                const float a32 = amax * kHtRs;
                n16 = amax > 0.f ? __half_as_ushort(__float2half_rn(a32)) : 0u;
                if (cg == 0) {
                    list(r < nv && amax > 0.f && near_fp16_tie_fast(a32), v0 + r, arg);
                    *reinterpret_cast<uint16_t *>(blk) = (uint16_t)n16;
                }
            } else {
                // ---- norm: float32 sum of squares of the row's inputs, four column groups added in order
                float sp = 0.f;
#pragma unroll
                for (int c = 0; c < CW / 8; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(at + ht_off(r, cg * CW + 8 * c));
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float e0 = ht_val<DT>(ws[k] & 0xFFFFu), e1 = ht_val<DT>(ws[k] >> 16);
                        sp = fmaf(e0, e0, sp);
                        sp = fmaf(e1, e1, sp);
                    }
                }
                part[cg * kHtRows + r] = sp;
                // the previous tile's bulk stores have read the blocks before they are rewritten
                if (bulk_out && cg == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                asm volatile("bar.sync %0, 128;" ::"r"(qbar) : "memory");
                const float ss = ((part[r] + part[kHtRows + r]) + part[2 * kHtRows + r]) + part[3 * kHtRows + r];
                float nrm = sqrtf(ss);
                float inv = ss > 0.f ? 1.f / nrm : 0.f;
                // outside float32's safe range (a zero row included): norm and scale from a double sum
                // of the exact squares, here (the four threads of the row see the same ss)
                const bool oor = r < nv && !(ss >= 7.888609052210118e-31f /* 2^-100 */ && ss <= 1.2676506002282294e30f);
                double nd = 0.0;
                if (oor) {
                    nd = sqrt(ht_row_sumsq_d<DT, D>(at, r));
                    inv = nd > 0.0 ? (float)(1.0 / nd) : 0.f;   // a zero row: y = 0, code L/2
                }
                // the row tile is read: the next load may take its place while this tile is quantised
                __syncwarp();
                if (lane == 0) tc_mbar_arrive(bars + 32 + 8 * st);
                ht_wait_ld(u);
                // the accumulator is in registers: the next products may take its place
                tc_fence_before();
                __syncwarp();
                if (lane == 0) tc_mbar_arrive(bars + 56 + 8 * st);
                // ---- quantise and pack: code = #{boundaries <= y} from the cell of G y and one comparison
                const float cs = a.grid * (HAD ? kHtRs : 1.f) * inv;
                const float2 cs2 = make_float2(cs, cs);
                const uint32_t cb_s = base_s + S::kCb;
                constexpr int B = BITS == 2 ? 2 : 4;   // accumulation width of a code (3-bit: nibbles)
                float csq = 0.f;                       // this thread's share of sum c[code]^2
#pragma unroll
                for (int g = 0; g < CW / 8; ++g) {
                    uint32_t w = 0;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float2 y = __fmul2_rn(make_float2(u[8 * g + e], u[8 * g + e + 1]), cs2);
                        const float2 t = __fadd2_rn(y, off2);
                        const float2 c0 = ht_lds_f2(tab_s + (__float_as_uint(t.x) & 0x3F8u));
                        const float2 c1 = ht_lds_f2(tab_s + (__float_as_uint(t.y) & 0x3F8u));
                        const uint32_t k0 = __float_as_uint(c0.y) - ht_set_ge(y.x, c0.x);
                        const uint32_t k1 = __float_as_uint(c1.y) - ht_set_ge(y.y, c1.x);
                        w |= (k0 << (B * e)) | (k1 << (B * e + B));
                        if (HAD && a.nc) {
                            float c0v, c1v;
                            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(c0v) : "r"(cb_s + 4 * k0));
                            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(c1v) : "r"(cb_s + 4 * k1));
                            csq = fmaf(c0v, c0v, csq);
                            csq = fmaf(c1v, c1v, csq);
                        }
                    }
                    const int j0 = cg * CW + 8 * g;   // first column of the 8
                    if constexpr (BITS == 4) {
                        uint16_t *o = reinterpret_cast<uint16_t *>(blk + 2 + j0 / 2);
                        o[0] = (uint16_t)w;
                        o[1] = (uint16_t)(w >> 16);
                    } else if constexpr (BITS == 2) {
                        *reinterpret_cast<uint16_t *>(blk + 2 + j0 / 4) = (uint16_t)w;
                    } else if (HAD && a.dense) {
                        // eight 3-bit codes (nibbles of w) into the 24 bits of group j0 / 8
                        uint32_t d3 = 0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) d3 |= ((w >> (4 * e)) & 7u) << (3 * e);
                        uint8_t *o = blk + 2 + 3 * (j0 / 8);
                        o[0] = (uint8_t)d3;
                        o[1] = (uint8_t)(d3 >> 8);
                        o[2] = (uint8_t)(d3 >> 16);
                    } else {
                        // low plane: bits 0-1 of nibble e to bits 2e, 2e + 1; high plane: bit 2 of nibble e to bit e
                        uint32_t lo = w & 0x33333333u;
                        lo = (lo | (lo >> 2)) & 0x0F0F0F0Fu;
                        lo = (lo | (lo >> 4)) & 0x00FF00FFu;
                        lo = (lo | (lo >> 8)) & 0x0000FFFFu;
                        uint32_t hb = (w >> 2) & 0x11111111u;
                        hb = (hb | (hb >> 3)) & 0x03030303u;
                        hb = (hb | (hb >> 6)) & 0x000F000Fu;
                        hb = (hb | (hb >> 12)) & 0x000000FFu;
                        *reinterpret_cast<uint16_t *>(blk + 2 + j0 / 4) = (uint16_t)lo;
                        blk[2 + D / 4 + j0 / 8] = (uint8_t)hb;
                    }
                }
                // the stored norm (norm-corrected: over the L2 norm of the row's centroids, the four
                // groups added in order); a zero row stores 0
                float stored = nrm, cq = 1.f;
                if (HAD && a.nc) {
                    part2[cg * kHtRows + r] = csq;
                    asm volatile("bar.sync %0, 128;" ::"r"(qbar) : "memory");
                    cq = ((part2[r] + part2[kHtRows + r]) + part2[2 * kHtRows + r]) + part2[3 * kHtRows + r];
                    stored = nrm / sqrtf(cq);
                }
                if (oor)   // (double precision only here: GB300's FP64 pipe is narrow)
                    n16 = nd > 0.0 ? __half_as_ushort(__double2half(nd / sqrt((double)cq))) : 0u;
                else
                    n16 = ss > 0.f ? __half_as_ushort(__float2half_rn(stored)) : 0u;
                // within 2^-20 of an fp16 rounding boundary: listed; rewritten after the loop
                if (cg == 0) {
                    list(r < nv && !oor && near_fp16_tie_fast(stored), v0 + r, 0);
                    *reinterpret_cast<uint16_t *>(blk) = (uint16_t)n16;
                }
            }
            if (bulk_out) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // blocks -> bulk copy
            asm volatile("bar.sync %0, 128;" ::"r"(qbar) : "memory");   // the quarter's 32 blocks are written

            // ---- store the quarter's 32 blocks
            uint8_t *dst = a.blocks + (v0 + 32 * grp) * BB;
            const uint8_t *src = sm_out + 32 * grp * BB;
            if (bulk_out && rows == 32) {
                // 32 blocks: 32 BB bytes (a multiple of 16) at a 16-byte aligned offset
                if (cg == 0 && lane == 0) {
                    const uint32_t ss_ = (uint32_t)__cvta_generic_to_shared(src);
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(ss_),
                                 "r"(32 * BB)
                                 : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                }
            } else {
                // a partial quarter (the last tile) or a 2-byte aligned destination: 2-byte pieces
                for (int q = 32 * cg + lane; q < rows * BB / 2; q += 128)
                    reinterpret_cast<uint16_t *>(dst)[q] = reinterpret_cast<const uint16_t *>(src)[q];
            }
        }
        // ---- the listed rows, once every block of this CTA is in memory (the bulk stores complete
        // and ordered before these writes); an overflowed list redoes every row of the CTA
        if (bulk_out && cg == 0 && lane == 0) {
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __threadfence_block();
        asm volatile("bar.sync 5, %0;" ::"n"(32 * kHtEpiWarps) : "memory");
        const bool all = fix[1] != 0;
        const int nfix = all ? 0 : min(fix[0], kHtFixCap);
        for (int q = warp; q < nfix; q += kHtEpiWarps) {
            if constexpr (BITS == 8) ht_fix_scale<DT>(a, (int64_t)fix[4 + 2 * q], fix[5 + 2 * q], lane);
            else ht_fix_norm<DT, D, BITS, BB>(a, (int64_t)fix[4 + 2 * q], lane);
        }
        if (all) {
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x)
                for (int rr = warp; rr < kHtRows; rr += kHtEpiWarps) {
                    const int64_t v = tile * kHtRows + rr;
                    if (v >= a.n_vec) continue;
                    if constexpr (BITS == 8) {
                        // (a zero row keeps its zero scale)
                        if (*reinterpret_cast<const uint16_t *>(a.blocks + v * BB) != 0) ht_fix_scale<DT>(a, v, -1, lane);
                    } else {
                        ht_fix_norm<DT, D, BITS, BB>(a, v, lane);
                    }
                }
        }
    }

    // ---- teardown: every product has completed (the producer waited for its last commit) and every
    // tensor-memory load completed
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kCols) : "memory");
}

// Tensor map of n_rows rows of D 16-bit elements, stride_bytes apart (a multiple of 16): boxes of
// 32 columns x 128 rows, 64-byte swizzle, rows past the end read as zero.
bool ht_make_map(CUtensorMap *map, const void *x, int dt, int64_t n_rows, int D, int64_t stride_bytes) {
    TensorMapEncodeTiledFn enc = tensor_map_encoder();
    if (!enc || n_rows <= 0 || n_rows > 0x7FFFFFFFLL - 128) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)n_rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)stride_bytes};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, dt == TQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
               const_cast<void *>(x), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Cell table of a codebook: with z = G y, cell j holds z + 64 in [j - 1/16, j + 15/16); G is the
// smallest integer above 1 / (the smallest gap between adjacent boundaries), so no cell holds two
// boundaries.  False when that G exceeds 62 (|z| <= G must stay inside the table).
bool ht_table(const tq_codebook *cb, HtArgs *a) {
    const int L = cb->levels;
    double gap = 1.0;
    for (int i = 0; i + 1 < L - 1; ++i) gap = std::min(gap, (double)cb->boundaries[i + 1] - (double)cb->boundaries[i]);
    const double g = std::floor(1.0 / gap) + 1.0;
    if (!(g <= 62.0)) return false;
    const float G = (float)g;
    a->grid = G;
    for (int j = 0; j < kHtBuckets; ++j) {
        uint32_t below = 0;
        float inner = INFINITY;
        for (int i = 0; i < L - 1; ++i) {
            const float z = G * cb->boundaries[i];
            if (z + 64.f < j - 0.0625f) ++below;
            else if (z + 64.f < j + 0.9375f) inner = z;
        }
        float codef;
        std::memcpy(&codef, &below, 4);
        a->table[j] = make_float2(inner, codef);
    }
    for (int i = 0; i < 16; ++i) a->c[i] = i < L ? cb->centroids[i] : 0.f;
    return true;
}

template <int ND, int DT, int BITS, bool HAD>
int ht_launch(const CUtensorMap &map, const HtArgs &a, cudaStream_t st) {
    using S = HtSmem<32 * ND, BITS, HAD>;
    static int done[64] = {0};
    if (set_smem_limit((const void *)encode_d_tc_kernel<ND, DT, BITS, HAD>, S::kTotal, done) != TQ_OK)
        return TQ_ERR_CUDA;
    const int64_t ntiles = (a.n_vec + kHtRows - 1) / kHtRows;
    const int grid = (int)std::min<int64_t>(ntiles, (int64_t)sm_count());
    encode_d_tc_kernel<ND, DT, BITS, HAD><<<grid, kHtThreads, S::kTotal, st>>>(map, a);
    return launch_status();
}

template <int ND, int DT>
int ht_launch_bits(const CUtensorMap &map, const HtArgs &a, int bits, cudaStream_t st) {
    switch (bits) {
        case 2: return ht_launch<ND, DT, 2, false>(map, a, st);
        case 3: return ht_launch<ND, DT, 3, false>(map, a, st);
        default: return ht_launch<ND, DT, 4, false>(map, a, st);
    }
}

template <int DT>
int ht_launch_dim(const CUtensorMap &map, const HtArgs &a, int d, int bits, cudaStream_t st) {
    switch (d) {
        case 64: return ht_launch_bits<2, DT>(map, a, bits, st);
        case 96: return ht_launch_bits<3, DT>(map, a, bits, st);
        case 128: return ht_launch_bits<4, DT>(map, a, bits, st);
        default: return ht_launch_bits<5, DT>(map, a, bits, st);
    }
}

template <int DT>
int ht_launch_ext(const CUtensorMap &map, const HtArgs &a, int bits, cudaStream_t st) {
    switch (bits) {
        case 2: return ht_launch<4, DT, 2, true>(map, a, st);
        case 3: return ht_launch<4, DT, 3, true>(map, a, st);
        case 4: return ht_launch<4, DT, 4, true>(map, a, st);
        default: return ht_launch<4, DT, 8, true>(map, a, st);
    }
}

}  // namespace

int hd_encode_tc(const void *x, int x_dtype, int64_t n_vec, int d, const tq_codebook *cb, const float *R,
                 uint8_t *blocks, cudaStream_t st) {
    if ((x_dtype != TQ_BF16 && x_dtype != TQ_F16) || n_vec < kHdTcMinRows || !aligned(x, 16) || !aligned(R, 4) ||
        !aligned(blocks, 2))
        return 1;
    if (d != 64 && d != 96 && d != 128 && d != 160) return 1;
    HtArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!ht_table(cb, &a)) return 1;
    CUtensorMap map;
    if (!ht_make_map(&map, x, x_dtype, n_vec, d, (int64_t)d * 2)) return 1;
    a.x = x;
    a.blocks = blocks;
    a.R = R;
    a.n_vec = n_vec;
    a.x_stride = (int64_t)d * 2;
    a.drop = drop_copies();
    return x_dtype == TQ_BF16 ? ht_launch_dim<TQ_BF16>(map, a, d, cb->bits, st)
                              : ht_launch_dim<TQ_F16>(map, a, d, cb->bits, st);
}

int ext_encode_tc(const void *x, int x_dtype, int64_t n_vec, int64_t x_stride_bytes, const tq_codebook *cb,
                  const uint32_t *signs, int nc, int dense, uint8_t *blocks, cudaStream_t st) {
    if ((x_dtype != TQ_BF16 && x_dtype != TQ_F16) || n_vec < kHdTcMinRows || !aligned(x, 16) ||
        (x_stride_bytes & 15) || !aligned(blocks, 2) || cb->head_dim != 128)
        return 1;
    HtArgs a;
    std::memset(&a, 0, sizeof(a));
    if (cb->bits != 8 && !ht_table(cb, &a)) return 1;
    CUtensorMap map;
    if (!ht_make_map(&map, x, x_dtype, n_vec, 128, x_stride_bytes)) return 1;
    a.x = x;
    a.blocks = blocks;
    a.n_vec = n_vec;
    a.x_stride = x_stride_bytes;
    a.nc = nc;
    a.dense = dense;
    for (int i = 0; i < 4; ++i) a.signs[i] = signs[i];
    a.drop = drop_copies();
    return x_dtype == TQ_BF16 ? ht_launch_ext<TQ_BF16>(map, a, cb->bits, st)
                              : ht_launch_ext<TQ_F16>(map, a, cb->bits, st);
}

int wait_failed_headdim(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

}  // namespace tq
