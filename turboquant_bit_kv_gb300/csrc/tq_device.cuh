// Device helpers shared by libtq's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int kD = 128;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

template <int BITS>
struct BlockFmt {
    static constexpr int kBytes = 2 + 16 * BITS;  // 34 / 50 / 66
    static constexpr int kWords = 4 * BITS;       // 32-bit code words after the norm
    static constexpr int kLevels = 1 << BITS;
};

template <int DT>
struct InFmt {
    static constexpr int kRowBytes = DT == TQ_F32 ? 512 : 256;
    static constexpr int kPitch = kRowBytes + 16;  // conflict-free 16-byte row reads
};


// Kernel-parameter copy of a codebook: centroids, boundaries and the
// non-negative boundaries b[L/2 .. L-2] ("positive" half; b[L/2 - 1] == 0).
struct DevCodebook {
    float c[16];
    float b[15];
    int bits;
};

__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
// a - b rounded once: fma(b, -1, a).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    return __ffma2_rn(b, make_float2(-1.f, -1.f), a);
}

// Unnormalised Walsh-Hadamard transform of 128 values held as 64 packed pairs
// p[i] = (e_i, e_{i+64}).  Stages 1..32 act on both halves at once with
// packed float2 adds; stage 64 combines the two halves of each pair.  The
// result is H e in Sylvester order (H[i][j] = (-1)^popcount(i & j)), in the
// same pair layout.
__device__ __forceinline__ void fwht128(float2 (&p)[64]) {
#pragma unroll
    for (int L = 1; L < 64; L <<= 1) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            if ((i & L) == 0) {
                float2 a = p[i], b = p[i + L];
                p[i] = add2(a, b);
                p[i + L] = sub2(a, b);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        float x = p[i].x, y = p[i].y;
        p[i] = make_float2(x + y, x - y);
    }
}

// Unnormalised Walsh-Hadamard transform (Sylvester order) of one 128-element
// vector shared by a thread pair (partner = lane ^ 1).  Thread h of the pair
// holds elements e(c, k) = 16c + 8h + k (c, k = 0..7) as packed pairs
// p[c'][k] = (e(c', k), e(c' + 4, k)); sgn = +1 for h = 0 and -1 for h = 1.
// Six stages (element bits 0-2, 4-6) run in registers; the stage on bit 3 is
// one exchange with the partner and one packed FMA, which leaves both
// threads with exact butterfly outputs.
__device__ __forceinline__ void fwht_pair128(float2 (&p)[4][8], float sgn) {
#pragma unroll
    for (int L = 1; L < 8; L <<= 1)              // element bits 0..2 (k)
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if ((k & L) == 0) {
                    const float2 a = p[c][k], b = p[c][k + L];
                    p[c][k] = __fadd2_rn(a, b);
                    p[c][k + L] = sub2(a, b);
                }
#pragma unroll
    for (int L = 1; L < 4; L <<= 1)              // element bits 4..5 (c')
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if ((c & L) == 0)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 a = p[c][k], b = p[c + L][k];
                    p[c][k] = __fadd2_rn(a, b);
                    p[c + L][k] = sub2(a, b);
                }
#pragma unroll
    for (int c = 0; c < 4; ++c)                  // element bit 6 (inside a pair)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float x = p[c][k].x, y = p[c][k].y;
            p[c][k] = make_float2(x + y, x - y);
        }
    // element bit 3: the partner holds e ^ 8.  h = 0 keeps e + partner,
    // h = 1 (partner holds e - 8) keeps partner - own: fma(own, sgn, partner).
    const float2 s2 = make_float2(sgn, sgn);
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float2 o;
            o.x = __shfl_xor_sync(0xffffffffu, p[c][k].x, 1);
            o.y = __shfl_xor_sync(0xffffffffu, p[c][k].y, 1);
            p[c][k] = __ffma2_rn(p[c][k], s2, o);
        }
}

// Value j (0..127) of the pair layout.
template <int J>
__device__ __forceinline__ float pair_get(const float2 (&p)[64]) {
    return J < 64 ? p[J & 63].x : p[J & 63].y;
}

__device__ __forceinline__ float bf16_bits_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_bits_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sum of squares of the 128 values by 8 packed accumulator chains and a
// pairwise tree (relative error below 12 * 2^-24 for these non-negative terms).
__device__ __forceinline__ float sumsq128(const float2 (&p)[64]) {
    float2 acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = __fmul2_rn(p[k], p[k]);
#pragma unroll
    for (int i = 8; i < 64; ++i) acc[i & 7] = __ffma2_rn(p[i], p[i], acc[i & 7]);
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1)
#pragma unroll
        for (int k = 0; k < s; ++k) acc[k] = add2(acc[k], acc[k + s]);
    return acc[0].x + acc[0].y;
}

// Error-free sum a + b = s + e (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// True when n (>= 0) lies within rel * n of a rounding boundary of fp16
// round-to-nearest, i.e. when a small error in n could change fp16(n).
__device__ __forceinline__ bool near_fp16_tie(float n, float rel) {
    __half h = __float2half_rn(n);
    unsigned short hb = __half_as_ushort(h);
    if (hb >= 0x7C00u) return n >= 65504.f * (1.f - 4.f * rel);   // overflow side
    float hv = __half2float(h);
    float tol = n * rel;
    if (hb > 0) {
        float lo = __half2float(__ushort_as_half((unsigned short)(hb - 1)));
        if (fabsf(n - 0.5f * (lo + hv)) <= tol) return true;
    }
    float hi = (hb + 1 >= 0x7C00u) ? 65520.f : __half2float(__ushort_as_half((unsigned short)(hb + 1)));
    return fabsf(n - 0.5f * (hv + hi)) <= tol;
}

// Conservative, integer-only form of near_fp16_tie(n, 2^-20): true when the
// 13 float bits below the fp16 mantissa are within 16 units of the half-way
// pattern 0x1000 (16 float ulps are 2^-20 .. 2^-19 of n), or when n is
// outside fp16's normal range (zero, subnormal, overflow).
__device__ __forceinline__ bool near_fp16_tie_fast(float n) {
    const uint32_t b = __float_as_uint(n);
    return ((b & 0x1FFFu) - 0x0FF0u) <= 0x20u || !(n >= 6.103515625e-05f && n < 65504.f);
}

// Double-float accumulation of a sum of squares (TwoProduct via FMA, TwoSum).
struct SumSq2 {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float v) {
        float pr = v * v;
        float pe = fmaf(v, v, -pr);
        float t, e;
        two_sum(s, pr, t, e);
        s = t;
        c += e + pe;
    }
    // sqrt of the sum, rounded once to fp16 (round to nearest even).
    __device__ __forceinline__ unsigned short sqrt_fp16() const {
        float hi, lo;
        two_sum(s, c, hi, lo);
        return __half_as_ushort(__double2half(sqrt((double)hi + (double)lo)));
    }
};

// fp16 of the L2 norm of a row of 128 values (dtype DT) held in shared memory,
// accurate to far below an fp16 rounding step.  Used only when the fast
// float estimate lies within 2^-20 of an fp16 rounding boundary; out of line
// because it is rare.
template <int DT>
__device__ __noinline__ unsigned short exact_norm_fp16_smem(const uint8_t *row) {
    SumSq2 acc;
    for (int j = 0; j < kD; ++j) {
        float v;
        if (DT == TQ_F32) v = reinterpret_cast<const float *>(row)[j];
        else if (DT == TQ_BF16) v = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(row)[j] << 16);
        else v = __half2float(reinterpret_cast<const __half *>(row)[j]);
        acc.add(v);
    }
    return acc.sqrt_fp16();
}

// Norm of a row of 128 values in shared memory, in double (exact squares).
template <int DT>
__device__ __noinline__ double norm_double_smem(const uint8_t *row) {
    double acc = 0.0;
    for (int j = 0; j < kD; ++j) {
        float v;
        if (DT == TQ_F32) v = reinterpret_cast<const float *>(row)[j];
        else if (DT == TQ_BF16) v = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(row)[j] << 16);
        else v = __half2float(reinterpret_cast<const __half *>(row)[j]);
        acc = fma((double)v, (double)v, acc);
    }
    return sqrt(acc);
}

// Norm of the vector whose (sign-flipped) values are in p and whose raw row
// is still in shared memory at `row`.  Returns the fp16 bits of ||x|| and, in
// n_out, a float32 norm in the same units as p on return.  When the sum of
// squares leaves [2^-100, 2^100] (tiny or huge vectors, where float32 squares
// underflow or overflow) p is first rescaled by an exact power of two so the
// transform and the quantiser work in range; codes do not depend on the
// scale, and the stored norm comes from a double-precision sum.
template <int DT>
__device__ __forceinline__ unsigned short norm_fp16(float2 (&p)[64], const uint8_t *row, float &n_out) {
    const float ss = sumsq128(p);
    if (ss >= 7.888609052210118e-31f /* 2^-100 */ && ss <= 1.2676506002282294e30f /* 2^100 */) {
        const float n = sqrtf(ss);
        n_out = n;
        if (!near_fp16_tie(n, 9.5367431640625e-07f /* 2^-20 */))
            return __half_as_ushort(__float2half_rn(n));
        return exact_norm_fp16_smem<DT>(row);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fmaxf(fabsf(p[i].x), fabsf(p[i].y)));
    if (amax == 0.f) {
        n_out = 0.f;
        return 0;
    }
    int e;
    frexpf(amax, &e);                       // amax = m 2^e, m in [0.5, 1)
    const int e1 = -e / 2, e2 = -e - e1;    // two factors, each a normal float
    const float2 s1 = make_float2(ldexpf(1.f, e1), ldexpf(1.f, e1));
    const float2 s2 = make_float2(ldexpf(1.f, e2), ldexpf(1.f, e2));
#pragma unroll
    for (int i = 0; i < 64; ++i) p[i] = __fmul2_rn(__fmul2_rn(p[i], s1), s2);
    n_out = sqrtf(sumsq128(p));
    return __half_as_ushort(__double2half(norm_double_smem<DT>(row)));
}

// 16-byte async copy global -> shared (L2 only, no L1 allocation).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Sticky record of a bounded wait that gave up.  Each translation unit that
// includes this header has its own word (there is no device-side linking
// between units); the units whose kernels wait on mbarriers expose a host
// reader of theirs, and tq_device_status combines them.
static __device__ unsigned int g_tq_wait_failed;

__device__ __forceinline__ void note_wait_failed() { atomicOr(&g_tq_wait_failed, 1u); }

// Host: this unit's word on the current device (reset when `clear`).
static inline int read_wait_failed(unsigned *v, bool clear) {
    if (cudaMemcpyFromSymbol(v, g_tq_wait_failed, sizeof(unsigned)) != cudaSuccess) return TQ_ERR_CUDA;
    const unsigned zero = 0;
    if (clear && cudaMemcpyToSymbol(g_tq_wait_failed, &zero, sizeof(unsigned)) != cudaSuccess) return TQ_ERR_CUDA;
    return TQ_OK;
}

// Wait for the phase of parity `parity` of the mbarrier at shared address
// `bar`.  mbarrier.try_wait suspends the warp in hardware for a while instead
// of spinning on issue slots; the wait gives up (false) after about 100 ms
// of device time (or 2^22 attempts), so a copy that never lands cannot hang
// the kernel.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns = 100000000ull) {
    uint64_t t0 = 0;
    for (int i = 0; i < (1 << 22); ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        uint64_t now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (i == 0) t0 = now;
        else if (now - t0 > limit_ns) break;
    }
    return false;
}

// Spin for about `ns` of device time (the drain of a kernel whose wait gave up:
// copies it may still have in flight land meanwhile).
__device__ __forceinline__ void spin_ns(uint64_t ns) {
    uint64_t t0, now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        __nanosleep(1000);
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    } while (now - t0 < ns);
}

// 32-bit word at a 2-byte aligned shared-memory address.
__device__ __forceinline__ uint32_t lds_u32_a2(const uint8_t *p) {
    const uint16_t *h = reinterpret_cast<const uint16_t *>(p);
    return (uint32_t)h[0] | ((uint32_t)h[1] << 16);
}

}  // namespace tq
