// tq_attn_prefill: attention of several new query tokens per sequence (a
// prefill chunk, or the draft tokens of a speculative verify step) over a
// packed cache that already holds them, with the causal mask, on the
// 5th-generation tensor cores.
//
// "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)", section 2
// (Requirements): the quantised KV cache is reachable only through the fused
// flash-attention path, prefill included; "TurboQuant KV Cache Compression —
// Spec", Optimization: Fused dequant-dot: the query is rotated once, keys are
// scored as norm x centroid in the rotated domain, values are accumulated in
// the rotated domain and the output is rotated back once.  With M query
// tokens and G query heads per KV head, the M x G query rows of a (sequence,
// KV head) meet every key, so the scores and the value sums are dense
// contractions: a CTA takes 128 of those rows and streams the keys in tiles
// of 64.
//
//   S[128 rows x 64 keys]  = Q[128 x 128 dims] K^T         (tcgen05, 3 products)
//   O[128 rows x 128 dims] += P[128 x 64 keys] V[64 x 128]  (tcgen05, 2 products)
//
// Precision as in the decode kernel: the rotated, scaled query, the key
// centroids and the probabilities are split x = hi + lo into fp16 halves
// (products hi.hi + hi.lo + lo.hi, float32 accumulate in tensor memory); the
// value centroids are single fp16.  Key norms scale the scores, value norms
// scale the probabilities.
//
// Warp roles (448 threads, one CTA per SM):
//   warps 0-7  row warps: threads (r, h) own query row r = tensor-memory
//              lane r, keys 32 h .. 32 h + 31 of each tile (warps w and w + 4
//              read the same lanes).  Per key tile: read S, apply key norms
//              and the causal mask, share the row maximum with the other
//              thread of the row, online softmax (the reference maximum
//              moves only when a row's maximum exceeds it by more than 8 in
//              log2 units, so that the accumulator in tensor memory is
//              rarely rescaled), write P (times the value norms) as fp16
//              hi / lo parts into tensor memory, the A operand of P V (two
//              stages, so the row warps wait for the products of tile j - 2,
//              not j - 1).  Epilogue: O / l, inverse rotation (its last
//              stage across the row's two threads), store.
//   warps 8-11 key warps: thread (k, h) dequantises dims 64 h .. + 63 of key
//              k of the tile into the K hi / lo tiles and the V tile
//              (centroid lookups in lane-replicated tables).
//   warp 12    producer: bulk copies of the tile's packed K and V blocks.
//   warp 13    one thread issues the tensor-core products.
// All warps prepare the rotated query rows in the prologue.
// Key tiles and their packed blocks are double-buffered, as are the score
// accumulators, so the products of tile j + 1 run while the row warps work on
// tile j.  Every mbarrier wait is bounded; a wait that gives up is recorded
// (tq_device_status) and the roles run their loops to the end without further
// waits or issues.

#include <cmath>

#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {
namespace {

constexpr int kPfRows = 128;                 // query rows per CTA (MMA M, tensor-memory lanes)
constexpr int kPfKeys = 64;                  // keys per tile (N of the scores, K of P V)
constexpr int kPfRowWarps = 8;               // two threads per query row (32 keys of a tile each)
constexpr int kPfKeyWarps = 4;               // two threads per key (64 dims each)
constexpr int kPfProducerWarp = kPfRowWarps + kPfKeyWarps;
constexpr int kPfMmaWarp = kPfProducerWarp + 1;
constexpr int kPfThreads = 32 * (kPfMmaWarp + 1);   // 448
// tensor memory: S[2] (64 columns each) at 0, O (128) at 128, P[2] at 256: each P stage holds the
// hi parts (32 columns: 64 keys of fp16 pairs) then the lo parts
constexpr uint32_t kPfCols = 512;
constexpr uint32_t kPfColO = 128;
constexpr uint32_t kPfColP = 256;

// Shared memory (offsets from a 1024-byte aligned base).  Operand tiles use the
// K-major 128-byte swizzle of tq_tc.cuh: 64-element blocks of rows x 128 bytes.
template <int KB, int VB>
struct PfSmem {
    static constexpr int kQhi = 0;                         // Q hi: 128 rows x 128 dims (two 16 KB blocks)
    static constexpr int kQlo = 32768;
    static constexpr int kKhi = 65536;                     // [2] keys: 64 rows x 128 dims (two 8 KB blocks)
    static constexpr int kKlo = 98304;                     // [2]
    static constexpr int kV = 131072;                      // [2] values: 64 keys x 128 dims, same layout
    static constexpr int kBlk = 163840;                    // [2] packed blocks: 64 K blocks | 64 V blocks
    static constexpr int kBlkBytes = kPfKeys * (2 + 16 * KB + 2 + 16 * VB);
    static constexpr int kNorm = kBlk + 2 * kBlkBytes;     // [2] kn[64] | vn[64] (float)
    static constexpr int kKTab = kNorm + 2 * 512;          // key centroids: 16 codes x 32 lanes x half2 (hi, lo)
    static constexpr int kVTab = kKTab + 2048;             // value centroids: 16 codes x 32 lanes x half2 (v, v)
    static constexpr int kXch = kVTab + 2048;              // row max / sum exchange: [2][2][128] float
    static constexpr int kBars = kXch + 2048;              // 24 mbarriers
    static constexpr int kSlot = kBars + 24 * 8;           // tensor-memory base address, failure flag
    static constexpr int kTotal = kSlot + 16 + 1024;       // + alignment slack of the base
    static_assert(kTotal <= 232448, "shared memory of one CTA");
};

// mbarriers
enum {
    kBlkFull = 0,    // [2] packed blocks landed (bulk copy bytes)
    kBlkEmpty = 2,   // [2] packed blocks read (4 key warps)
    kKvReady = 4,    // [2] K / V tiles written (4 key warps)
    kKvFree = 6,     // [2] the products that read the K / V tiles completed (commit)
    kSReady = 8,     // [2] scores in tensor memory (commit)
    kSFree = 10,     // [2] scores read (4 row warps)
    kPReady = 12,    // [2] P written, O rescaled if needed (8 row warps)
    kPvDone = 14,    // [2] P V completed: P stage free, O current (commit)
    kDrain = 16      // the issuing thread's last commit before teardown
};

struct PfArgs {
    const void *q;          // [B][M][Hq][128]
    const uint8_t *k;       // [B][Hkv][T_cap] key blocks
    const uint8_t *v;       // [B][Hkv][T_cap] value blocks
    const int32_t *seq_lens;
    float *out;             // [B][M][Hq][128]
    int q_dtype, B, M, Hq, Hkv, G, T_cap, T, kbb, vbb, row_tiles;
    float qscale;           // scale * log2(e)
    float kc[16], vc[16];
    uint32_t signs[4];
    int drop;               // test hook: issue no bulk copies (the waits for them run out)
    // paged cache (NULL table: contiguous [B][Hkv][T_cap]): pages of `page` tokens in pools
    // [pages][Hkv][page]; token t of sequence b is slot t % page of page table[b * max_pages + t / page]
    const int32_t *table;
    int max_pages, page;
};

__device__ __forceinline__ uint64_t pf_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: float32 accumulator, fp16 A and B, A
// K-major, B K-major (tb = 0) or MN-major (tb = 1), M = 128, N = n.
__host__ __device__ constexpr uint32_t pf_idesc(uint32_t n, uint32_t tb) {
    return (1u << 4) | (tb << 16) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void pf_sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void pf_bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// D (+)= A B with A (M 128 x K 16, fp16) in tensor memory at column a_tmem (rows in lanes, K pairs
// packed per 32-bit column) and B from a shared-memory descriptor.
__device__ __forceinline__ void pf_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::
            "r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
        "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
        "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
        "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

__device__ __forceinline__ uint32_t pf_lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t pf_lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t pf_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pf_pack(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Code words of dims 32 q .. 32 q + 31 of the block at shared address `blk`
// (2-byte aligned): 8-bit (turboq8): 8 words; 4-bit: 4 words; 2-bit: 2
// words; 3-bit: 2 low-plane words then 1 high-plane word.
template <int BITS>
__device__ __forceinline__ void pf_code_words(uint32_t blk, int q, uint32_t (&w)[8]) {
    auto word = [&](uint32_t at) { return pf_lds16(at) | (pf_lds16(at + 2) << 16); };
    if constexpr (BITS == 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = word(blk + 2 + 32 * q + 4 * i);
    } else if constexpr (BITS == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = word(blk + 2 + 16 * q + 4 * i);
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) w[i] = word(blk + 2 + 8 * q + 4 * i);
        if constexpr (BITS == 3) w[2] = word(blk + 34 + 4 * q);
    }
}

// Code of relative dim e (0..31) from the words above.
template <int BITS>
__device__ __forceinline__ uint32_t pf_code(const uint32_t (&w)[8], int e) {
    if constexpr (BITS == 8) return (w[e >> 2] >> (8 * (e & 3))) & 255u;
    else if constexpr (BITS == 4) return (w[e >> 3] >> (4 * (e & 7))) & 15u;
    else if constexpr (BITS == 2) return (w[e >> 4] >> (2 * (e & 15))) & 3u;
    else return ((w[e >> 4] >> (2 * (e & 15))) & 3u) | (((w[2] >> e) & 1u) << 2);
}

// 2^x (the special-function unit's approximation, a few ulp; 2^-inf = 0).
__device__ __forceinline__ float pf_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (hi, lo) fp16 splits of two floats, packed as half2 words: x = hi + lo to about 2^-22.
__device__ __forceinline__ void pf_split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// turboq8 entry of code i: the grid level (i - 127.5) / 127.5 is (2 i - 255) / 255; the integer
// 2 i - 255 is exact in fp16, the 1 / 255 goes into the block's norm factor (no lo half needed).
__device__ __forceinline__ uint32_t pf_q8_entry(uint32_t i, bool dup) {
    const uint32_t h = __half_as_ushort(__int2half_rn((int)(2 * i) - 255));
    return dup ? (h | (h << 16)) : h;
}

template <int KB, int VB>
__global__ void __launch_bounds__(kPfThreads, 1) attn_prefill_kernel(const __grid_constant__ PfArgs a) {
    using S = PfSmem<KB, VB>;
    extern __shared__ __align__(16) uint8_t pf_smem_raw[];
    const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(pf_smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = pf_smem_raw + (base_s - raw_s);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bars = base_s + S::kBars;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile int *fail_s = reinterpret_cast<volatile int *>(smem + S::kSlot + 4);

    // ---- the CTA's rows and key range
    const int rt = blockIdx.x % a.row_tiles;
    const int seg = blockIdx.x / a.row_tiles;
    const int b = seg / a.Hkv, kvh = seg % a.Hkv;
    int L = a.T;
    if (a.seq_lens) {
        const int sl = a.seq_lens[b];
        L = sl < 0 ? 0 : (sl > a.T ? a.T : sl);
    }
    const int rows_total = a.M * a.G;
    const int r0 = rt * kPfRows;
    const int i_hi = min(a.M - 1, (min(r0 + kPfRows, rows_total) - 1) / a.G);
    const int p_max = L - a.M + i_hi;                      // last key any row of the CTA sees
    const int n_tiles = p_max < 0 ? 0 : (p_max + kPfKeys) / kPfKeys;
    const int n_keys8 = p_max < 0 ? 0 : ((p_max + 8) & ~7);   // keys copied, a multiple of 8 (<= T_cap)

    // ---- setup: centroid tables, rotated query rows, barriers, tensor memory
    for (int q = tid; q < 16 * 32; q += kPfThreads) {
        const int e = q >> 5, l = q & 31;
        const float c = a.kc[e];
        const __half h = __float2half_rn(c);
        const __half lo = __float2half_rn(c - __half2float(h));
        *reinterpret_cast<__half2 *>(smem + S::kKTab + e * 128 + l * 4) = __halves2half2(h, lo);
        const __half vh = __float2half_rn(a.vc[e]);
        *reinterpret_cast<__half2 *>(smem + S::kVTab + e * 128 + l * 4) = __halves2half2(vh, vh);
    }
    // query rows: one warp per row; lane holds dims 4 lane .. + 3; R q = H (D q) / sqrt(128), times scale log2(e)
    for (int r = warp; r < kPfRows; r += kPfThreads / 32) {
        const int rg = r0 + r;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (rg < rows_total) {
            const int i = rg / a.G, hq = kvh * a.G + rg % a.G;
            const int64_t base = (((int64_t)b * a.M + i) * a.Hq + hq) * kD + 4 * lane;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float x;
                if (a.q_dtype == TQ_F32) x = reinterpret_cast<const float *>(a.q)[base + k];
                else if (a.q_dtype == TQ_BF16) x = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.q)[base + k]);
                else x = __half2float(reinterpret_cast<const __half *>(a.q)[base + k]);
                const int d = 4 * lane + k;
                v[k] = ((a.signs[d >> 5] >> (d & 31)) & 1u) ? -x : x;
            }
        }
        const float x0 = v[0] + v[1], x1 = v[0] - v[1], x2 = v[2] + v[3], x3 = v[2] - v[3];
        v[0] = x0 + x2;
        v[2] = x0 - x2;
        v[1] = x1 + x3;
        v[3] = x1 - x3;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float o = __shfl_xor_sync(0xffffffffu, v[k], m);
                v[k] = (lane & m) ? (o - v[k]) : (v[k] + o);
            }
        }
        const float f = a.qscale * 0.08838834764831845f;
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) pf_split2(v[2 * k] * f, v[2 * k + 1] * f, hi[k], lo[k]);
        // dims 4 lane .. + 3: block lane >> 4, 16-byte chunk (lane & 15) >> 1, half of it lane & 1
        const int off = (lane >> 4) * 16384 + r * 128 + ((((lane & 15) >> 1) ^ (r & 7)) << 4) + (lane & 1) * 8;
        *reinterpret_cast<uint2 *>(smem + S::kQhi + off) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2 *>(smem + S::kQlo + off) = make_uint2(lo[0], lo[1]);
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            tc_mbar_init(bar(kBlkFull + s), 1);
            tc_mbar_init(bar(kBlkEmpty + s), kPfKeyWarps);
            tc_mbar_init(bar(kKvReady + s), kPfKeyWarps);
            tc_mbar_init(bar(kKvFree + s), 1);
            tc_mbar_init(bar(kSReady + s), 1);
            tc_mbar_init(bar(kSFree + s), kPfRowWarps);
        }
        for (int s = 0; s < 2; ++s) {
            tc_mbar_init(bar(kPReady + s), kPfRowWarps);
            tc_mbar_init(bar(kPvDone + s), 1);
        }
        tc_mbar_init(bar(kDrain), 1);
        *fail_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base_s + S::kSlot),
                     "r"(kPfCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the query tiles were written by ordinary stores and are read by the tensor cores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + S::kSlot);

    // a bounded wait; one that gives up is recorded, and the caller's role makes no further waits
    auto wait = [&](bool &ok, int b_idx, uint32_t parity) {
        if (ok && !tc_mbar_wait(bar(b_idx), parity)) {
            ok = false;
            *fail_s = 1;
            note_wait_failed();
        }
    };

    if (warp == kPfProducerWarp) {
        // ---- producer: packed K and V blocks of each tile
        if (lane == 0) {
            bool ok = true;
            const int64_t row0 = (int64_t)seg * a.T_cap;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j & 1, u = j >> 1;
                if (u >= 1) wait(ok, kBlkEmpty + s, (uint32_t)(u - 1) & 1u);
                if (!ok) break;
                const int t0 = j * kPfKeys;
                const int nk = min(kPfKeys, n_keys8 - t0);
                const uint32_t dst = base_s + S::kBlk + s * S::kBlkBytes;
                if (!a.drop) {   // (test hook: no copy, so the key warps' wait runs out)
                    tc_mbar_expect_tx(bar(kBlkFull + s), (uint32_t)(nk * (a.kbb + a.vbb)));
                    if (!a.table) {
                        pf_bulk_g2s(dst, a.k + (row0 + t0) * a.kbb, (uint32_t)(nk * a.kbb), bar(kBlkFull + s));
                        pf_bulk_g2s(dst + kPfKeys * a.kbb, a.v + (row0 + t0) * a.vbb, (uint32_t)(nk * a.vbb),
                                    bar(kBlkFull + s));
                    } else {
                        // one pair of copies per page the tile touches (pieces of a multiple of 8 tokens)
                        for (int t = t0; t < t0 + nk;) {
                            const int pg = t / a.page, off = t - pg * a.page;
                            const int n = min(t0 + nk - t, a.page - off);
                            const int64_t slot = ((int64_t)a.table[(int64_t)b * a.max_pages + pg] * a.Hkv + kvh) *
                                                     a.page + off;
                            pf_bulk_g2s(dst + (t - t0) * a.kbb, a.k + slot * a.kbb, (uint32_t)(n * a.kbb),
                                        bar(kBlkFull + s));
                            pf_bulk_g2s(dst + kPfKeys * a.kbb + (t - t0) * a.vbb, a.v + slot * a.vbb,
                                        (uint32_t)(n * a.vbb), bar(kBlkFull + s));
                            t += n;
                        }
                    }
                }
            }
        }
    } else if (warp == kPfMmaWarp) {
        // ---- the tensor-core products
        if (lane == 0) {
            bool ok = true;
            const uint32_t id_s = pf_idesc(kPfKeys, 0), id_pv = pf_idesc(128, 1);
            auto scores = [&](int j) {
                const int s = j & 1;
                const uint32_t d = tmem + (uint32_t)(s * kPfKeys);
                const uint32_t kh = base_s + S::kKhi + s * 16384, kl = base_s + S::kKlo + s * 16384;
                // turboq8 keys are exact in fp16: no lo product
                constexpr int kParts = KB == 8 ? 2 : 3;
#pragma unroll
                for (int part = 0; part < kParts; ++part) {
                    const uint32_t qa = base_s + ((part == 2 || (KB == 8 && part == 1)) ? S::kQlo : S::kQhi);
                    const uint32_t kb = (KB != 8 && part == 1) ? kl : kh;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t qo = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32);
                        const uint32_t ko = (uint32_t)((ks >> 2) * 8192 + (ks & 3) * 32);
                        tc_mma(d, pf_desc(qa + qo, 16, 1024), pf_desc(kb + ko, 16, 1024), id_s,
                               (part > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                tc_commit(bar(kSReady + s));
            };
            auto values = [&](int j) {
                const int s = j & 1;
                const uint32_t vs = base_s + S::kV + s * 16384;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    // A = P of stage s in tensor memory (rows in lanes, 16 keys = 8 columns per step)
                    const uint32_t pa = tmem + kPfColP + 64u * (uint32_t)s + 32u * (uint32_t)part;
#pragma unroll
                    for (int ks = 0; ks < kPfKeys / 16; ++ks)
                        pf_mma_ts(tmem + kPfColO, pa + 8u * (uint32_t)ks, pf_desc(vs + ks * 2048, 8192, 1024), id_pv,
                                  (j > 0 || part > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(bar(kPvDone + s));
                tc_commit(bar(kKvFree + s));
            };
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j & 1, u = j >> 1;
                wait(ok, kKvReady + s, (uint32_t)u & 1u);
                if (u >= 1) wait(ok, kSFree + s, (uint32_t)(u - 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                scores(j);
                if (j >= 1) {
                    wait(ok, kPReady + ((j - 1) & 1), (uint32_t)((j - 1) >> 1) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    values(j - 1);
                }
            }
            if (ok && n_tiles > 0) {
                wait(ok, kPReady + ((n_tiles - 1) & 1), (uint32_t)((n_tiles - 1) >> 1) & 1u);
                if (ok) {
                    tc_fence_after();
                    values(n_tiles - 1);
                }
            }
            // before teardown: every product issued here has completed
            tc_commit(bar(kDrain));
            tc_mbar_wait(bar(kDrain), 0u);
        }
    } else if (warp >= kPfRowWarps) {
        // ---- key warps: thread (k, hk) = dims 64 hk .. 64 hk + 63 of key k of the tile, taken as the
        // 32-dim quarters q = 2 hk, 2 hk + 1
        const int kt = tid - 32 * kPfRowWarps, k = kt >> 1, hk = kt & 1;
        const uint32_t ktab = base_s + S::kKTab + 4u * lane, vtab = base_s + S::kVTab + 4u * lane;
        float *norms = reinterpret_cast<float *>(smem + S::kNorm);
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int s = j & 1, u = j >> 1;
            wait(ok, kBlkFull + s, (uint32_t)u & 1u);
            if (u >= 1) wait(ok, kKvFree + s, (uint32_t)(u - 1) & 1u);
            const uint32_t blk = base_s + S::kBlk + s * S::kBlkBytes;
            const uint32_t kblk = blk + k * a.kbb, vblk = blk + kPfKeys * a.kbb + k * a.vbb;
            // dims 32 q .. + 31: 64-dim block q >> 1, 16-byte chunks 4 (q & 1) .. + 3 of row k
            const uint32_t row = (uint32_t)(hk * 8192 + k * 128);
#pragma unroll
            for (int q = 2 * hk; q < 2 * hk + 2; ++q) {
                uint32_t w[8];
                pf_code_words<KB>(kblk, q, w);
                const uint32_t khi = base_s + S::kKhi + s * 16384 + row, klo = base_s + S::kKlo + s * 16384 + row;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t e[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        e[i] = KB == 8 ? pf_q8_entry(pf_code<KB>(w, 8 * c + i), false)
                                       : pf_lds32(ktab + pf_code<KB>(w, 8 * c + i) * 128u);
                    const uint32_t sw = (uint32_t)((((4 * (q & 1) + c) ^ (k & 7)) << 4));
                    pf_sts128(khi + sw, pf_prmt(e[0], e[1], 0x5410), pf_prmt(e[2], e[3], 0x5410),
                              pf_prmt(e[4], e[5], 0x5410), pf_prmt(e[6], e[7], 0x5410));
                    if constexpr (KB != 8)
                        pf_sts128(klo + sw, pf_prmt(e[0], e[1], 0x7632), pf_prmt(e[2], e[3], 0x7632),
                                  pf_prmt(e[4], e[5], 0x7632), pf_prmt(e[6], e[7], 0x7632));
                }
            }
#pragma unroll
            for (int q = 2 * hk; q < 2 * hk + 2; ++q) {
                uint32_t w[8];
                pf_code_words<VB>(vblk, q, w);
                const uint32_t vt = base_s + S::kV + s * 16384 + row;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t e[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        e[i] = VB == 8 ? pf_q8_entry(pf_code<VB>(w, 8 * c + i), true)
                                       : pf_lds32(vtab + pf_code<VB>(w, 8 * c + i) * 128u);
                    pf_sts128(vt + (uint32_t)((((4 * (q & 1) + c) ^ (k & 7)) << 4)), pf_prmt(e[0], e[1], 0x5410),
                              pf_prmt(e[2], e[3], 0x5410), pf_prmt(e[4], e[5], 0x5410), pf_prmt(e[6], e[7], 0x5410));
                }
            }
            if (hk == 0) {
                // the block's norm (turboq8: its scale over 255, the grid's step factor)
                const float kf = KB == 8 ? (1.f / 255.f) : 1.f, vf = VB == 8 ? (1.f / 255.f) : 1.f;
                norms[s * 128 + k] = __half2float(__ushort_as_half((unsigned short)pf_lds16(kblk))) * kf;
                norms[s * 128 + 64 + k] = __half2float(__ushort_as_half((unsigned short)pf_lds16(vblk))) * vf;
            }
            // the tiles were written by ordinary stores and are read by the tensor cores
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                tc_mbar_arrive(bar(kBlkEmpty + s));
                tc_mbar_arrive(bar(kKvReady + s));
            }
        }
    } else {
        // ---- row warps: thread (r, h) = keys 32 h .. 32 h + 31 of each tile for query row r0 + r
        // (tensor-memory lane r); the two threads of a row meet through shared memory on named
        // barrier 1 (the eight row warps) to share the row maximum, the row sum and the output
        const int r = tid & 127, h = tid >> 7, rg = r0 + r;
        const bool row_valid = rg < rows_total;
        const int qi = row_valid ? rg / a.G : 0;
        const int pos = L - a.M + qi;                  // this row's query position (keys 0 .. pos)
        const uint32_t lane_t = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const float *norms = reinterpret_cast<const float *>(smem + S::kNorm);
        float *xch = reinterpret_cast<float *>(smem + S::kXch);   // [tile parity][half][128 rows]
        auto rows_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kPfRowWarps) : "memory"); };
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int s = j & 1, u = j >> 1;
            wait(ok, kSReady + s, (uint32_t)u & 1u);
            tc_fence_after();
            float sv[32];
            tc_ld32(lane_t + (uint32_t)(s * kPfKeys + 32 * h), sv);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bar(kSFree + s));
            // key norms and the causal mask (key t visible to the row iff t <= pos); a warp whose 32
            // keys are all visible to all its rows (every tile but the last few) skips the mask
            const int t0 = j * kPfKeys + 32 * h;
            const float4 *kn4 = reinterpret_cast<const float4 *>(norms + s * 128 + 32 * h);
            const float4 *vn4 = reinterpret_cast<const float4 *>(norms + s * 128 + 64 + 32 * h);
            const bool full = __all_sync(0xffffffffu, row_valid && t0 + 31 <= pos);
            float mx = -INFINITY;
            if (full) {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 n = kn4[q4];
                    const float2 a = __fmul2_rn(make_float2(sv[4 * q4], sv[4 * q4 + 1]), make_float2(n.x, n.y));
                    const float2 b = __fmul2_rn(make_float2(sv[4 * q4 + 2], sv[4 * q4 + 3]), make_float2(n.z, n.w));
                    sv[4 * q4] = a.x;
                    sv[4 * q4 + 1] = a.y;
                    sv[4 * q4 + 2] = b.x;
                    sv[4 * q4 + 3] = b.y;
                    mx = fmaxf(mx, fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y)));
                }
            } else {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 n = kn4[q4];
                    const float nn[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * q4 + e;
                        const bool vis = row_valid && t0 + c <= pos;
                        sv[c] = vis ? sv[c] * nn[e] : -INFINITY;
                        mx = fmaxf(mx, sv[c]);
                    }
                }
            }
            xch[(s * 2 + h) * 128 + r] = mx;
            rows_sync();
            mx = fmaxf(mx, xch[(s * 2 + (h ^ 1)) * 128 + r]);
            // the reference maximum moves when the row's maximum exceeds it by more than 8 (log2
            // units), so probabilities stay below 2^8 and O is rarely rescaled
            const bool move = mx > m_ref + 8.f;
            const float m_new = move ? mx : m_ref;
            const float factor = move ? (m_ref == -INFINITY ? 0.f : exp2f(m_ref - m_new)) : 1.f;
            // P stage s is free once the products of tile j - 2 have completed; O is rescaled only
            // after those of tile j - 1, so that it holds exactly the earlier tiles
            if (j >= 2) wait(ok, kPvDone + s, (uint32_t)((j - 2) >> 1) & 1u);
            const bool resc = j >= 1 && __any_sync(0xffffffffu, move);
            if (resc) wait(ok, kPvDone + ((j - 1) & 1), (uint32_t)((j - 1) >> 1) & 1u);
            tc_fence_after();
            if (resc) {
#pragma unroll
                for (int c4 = 0; c4 < 2; ++c4) {
                    float o32[32];
                    const uint32_t col = kPfColO + 64u * h + 32u * c4;
                    tc_ld32(lane_t + col, o32);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o32[c] *= factor;
                    tc_st32(lane_t + col, o32);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            float2 sum2 = make_float2(0.f, 0.f);
            uint32_t hw[16], lw[16];   // P of keys 32 h .. + 31 as fp16 pairs: hi and lo parts
            // (a row that has seen no visible key yet has m_new = -inf and only masked keys here)
            const float mref = m_new == -INFINITY ? 0.f : m_new;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int c = 8 * c8 + 2 * qq;
                    // p = 2^(s - m): exp2 of -inf is 0, so masked keys give p = 0; their value norms may
                    // be anything (keys past the copied ones), hence the select on the product
                    const float2 p = make_float2(pf_ex2(sv[c] - mref), pf_ex2(sv[c + 1] - mref));
                    sum2 = __fadd2_rn(sum2, p);
                    const float4 vn = vn4[c >> 2];
                    const float2 nv = (c & 2) ? make_float2(vn.z, vn.w) : make_float2(vn.x, vn.y);
                    float2 pp = __fmul2_rn(p, nv);
                    if (!full) {
                        pp.x = sv[c] == -INFINITY ? 0.f : pp.x;
                        pp.y = sv[c + 1] == -INFINITY ? 0.f : pp.y;
                    }
                    pf_split2(pp.x, pp.y, hw[4 * c8 + qq], lw[4 * c8 + qq]);
                }
            }
            // P of stage s: this row's lane, keys 32 h .. + 31 = columns 16 h .. + 15 of each part
            tc_st16u(lane_t + kPfColP + 64u * (uint32_t)s + 16u * (uint32_t)h, hw);
            tc_st16u(lane_t + kPfColP + 64u * (uint32_t)s + 32u + 16u * (uint32_t)h, lw);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            l = l * factor + (sum2.x + sum2.y);
            m_ref = m_new;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) tc_mbar_arrive(bar(kPReady + s));
        }
        // ---- epilogue: o = O / l, rotated back: D H o / sqrt(128); this thread holds dims 64 h .. + 63
        if (n_tiles > 0) wait(ok, kPvDone + ((n_tiles - 1) & 1), (uint32_t)((n_tiles - 1) >> 1) & 1u);
        tc_fence_after();
        // (the exchange slot of parity n_tiles was last read before the last tile's barrier)
        const int se = n_tiles & 1;
        xch[(se * 2 + h) * 128 + r] = l;
        rows_sync();
        const float lt = l + xch[(se * 2 + (h ^ 1)) * 128 + r];
        float o[64];
        if (n_tiles > 0) {
#pragma unroll
            for (int c4 = 0; c4 < 2; ++c4) {
                float o32[32];
                tc_ld32(lane_t + kPfColO + 64u * h + 32u * c4, o32);
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) o[32 * c4 + c] = o32[c];
            }
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = 0.f;
        }
        const float inv = (lt > 0.f && ok) ? 0.08838834764831845f / lt : (ok ? 0.f : __int_as_float(0x7fc00000));
#pragma unroll
        for (int m = 1; m < 64; m <<= 1) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                if ((c & m) == 0) {
                    const float x = o[c], y = o[c + m];
                    o[c] = x + y;
                    o[c + m] = x - y;
                }
            }
        }
        // the last butterfly stage pairs dim d of the low half with d + 64 of the high half: through
        // shared memory (the query tiles, no longer read once every product has completed)
        float *ox = reinterpret_cast<float *>(smem + S::kQhi);   // [128 rows][2 halves][64]
#pragma unroll
        for (int c = 0; c < 64; ++c) ox[(r * 2 + h) * 64 + ((c + r) & 63)] = o[c];
        rows_sync();
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float other = ox[(r * 2 + (h ^ 1)) * 64 + ((c + r) & 63)];
            o[c] = h ? (other - o[c]) : (o[c] + other);
        }
        if (row_valid) {
            const int hq = kvh * a.G + rg % a.G;
            float4 *dst = reinterpret_cast<float4 *>(a.out + (((int64_t)b * a.M + qi) * a.Hq + hq) * kD + 64 * h);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                float e[4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int d = 64 * h + 4 * c4 + qq;
                    const float x = o[4 * c4 + qq] * inv;
                    e[qq] = ((a.signs[d >> 5] >> (d & 31)) & 1u) ? -x : x;
                }
                dst[c4] = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
    }

    // ---- teardown: every product completed (the issuing thread waited for its last commit), every
    // tensor-memory access completed; copies still in flight after a failed wait land first
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*fail_s) {
        if (tid == 0) spin_ns(100000000ull);
        __syncthreads();
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPfCols) : "memory");
}

template <int KB, int VB>
int launch_prefill(const PfArgs &a, int grid, cudaStream_t st) {
    using S = PfSmem<KB, VB>;
    static int done[64] = {0};
    if (set_smem_limit((const void *)attn_prefill_kernel<KB, VB>, S::kTotal, done) != TQ_OK) return TQ_ERR_CUDA;
    attn_prefill_kernel<KB, VB><<<grid, kPfThreads, S::kTotal, st>>>(a);
    return launch_status();
}

// Key / value widths served: 2, 3, 4 with each other; turboq8 keys with 2/3/4-bit values and
// 4-bit keys with turboq8 values (the asymmetric pairs of the fork page; 8/8 does not fit the
// shared memory of one CTA).
template <int KB>
int launch_prefill_v(const PfArgs &a, int vb, int grid, cudaStream_t st) {
    switch (vb) {
        case 2: return launch_prefill<KB, 2>(a, grid, st);
        case 3: return launch_prefill<KB, 3>(a, grid, st);
        case 4: return launch_prefill<KB, 4>(a, grid, st);
        case 8:
            if constexpr (KB == 4) return launch_prefill<4, 8>(a, grid, st);
            return TQ_ERR_UNSUPPORTED;
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace

int wait_failed_prefill(unsigned *v, bool clear) { return read_wait_failed(v, clear); }

}  // namespace tq

using namespace tq;

namespace {

int prefill_call(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb, const uint8_t *v_blocks,
                 const tq_codebook *vcb, const int32_t *seq_lens, int B, int M, int Hq, int Hkv, int T_cap, int T,
                 float scale, tq_signs signs, float *out, const int32_t *table, int max_pages, int page,
                 void *stream) {
    if (!q || !k_blocks || !kcb || !v_blocks || !vcb || !out) return TQ_ERR_ARG;
    if (B <= 0 || M <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T_cap <= 0 || T < 1 || T > T_cap || (T_cap & 7))
        return TQ_ERR_ARG;
    if (!std::isfinite(scale)) return TQ_ERR_ARG;
    auto book_ok = [](const tq_codebook *cb) {
        return codebook_ok(cb) || (cb->head_dim == kD && cb->bits == 8 && cb->levels == 256);
    };
    if (dtype_bytes(q_dtype) == 0 || !book_ok(kcb) || !book_ok(vcb)) return TQ_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_blocks, 16) || !aligned(v_blocks, 16) || !aligned(out, 16)) return TQ_ERR_ALIGN;
    PfArgs a;
    a.q = q;
    a.q_dtype = q_dtype;
    a.k = k_blocks;
    a.v = v_blocks;
    a.seq_lens = seq_lens;
    a.out = out;
    a.B = B;
    a.M = M;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.T_cap = T_cap;
    a.T = T;
    a.kbb = 2 + 16 * kcb->bits;
    a.vbb = 2 + 16 * vcb->bits;
    a.qscale = scale * 1.4426950408889634f;
    for (int i = 0; i < 16; ++i) {
        a.kc[i] = (kcb->bits != 8 && i < kcb->levels) ? kcb->centroids[i] : 0.f;
        a.vc[i] = (vcb->bits != 8 && i < vcb->levels) ? vcb->centroids[i] : 0.f;
    }
    for (int i = 0; i < 4; ++i) a.signs[i] = signs.w[i];
    a.drop = drop_copies();
    a.table = table;
    a.max_pages = max_pages;
    a.page = page;
    const int64_t rows = (int64_t)M * a.G;
    a.row_tiles = (int)((rows + kPfRows - 1) / kPfRows);
    const int64_t grid = (int64_t)B * Hkv * a.row_tiles;
    if (grid > 0x7FFFFFFF || (int64_t)B * M * Hq > ((int64_t)1 << 40)) return TQ_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (kcb->bits) {
        case 2: return launch_prefill_v<2>(a, vcb->bits, (int)grid, st);
        case 3: return launch_prefill_v<3>(a, vcb->bits, (int)grid, st);
        case 4: return launch_prefill_v<4>(a, vcb->bits, (int)grid, st);
        case 8: return vcb->bits == 8 ? TQ_ERR_UNSUPPORTED : launch_prefill_v<8>(a, vcb->bits, (int)grid, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace

extern "C" int tq_attn_prefill(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                               const uint8_t *v_blocks, const tq_codebook *vcb, const int32_t *seq_lens, int B,
                               int M, int Hq, int Hkv, int T_cap, int T, float scale, tq_signs signs, float *out,
                               void *stream) {
    return prefill_call(q, q_dtype, k_blocks, kcb, v_blocks, vcb, seq_lens, B, M, Hq, Hkv, T_cap, T, scale, signs,
                        out, nullptr, 0, 0, stream);
}

extern "C" int tq_attn_prefill_paged(const void *q, int q_dtype, const uint8_t *k_pool, const tq_codebook *kcb,
                                     const uint8_t *v_pool, const tq_codebook *vcb, const int32_t *block_table,
                                     int max_pages, int page_tokens, const int32_t *seq_lens, int B, int M, int Hq,
                                     int Hkv, int T, float scale, tq_signs signs, float *out, void *stream) {
    if (!block_table || max_pages <= 0 || page_tokens <= 0 || (page_tokens & 7)) return TQ_ERR_ARG;
    if ((int64_t)max_pages * page_tokens < T || (int64_t)max_pages * page_tokens > 0x7FFFFFFF) return TQ_ERR_ARG;
    // the kernel's key range never passes T: T_cap = T rounded up to 8 stands for the table's span
    const int T_cap = (T + 7) & ~7;
    return prefill_call(q, q_dtype, k_pool, kcb, v_pool, vcb, seq_lens, B, M, Hq, Hkv, T_cap, T, scale, signs, out,
                        block_table, max_pages, page_tokens, stream);
}
