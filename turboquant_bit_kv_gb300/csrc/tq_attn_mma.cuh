// Tensor-core decode attention over packed caches (sm_103a).
//
// Same computation as attn_split_kernel ("TurboQuant KV Cache Compression —
// Spec", Optimization: Fused dequant-dot; "RotorQuant KV Cache Compression",
// The QJL Estimator Formula and Fused Kernel Logic): rotated query, scores
// against dequantised rotated keys (plus the QJL sign term), online softmax,
// values accumulated in the rotated domain (raw values as they are), one
// inverse rotation per output (in the combine kernel).
//
// Once a tile of codes is looked up, every product is a dense contraction,
// run as mma.sync m16n8k16 (fp16 operands, float32 accumulate; the G <= 8
// query heads sharing a KV head fill N = 8, zero-padded; the query and P are
// split hi + lo: with G <= 4 the n-tile's 8 columns are 4 heads x (hi, lo),
// with G = 5..8 they are the 8 heads and the hi and lo parts go through
// separate products into the same accumulators -- Khi Qhi, Khi Qlo, Klo Qhi
// for the scores, V Phi and V Plo for the values):
//   scores  S[16 tokens x 8 heads]  = Khat[16 x 128] * Qrot^T[128 x 8]
//   QJL     S2[16 tokens x 8 heads] = Sgn[16 x 128] * (S q)^T[128 x 8]
//   values  O[128 dims x 8 heads]  += Vhat^T[128 x 16] * P[16 tokens x 8]
//   * Keys: a thread reads the code slice of its dims 32t..32t+31 per token
//     (the MMA's k-columns permuted to match) and turns each pair of codes
//     into the (hi, lo) pair of half2 fragment registers: two 4-byte lookups
//     in a table with a copy per lane and the hi and lo halves in separate
//     128-byte halves of each 256-byte row (so each lands straight in its
//     MMA operand register), or, where the rows share space with the 2-bit
//     value pairs or only 128-byte rows fit, one 8-byte lookup in a table
//     replicated for 16 lanes; one byte permute yields the lookup offset
//     (entry * 256 + lane offset).  The pair's table index is the code byte
//     (4-bit), the nibble (2-bit), or the low nibble of the 2-bit plane plus
//     the two high-plane bits (3-bit).
//   * 2-bit values: a thread owns dims 16g..16g+15 (the MMA's m-rows
//     permuted so that the two rows of an m-tile are dims d and d + 1), one
//     32-bit code word per token; the code words of two tokens are
//     interleaved by nibbles so that one byte holds the codes of both dims
//     of both tokens, and one 8-byte lookup in a 256-entry pair table (the
//     upper halves of the key table's rows) yields both fragment registers.
//   * 3- and 4-bit values: each lane dequantises half of one token's row
//     into an fp16 tile in shared memory (pairs of dims through the same
//     kind of table as keys), and the fragments are read back transposed
//     with ldmatrix.trans; raw fp16 values are staged straight into that
//     layout.
//   * QJL: sign bits become +-1 fragments through a 16-entry nibble table;
//     S q is computed once per (sequence, KV head) and query head.
//   * Softmax runs on the score accumulators per 32-token chunk; the value
//     norm is folded into P, which is transposed into the PV operand layout
//     with movmatrix.
//
// Work partition: the B * Hkv * ceil(T / 32) chunks, ordered by (sequence,
// KV head, position), are cut into W equal contiguous ranges, one per warp
// of the grid (all CTAs resident), so every warp does the same work (to one
// chunk) and there is no wave tail.  Each warp works on its own: a two- or
// three-stage ring of bulk copies on its own mbarriers, its own softmax
// state, and one partial per query head for every (sequence, KV head)
// segment its range touches, written to slot (warp - first warp of the
// segment).  The query fragments come from attn_prep_mma_kernel (rotated,
// scaled, split hi | lo once per segment); attn_combine_mma_kernel merges
// each segment's slots and applies the inverse rotation.  The three kernels
// are chained as programmatic dependents, so each one's launch and prologue
// (the first copies, the lookup tables) overlap the previous one.
//
// This header holds the kernel template; tq_attn_mma_k{2,3,4}.cu instantiate
// it per key width and tq_attn_mma.cu plans and dispatches.

#pragma once

#include <cmath>

#include "tq_attn.cuh"
#include "tq_attn_mma.h"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kVtPitch = 272;                  // fp16 value tile row: 256 B + 16 B pad (conflict-free)
constexpr unsigned kFull = 0xffffffffu;

constexpr int align16(int x) { return (x + 15) & ~15; }

// NT: 1 serves up to 4 query heads per KV head with n-tiles of 8 columns =
// 4 heads x (hi, lo) fp16 parts (query, sketched query and P are split
// x = hi + lo so their products keep float32 precision); NT = 2 serves 5 to 8
// heads with one n-tile of the 8 heads, the hi and lo parts as two operands
// (kH8).
template <int KB, int VB, bool QJL, int NT, bool WIDE = true>
struct Cfg {
    // 2-bit values with one n-tile fit in 128 registers: one CTA of 16 warps
    // per SM (WIDE; below 32 chunks per warp at that width, 12 warps -- fewer,
    // longer ranges -- measured 4% faster); two n-tiles of packed values fit in
    // 168 (12 warps; measured 5% faster than 8 at 7 query heads per KV head);
    // the rest, and every turboq8 configuration (130-byte blocks: larger
    // stages), run 8 warps.
    static constexpr int kW = (KB == 8 || VB == 8) ? 8
                              : (VB == 2 && NT == 1) ? (WIDE ? 16 : 12) : (NT == 2 && VB != 16) ? 12 : 8;
    static constexpr int kThreads = kW * 32;
    static constexpr bool kH8 = NT == 2;   // one n-tile of 8 heads; hi / lo parts as separate products
    static constexpr int kNO = kH8 ? 1 : NT;   // accumulator n-tiles
    // turboq8 blocks: [fp16 scale][128 code bytes]
    static constexpr int kKBytes = KB == 8 ? 130 : 2 + 16 * KB;
    static constexpr bool kRawV = VB == 16;
    static constexpr bool kRegV = VB == 2;                 // value fragments straight from a pair table
    static constexpr int kVBytes = kRawV ? 256 : VB == 8 ? 130 : 2 + 16 * VB;
    static constexpr int kKStage = align16(kMmaChunk * kKBytes);
    static constexpr int kVStage = kRawV ? kMmaChunk * kVtPitch : align16(kMmaChunk * kVBytes);
    static constexpr int kSStage = QJL ? kMmaChunk * 16 : 0;      // sign bits
    static constexpr int kRStage = QJL ? kMmaChunk * 2 : 0;       // fp16 residual norms
    // +16: word reads past a 2-byte aligned slice stay inside the warp's stage
    static constexpr int kWarpStage = kKStage + kVStage + kSStage + kRStage + 16;
    static constexpr int kVtile = (kRegV || kRawV) ? 0 : 16 * kVtPitch;   // per-warp dequantised tile
    // turboq8 codes need no table: the level 2i - 255 is an integer, exact in fp16 (the 1 / 255
    // goes into the block's norm factor)
    static constexpr int kKLutEntries = KB == 8 ? 0 : KB == 4 ? 256 : KB == 3 ? 64 : 16;
    static constexpr int kVLutEntries = VB == 4 ? 256 : VB == 3 ? 64 : 0;
    // value-pair table rows: 256 bytes for 3-bit values (one byte permute yields entry * 256 + lane
    // offset), 128 for the 256 entries of 4-bit values (offset by a multiply)
    static constexpr int kVRow = VB == 3 ? 256 : 128;
    static constexpr int kVLutBytes = kVLutEntries * kVRow + (QJL ? 16 * 256 : 0);
    static constexpr int kVtileBytes = kW * kVtile + kW * 3 * 8;
    // key-table rows of 256 bytes (offset from one byte permute) where they fit, else 128
    static constexpr int kKRow =
        (kRegV ? 256 : kKLutEntries) * 256 + kVLutBytes + kVtileBytes + kW * 2 * kWarpStage <= 227 * 1024 ? 256
                                                                                                    : 128;
    // 2-bit values: 256 rows, key entries in the lower and value-pair entries in the upper half
    static constexpr int kKRows = kRegV ? 256 : kKLutEntries;
    static constexpr int kSmemKLut = 0;
    static constexpr int kSmemVLut = kSmemKLut + kKRows * kKRow;
    static constexpr int kSmemSLut = kSmemVLut + kVLutEntries * kVRow;
    static constexpr int kSmemVt = kSmemSLut + (QJL ? 16 * 256 : 0);
    static constexpr int kSmemBars = kSmemVt + kW * kVtile;
    static constexpr int kFixed = kSmemBars + kW * 3 * 8;                 // up to 3 mbarriers per warp
    // pipeline depth: three stages per warp where they fit, else two
    static constexpr int kStages = kFixed + kW * 3 * kWarpStage <= 227 * 1024 ? 3 : 2;
    static constexpr int kSmemStages = kFixed;
    // bytes a full chunk brings in (bulk copies, one mbarrier phase)
    static constexpr int kChunkBytes = kMmaChunk * kKBytes + kMmaChunk * (kRawV ? 256 : kVBytes) +
                                       (QJL ? kMmaChunk * 16 + kMmaChunk * 2 : 0);
    static constexpr int kSmemTotal = kSmemStages + kW * kStages * kWarpStage;
    static constexpr int kMinBlocks = (kW == 8 && NT == 1 && kSmemTotal <= 113 * 1024) ? 2 : 1;
    static_assert(kSmemTotal <= 227 * 1024, "shared memory");
    static_assert(!kRegV || kKRow == 256, "2-bit value pairs live in the upper half of 256-byte rows");
    // key rows of 256 bytes not shared with value pairs hold the hi and lo halves in separate
    // 128-byte halves, one word per lane: two 4-byte loads put them straight into the MMA's
    // operand registers (an 8-byte (hi, lo) load would need register moves to regroup them)
    static constexpr bool kKSplit = !kRegV && kKRow == 256;
    static_assert(kW * kMinBlocks <= kMmaMaxWarpsPerSm, "warps per SM");
};


__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Dynamic shared memory of the kernel.  Loads are plain C++ dereferences
// (shared-window address minus the base), which the compiler can schedule
// and fold into immediate offsets; the bounded mbarrier waits, __syncwarp
// and the asm stores (memory clobbers) still order them.
extern __shared__ __align__(16) uint8_t tq_attn_dsmem[];

template <class T>
__device__ __forceinline__ T lds(uint32_t addr) {
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(tq_attn_dsmem);
    return *reinterpret_cast<const T *>(tq_attn_dsmem + (addr - base));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) { return lds<uint32_t>(addr); }

__device__ __forceinline__ uint2 lds64(uint32_t addr) { return lds<uint2>(addr); }

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) { return lds<unsigned short>(addr); }

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
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
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
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

// ---- bulk (TMA engine) copies completing on an mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Wait for the phase with parity `parity` to complete (bounded; false when
// it gave up).  After a wait of this lane gave up (ok false) later waits make
// a single attempt, so the loop runs on to its end without stalling.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, bool ok) {
    return mbar_wait_bounded(bar, parity, ok ? 100000000ull : 0ull);
}

// Codes of the two dims of a table entry.  4-bit: entry = byte (low nibble
// first dim); 2-bit: entry = nibble; 3-bit: entry = the pair's 2-bit-plane
// nibble | high-plane bits << 4.
template <int BITS>
__device__ __forceinline__ void pair_codes(int e, int &c0, int &c1) {
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

// Lane-replicated half2 table of a codebook in rows of ROW bytes: word
// e * ROW / 4 + l = (c[c0(e)], c[c1(e)]) for every lane l; stores rotated by
// e so a warp's stores are conflict-free.
template <int BITS, int ROW>
__device__ __forceinline__ void build_pair_lut(uint32_t *lut, const float *cb, int tid, int nthreads) {
    constexpr int E = BITS == 4 ? 256 : BITS == 3 ? 64 : 16;
    for (int e = tid; e < E; e += nthreads) {
        int c0, c1;
        pair_codes<BITS>(e, c0, c1);
        const uint32_t val = pack_half2(cb[c0], cb[c1]);
#pragma unroll 8
        for (int j = 0; j < 32; ++j) lut[e * (ROW / 4) + ((j + e) & 31)] = val;
    }
}

// Split table of a codebook for the keys: entry e at byte e * row + l * 8 for
// l = 0..15 (lanes l and l + 16 share a copy; an 8-byte load serves half a
// warp per pass, so this is conflict-free; with 256-byte rows the upper half
// is unused and one byte permute yields the offset e * 256 + l * 8) holds
// (hi, lo) half2 words with hi = fp16(c), lo = fp16(c - hi): hi + lo
// carries c to about 2^-22.
template <int BITS>
__device__ __forceinline__ void build_split_lut(uint2 *lut, const float *cb, int tid, int nthreads, int row_words) {
    constexpr int E = BITS == 4 ? 256 : BITS == 3 ? 64 : 16;
    for (int q = tid; q < E * 16; q += nthreads) {
        const int e = q >> 4, l = q & 15;
        int c0, c1;
        pair_codes<BITS>(e, c0, c1);
        const __half h0 = __float2half_rn(cb[c0]), h1 = __float2half_rn(cb[c1]);
        const uint32_t hi = pack_half2(__half2float(h0), __half2float(h1));
        const uint32_t lo = pack_half2(cb[c0] - __half2float(h0), cb[c1] - __half2float(h1));
        lut[e * row_words + l] = make_uint2(hi, lo);
    }
}

// The same table with 256-byte rows split by half: entry e holds hi at byte
// e * 256 + 4 l and lo at e * 256 + 128 + 4 l for every lane l (conflict-free
// 4-byte loads, one word per lane).
template <int BITS>
__device__ __forceinline__ void build_split_lut_hl(uint32_t *lut, const float *cb, int tid, int nthreads) {
    constexpr int E = BITS == 4 ? 256 : BITS == 3 ? 64 : 16;
    for (int q = tid; q < E * 32; q += nthreads) {
        const int e = q >> 5, l = q & 31;
        int c0, c1;
        pair_codes<BITS>(e, c0, c1);
        const __half h0 = __float2half_rn(cb[c0]), h1 = __float2half_rn(cb[c1]);
        lut[e * 64 + l] = pack_half2(__half2float(h0), __half2float(h1));
        lut[e * 64 + 32 + l] = pack_half2(cb[c0] - __half2float(h0), cb[c1] - __half2float(h1));
    }
}

// (hi, lo) fp16 splits of two floats, packed as the half2 words hi = (hi0,
// hi1) and lo = (lo0, lo1): x = hi + lo to about 2^-22.
__device__ __forceinline__ void split2_half2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// (hi, lo) fp16 split of x packed as one half2: x = hi + lo to about 2^-22.
__device__ __forceinline__ uint32_t split_half2(float x) {
    const __half h = __float2half_rn(x);
    return pack_half2(__half2float(h), x - __half2float(h));
}

// 3-bit pair indices of 8 pairs from one 2-bit-plane word L (dims 16h..16h+15
// of the slice, pairs 8h..8h+7) and the 16 high-plane bits Hh of the same
// dims: even pairs (8h + 2i) in byte i of `ev`, odd pairs in byte i of `od`.
__device__ __forceinline__ void pair_index3(uint32_t L, uint32_t Hh, uint32_t &ev, uint32_t &od) {
    const uint32_t v = prmt(Hh, 0, 0x1100u);   // bytes [Hh1, Hh1, Hh0, Hh0]
    ev = (L & 0x0F0F0F0Fu) | ((v << 4) & 0x00300030u) | (v & 0x30003000u);
    od = ((L >> 4) & 0x0F0F0F0Fu) | ((v << 2) & 0x00300030u) | ((v >> 2) & 0x30003000u);
}

// half2(2 i - 255) of the two turboq8 codes i that selector `sel` (0x4140:
// bytes 0, 1 of w; 0x4342: bytes 2, 3) picks: one byte permute makes the fp16
// bit patterns of 1024 + i (exponent byte 0x64 over the code byte), then
// (1024 + i) - 1024 and 2 i - 255, each exact (2303 itself has no fp16).
__device__ __forceinline__ uint32_t q8_levels(uint32_t w, uint32_t sel) {
    const uint32_t p = prmt(w, 0x64u, sel);
    const __half2 i2 = __hsub2(*reinterpret_cast<const __half2 *>(&p), __floats2half2_rn(1024.f, 1024.f));
    const __half2 l2 = __hfma2(i2, __floats2half2_rn(2.f, 2.f), __floats2half2_rn(-255.f, -255.f));
    return *reinterpret_cast<const uint32_t *>(&l2);
}

// Half2 key fragments for k-step ks of one token row: pairs 2ks (dims
// 32t + 4ks + {0, 1}) and 2ks + 1 (dims 32t + 4ks + {2, 3}) of the slice.
template <int KB>
struct KeySlice {
    // 8-bit: the 32 code bytes; 4-bit: the 16 code bytes; 2/3-bit: even / odd pair indices of
    // halves 0, 1
    uint32_t w[KB == 8 ? 8 : 4];

    __device__ __forceinline__ void load(uint32_t row_s, int t) {
        if constexpr (KB == 8) {
            lds_words_a2<8>(row_s + 2 + 32 * t, w);
        } else if constexpr (KB == 4) {
            lds_words_a2<4>(row_s + 2 + 16 * t, w);
        } else if constexpr (KB == 2) {
            uint32_t c[2];
            lds_words_a2<2>(row_s + 2 + 8 * t, c);
            w[0] = c[0] & 0x0F0F0F0Fu;
            w[1] = (c[0] >> 4) & 0x0F0F0F0Fu;
            w[2] = c[1] & 0x0F0F0F0Fu;
            w[3] = (c[1] >> 4) & 0x0F0F0F0Fu;
        } else {
            uint32_t c[2], hb[1];
            lds_words_a2<2>(row_s + 2 + 8 * t, c);
            lds_words_a2<1>(row_s + 34 + 4 * t, hb);
            pair_index3(c[0], hb[0], w[0], w[1]);
            pair_index3(c[1], hb[0] >> 16, w[2], w[3]);
        }
    }
    // turboq8: the fragment words of pair 2ks (x) and pair 2ks + 1 (y) themselves, half2(2 i - 255)
    // per code i (see q8_levels)
    __device__ __forceinline__ void levels(int ks, uint32_t &x, uint32_t &y) const {
        x = q8_levels(w[ks], 0x4140u);
        y = q8_levels(w[ks], 0x4342u);
    }
    // key-table byte offsets of pair 2ks (x) and pair 2ks + 1 (y) for rows of
    // ROW bytes: with 256-byte rows one byte permute puts the pair index in
    // byte 1 and the lane offset lo8 in byte 0
    template <int ROW>
    __device__ __forceinline__ void pick(int ks, uint32_t lo8, uint32_t &x, uint32_t &y) const {
        uint32_t wx, wy, bx, by;
        if constexpr (KB == 4) {
            wx = wy = w[ks >> 1];
            bx = 2 * (ks & 1);
            by = bx + 1;
        } else {
            const int h = ks >> 2;
            wx = w[2 * h];
            wy = w[2 * h + 1];
            bx = by = ks & 3;
        }
        if constexpr (ROW == 256) {
            x = prmt(wx, lo8, 0x6504u + bx * 16);
            y = prmt(wy, lo8, 0x6504u + by * 16);
        } else {
            x = prmt(wx, 0, 0x4440u + bx) * ROW + lo8;
            y = prmt(wy, 0, 0x4440u + by) * ROW + lo8;
        }
    }
};

// One lane dequantises 64 dims (half `hf`) of one token's packed value block
// into an fp16 row of the value tile (pairs through the pair table).
template <int VB>
__device__ __forceinline__ void dequant_value_half(uint32_t blk_s, int hf, uint32_t lut_s, uint32_t row_s) {
    if constexpr (VB == 8) {
        // turboq8: half2(2 i - 255) per code pair (q8_levels), no table
        uint32_t c[16];
        lds_words_a2<16>(blk_s + 2 + 64 * hf, c);
        uint32_t h[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            h[2 * i] = q8_levels(c[i], 0x4140u);
            h[2 * i + 1] = q8_levels(c[i], 0x4342u);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) sts128(row_s + 128 * hf + 16 * q, h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    } else if constexpr (VB == 4) {
        uint32_t c[8];
        lds_words_a2<8>(blk_s + 2 + 32 * hf, c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = lds32(lut_s + prmt(c[2 * q + (j >> 2)], 0, 0x4440u + (j & 3)) * 128u);
            sts128(row_s + 128 * hf + 32 * q, h[0], h[1], h[2], h[3]);
            sts128(row_s + 128 * hf + 32 * q + 16, h[4], h[5], h[6], h[7]);
        }
    } else {  // VB == 3: 256-byte rows, one byte permute yields entry * 256 + the lane offset
        uint32_t c[4], hb[2];
        lds_words_a2<4>(blk_s + 2 + 16 * hf, c);
        lds_words_a2<2>(blk_s + 34 + 8 * hf, hb);
        const uint32_t lo8 = (threadIdx.x & 31) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t ev, od;
            pair_index3(c[q], hb[q >> 1] >> (16 * (q & 1)), ev, od);
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[2 * i] = lds32(lut_s + prmt(ev, lo8, 0x6504u + 16u * i));
                h[2 * i + 1] = lds32(lut_s + prmt(od, lo8, 0x6504u + 16u * i));
            }
            sts128(row_s + 128 * hf + 32 * q, h[0], h[1], h[2], h[3]);
            sts128(row_s + 128 * hf + 32 * q + 16, h[4], h[5], h[6], h[7]);
        }
    }
}

// Dim of accumulator row `r` (0: fragment row g, 1: row g + 8) of m-tile m.
template <bool REGV>
__device__ __forceinline__ int acc_dim(int m, int r, int g) {
    return REGV ? 16 * g + 2 * m + r : 16 * m + g + 8 * r;
}

// Pair table of a 2-bit value codebook: entry e = [code of token A, dim d |
// A, d + 1 | token B, d | B, d + 1] (2 bits each, lowest first) holds the
// fragment words half2(c[A, d], c[B, d]) and half2(c[A, d + 1], c[B, d + 1]);
// stored at byte e * 256 + 128 + l * 8 for l = 0..15 (the upper half of the
// key table's 256-byte rows).
__device__ __forceinline__ void build_value_pair_lut(uint8_t *rows, const float *cb, int tid, int nthreads) {
    for (int q = tid; q < 256 * 16; q += nthreads) {
        const int e = q >> 4, l = q & 15;
        const uint32_t x = pack_half2(cb[e & 3], cb[(e >> 4) & 3]);
        const uint32_t y = pack_half2(cb[(e >> 2) & 3], cb[(e >> 6) & 3]);
        *reinterpret_cast<uint2 *>(rows + e * 256 + 128 + l * 8) = make_uint2(x, y);
    }
}


// Paged cache: the chunk of segment j starting at token t0 lies in one page (pages are multiples of
// 32 tokens); the slot of token t0 in the pools, less t0 (so that row0 + t0 is that slot).
__device__ __forceinline__ int64_t paged_row0(const AttnArgs &a, int j, int t0) {
    const int pg = t0 / a.page;
    return ((int64_t)a.table[(int64_t)(j / a.Hkv) * a.max_pages + pg] * a.Hkv + j % a.Hkv) * a.page +
           (t0 - pg * a.page) - t0;
}

template <int KB, int VB, bool QJL, int NT, bool WIDE, bool PAGED = false>
__global__ void __launch_bounds__(Cfg<KB, VB, QJL, NT, WIDE>::kThreads, Cfg<KB, VB, QJL, NT, WIDE>::kMinBlocks)
    attn_mma_kernel(const __grid_constant__ AttnArgs a, const MmaPlan plan) {
    using C = Cfg<KB, VB, QJL, NT, WIDE>;
    constexpr int kS = C::kStages;
    uint8_t *smem = tq_attn_dsmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const uint32_t smem_s = (uint32_t)__cvta_generic_to_shared(smem);
    const uint32_t stage_s = smem_s + C::kSmemStages + warp * kS * C::kWarpStage;
    const uint32_t bar_s = smem_s + C::kSmemBars + warp * 3 * 8;
    if (lane == 0) {
        // (test hook: a second arrival that never comes keeps every phase from completing, so the
        // first wait runs out while the copies still land)
#pragma unroll
        for (int s = 0; s < kS; ++s) mbar_init(bar_s + 8 * s, a.drop ? 2 : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // the combine kernel may take its (idle) place on the SMs now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");

    // this warp's chunks [lo, hi) in (segment, position) order: segments j0 .. j1, from chunk cb0
    // of segment j0 to chunk ce1 (exclusive) of segment j1
    const int gw = warp * plan.P + blockIdx.x;
    const bool active = gw < plan.W;
    int j0 = 0, j1 = -1, cb0 = 0, ce1 = 0;
    if (active) {
        const int64_t lo = (int64_t)gw * plan.Ctot / plan.W, hi = ((int64_t)gw + 1) * plan.Ctot / plan.W;
        j0 = (int)(lo / plan.C);
        j1 = (int)((hi - 1) / plan.C);
        cb0 = (int)(lo - (int64_t)j0 * plan.C);
        ce1 = (int)(hi - (int64_t)j1 * plan.C);
    }
    // live tokens of segment j: its sequence's length clamped to [0, T]
    auto seg_len = [&](int j) {
        int L = a.T;
        if (a.seq_lens) {
            const int sl = a.seq_lens[j / a.Hkv];
            L = sl < 0 ? 0 : (sl > a.T ? a.T : sl);
        }
        return L;
    };

    uint32_t phase = 0;        // bit s: parity of the next completion of barrier s
    uint32_t bulk_mask = 0;    // bit s: stage s was filled by bulk copies
    bool copies_ok = true;

    // stage of chunk ci of segment j: K blocks | V blocks (raw: 272-byte rows) | sign rows | residual norms
    auto issue = [&](int buf, int j, int ci, int L) {
        const int t0 = ci * kMmaChunk;
        const int n = min(kMmaChunk, L - t0);
        const int64_t row0 = PAGED ? paged_row0(a, j, t0) : (int64_t)j * a.T_cap;
        const uint8_t *kbase = a.k + row0 * C::kKBytes;
        const uint8_t *vbase = a.v + row0 * C::kVBytes;
        const uint8_t *sgbase = QJL ? a.qjl_bits + row0 * 16 : nullptr;
        const uint8_t *rnbase = QJL ? reinterpret_cast<const uint8_t *>(a.rn + row0) : nullptr;
        const uint32_t dk = stage_s + buf * C::kWarpStage, dv = dk + C::kKStage;
        const uint8_t *sk = kbase + (int64_t)t0 * C::kKBytes, *sv = vbase + (int64_t)t0 * C::kVBytes;
        if (n == kMmaChunk) {
            // full chunk: contiguous 16-byte aligned ranges, bulk copies on barrier `buf`
            const uint32_t bar = bar_s + 8 * buf;
            if (lane == 0) mbar_expect_tx(bar, C::kChunkBytes);
            __syncwarp();
            if (lane == 0) {
                bulk_g2s(dk, sk, kMmaChunk * C::kKBytes, bar);
                if constexpr (!C::kRawV) bulk_g2s(dv, sv, kMmaChunk * C::kVBytes, bar);
                if constexpr (QJL) {
                    const uint32_t ds = dv + C::kVStage;
                    bulk_g2s(ds, sgbase + (int64_t)t0 * 16, kMmaChunk * 16, bar);
                    bulk_g2s(ds + C::kSStage, rnbase + (int64_t)t0 * 2, kMmaChunk * 2, bar);
                }
            }
            if constexpr (C::kRawV) bulk_g2s(dv + lane * kVtPitch, sv + lane * 256, 256, bar);
            bulk_mask |= 1u << buf;
            return;
        }
        // partial chunk (the end of a sequence): 16-byte cp.async pieces, zero-filled past the tokens
        bulk_mask &= ~(1u << buf);
        // (the address given with a zero-byte copy: the segment's start, or under paging the chunk's own)
        const uint8_t *kz = PAGED ? sk : kbase, *vz = PAGED ? sv : vbase;
        const int nk = (n * C::kKBytes + 15) >> 4;
        for (int q = lane; q < C::kKStage / 16; q += 32) cp16_zfill(dk + 16 * q, q < nk ? sk + 16 * q : kz, q < nk);
        if constexpr (C::kRawV) {
            for (int q = lane; q < kMmaChunk * 16; q += 32) {
                const int r = q >> 4, col = q & 15;
                cp16_zfill(dv + r * kVtPitch + 16 * col, r < n ? sv + r * 256 + 16 * col : vz, r < n);
            }
        } else {
            const int nvb = (n * C::kVBytes + 15) >> 4;
            for (int q = lane; q < C::kVStage / 16; q += 32)
                cp16_zfill(dv + 16 * q, q < nvb ? sv + 16 * q : vz, q < nvb);
        }
        if constexpr (QJL) {
            const uint32_t ds = dv + C::kVStage, dr = ds + C::kSStage;
            const uint8_t *ss = sgbase + (int64_t)t0 * 16, *sr = rnbase + (int64_t)t0 * 2;
            cp16_zfill(ds + 16 * lane, lane < n ? ss + 16 * lane : sgbase, lane < n);
            const int nr = (2 * n + 15) >> 4;
            if (lane < 4) cp16_zfill(dr + 16 * lane, lane < nr ? sr + 16 * lane : rnbase, lane < nr);
        }
        cp_async_commit();
    };

    // live chunks [cb, ce) of segment j within this warp's range
    auto seg_end = [&](int j, int L) { return min(j == j1 ? ce1 : plan.C, (L + kMmaChunk - 1) / kMmaChunk); };
    // issue cursor: chunk ici of segment ij, always at a live chunk (ici < iend) unless past the range
    int ij = j0, ici = cb0, iL = 0, iend = 0;
    if (active) {
        iL = seg_len(j0);
        iend = seg_end(j0, iL);
    }
    auto settle = [&]() {
        while (ici >= iend && ij < j1) {
            ++ij;
            ici = 0;
            iL = seg_len(ij);
            iend = seg_end(ij, iL);
        }
    };
    int ist = 0;   // stage of the next issue
    auto issue_next = [&]() {
        if (ici < iend) {
            issue(ist, ij, ici, iL);
            ++ici;
            settle();
        }
        ist = ist + 1 == kS ? 0 : ist + 1;
    };
    // the first chunks are on their way while the tables are built
    if (active) {
        settle();
#pragma unroll
        for (int s = 0; s + 1 < kS; ++s) issue_next();
    }

    if constexpr (KB == 8) {
        // (turboq8 keys: no table)
    } else if constexpr (C::kKSplit) {
        build_split_lut_hl<KB>(reinterpret_cast<uint32_t *>(smem + C::kSmemKLut), a.kc, tid, C::kThreads);
    } else {
        build_split_lut<KB>(reinterpret_cast<uint2 *>(smem + C::kSmemKLut), a.kc, tid, C::kThreads, C::kKRow / 8);
    }
    if constexpr (VB == 3 || VB == 4)
        build_pair_lut<VB, C::kVRow>(reinterpret_cast<uint32_t *>(smem + C::kSmemVLut), a.vc, tid, C::kThreads);
    if constexpr (QJL) {
        // sign table: entry e (4 sign bits) = (half2(s0, s1), half2(s2, s3)), s = bit ? +1 : -1,
        // at byte e * 256 + lane * 8
        uint32_t *sl = reinterpret_cast<uint32_t *>(smem + C::kSmemSLut);
        for (int q = tid; q < 16 * 32; q += C::kThreads) {
            const int e = q >> 5, l = q & 31;
            const uint32_t p0 = (e & 1) ? 0x3C00u : 0xBC00u, p1 = (e & 2) ? 0x3C00u : 0xBC00u;
            const uint32_t p2 = (e & 4) ? 0x3C00u : 0xBC00u, p3 = (e & 8) ? 0x3C00u : 0xBC00u;
            sl[e * 64 + 2 * l] = p0 | (p1 << 16);
            sl[e * 64 + 2 * l + 1] = p2 | (p3 << 16);
        }
    }
    if constexpr (C::kRegV) build_value_pair_lut(smem + C::kSmemKLut, a.vc, tid, C::kThreads);
    const uint32_t klut_s = smem_s + C::kSmemKLut, klane = C::kKSplit ? lane * 4 : (lane & 15) * 8;
    const uint32_t vlane = 128 + (lane & 15) * 8;
    const uint32_t vlut_s = smem_s + C::kSmemVLut + (C::kVRow == 256 ? 0 : lane * 4);
    const uint32_t slut_s = smem_s + C::kSmemSLut + lane * 8;
    const uint32_t vt_s = smem_s + C::kSmemVt + warp * C::kVtile;
    __syncthreads();
    // the query fragments come from the prep kernel this one depends on
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int cst = 0;   // stage of the next chunk to compute
    for (int j = j0; j <= j1; ++j) {
        const int L = seg_len(j);
        const int cb = j == j0 ? cb0 : 0, ce = seg_end(j, L);
        const int b = j / a.Hkv, kvh = j % a.Hkv;
        // B fragments (k-step ks) of the rotated, scaled query and of S q: n-tile nt of 4 heads x
        // (hi, lo), or (kH8) nt = 0: the 8 heads' hi parts, nt = 1: their lo parts
        uint32_t qb[NT][8][2];
        uint32_t sb[QJL ? 8 : 1][2];
        {
            const uint4 *fr = reinterpret_cast<const uint4 *>(a.ws + plan.frag_off + (int64_t)j * kFragWords) + lane * 4;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = fr[nt * 128 + q];
                    qb[nt][2 * q][0] = w.x;
                    qb[nt][2 * q][1] = w.y;
                    qb[nt][2 * q + 1][0] = w.z;
                    qb[nt][2 * q + 1][1] = w.w;
                }
            if constexpr (QJL) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = fr[2 * 128 + q];
                    sb[2 * q][0] = w.x;
                    sb[2 * q][1] = w.y;
                    sb[2 * q + 1][0] = w.z;
                    sb[2 * q + 1][1] = w.w;
                }
            }
        }

        // accumulators: n-tile nt, m-tile m; columns (2t, 2t+1) = head 4 nt + t, (hi, lo) parts, or
        // (kH8) heads 2t, 2t + 1.  Softmax slot i of this thread: head 4 i + t, or (kH8) 2t + i.
        float o[C::kNO][8][4];
#pragma unroll
        for (int nt = 0; nt < C::kNO; ++nt)
#pragma unroll
            for (int m = 0; m < 8; ++m) o[nt][m][0] = o[nt][m][1] = o[nt][m][2] = o[nt][m][3] = 0.f;
        float mrun[NT], lrun[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mrun[nt] = -INFINITY;
            lrun[nt] = 0.f;
        }

        for (int ci = cb; ci < ce; ++ci) {
            issue_next();
            if (bulk_mask & (1u << cst)) {
                copies_ok &= mbar_wait(bar_s + 8 * cst, (phase >> cst) & 1u, copies_ok);
                phase ^= 1u << cst;
            } else {
                cp_async_wait<0>();
            }
            __syncwarp();
            const int nvalid = min(kMmaChunk, L - ci * kMmaChunk);
            const uint32_t ks_s = stage_s + cst * C::kWarpStage, vs_s = ks_s + C::kKStage;
            const uint32_t sg_s = vs_s + C::kVStage, rn_s = sg_s + C::kSStage;

            // ---- scores of 2 tiles of 16 tokens (rows g, g + 8): (Khi + Klo) x (Qhi | Qlo)
            KeySlice<KB> ksl[2][2];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) ksl[mt][rh].load(ks_s + (16 * mt + g + 8 * rh) * C::kKBytes, t);
            float acc[C::kNO][2][4];             // [n-tile][m-tile][fragment]
#pragma unroll
            for (int nt = 0; nt < C::kNO; ++nt)
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t x0, y0, x1, y1;
                    if constexpr (KB == 8) {
                        // turboq8 keys: exact fp16 levels, no lo part
                        ksl[mt][0].levels(ks, x0, y0);
                        ksl[mt][1].levels(ks, x1, y1);
                        if constexpr (C::kH8) {
                            mma16816(acc[0][mt], x0, x1, y0, y1, qb[0][ks][0], qb[0][ks][1]);
                            mma16816(acc[0][mt], x0, x1, y0, y1, qb[1][ks][0], qb[1][ks][1]);
                        } else {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816(acc[nt][mt], x0, x1, y0, y1, qb[nt][ks][0], qb[nt][ks][1]);
                        }
                        continue;
                    }
                    ksl[mt][0].template pick<C::kKRow>(ks, klane, x0, y0);
                    ksl[mt][1].template pick<C::kKRow>(ks, klane, x1, y1);
                    if constexpr (C::kKSplit) {
                        const uint32_t h0 = lds32(klut_s + x0), h1 = lds32(klut_s + x1);
                        const uint32_t h2 = lds32(klut_s + y0), h3 = lds32(klut_s + y1);
                        const uint32_t l0 = lds32(klut_s + x0 + 128), l1 = lds32(klut_s + x1 + 128);
                        const uint32_t l2 = lds32(klut_s + y0 + 128), l3 = lds32(klut_s + y1 + 128);
                        if constexpr (C::kH8) {
                            mma16816(acc[0][mt], h0, h1, h2, h3, qb[0][ks][0], qb[0][ks][1]);
                            mma16816(acc[0][mt], h0, h1, h2, h3, qb[1][ks][0], qb[1][ks][1]);
                            mma16816(acc[0][mt], l0, l1, l2, l3, qb[0][ks][0], qb[0][ks][1]);
                        } else {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                mma16816(acc[nt][mt], h0, h1, h2, h3, qb[nt][ks][0], qb[nt][ks][1]);
                                mma16816(acc[nt][mt], l0, l1, l2, l3, qb[nt][ks][0], qb[nt][ks][1]);
                            }
                        }
                    } else if constexpr (C::kH8) {
                        const uint2 a0 = lds64(klut_s + x0), a2 = lds64(klut_s + y0);
                        const uint2 a1 = lds64(klut_s + x1), a3 = lds64(klut_s + y1);
                        mma16816(acc[0][mt], a0.x, a1.x, a2.x, a3.x, qb[0][ks][0], qb[0][ks][1]);
                        mma16816(acc[0][mt], a0.x, a1.x, a2.x, a3.x, qb[1][ks][0], qb[1][ks][1]);
                        mma16816(acc[0][mt], a0.y, a1.y, a2.y, a3.y, qb[0][ks][0], qb[0][ks][1]);
                    } else {
                        const uint2 a0 = lds64(klut_s + x0), a2 = lds64(klut_s + y0);
                        const uint2 a1 = lds64(klut_s + x1), a3 = lds64(klut_s + y1);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816(acc[nt][mt], a0.x, a1.x, a2.x, a3.x, qb[nt][ks][0], qb[nt][ks][1]);
                            mma16816(acc[nt][mt], a0.y, a1.y, a2.y, a3.y, qb[nt][ks][0], qb[nt][ks][1]);
                        }
                    }
                }
            }
            float acc2[QJL ? 2 : 1][4];
            if constexpr (QJL) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    acc2[mt][0] = acc2[mt][1] = acc2[mt][2] = acc2[mt][3] = 0.f;
                    const uint32_t wa = lds32(sg_s + (16 * mt + g) * 16 + 4 * t);
                    const uint32_t wb = lds32(sg_s + (16 * mt + g + 8) * 16 + 4 * t);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint2 fa = lds64(slut_s + ((wa >> (4 * ks)) & 15u) * 256u);
                        const uint2 fb = lds64(slut_s + ((wb >> (4 * ks)) & 15u) * 256u);
                        mma16816(acc2[mt], fa.x, fb.x, fa.y, fb.y, sb[ks][0], sb[ks][1]);
                    }
                }
            }
            // s[i][mt][r]: softmax slot i, token 16 mt + g + 8 r
            float s[NT][2][2];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int ta = 16 * mt + g, tb = ta + 8;
                // the block norms (turboq8: the scale over 255, the grid's step factor)
                constexpr float kf = KB == 8 ? 1.f / 255.f : 1.f;
                const float na = __half2float(__ushort_as_half((unsigned short)lds_u16(ks_s + ta * C::kKBytes))) * kf;
                const float nb = __half2float(__ushort_as_half((unsigned short)lds_u16(ks_s + tb * C::kKBytes))) * kf;
                float ra = 0.f, rb = 0.f;
                if constexpr (QJL) {
                    ra = __half2float(__ushort_as_half((unsigned short)lds_u16(rn_s + 2 * ta)));
                    rb = __half2float(__ushort_as_half((unsigned short)lds_u16(rn_s + 2 * tb)));
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float ea = (C::kH8 ? acc[0][mt][nt] : acc[nt][mt][0] + acc[nt][mt][1]) * na;
                    float eb = (C::kH8 ? acc[0][mt][2 + nt] : acc[nt][mt][2] + acc[nt][mt][3]) * nb;
                    if constexpr (QJL) {
                        ea = fmaf(acc2[mt][0] + acc2[mt][1], ra, ea);
                        eb = fmaf(acc2[mt][2] + acc2[mt][3], rb, eb);
                    }
                    s[nt][mt][0] = ta < nvalid ? ea : -INFINITY;
                    s[nt][mt][1] = tb < nvalid ? eb : -INFINITY;
                }
            }
            // ---- online softmax per head (max over the rows g of the warp)
            bool moved = false;
            float corr[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float mx = fmaxf(fmaxf(s[nt][0][0], s[nt][0][1]), fmaxf(s[nt][1][0], s[nt][1][1]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
                const float mn = fmaxf(mrun[nt], mx);
                moved |= mn != mrun[nt];
                corr[nt] = mn == -INFINITY ? 1.f : exp2f(mrun[nt] - mn);
                mrun[nt] = mn;
                lrun[nt] *= corr[nt];
            }
            if (__any_sync(kFull, moved)) {   // the running max rarely moves once it has settled
#pragma unroll
                for (int nt = 0; nt < C::kNO; ++nt)
#pragma unroll
                    for (int m = 0; m < 8; ++m)
#pragma unroll
                        for (int q = 0; q < 4; ++q) o[nt][m][q] *= corr[C::kH8 ? (q & 1) : nt];
            }
            // ---- P (times the value norm, split hi | lo) and P V for each 16-token tile
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int ta = 16 * mt + g, tb = ta + 8;
                float nva = 1.f, nvb = 1.f;
                if constexpr (!C::kRawV) {
                    constexpr float vf = VB == 8 ? 1.f / 255.f : 1.f;
                    nva = __half2float(__ushort_as_half((unsigned short)lds_u16(vs_s + ta * C::kVBytes))) * vf;
                    nvb = __half2float(__ushort_as_half((unsigned short)lds_u16(vs_s + tb * C::kVBytes))) * vf;
                }
                // B fragments of P (8 x 8 blocks of token rows g / g + 8, transposed): per n-tile, or
                // (kH8) index 0: the hi parts of the 8 heads, 1: the lo parts
                uint32_t b0[NT], b1[NT];
                float pa[NT], pb[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float mm = mrun[nt];
                    pa[nt] = mm == -INFINITY ? 0.f : exp2f(s[nt][mt][0] - mm);
                    pb[nt] = mm == -INFINITY ? 0.f : exp2f(s[nt][mt][1] - mm);
                    lrun[nt] += pa[nt] + pb[nt];
                }
                if constexpr (C::kH8) {
                    uint32_t ha, la, hb, lb;
                    split2_half2(pa[0] * nva, pa[1] * nva, ha, la);
                    split2_half2(pb[0] * nvb, pb[1] * nvb, hb, lb);
                    b0[0] = movmatrix_trans(ha);
                    b1[0] = movmatrix_trans(hb);
                    b0[1] = movmatrix_trans(la);
                    b1[1] = movmatrix_trans(lb);
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        b0[nt] = movmatrix_trans(split_half2(pa[nt] * nva));
                        b1[nt] = movmatrix_trans(split_half2(pb[nt] * nvb));
                    }
                }
                if constexpr (C::kRegV) {
                    // value codes of tokens 2t, 2t+1, 2t+8, 2t+9 of the tile: dims 16g..16g+15
                    uint32_t w0[1], w1[1], w2[1], w3[1];
                    lds_words_a2<1>(vs_s + (16 * mt + 2 * t) * C::kVBytes + 2 + 4 * g, w0);
                    lds_words_a2<1>(vs_s + (16 * mt + 2 * t + 1) * C::kVBytes + 2 + 4 * g, w1);
                    lds_words_a2<1>(vs_s + (16 * mt + 2 * t + 8) * C::kVBytes + 2 + 4 * g, w2);
                    lds_words_a2<1>(vs_s + (16 * mt + 2 * t + 9) * C::kVBytes + 2 + 4 * g, w3);
                    // interleave the two tokens of each register pair by nibbles: byte j of xl =
                    // [2t: dims 4j, 4j+1 | 2t+1: dims 4j, 4j+1], of xh the same for dims 4j+2, 4j+3
                    const uint32_t xl = (w0[0] & 0x0F0F0F0Fu) | ((w1[0] << 4) & 0xF0F0F0F0u);
                    const uint32_t xh = ((w0[0] >> 4) & 0x0F0F0F0Fu) | (w1[0] & 0xF0F0F0F0u);
                    const uint32_t yl = (w2[0] & 0x0F0F0F0Fu) | ((w3[0] << 4) & 0xF0F0F0F0u);
                    const uint32_t yh = ((w2[0] >> 4) & 0x0F0F0F0Fu) | (w3[0] & 0xF0F0F0F0u);
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        // m-tile m: rows g, g + 8 <-> dims 16g + 2m, + 1: one byte of xl / xh (yl / yh)
                        // is the pair-table entry of both rows (tokens 2t, 2t+1; 2t+8, 2t+9)
                        const uint32_t xs = (m & 1) ? xh : xl, ys = (m & 1) ? yh : yl;
                        const uint32_t sel = 0x6504u + 16u * (uint32_t)(m >> 1);
                        const uint2 p = lds64(klut_s + prmt(xs, vlane, sel));
                        const uint2 r = lds64(klut_s + prmt(ys, vlane, sel));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(o[C::kH8 ? 0 : nt][m], p.x, p.y, r.x, r.y, b0[nt], b1[nt]);
                    }
                } else {
                    uint32_t tile_s;
                    if constexpr (C::kRawV) {
                        tile_s = vs_s + 16 * mt * kVtPitch;
                    } else {
                        // lane -> token (lane & 15) of the tile, dims 64 (lane >> 4) .. + 63
                        dequant_value_half<VB>(vs_s + (16 * mt + (lane & 15)) * C::kVBytes, lane >> 4, vlut_s,
                                               vt_s + (lane & 15) * kVtPitch);
                        __syncwarp();
                        tile_s = vt_s;
                    }
                    // A = Vhat^T of m-tile m (dims 16m..16m+15 x the 16 tokens), read transposed
                    const uint32_t arow = tile_s + ((lane & 7) + 8 * (lane >> 4)) * kVtPitch + 16 * ((lane >> 3) & 1);
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(arow + 32 * m, a0, a1, a2, a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(o[C::kH8 ? 0 : nt][m], a0, a1, a2, a3, b0[nt], b1[nt]);
                    }
                    if constexpr (!C::kRawV) __syncwarp();   // the tile is rewritten for the next 16 tokens
                }
            }

            __syncwarp();
            cst = cst + 1 == kS ? 0 : cst + 1;
        }

        // ---- this warp's partial of segment j: fold the (hi, lo) columns (G <= 4), sum l over the rows g
        const bool ok = __all_sync(kFull, copies_ok);
        const int slot = (int)(gw - mma_worker_of_chunk((int64_t)j * plan.C, plan));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float l = lrun[nt];
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) l += __shfl_xor_sync(kFull, l, off);
            const int head = C::kH8 ? 2 * t + nt : 4 * nt + t;
            // output of this slot's head at accumulator n-tile no, fragment entries 2r (+ 1)
            const int no = C::kH8 ? 0 : nt;
            auto out_at = [&](int m, int r) {
                return C::kH8 ? o[0][m][2 * r + nt] : o[no][m][2 * r] + o[no][m][2 * r + 1];
            };
            if (head < a.G) {
                float *pr = a.ws + (((int64_t)b * a.Hq + kvh * a.G + head) * plan.Smax + slot) * kPartialFloats;
                if constexpr (C::kRegV) {
                    // dims 16g .. 16g + 15: float4 q holds dims 16g + 4q .. + 3 = m-tiles 2q, 2q + 1, rows g, g + 8
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int m0 = 2 * q;
                        reinterpret_cast<float4 *>(pr + 4 + 16 * g)[q] =
                            make_float4(out_at(m0, 0), out_at(m0, 1), out_at(m0 + 1, 0), out_at(m0 + 1, 1));
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 8; ++m)
#pragma unroll
                        for (int r = 0; r < 2; ++r) pr[4 + acc_dim<false>(m, r, g)] = out_at(m, r);
                }
                if (g == 0) {
                    pr[0] = mrun[nt];
                    pr[1] = ok ? l : __int_as_float(0x7fc00000);   // NaN marks a failed copy
                }
            }
        }
    }
    if (!__all_sync(kFull, copies_ok)) {
        // a wait gave up: the event is recorded, and copies this warp may still have in flight land
        // before it exits (about 0.1 s)
        if (lane == 0) note_wait_failed();
        spin_ns(100000000ull);
    }
}

template <int KB, int VB, bool QJL, int NT, bool WIDE, bool PAGED = false>
int launch_cfg_w(const AttnArgs &a, MmaPlan &plan, cudaStream_t st) {
    static_assert(!QJL || NT == 1, "the QJL term covers up to 4 query heads per KV head");
    static_assert(!(QJL && PAGED), "paged caches hold packed keys and values only");
    using C = Cfg<KB, VB, QJL, NT, WIDE>;
    static int done[64] = {0};
    if (set_smem_limit((const void *)attn_mma_kernel<KB, VB, QJL, NT, WIDE, PAGED>, C::kSmemTotal, done) != TQ_OK)
        return TQ_ERR_CUDA;
    // a programmatic dependent of the query-prep kernel: its prologue (first copies, tables) overlaps it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.P);
    cfg.blockDim = dim3((unsigned)C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemTotal;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn_mma_kernel<KB, VB, QJL, NT, WIDE, PAGED>, a, plan) != cudaSuccess)
        return TQ_ERR_CUDA;
    return launch_status();
}

// Only 2-bit values with one n-tile have a narrow (12-warp) variant.
template <int KB, int VB, bool QJL, int NT, bool PAGED = false>
int launch_cfg(const AttnArgs &a, MmaPlan &plan, cudaStream_t st) {
    if constexpr (VB == 2 && NT == 1) {
        if (!plan.wide) return launch_cfg_w<KB, VB, QJL, NT, false, PAGED>(a, plan, st);
    }
    return launch_cfg_w<KB, VB, QJL, NT, true, PAGED>(a, plan, st);
}

template <int KB, int VB, bool QJL, int NT>
void shape_of(bool wide, int *ctas_per_sm, int *warps) {
    if constexpr (VB == 2 && NT == 1) {
        if (!wide) {
            *ctas_per_sm = Cfg<KB, VB, QJL, NT, false>::kMinBlocks;
            *warps = Cfg<KB, VB, QJL, NT, false>::kW;
            return;
        }
    }
    *ctas_per_sm = Cfg<KB, VB, QJL, NT, true>::kMinBlocks;
    *warps = Cfg<KB, VB, QJL, NT, true>::kW;
}

}  // namespace
}  // namespace tq
