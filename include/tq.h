/*
 * tq.h -- C ABI of libtq: GB300-native TurboQuant KV-cache compression.
 *
 * The operations restate these pages:
 *   [spec]   "TurboQuant KV Cache Compression — Spec" (Foundry attention/spec.md)
 *   [fork]   "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)" (llama.cpp fork,
 *            turboquant-kv-base.md)
 *   [rotor]  "RotorQuant KV Cache Compression" (RotorQuant docs)
 *   [serde]  "lmcache.v1.distributed.serde.turboquant" (LMCache serde design)
 *
 * Conventions for every call:
 *   - head_dim is 128 ([fork] section 2, "head_dim multiple of 128": the block
 *     size of all types is 128); any other value returns TQ_ERR_UNSUPPORTED.
 *   - bits is 2, 3 or 4 ([spec] fa_tq_config); blocks are 2 + 16*bits bytes:
 *     34 / 50 / 66 ([fork] section 4 block structures, without the legacy rnorm).
 *   - Every device buffer is owned by the caller.  The library allocates no
 *     device memory and keeps no per-call state; codebooks and signs travel
 *     by value into the kernels.
 *   - Calls that take a `stream` (a cudaStream_t, NULL = legacy default
 *     stream) only enqueue work and return without synchronising.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check returns a negative tq_status and enqueues nothing.  A CUDA
 *     launch error returns TQ_ERR_CUDA.  Nothing throws across this ABI and no
 *     kernel traps or asserts.
 *   - Every wait inside a kernel (for a bulk or TMA copy, or a tensor-core
 *     product) is bounded at about 0.1 s of device time.  A kernel whose wait
 *     runs out stops issuing copies and waiting, lets the copies it already
 *     issued land, finishes without hanging (its output is then invalid) and
 *     records the event in a sticky per-device status that tq_device_status
 *     returns as TQ_ERR_TIMEOUT.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TQ_OK = 0,
    TQ_ERR_ARG = -1,          /* null pointer, negative count, bad stride, T range */
    TQ_ERR_UNSUPPORTED = -2,  /* head_dim != 128, bits not in {2,3,4}, dtype, G > 8 */
    TQ_ERR_ALIGN = -3,        /* a base pointer or stride breaks the stated alignment */
    TQ_ERR_WORKSPACE = -4,    /* workspace smaller than tq_attn_workspace_bytes() */
    TQ_ERR_CUDA = -5,         /* a CUDA runtime call or kernel launch failed */
    TQ_ERR_TIMEOUT = -6       /* a kernel gave up a bounded wait (tq_device_status) */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

/* Lloyd-Max codebook of one (head_dim, bits) pair ([spec] Algorithm Detail,
 * Step 2, fa_tq_codebook, plus head_dim).  Values are in the unit-sphere
 * coordinate y = 2u - 1, u ~ Beta(d/2, d/2), ascending; boundaries[i] lies
 * between centroids[i] and centroids[i+1]; only the first `levels` centroids
 * and `levels - 1` boundaries are meaningful. */
typedef struct {
    int head_dim;
    int bits;
    int levels;
    float centroids[16];
    float boundaries[15];
} tq_codebook;

/* Random sign diagonal D of the rotation R x = H (D x) / sqrt(d) ([spec]
 * As-Built Notes, Step 1).  Bit j of the 128-bit mask (word j / 32, bit
 * j % 32) set means D_jj = -1. */
typedef struct {
    uint32_t w[4];
} tq_signs;

/* Fill *out with the Lloyd-Max codebook of Beta(head_dim/2, head_dim/2)
 * for `bits` ([spec] Codebook Generation: conditional means of cells,
 * midpoint boundaries, iterated to a fixed point).  Host only; the first
 * call per (head_dim, bits) runs the iteration (milliseconds) and caches it;
 * thread-safe.  head_dim 64, 96, 128 or 160 ([spec] Types / Codebook
 * Generation: the target dimensions) for bits 2-4; 128 for bits 8
 * (turboq8).  Errors: TQ_ERR_ARG (out NULL), TQ_ERR_UNSUPPORTED. */
int tq_codebook_load(int head_dim, int bits, tq_codebook *out);

/* Fill *out with the sign diagonal drawn from `seed` ([spec] Lifecycle,
 * fa_tq_init(head_dim, config, seed)): output j of splitmix64 started at
 * `seed` gives sign j, top bit set => -1.  Host only. */
int tq_signs_from_seed(uint64_t seed, int head_dim, tq_signs *out);

/* Bytes of one 128-element block: 34, 50 or 66; 0 for unsupported bits. */
size_t tq_block_bytes(int bits);

/* Quantise-on-insert ([spec] As-Built Notes and Steps 1-3; [fork] section 4
 * encode pipeline steps 1-3): for each of n_vec rows x of 128 elements,
 * n = ||x||, y = H (D x) / (sqrt(128) n), code_j = #{i : boundaries[i] <= y_j},
 * codes bit-packed after the fp16 (round-to-nearest-even) norm n.
 *   x                 device, row i at x + i * x_stride_elems elements, dtype
 *                     x_dtype (TQ_F32 / TQ_BF16 / TQ_F16); base 16-byte aligned,
 *                     x_stride_elems * sizeof(dtype) a multiple of 16.
 *   cb, signs         codebook (cb->bits selects 2/3/4) and sign diagonal.
 *   blocks            device output; block of row i at
 *                     blocks + dst(i) * block_stride_bytes, dst(i) = i or
 *                     dst_index[i] (device int64, n_vec entries) when given;
 *                     block_stride_bytes >= tq_block_bytes(bits) and even,
 *                     blocks 2-byte aligned.  Rows must not share a block.
 *   n_vec == 0 is a no-op.  Zero rows store norm 0 and every code = levels/2.
 * Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_encode_kv(const void *x, int x_dtype, int64_t n_vec, int64_t x_stride_elems,
                 const tq_codebook *cb, tq_signs signs,
                 uint8_t *blocks, int64_t block_stride_bytes,
                 const int64_t *dst_index, void *stream);

/* Dequantise ([spec] Overview "look up reconstruction values, then rotate
 * back"; Quantize / Dequantize fa_tq_dequantize): x_hat = n16 * D H c[code]
 * / sqrt(128) for n_vec blocks, written as out_dtype (float32, or bf16 / fp16
 * rounded to nearest even) at out + i * out_stride_elems elements.
 *   blocks            device, block i at blocks + i * block_stride_bytes
 *                     (even stride >= block bytes; base 2-byte aligned).
 *   out               device, base 16-byte aligned, out_stride_elems *
 *                     sizeof(out_dtype) a multiple of 16.
 * Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_decode_kv(const uint8_t *blocks, int64_t block_stride_bytes, int64_t n_vec,
                 const tq_codebook *cb, tq_signs signs,
                 void *out, int out_dtype, int64_t out_stride_elems, void *stream);

/* Further block formats ([fork] section 4, Encode pipeline step 4: the
 * corrected norm; [spec] Algorithm Detail Step 3: eight 3-bit values in
 * three bytes; [fork] At a glance and the turboq8 paragraph: the 8-bit
 * codec), selected by `flags` of the _ex calls:
 *   TQ_FMT_NORM_CORRECT  bits 2..4: the stored norm is ||x|| / ||c[idx]||
 *                        (rounded once to fp16), so the block decodes to a
 *                        vector of the input's norm; codes, layout and
 *                        decoding are those of the plain block.
 *   TQ_FMT_DENSE3        bits 3: 50-byte block [fp16 norm][16 x 3 bytes], the
 *                        codes of elements 8g .. 8g + 7 in the 24-bit
 *                        little-endian word of group g, element 8g + p in
 *                        bits 3p .. 3p + 2.
 * turboq8 (a codebook of bits 8 from tq_codebook_load(128, 8), no flags):
 * u = R x, a = max |u_j|, code i_j = nearest level of the grid
 * (i - 127.5) / 127.5 to u_j / a (decided in float32, ties to the upper),
 * block [fp16(a)][128 code bytes] (130 bytes); decode x_hat = R^T (a16 (i -
 * 127.5) / 127.5).  tq_encode_kv / tq_decode_kv accept turboq8 codebooks
 * as well. */
#define TQ_FMT_NORM_CORRECT 1
#define TQ_FMT_DENSE3 2

/* Block bytes of a format: 34 / 50 / 66 for bits 2 / 3 / 4 (any valid
 * flags), 130 for bits 8; 0 for an invalid combination. */
size_t tq_block_bytes_ex(int bits, int flags);

/* tq_encode_kv with `flags` (above); same arguments, layout, alignment and
 * errors, plus TQ_ERR_ARG for unknown flags and TQ_ERR_UNSUPPORTED for a
 * flag the bit width does not take. */
int tq_encode_kv_ex(const void *x, int x_dtype, int64_t n_vec, int64_t x_stride_elems,
                    const tq_codebook *cb, tq_signs signs,
                    uint8_t *blocks, int64_t block_stride_bytes,
                    const int64_t *dst_index, int flags, void *stream);

/* tq_decode_kv with `flags` (TQ_FMT_DENSE3 selects the dense 3-bit layout;
 * TQ_FMT_NORM_CORRECT changes nothing in decoding). */
int tq_decode_kv_ex(const uint8_t *blocks, int64_t block_stride_bytes, int64_t n_vec,
                    const tq_codebook *cb, tq_signs signs,
                    void *out, int out_dtype, int64_t out_stride_elems, int flags, void *stream);

/* QJL residual sketch of keys ([rotor] Implementation Requirements 1-2):
 * k_mse = decode(k_blocks[i]), r = k - k_mse, res_norm_f16[i] = fp16(||r||),
 * bit j of qjl_bits[i] (byte j / 8, position j % 8) = [(S r)_j >= 0].
 *   k                 device original keys (dtype k_dtype, same alignment
 *                     rules as tq_encode_kv's x).
 *   k_blocks          device blocks of the same keys made by tq_encode_kv
 *                     with the same cb / signs.
 *   S                 device float32 [128][128] row-major sketch, m = 128.
 *   qjl_bits          device [n_vec][16] bytes; res_norm_f16 device [n_vec].
 * Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_qjl_encode(const void *k, int k_dtype, int64_t n_vec, int64_t k_stride_elems,
                  const uint8_t *k_blocks, int64_t block_stride_bytes,
                  const tq_codebook *cb, tq_signs signs, const float *S,
                  uint8_t *qjl_bits, uint16_t *res_norm_f16, void *stream);

/* Workspace bytes tq_attn_decode needs for this shape (split-K partials)
 * on the current device (the split depends on its SM count).  Host only.
 * Returns 0 for an invalid shape. */
size_t tq_attn_workspace_bytes(int B, int Hq, int Hkv, int T_cap);

/* The same for a GPU of `sms` SMs (sms <= 0: the current device), for
 * sizing buffers ahead of time or on a machine without the GPU.  Host only;
 * touches no device memory.  Returns 0 for an invalid shape. */
size_t tq_attn_workspace_bytes_sms(int B, int Hq, int Hkv, int T_cap, int sms);

/* The work partition tq_attn_decode's tensor-core path uses for a shape
 * (split-K over the context, [spec] Optimization: Fused dequant-dot), for
 * tests and tuning.  value_bits 16 stands for raw fp16 values; qjl != 0 for
 * the two-term score; sms <= 0 takes the current device's SM count.  Fills
 * out[7] (host memory):
 *   out[0] C     chunks of 32 tokens per (sequence, KV head) segment,
 *   out[1] Ctot  B * Hkv * C, chunks ordered by (sequence, KV head, position),
 *   out[2] P     CTAs,
 *   out[3] W     warp workers; worker w owns chunks [w Ctot / W, (w+1) Ctot / W),
 *   out[4] Smax  partial slots per (sequence, query head): no segment meets
 *                more worker ranges,
 *   out[5]       slot groups of 128 threads in a combine CTA,
 *   out[6]       warps per CTA.
 * Host only: touches no device memory.  TQ_ERR_ARG for a bad shape or a NULL
 * out; TQ_ERR_UNSUPPORTED for invalid bits or a shape that takes the CUDA-core
 * split path instead. */
int tq_attn_plan(int B, int Hq, int Hkv, int T, int key_bits, int value_bits, int qjl, int sms, int64_t *out);

/* The context splits tq_attn_decode_d makes for B sequences x Hkv KV heads
 * over T tokens when ctas_resident attention CTAs of warps_per_cta warps fit
 * on the device at once (its tensor-core attention kernel runs 4 warps per
 * CTA; ctas_resident is the SM count times its CTAs per SM): of the split
 * counts s = 1 .. max(1, ceil(T / 32) / 16) (every split keeps at least 16
 * chunks of 32 tokens), the first with the fewest waves of CTAs times
 * 32-token steps per warp (plus one); then tokens per split = ceil(ceil(T /
 * 32) / s) * 32 and splits = ceil(T / tokens per split).
 *   out[0] splits, out[1] tokens per split (a multiple of 32), out[2] the most
 *   splits a context of T tokens takes.
 * Host only.  TQ_ERR_ARG for a non-positive size or a NULL out. */
int tq_attn_plan_d(int B, int Hkv, int T, int ctas_resident, int warps_per_cta, int32_t *out);

/* Fused decode attention over a packed cache ([spec] Optimization: Fused
 * dequant-dot; [fork] section 2 "fused flash-attention path required";
 * [rotor] Fused Kernel Logic for the QJL term).  One query token per
 * (batch, query head):
 *   s_t = scale * ( n_t * <R q, cK[code_t]> + term2_t ),
 *   term2_t = rn_t * sqrt(pi/2) / 128 * <S q, sign_t>   (only when qjl_bits),
 *   o = sum_t softmax(s)_t * v_hat_t,  v_hat_t = R^T (nv_t cV[vcode_t])
 *                                     (or the raw fp16 value when vcb NULL),
 * computed as: rotate q once, score in the rotated domain, online softmax,
 * accumulate values in the rotated domain, one inverse rotation per output.
 *   q           device [B][Hq][128], dtype q_dtype (TQ_F32 / TQ_BF16 / TQ_F16).
 *   k_blocks    device [B][Hkv][T_cap] blocks of kcb->bits, contiguous.
 *   v           device: [B][Hkv][T_cap] blocks of vcb->bits, or, when vcb is
 *               NULL, raw fp16 values [B][Hkv][T_cap][128].
 *   seq_lens    device int32 [B] (each clamped to [0, T]; length 0 gives a
 *               zero output row) or NULL for T tokens in every sequence.
 *   Hq % Hkv == 0, G = Hq / Hkv <= 8 (query head h reads KV head h / G);
 *   1 <= T <= T_cap; T_cap a multiple of 8; k_blocks, v, q and out 16-byte
 *   aligned.
 *   qjl_bits    device [B][Hkv][T_cap][16], res_norm_f16 device [B][Hkv][T_cap],
 *               S device float32 [128][128]: all three NULL (plain score) or
 *               all three set (two-term score).
 *   out         device float32 [B][Hq][128].
 *   workspace   device scratch of >= tq_attn_workspace_bytes(B, Hq, Hkv, T_cap)
 *               bytes, 16-byte aligned (TQ_ERR_ALIGN otherwise); clobbered;
 *               calls that overlap on the GPU must use different workspaces.
 *   turboq8 keys with 2/3/4-bit values, or 4-bit keys with turboq8 values
 *   ([fork] section 2, Asymmetric K/V), run on the same split-K tensor-core
 *   path when workspace holds tq_attn_workspace_bytes(...) bytes (16-byte
 *   aligned, G <= 8); with a smaller or NULL workspace they are served as
 *   the one-token case of tq_attn_prefill (the workspace is then unused).
 *   Other combinations with turboq8, and QJL with turboq8, return
 *   TQ_ERR_UNSUPPORTED.
 * Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_WORKSPACE,
 * TQ_ERR_CUDA. */
int tq_attn_decode(const void *q, int q_dtype,
                   const uint8_t *k_blocks, const tq_codebook *kcb,
                   const void *v, const tq_codebook *vcb,
                   const int32_t *seq_lens, int B, int Hq, int Hkv, int T_cap, int T,
                   float scale, tq_signs signs,
                   const uint8_t *qjl_bits, const uint16_t *res_norm_f16, const float *S,
                   float *out, void *workspace, size_t workspace_bytes, void *stream);

/* Attention of M new query tokens per sequence over a packed cache that
 * already holds them, with the causal mask: a prefill chunk, or the draft
 * tokens of a speculative verify step ([fork] section 2, Requirements: the
 * quantised cache is reachable only through the fused flash-attention path;
 * [spec] Optimization: Fused dequant-dot for the rotated-domain scores and
 * value sums).  Query token i of sequence b sits at position
 * p = L_b - M + i (L_b its length) and attends to the keys at positions
 * 0 .. p:
 *   s_t = scale * n_t * <R q, cK[code_t]>,  o = sum_{t <= p} softmax(s)_t v_hat_t,
 * a query with p < 0 gives a zero output row.
 *   q         device [B][M][Hq][128] of q_dtype (TQ_F32 / TQ_BF16 / TQ_F16).
 *   k_blocks  device [B][Hkv][T_cap] blocks of kcb->bits; v_blocks the same
 *             for vcb->bits (packed values only).  Widths: 2, 3, 4 with each
 *             other, turboq8 (bits 8) keys with 2/3/4-bit values, 4-bit keys
 *             with turboq8 values.
 *   seq_lens  device int32 [B] (each clamped to [0, T]) or NULL for T.
 *   Hq % Hkv == 0 (query head h reads KV head h / (Hq / Hkv)); 1 <= T <=
 *   T_cap, T_cap a multiple of 8; q, k_blocks, v_blocks, out 16-byte aligned.
 *   out       device float32 [B][M][Hq][128].
 * No workspace.  Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN,
 * TQ_ERR_CUDA. */
int tq_attn_prefill(const void *q, int q_dtype,
                    const uint8_t *k_blocks, const tq_codebook *kcb,
                    const uint8_t *v_blocks, const tq_codebook *vcb,
                    const int32_t *seq_lens, int B, int M, int Hq, int Hkv, int T_cap, int T,
                    float scale, tq_signs signs, float *out, void *stream);

/* tq_attn_prefill over a paged cache: the serde page's "block/slot mapping"
 * (Limitations) and the spec's per-position packed cache (Integration
 * Points).  Packed blocks live in pools of pages of `page_tokens` tokens
 * (a multiple of 8): k_pool / v_pool are device [num_pages][Hkv][page_tokens]
 * blocks, and token t of sequence b is slot t % page_tokens of page
 * block_table[b * max_pages + t / page_tokens] (device int32 [B][max_pages];
 * the entries for the pages covering tokens 0 .. L_b - 1 must name pages of
 * the pools).  max_pages * page_tokens >= T; the other arguments, the
 * causal rule and the errors as tq_attn_prefill. */
int tq_attn_prefill_paged(const void *q, int q_dtype,
                          const uint8_t *k_pool, const tq_codebook *kcb,
                          const uint8_t *v_pool, const tq_codebook *vcb,
                          const int32_t *block_table, int max_pages, int page_tokens,
                          const int32_t *seq_lens, int B, int M, int Hq, int Hkv, int T,
                          float scale, tq_signs signs, float *out, void *stream);

/* Decode attention (one query token per sequence, q [B][Hq][128], out
 * [B][Hq][128]) over a paged cache laid out as for tq_attn_prefill_paged.
 * With 2/3/4-bit keys and values, pages of a multiple of 32 tokens and a
 * workspace of >= tq_attn_workspace_bytes(B, Hq, Hkv, T rounded up to 8)
 * bytes (16-byte aligned; clobbered), it runs the split-K tensor-core decode
 * kernels of tq_attn_decode through the block table; otherwise (no
 * workspace, other page sizes, turboq8) the one-token case of
 * tq_attn_prefill_paged.  Errors as tq_attn_decode. */
int tq_attn_decode_paged(const void *q, int q_dtype,
                         const uint8_t *k_pool, const tq_codebook *kcb,
                         const uint8_t *v_pool, const tq_codebook *vcb,
                         const int32_t *block_table, int max_pages, int page_tokens,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int T,
                         float scale, tq_signs signs, float *out,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Size of the device array that tq_attn_decode_noalloc uses as its split-K
 * scratch: 16 MiB.  On GPUs of 148 to 160 SMs that covers, at any context,
 * batch 64 x 28 query heads over 4 KV heads (about 11.4 MiB), batch 64 x 32
 * over 8 (about 9.2 MiB) and batch 128 x 32 over 8 (about 14.3 MiB); batch
 * 256 x 32 over 8 needs about 24.4 MiB and is refused.
 * tq_attn_workspace_bytes_sms gives the figure for any shape. */
#define TQ_ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)

/* tq_attn_decode for callers that cannot allocate device memory (the pages
 * have no counterpart: this is a library convenience).  A serving engine
 * that owns all device memory in its own pool, or a plugin interface that
 * passes a kernel only its inputs and outputs, cannot supply the split-K
 * workspace, and a cudaMalloc inside a latency-critical decode loop is not
 * acceptable either.  This call takes the same arguments as tq_attn_decode
 * minus the workspace and uses a fixed TQ_ATTN_NOALLOC_SCRATCH_BYTES array of
 * device memory inside the library instead; it allocates nothing.
 *   - Shapes whose workspace (tq_attn_workspace_bytes) exceeds the array
 *     return TQ_ERR_WORKSPACE; an invalid shape returns TQ_ERR_ARG.
 *   - The array's device address is looked up once per device, on the first
 *     call made with that device current; make that first call before any
 *     stream capture.  The address is kept until process exit: after a
 *     cudaDeviceReset, load the library afresh before calling this again.
 *   - All calls share the array, which keeps the last call's contents (no
 *     part of it needs to start at zero); calls that overlap on the GPU race
 *     on it, so serialise them (one stream, or events).
 *   - Every GPU that loads the library holds the array until process exit.
 * Errors: as tq_attn_decode. */
int tq_attn_decode_noalloc(const void *q, int q_dtype,
                           const uint8_t *k_blocks, const tq_codebook *kcb,
                           const void *v, const tq_codebook *vcb,
                           const int32_t *seq_lens, int B, int Hq, int Hkv, int T_cap, int T,
                           float scale, tq_signs signs,
                           const uint8_t *qjl_bits, const uint16_t *res_norm_f16, const float *S,
                           float *out, void *stream);

/* Serialised size of one KV object ([serde] Tensor Layout and
 * estimate_serialized_size): raw first layers | compressed middle layers |
 * raw last layers, with quant_start = min(skip_first, L) and quant_end =
 * max(quant_start, L - skip_last) ([serde] Configuration); compressed layers
 * are [L_c][ceil(T / block_size)][block_size][hidden / 128][slot], slot =
 * key block + value block bytes.  elem_bytes is 2 (bf16 / fp16).  Returns 0
 * for invalid arguments. */
size_t tq_serde_size(int num_layers, int num_tokens, int hidden_dim, int head_dim,
                     int block_size, int skip_first, int skip_last,
                     int key_bits, int value_bits, int elem_bytes);

/* Serialise src (device, [2][L][T][hidden] of elem_dtype TQ_BF16 / TQ_F16,
 * 16-byte aligned) into dst (device, tq_serde_size() bytes, 16-byte aligned):
 * raw layers copied byte for byte, middle layers encoded with kcb / vcb.
 * Token slots past T in the last token block are written as zero bytes.
 * Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_serde_serialize(const void *src, int elem_dtype, int num_layers, int num_tokens,
                       int hidden_dim, int head_dim, int block_size,
                       int skip_first, int skip_last,
                       const tq_codebook *kcb, const tq_codebook *vcb, tq_signs signs,
                       uint8_t *dst, void *stream);

/* Inverse of tq_serde_serialize ([serde] Decompression Path): restores the
 * [2][L][T][hidden] tensor in dst (raw layers byte-identical, middle layers
 * dequantised and rounded to elem_dtype). */
int tq_serde_deserialize(const uint8_t *src, int elem_dtype, int num_layers, int num_tokens,
                         int hidden_dim, int head_dim, int block_size,
                         int skip_first, int skip_last,
                         const tq_codebook *kcb, const tq_codebook *vcb, tq_signs signs,
                         void *dst, void *stream);

/* Sticky status of the kernels' bounded waits on the current device: waits
 * for the work already enqueued on `stream` (cudaStreamSynchronize), then
 * returns TQ_ERR_TIMEOUT if any kernel of this library gave up a wait on this
 * device since the status was last cleared, else TQ_OK (TQ_ERR_CUDA if a
 * CUDA call fails).  clear != 0 resets it.  Host call; it synchronises, so it
 * belongs in diagnostics and tests rather than in a decode loop. */
int tq_device_status(int clear, void *stream);

/* Fault injection for tests of the bounded waits (the pages have no
 * counterpart).  While on != 0, kernels launched afterwards with bounded
 * waits (the tensor-core encode and QJL encode issue none of their TMA
 * loads; the tensor-core attention sets up its copy barriers to wait for an
 * arrival that never comes) find their first wait unsatisfiable, so it runs
 * out after about 0.1 s, as it would for a copy that never lands; their
 * outputs are then invalid and tq_device_status reports TQ_ERR_TIMEOUT.  No
 * memory is touched outside the call's own buffers.  Host only; returns
 * TQ_OK. */
int tq_debug_drop_copies(int on);

/* Static, human-readable name of a tq_status value. */
const char *tq_status_string(int status);

/* ---- Head dims other than 128 ([spec] Types / Codebook Generation: target
 * dimensions 64, 96, 128, 160; Hadamard Transform Detail: for a head dim that
 * is not a power of two, "a dense random orthogonal matrix").  The rotation
 * is an input: R, a device float32 [head_dim][head_dim] row-major orthogonal
 * matrix (R R^T = I), owned by the caller; y = R x / ||x||, and a block
 * decodes to n16 R^T c[code].  Blocks: [fp16 norm][codes], 2-bit four per
 * byte, 4-bit two per byte, 3-bit a 2-bit low plane of head_dim / 4 bytes
 * then a 1-bit high plane of head_dim / 8 bytes (the 128-element layout
 * generalised); 2 + head_dim * bits / 8 bytes, back to back.  head_dim is
 * 64, 96, 128 or 160 and the codebook one of tq_codebook_load(head_dim, .).
 * The encode of 1024 or more bf16 / fp16 rows and the decode attention run
 * on the tensor cores, the rest of the encode and the decode on CUDA cores
 * (the rotation as a dense product per row); the 128-element entry points
 * above remain the fast path for head_dim 128 (the rotation there is the
 * exact H D transform). */

/* Bytes of one block at head_dim: 2 + head_dim * bits / 8; 0 if unsupported. */
size_t tq_block_bytes_d(int head_dim, int bits);

/* Host: R = H D / sqrt(head_dim) for a power-of-two head_dim (64 or 128),
 * H the Sylvester-Hadamard matrix, D the first head_dim signs of `signs`
 * (bit set = -1), written row-major to R_host [head_dim * head_dim].
 * Errors: TQ_ERR_ARG, TQ_ERR_UNSUPPORTED (other head dims). */
int tq_rotation_hadamard(int head_dim, tq_signs signs, float *R_host);

/* Encode n_vec rows x [n_vec][head_dim] (x_dtype TQ_F32 / TQ_BF16 / TQ_F16)
 * into blocks [n_vec][tq_block_bytes_d(head_dim, cb->bits)].  Codes decided
 * in float32 (y = R x / ||x|| against the float32 boundaries); the norm is
 * rounded once to fp16 (recomputed in double precision near an fp16
 * rounding boundary); a zero row stores norm 0 and code L/2.  n_vec 0 is a
 * no-op.  x 4-byte aligned, R 16-byte aligned.  Errors: TQ_ERR_ARG,
 * TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGN, TQ_ERR_CUDA. */
int tq_encode_kv_d(const void *x, int x_dtype, int64_t n_vec, int head_dim, const tq_codebook *cb,
                   const float *R, uint8_t *blocks, void *stream);

/* Decode blocks back to rows out [n_vec][head_dim] of out_dtype:
 * x_hat = n16 R^T c[code] (float32 arithmetic, one rounding to the output
 * type).  Errors as tq_encode_kv_d. */
int tq_decode_kv_d(const uint8_t *blocks, int64_t n_vec, int head_dim, const tq_codebook *cb, const float *R,
                   void *out, int out_dtype, void *stream);

/* Scratch bytes tq_attn_decode_d needs (0 for a bad shape). */
size_t tq_attn_workspace_bytes_d(int B, int Hq, int Hkv, int T_cap, int head_dim);

/* Decode attention at head_dim (one query token per sequence and query
 * head), the same computation as tq_attn_decode: q rotated once (R q),
 * scores n_t <R q, cK[code_t]> in the rotated domain, online softmax, values
 * accumulated there, one inverse rotation per output; split over the
 * context with a merge.  q [B][Hq][head_dim] (q_dtype), k_blocks / v_blocks
 * [B][Hkv][T_cap] blocks of kcb->bits / vcb->bits at head_dim (both arrays
 * 16-byte aligned, T_cap a multiple of 8: the kernel copies 32-block runs
 * in 16-byte pieces), seq_lens as for tq_attn_decode, 1 <= T <= T_cap,
 * G = Hq / Hkv <= 8 (B, Hkv <= 65535, B * Hq <= 1048560), out float32
 * [B][Hq][head_dim], workspace >= tq_attn_workspace_bytes_d(...) bytes
 * (16-byte aligned).  Errors:
 * TQ_ERR_ARG (T_cap not a multiple of 8 among them), TQ_ERR_UNSUPPORTED,
 * TQ_ERR_ALIGN, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
int tq_attn_decode_d(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                     const uint8_t *v_blocks, const tq_codebook *vcb, const int32_t *seq_lens, int B, int Hq,
                     int Hkv, int T_cap, int T, int head_dim, float scale, const float *R, float *out,
                     void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
