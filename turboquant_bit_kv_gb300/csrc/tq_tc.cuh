// 5th-generation tensor-core (tcgen05), TMA and mbarrier helpers for sm_103a,
// shared by the tensor-core encode and QJL kernels, plus the host-side
// tensor map of a [rows x 128] matrix of 16-bit elements.
//
// Conventions: operands are K-major in the 128-byte swizzle layout (the
// layout a TMA box of 64 columns x R rows lands in with SWIZZLE_128B): a
// 128-column row tile is two 64-column blocks of R * 128 bytes, row m at
// m * 128 within its block, 16-byte chunk c of the row at ((c ^ (m & 7)) << 4).
// Every mbarrier wait is bounded (about 100 ms) and reports failure.

#pragma once

#include <cuda.h>   // CUtensorMap and its enums (the encoder itself comes from the driver entry point)
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "tq.h"
#include "tq_device.cuh"

namespace tq {


__device__ __forceinline__ void tc_mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void tc_mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tc_mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for the phase of parity `parity`; false when it gave up.
__device__ __forceinline__ bool tc_mbar_wait(uint32_t bar, uint32_t parity) { return mbar_wait_bounded(bar, parity); }

__device__ __forceinline__ void tc_tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: start address >> 4, leading byte offset 1 (unused with this
// swizzle), stride byte offset 1024 >> 4 (8 rows of 128 bytes), descriptor
// version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: float32 accumulator, A and B of dtype
// DT (bf16 = 1, fp16 = 0), both K-major, N = 128, M = 128.
template <int DT>
__host__ __device__ constexpr uint32_t tc_idesc() {
    return (1u << 4) | ((DT == TQ_BF16 ? 1u : 0u) << 7) | ((DT == TQ_BF16 ? 1u : 0u) << 10) | ((128u >> 3) << 17) |
           ((128u >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The 128 x 128 x 128 product D (+)= A * B^T of two swizzled K-major tiles
// (A: 128 rows, B: 128 rows = N) as eight K = 16 steps.
template <int DT>
__device__ __forceinline__ void tc_mma_tile(uint32_t d_tmem, uint32_t a_s, uint32_t b_s, bool accumulate) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32);
        tc_mma(d_tmem, tc_desc_sw128(a_s + off), tc_desc_sw128(b_s + off), tc_idesc<DT>(),
               (accumulate || ks > 0) ? 1u : 0u);
    }
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive float32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

typedef CUresult (*TensorMapEncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                           const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                           const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                           CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (the library links only the runtime).
inline TensorMapEncodeTiledFn tensor_map_encoder() {
    static TensorMapEncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TensorMapEncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of n_rows rows of 128 16-bit elements (dtype dt: bf16 or fp16)
// at x, row stride stride_bytes (a multiple of 16, x 16-byte aligned): boxes
// of 64 columns x 128 rows, 128-byte swizzle, rows past the end read as zero.
// False when no encoder is available or the driver rejects the layout.
inline bool make_row_tile_map(CUtensorMap *map, const void *x, int dt, int64_t n_rows, int64_t stride_bytes) {
    TensorMapEncodeTiledFn enc = tensor_map_encoder();
    if (!enc || n_rows <= 0 || n_rows > 0x7FFFFFFFLL - 128) return false;
    const cuuint64_t gdim[2] = {128, (cuuint64_t)n_rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)stride_bytes};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, dt == TQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
               const_cast<void *>(x), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tq
