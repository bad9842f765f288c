// Host-side helpers shared by libtq's CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

inline bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

inline int dtype_bytes(int dt) {
    switch (dt) {
        case TQ_F32: return 4;
        case TQ_BF16: return 2;
        case TQ_F16: return 2;
        default: return 0;
    }
}

// Codebook sanity (head_dim 128, bits 2..4, levels 2^bits).
bool codebook_ok(const tq_codebook *cb);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Raise a kernel's dynamic shared-memory limit once per process and device.
int set_smem_limit(const void *kernel, int bytes, int *done_for_device);

// QJL sketch of bf16 / fp16 keys on the tensor cores (tq_qjl.cu).  Returns 1
// when it does not handle the call (other key dtypes, or rows no tensor map
// can describe), else a TQ_ status.
int qjl_encode_tc(const void *k, int k_dtype, int64_t n_vec, int64_t k_stride_bytes, const uint8_t *blocks,
                  int64_t block_stride, int bits, const float *centroids, const uint32_t *signs, const float *S,
                  uint8_t *qjl_bits, uint16_t *res_norm_f16, cudaStream_t st);

// Paired encode into 2 BB-byte slots (tq_encode.cu): k rows into the first,
// v rows into the second half of each slot.  Returns 1 when the call is not
// of the form it covers (then nothing was enqueued), else a TQ_ status.
int encode_kv_pair(const void *k, const void *v, int x_dtype, int64_t n_vec, int64_t x_stride_elems,
                   const tq_codebook *cb, tq_signs signs, uint8_t *slots, cudaStream_t st);

// Test hook (tq_debug_drop_copies): kernels with bounded waits issue none of
// their bulk / TMA copies while this is set (tq_status.cu).
int drop_copies();

// Host readers of the bounded-wait failure word of the units whose kernels
// wait on mbarriers (see tq_device.cuh).
int wait_failed_encode(unsigned *v, bool clear);
int wait_failed_qjl(unsigned *v, bool clear);
int wait_failed_attn_k2(unsigned *v, bool clear);
int wait_failed_attn_k3(unsigned *v, bool clear);
int wait_failed_attn_k4(unsigned *v, bool clear);
int wait_failed_attn_k8(unsigned *v, bool clear);
int wait_failed_prefill(unsigned *v, bool clear);
int wait_failed_headdim(unsigned *v, bool clear);

// Encode at head dims 64 / 96 / 128 / 160 with the caller's rotation R on
// the tensor cores (tq_headdim_tc.cu): bf16 / fp16 rows, at least
// kHdTcMinRows of them, contiguous.  Returns 1 when it does not handle the
// call (then nothing was enqueued), else a TQ_ status.
constexpr int64_t kHdTcMinRows = 1024;
int hd_encode_tc(const void *x, int x_dtype, int64_t n_vec, int d, const tq_codebook *cb, const float *R,
                 uint8_t *blocks, cudaStream_t st);

// The further formats at d = 128 on the same tensor-core encode (tq_headdim_tc.cu), rotation H D:
// norm-corrected and dense 3-bit blocks of a 2/3/4-bit codebook, or turboq8 (bits 8); bf16 / fp16
// rows, at least kHdTcMinRows of them, blocks back to back.  Returns 1 when it does not handle the
// call (then nothing was enqueued), else a TQ_ status.
int ext_encode_tc(const void *x, int x_dtype, int64_t n_vec, int64_t x_stride_bytes, const tq_codebook *cb,
                  const uint32_t *signs, int nc, int dense, uint8_t *blocks, cudaStream_t st);

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace tq
