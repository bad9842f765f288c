// tq_attn_decode_noalloc: decode attention for callers that cannot allocate
// device memory.
//
// Some callers of this library never get to call cudaMalloc: a serving engine
// that reserves all of its device memory up front in its own pool, or a plugin
// interface that hands a kernel only its input and output buffers, has no way
// to provide the extra split-K scratch that tq_attn_decode needs; in a
// latency-critical decode loop a cudaMalloc (which may synchronise the
// device) is not acceptable either.  For them this entry point keeps that
// scratch in a fixed array of device memory that is part of the library
// itself, so the caller passes only inputs and outputs.
//
// The array is TQ_ATTN_NOALLOC_SCRATCH_BYTES bytes.  Every GPU that loads
// the library holds it until the process exits.  Shapes whose scratch would
// not fit are rejected with TQ_ERR_WORKSPACE.
//
// Host code cannot use the array's name as a device address (in host code it
// is only a stand-in), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device; that first call should therefore come before any stream
// capture.  The looked-up address is kept for the life of the process: after
// a cudaDeviceReset (or anything else that destroys and re-creates the
// device's primary context) the library must be loaded afresh before this
// entry point is called again.  All calls share the one array and it keeps
// what the last call wrote: nothing in it has to start at zero, because each
// call rewrites every partial result it later reads, but calls that overlap
// on the GPU (other streams, other threads) race on it.

#include <mutex>

#include "tq.h"

static __device__ __align__(256) unsigned char g_tq_attn_scratch[TQ_ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tq_attn_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return TQ_OK;
}

}  // namespace

extern "C" int tq_attn_decode_noalloc(const void *q, int q_dtype, const uint8_t *k_blocks, const tq_codebook *kcb,
                                      const void *v, const tq_codebook *vcb, const int32_t *seq_lens, int B, int Hq,
                                      int Hkv, int T_cap, int T, float scale, tq_signs signs,
                                      const uint8_t *qjl_bits, const uint16_t *res_norm_f16, const float *S,
                                      float *out, void *stream) {
    const size_t need = tq_attn_workspace_bytes(B, Hq, Hkv, T_cap);
    if (need == 0) return TQ_ERR_ARG;
    if (need > (size_t)TQ_ATTN_NOALLOC_SCRATCH_BYTES) return TQ_ERR_WORKSPACE;
    void *scratch = nullptr;
    int r = noalloc_scratch(&scratch);
    if (r != TQ_OK) return r;
    return tq_attn_decode(q, q_dtype, k_blocks, kcb, v, vcb, seq_lens, B, Hq, Hkv, T_cap, T, scale, signs, qjl_bits,
                          res_norm_f16, S, out, scratch, (size_t)TQ_ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
