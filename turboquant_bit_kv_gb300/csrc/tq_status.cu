// tq_device_status / tq_debug_drop_copies: the host side of the kernels'
// bounded waits.  A kernel whose wait runs out records it in its unit's
// failure word (tq_device.cuh); this unit reads and clears those words, and
// holds the test hook that makes kernels issue no copies.

#include <atomic>

#include "tq_internal.h"

namespace tq {
namespace {
std::atomic<int> g_drop_copies{0};
}  // namespace

int drop_copies() { return g_drop_copies.load(std::memory_order_relaxed); }

}  // namespace tq

using namespace tq;

extern "C" int tq_debug_drop_copies(int on) {
    g_drop_copies.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
    return TQ_OK;
}

extern "C" int tq_device_status(int clear, void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TQ_ERR_CUDA;
    int (*const readers[])(unsigned *, bool) = {wait_failed_encode, wait_failed_qjl, wait_failed_attn_k2,
                                               wait_failed_attn_k3, wait_failed_attn_k4, wait_failed_attn_k8,
                                               wait_failed_prefill, wait_failed_headdim};
    unsigned any = 0;
    for (auto rd : readers) {
        unsigned v = 0;
        const int r = rd(&v, clear != 0);
        if (r != TQ_OK) return r;
        any |= v;
    }
    return any ? TQ_ERR_TIMEOUT : TQ_OK;
}
