// qk_mmq_noalloc.cu -- qk_mmq_q4k with a workspace that is part of the
// library image instead of a caller buffer.
//
// Some callers cannot hand the MMQ a workspace: a plain C host with no device
// allocator of its own, code that must not call cudaMalloc in its steady
// state (cudaMalloc can synchronise the device and take locks, which a
// latency-bound prefill loop or a real-time thread cannot afford), or a caller
// that sizes nothing per call.  For them this entry point uses one
// statically allocated device array, reserved when the module is loaded, as
// the workspace of every call.  It allocates nothing and frees nothing.
//
// Limits and rules:
//  - the array holds QK_MMQ_STATIC_WS_BYTES bytes (32 MiB); a problem whose
//    qk_mmq_workspace_bytes(M, N, K) exceeds it is rejected with
//    QK_E_WORKSPACE before anything is launched;
//  - nothing in the array needs to start at zero: every call writes each byte
//    it reads before reading it;
//  - the array is shared by all calls on a device, so calls whose kernels can
//    overlap (different streams, or different host threads without ordering)
//    race on it; issue them on one stream;
//  - the array's device address is looked up with cudaGetSymbolAddress on the
//    first call on each device and cached; that first call must not be made
//    while the stream is being captured into a CUDA graph.
#include "qk_common.cuh"

#include <atomic>

namespace {

constexpr size_t kStaticWsBytes = QK_MMQ_STATIC_WS_BYTES;

static __device__ __align__(256) uint8_t g_mmq_static_ws[kStaticWsBytes];

// per-device cache of the array's address
void *static_ws_address()
{
    static std::atomic<void *> cache[qk::kMaxDevices];
    const int dev = qk::device_slot();
    if (dev < 0) return nullptr;
    void *p = cache[dev].load(std::memory_order_acquire);
    if (p) return p;
    if (cudaGetSymbolAddress(&p, g_mmq_static_ws) != cudaSuccess || !p) return nullptr;
    cache[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace

extern "C" int qk_mmq_q4k_noalloc(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                                  int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    size_t need = 0;
    const int st = qk_mmq_workspace_bytes(M, N, K, &need);
    if (st != QK_OK) return st;
    if (M == 0) return QK_OK;
    // the static array runs the call unsplit when it cannot also hold the split-K scratch
    if (qk::mmq_base_workspace_bytes(M, K) > kStaticWsBytes) return QK_E_WORKSPACE;
    void *ws = static_ws_address();
    if (!ws) return QK_E_CUDA;
    return qk_mmq_q4k(w, codes, scales, M, N, K, residual, y, ws, kStaticWsBytes, flags, stream);
}
