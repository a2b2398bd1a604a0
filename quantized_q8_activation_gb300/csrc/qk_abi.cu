// qk_abi.cu -- library-wide entry points of the C ABI (version, status
// strings) and the per-device SM count used to size persistent grids.
#include "qk_common.cuh"

#include <atomic>

namespace qk {

int sm_count()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

size_t max_smem_optin()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 48 * 1024;
    if (dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return (size_t)v;
    }
    int n = 48 * 1024;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || n < 1)
        n = 48 * 1024;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return (size_t)n;
}

}  // namespace qk

extern "C" int qk_version(void) { return 100; }   // 0.1.0

extern "C" const char *qk_status_string(int status)
{
    switch (status) {
    case QK_OK: return "ok";
    case QK_E_NULL: return "a required pointer is NULL";
    case QK_E_SHAPE: return "shape out of range (M, N, K; K must be a multiple of 256)";
    case QK_E_ALIGN: return "pointer or leading dimension misaligned";
    case QK_E_ALIAS: return "output overlaps an input";
    case QK_E_TYPE: return "unknown quantization type";
    case QK_E_WORKSPACE: return "workspace too small";
    case QK_E_CUDA: return "CUDA runtime error";
    default: return "unknown status";
    }
}
