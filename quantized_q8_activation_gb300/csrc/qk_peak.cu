// qk_peak.cu -- tensor-core peak micro-benchmarks (declared in include/qk_peak.h).
//
// The prefill MMQ reports its rate against two ceilings measured here on the
// device itself: the legacy warp-level int8 MMA (mma.sync m16n8k32 s8, the
// instruction an int8 MMQ would use on this part) and the tcgen05 f16 MMA that
// the library's MMQ issues (128 x 256 x 16, f32 accumulator in tensor memory).
// Both loops keep their operands on chip, so the figure is the tensor pipe's
// own rate, not a memory rate.
#include "qk_common.cuh"
#include "qk_peak.h"
#include "qk_tc.cuh"

#include <atomic>

namespace {

using namespace qk::tc;

__device__ unsigned g_peak_errors;       // a bounded wait of the tcgen05 loop gave up
__device__ int g_peak_sink;              // keeps the int8 results observable

constexpr int kS8Warps = 16, kS8Acc = 8;
constexpr int kOneCtaSmem = 120 * 1024;  // dynamic shared memory that keeps one CTA per SM
constexpr int TC_M = 128, TC_N = 256, TC_K = 16;

// mma.sync s8: every warp runs kS8Acc independent accumulator chains of m16n8k32
__global__ void __launch_bounds__(kS8Warps * 32, 1) peak_s8_kernel(int64_t iters, int magic)
{
    const uint32_t t = threadIdx.x;
    const uint32_t a0 = t * 0x01010101u, a1 = a0 ^ 0x5a5a5a5au, a2 = a0 + 0x13131313u, a3 = ~a0;
    const uint32_t b0 = a0 ^ 0x33333333u, b1 = a1 + 0x07070707u;
    int acc[kS8Acc][4];
#pragma unroll
    for (int j = 0; j < kS8Acc; j++) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0;
    for (int64_t i = 0; i < iters; i++) {
#pragma unroll
        for (int j = 0; j < kS8Acc; j++)
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                         "{%0,%1,%2,%3};"
                         : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kS8Acc; j++) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
    if (s == magic) g_peak_sink = s;
}

// tcgen05 kind::f16: thread 0 of one CTA per SM issues 2 * iters MMAs of 128 x 256 x 16 into one
// tensor-memory accumulator (operand tiles of zeros, K-major with the 64-byte swizzle), commits,
// and waits (bounded) before the tensor memory is released
__global__ void __launch_bounds__(128, 1) peak_tc_kernel(int64_t iters)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int ATILE = TC_M * 64, BTILE = TC_N * 64;        // 32 f16 of K per row: two K-steps
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + ATILE + BTILE);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + ATILE + BTILE + 8);
    for (int i = threadIdx.x; i < (ATILE + BTILE) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tmem_ptr, TC_N);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_ptr;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = idesc_f16_f32(TC_M, TC_N);
        const uint32_t sa = smem_u32(smem), sb = sa + ATILE;
        for (int64_t i = 0; i < iters; i++) {
#pragma unroll
            for (int kk = 0; kk < 2; kk++)
                mma_f16(tmem, smem_desc(sa + 32 * kk, 16, 512, kLayoutSw64), smem_desc(sb + 32 * kk, 16, 512, kLayoutSw64),
                        idesc, (i | kk) != 0);
        }
        mma_commit(bar);
        mbar_wait(bar, 0, &g_peak_errors);
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        fence_after_sync();
        tmem_dealloc(tmem, TC_N);
    }
}

template <typename Kern>
int one_cta_per_sm(Kern kern, std::atomic<int> (&done)[qk::kMaxDevices])
{
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    if (done[dev].load()) return QK_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kOneCtaSmem) != cudaSuccess)
        return QK_E_CUDA;
    done[dev].store(1);
    return QK_OK;
}

// warm-up launch, then `reps` launches between two events on `stream`; elapsed milliseconds in *ms
template <typename Launch>
int timed(Launch launch_once, int reps, cudaStream_t st, double *ms)
{
    int s = launch_once();
    if (s != QK_OK) return s;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return QK_E_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return QK_E_CUDA;
    }
    cudaError_t e = cudaEventRecord(e0, st);
    for (int r = 0; r < reps && e == cudaSuccess && s == QK_OK; r++) s = launch_once();
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float f = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&f, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (s != QK_OK) return s;
    if (e != cudaSuccess) return QK_E_CUDA;
    *ms = f;
    return QK_OK;
}

std::atomic<int> g_s8_set[qk::kMaxDevices], g_tc_set[qk::kMaxDevices];

}  // namespace

extern "C" int qk_peak_mma_s8(int64_t iters, int reps, double *rate, double *ms, void *stream)
{
    if (!rate || !ms) return QK_E_NULL;
    if (iters < 1 || iters > ((int64_t)1 << 40) || reps < 1 || reps > 1000) return QK_E_SHAPE;
    int s = one_cta_per_sm(peak_s8_kernel, g_s8_set);
    if (s != QK_OK) return s;
    const int sms = qk::sm_count();
    cudaStream_t st = (cudaStream_t)stream;
    s = timed([&] { return qk::launch(peak_s8_kernel, dim3(sms), dim3(kS8Warps * 32), kOneCtaSmem, st, false,
                                      iters, 0x7eadbeef); },
              reps, st, ms);
    if (s != QK_OK) return s;
    const double ops = (double)reps * sms * kS8Warps * (double)iters * kS8Acc * (2.0 * 16 * 8 * 32);
    *rate = ops / (*ms * 1e-3) / 1e12;
    return QK_OK;
}

extern "C" int qk_peak_tcgen05_f16(int64_t iters, int reps, double *rate, double *ms, void *stream)
{
    if (!rate || !ms) return QK_E_NULL;
    if (iters < 1 || iters > ((int64_t)1 << 24) || reps < 1 || reps > 1000) return QK_E_SHAPE;
    int s = one_cta_per_sm(peak_tc_kernel, g_tc_set);
    if (s != QK_OK) return s;
    const int sms = qk::sm_count();
    cudaStream_t st = (cudaStream_t)stream;
    s = timed([&] { return qk::launch(peak_tc_kernel, dim3(sms), dim3(128), kOneCtaSmem, st, false, iters); }, reps,
              st, ms);
    if (s != QK_OK) return s;
    unsigned err = 0;
    if (cudaMemcpyFromSymbol(&err, g_peak_errors, sizeof(err)) != cudaSuccess) return QK_E_CUDA;
    if (err) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_peak_errors, &z, sizeof(z));
        return QK_E_CUDA;
    }
    const double flops = (double)reps * sms * 2.0 * (double)iters * (2.0 * TC_M * TC_N * TC_K);
    *rate = flops / (*ms * 1e-3) / 1e12;
    return QK_OK;
}
