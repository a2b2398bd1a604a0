// qk_quantize.cu -- f32 activations -> q8_1 blocks.
//
// Method: leone-cuda "CUDA kernel design" (a q8_1 block holds 32 signed
// codes, an f16 scale and an f16 source sum; the activation is quantized once
// per GEMV input) with d = amax/127 and s = d*sum(q).  Each lane handles four
// consecutive values (one 16-byte load), eight lanes one 32-value block; the
// block max and the integer code sum are exact 8-lane shuffle reductions.
// HBM-bound: 4 bytes read and 1.125 bytes written per value.
#include "qk_common.cuh"

#include <atomic>

namespace {

constexpr int kThreads = 256;              // 32 q8_1 blocks per CTA

__global__ void __launch_bounds__(kThreads) quantize_q8_1_kernel(const float *__restrict__ x, int64_t ldx,
                                                                 int64_t nblocks, int nb_row,
                                                                 int8_t *__restrict__ codes,
                                                                 __half2 *__restrict__ scales, int64_t K)
{
    qk::pdl_launch_dependents();            // let the consumer start its weight prefetch
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * (kThreads / 8) + (threadIdx.x >> 3);   // q8_1 block id
    const bool live = blk < nblocks;
    const int64_t m = live ? blk / nb_row : 0;
    const int b = live ? (int)(blk - m * nb_row) : 0;
    const int sub = lane & 7;               // lane within the block's 8-lane group
    const float *src = x + m * ldx + 32 * b + 4 * sub;
    // x may come from the previous kernel: read it only after the wait, but request its
    // lines into L2 now (the first and last lane of a block cover the block's 128 bytes);
    // L2 is where the producer's stores land, so the reads after the wait are current
    if (live && (sub == 0 || sub == 7)) qk::prefetch_l2(src);
    qk::pdl_wait();
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) v = *reinterpret_cast<const float4 *>(src);
    float d;
    int sum;
    const uint32_t packed = qk::q81_quant8(v, d, sum);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    if (live) {
        *reinterpret_cast<uint32_t *>(codes + m * K + 32 * b + 4 * sub) = packed;
        if (sub == 0) scales[blk] = __halves2half2(qk::f16_sat(d), qk::q81_sum_f16(d, sum));
    }
}

}  // namespace

extern "C" int qk_q8_1_bytes(int64_t M, int64_t K, size_t *codes_bytes, size_t *scales_bytes)
{
    if (!codes_bytes || !scales_bytes) return QK_E_NULL;
    if (M < 0 || K <= 0 || K % 32 != 0) return QK_E_SHAPE;
    *codes_bytes = (size_t)M * (size_t)K;
    *scales_bytes = (size_t)M * (size_t)(K / 32) * 4;
    return QK_OK;
}

extern "C" int qk_quantize_q8_1(const float *x, int64_t ldx, int64_t M, int64_t K, int8_t *codes,
                                void *scales, unsigned flags, void *stream)
{
    if (M < 0 || K <= 0 || K % 32 != 0 || ldx < K || K > (int64_t)1 << 30) return QK_E_SHAPE;
    if (M == 0) return QK_OK;
    if (!x || !codes || !scales) return QK_E_NULL;
    if (!qk::aligned(x, 16) || ldx % 4 != 0 || !qk::aligned(codes, 16) || !qk::aligned(scales, 16))
        return QK_E_ALIGN;
    const size_t xbytes = ((size_t)(M - 1) * (size_t)ldx + (size_t)K) * 4;
    const size_t cbytes = (size_t)M * (size_t)K, sbytes = (size_t)M * (size_t)(K / 32) * 4;
    if (qk::overlaps(x, xbytes, codes, cbytes) || qk::overlaps(x, xbytes, scales, sbytes) ||
        qk::overlaps(codes, cbytes, scales, sbytes))
        return QK_E_ALIAS;
    static std::atomic<int> carveout_set[qk::kMaxDevices];          // per device
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    if (!carveout_set[dev].load(std::memory_order_relaxed)) {
        if (qk::max_carveout(quantize_q8_1_kernel) != cudaSuccess) return QK_E_CUDA;
        carveout_set[dev].store(1, std::memory_order_relaxed);
    }
    const int nb_row = (int)(K / 32);
    const int64_t nblocks = M * nb_row;
    const int64_t grid = (nblocks + kThreads / 8 - 1) / (kThreads / 8);
    if (grid > 0x7fffffffLL) return QK_E_SHAPE;
    return qk::launch(quantize_q8_1_kernel, dim3((unsigned)grid), dim3(kThreads), 0, (cudaStream_t)stream,
                      (flags & QK_LAUNCH_PDL) != 0, x, ldx, nblocks, nb_row, codes,
                      reinterpret_cast<__half2 *>(scales), K);
}
