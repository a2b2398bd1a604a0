// qk_producers.cu -- the producers of GEMV/MMQ inputs with the q8_1 pack fused
// into their write-out: RMSNorm -> q8_1 and SwiGLU -> q8_1.
//
// Method: leone-cuda "CUDA kernel design" -- RMSNorm and SwiGLU write their
// dense output and its q8_1 blocks in the same kernel, so no standalone
// quantization runs before the next GEMV; RMSNorm reduces the squares in a
// fixed order and uses sqrtf (not an approximate reciprocal square root); the
// residual variant normalizes left + right.  minfer "15 . The CUDA backend"
// sec. 3.2.5 (decode producers fuse an int8 quantize epilogue so the following
// MMVQ skips its quantize launch).
//
// Both kernels quantize with the library's q8_1 block quantizer (eight lanes
// per 32-value block, four values per lane), so their codes are those of
// qk_quantize_q8_1 applied to the binary32 output they compute.
//
//  rmsnorm_q8_1_kernel: one CTA of 256 threads per row.  Thread t owns the
//    float4 chunks t, t + 256, ... of the row (kept in registers when the row
//    has at most 8 chunks per thread, re-read otherwise).  s = x (+ r),
//    ss = sum s^2 in a fixed order (per thread in chunk order, then a fixed
//    xor tree per warp, then warp 0 over the eight warp sums), then
//    inv = 1 / sqrtf(ss / K + eps) and y = (s * inv) * g, all IEEE binary32.
//  swiglu_q8_1_kernel: one thread per four output values,
//    h = (g / (1 + expf(-g))) * u in binary32 (expf is the CUDA math library's
//    accurate exponential), gate g and up u read from the two halves of the
//    gate||up GEMV output row.
#include "qk_common.cuh"

#include <atomic>

namespace {

constexpr int kThreads = 256;

// quantize one float4 per lane (eight lanes per 32-value block) and store codes, scales and,
// when asked, the binary32 values; `live` lanes hold real data, the others zeros
__device__ __forceinline__ void pack_store(float4 v, bool live, int8_t *codes, __half2 *scale, float *out)
{
    float d;
    int sum;
    const uint32_t packed = qk::q81_quant8(v, d, sum);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    if (!live) return;
    *reinterpret_cast<uint32_t *>(codes) = packed;
    if ((threadIdx.x & 7) == 0) *scale = __halves2half2(qk::f16_sat(d), qk::q81_sum_f16(d, sum));
    if (out) *reinterpret_cast<float4 *>(out) = v;
}

struct NormArgs {
    const float *x, *r, *g;
    int64_t ldx;
    float eps;
    int K;
    float *h_out, *y;
    int8_t *codes;
    __half2 *scales;
};

__device__ __forceinline__ float4 add4(float4 a, float4 b)
{
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

// U: float4 chunks per thread held in registers (0: any count, re-read from memory)
template <int U>
__global__ void __launch_bounds__(kThreads) rmsnorm_q8_1_kernel(const NormArgs a)
{
    qk::pdl_launch_dependents();
    __shared__ float s_part[kThreads / 32];
    __shared__ float s_inv;
    const int64_t m = blockIdx.x;
    const int K = a.K, nc = K >> 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *xr = a.x + m * a.ldx;
    const float *rr = a.r ? a.r + m * (int64_t)K : nullptr;
    qk::pdl_wait();                                  // x and r may come from the previous kernel

    auto load = [&](int c) -> float4 {
        float4 v = *reinterpret_cast<const float4 *>(xr + 4 * c);
        if (rr) v = add4(v, *reinterpret_cast<const float4 *>(rr + 4 * c));
        return v;
    };
    constexpr int UR = U > 0 ? U : 1;
    float4 sv[UR];
    float ss = 0.0f;
    if (U > 0) {
#pragma unroll
        for (int u = 0; u < UR; u++) {
            const int c = threadIdx.x + kThreads * u;
            sv[u] = c < nc ? load(c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < UR; u++) {
            const float4 v = sv[u];
            ss = __fadd_rn(ss, __fadd_rn(__fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y)),
                                         __fadd_rn(__fmul_rn(v.z, v.z), __fmul_rn(v.w, v.w))));
        }
    } else {
        for (int c = threadIdx.x; c < nc; c += kThreads) {
            const float4 v = load(c);
            ss = __fadd_rn(ss, __fadd_rn(__fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y)),
                                         __fadd_rn(__fmul_rn(v.z, v.z), __fmul_rn(v.w, v.w))));
        }
    }
    // fixed reduction order: xor tree in each warp, then warp 0 over the warps in index order
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (lane == 0) s_part[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = s_part[0];
        for (int w = 1; w < kThreads / 32; w++) t = __fadd_rn(t, s_part[w]);
        const float ms = __fdiv_rn(t, (float)K);
        s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
    }
    __syncthreads();
    const float inv = s_inv;

    float *yr = a.y ? a.y + m * (int64_t)K : nullptr;
    float *hr = a.h_out ? a.h_out + m * (int64_t)K : nullptr;
    int8_t *cr = a.codes + m * (int64_t)K;
    __half2 *sr = a.scales + m * (int64_t)(K >> 5);
    // every lane of a warp runs the same number of chunk rounds (the quantizer shuffles within
    // each 8-lane block); chunks past the row end quantize zeros and store nothing
    const int rounds = (nc + kThreads - 1) / kThreads;
    for (int u = 0; u < rounds; u++) {
        const int c = threadIdx.x + kThreads * u;
        const bool live = c < nc;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (U > 0) {
#pragma unroll
            for (int v = 0; v < UR; v++)
                if (v == u) s = sv[v];
        } else if (live) {
            s = load(c);
        }
        float4 y = s;
        if (live) {
            const float4 g = *reinterpret_cast<const float4 *>(a.g + 4 * c);
            y = make_float4(__fmul_rn(__fmul_rn(s.x, inv), g.x), __fmul_rn(__fmul_rn(s.y, inv), g.y),
                            __fmul_rn(__fmul_rn(s.z, inv), g.z), __fmul_rn(__fmul_rn(s.w, inv), g.w));
            if (hr) *reinterpret_cast<float4 *>(hr + 4 * c) = s;
        }
        pack_store(y, live, cr + 4 * c, sr + (c >> 3), yr ? yr + 4 * c : nullptr);
    }
}

__global__ void __launch_bounds__(kThreads) swiglu_q8_1_kernel(const float *__restrict__ gu, int64_t ld, int F,
                                                               float *__restrict__ h, int8_t *__restrict__ codes,
                                                               __half2 *__restrict__ scales)
{
    qk::pdl_launch_dependents();
    const int64_t m = blockIdx.y;
    const int c = blockIdx.x * kThreads + threadIdx.x;      // float4 chunk of the output row
    const bool live = c < (F >> 2);
    qk::pdl_wait();                                           // gu comes from the previous kernel
    float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
        const float *row = gu + m * ld;
        const float4 g = *reinterpret_cast<const float4 *>(row + 4 * c);
        const float4 u = *reinterpret_cast<const float4 *>(row + F + 4 * c);
        auto silu_mul = [](float gv, float uv) {
            return __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv))), uv);
        };
        out = make_float4(silu_mul(g.x, u.x), silu_mul(g.y, u.y), silu_mul(g.z, u.z), silu_mul(g.w, u.w));
    }
    pack_store(out, live, codes + m * F + 4 * c, scales + m * (F >> 5) + (c >> 3), h ? h + m * F + 4 * c : nullptr);
}

template <typename Kern>
int carveout_once(Kern kern, std::atomic<int> &flag)
{
    if (flag.load(std::memory_order_relaxed)) return QK_OK;
    if (qk::max_carveout(kern) != cudaSuccess) return QK_E_CUDA;
    flag.store(1, std::memory_order_relaxed);
    return QK_OK;
}

std::atomic<int> g_carve[qk::kMaxDevices][6];     // per device and kernel

}  // namespace

extern "C" int qk_rmsnorm_q8_1(const float *x, int64_t ldx, const float *r, const float *g, float eps, int64_t M,
                               int64_t K, float *h_out, float *y, int8_t *codes, void *scales, unsigned flags,
                               void *stream)
{
    if (M < 0 || K <= 0 || K % 32 != 0 || ldx < K || K > (int64_t)1 << 30 || M > 0x7fffffffLL) return QK_E_SHAPE;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return QK_E_SHAPE;           // also rejects NaN
    if (M == 0) return QK_OK;
    if (!x || !g || !codes || !scales) return QK_E_NULL;
    if (!qk::aligned(x, 16) || ldx % 4 != 0 || (r && !qk::aligned(r, 16)) || !qk::aligned(g, 16) ||
        (h_out && !qk::aligned(h_out, 16)) || (y && !qk::aligned(y, 16)) || !qk::aligned(codes, 16) ||
        !qk::aligned(scales, 16))
        return QK_E_ALIGN;
    const size_t xb = ((size_t)(M - 1) * (size_t)ldx + (size_t)K) * 4, rb = (size_t)M * K * 4, gb = (size_t)K * 4;
    const size_t cb = (size_t)M * K, sb = (size_t)M * (K / 32) * 4;
    const void *ins[3] = {x, r, g};
    const size_t inb[3] = {xb, rb, gb};
    void *outs[4] = {h_out, y, codes, scales};
    const size_t outb[4] = {rb, rb, cb, sb};
    for (int i = 0; i < 4; i++) {
        for (int j = 0; j < 3; j++)
            if (qk::overlaps(outs[i], outb[i], ins[j], inb[j])) return QK_E_ALIAS;
        for (int j = i + 1; j < 4; j++)
            if (qk::overlaps(outs[i], outb[i], outs[j], outb[j])) return QK_E_ALIAS;
    }
    NormArgs a{x, r, g, ldx, eps, (int)K, h_out, y, codes, reinterpret_cast<__half2 *>(scales)};
    const int per = (int)((K / 4 + kThreads - 1) / kThreads);
    const bool pdl = (flags & QK_LAUNCH_PDL) != 0;
    const dim3 grid((unsigned)M), block(kThreads);
    cudaStream_t st = (cudaStream_t)stream;
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    int s;
    if (per <= 1) {
        if ((s = carveout_once(rmsnorm_q8_1_kernel<1>, g_carve[dev][0])) != QK_OK) return s;
        return qk::launch(rmsnorm_q8_1_kernel<1>, grid, block, 0, st, pdl, a);
    }
    if (per <= 2) {
        if ((s = carveout_once(rmsnorm_q8_1_kernel<2>, g_carve[dev][1])) != QK_OK) return s;
        return qk::launch(rmsnorm_q8_1_kernel<2>, grid, block, 0, st, pdl, a);
    }
    if (per <= 4) {
        if ((s = carveout_once(rmsnorm_q8_1_kernel<4>, g_carve[dev][2])) != QK_OK) return s;
        return qk::launch(rmsnorm_q8_1_kernel<4>, grid, block, 0, st, pdl, a);
    }
    if (per <= 8) {
        if ((s = carveout_once(rmsnorm_q8_1_kernel<8>, g_carve[dev][3])) != QK_OK) return s;
        return qk::launch(rmsnorm_q8_1_kernel<8>, grid, block, 0, st, pdl, a);
    }
    if ((s = carveout_once(rmsnorm_q8_1_kernel<0>, g_carve[dev][4])) != QK_OK) return s;
    return qk::launch(rmsnorm_q8_1_kernel<0>, grid, block, 0, st, pdl, a);
}

extern "C" int qk_swiglu_q8_1(const float *gu, int64_t ldgu, int64_t M, int64_t F, float *h, int8_t *codes,
                              void *scales, unsigned flags, void *stream)
{
    if (M < 0 || F <= 0 || F % 32 != 0 || ldgu < 2 * F || F > (int64_t)1 << 30 || M > 65535) return QK_E_SHAPE;
    if (M == 0) return QK_OK;
    if (!gu || !codes || !scales) return QK_E_NULL;
    if (!qk::aligned(gu, 16) || ldgu % 4 != 0 || (h && !qk::aligned(h, 16)) || !qk::aligned(codes, 16) ||
        !qk::aligned(scales, 16))
        return QK_E_ALIGN;
    const size_t gb = ((size_t)(M - 1) * (size_t)ldgu + (size_t)(2 * F)) * 4, hb = (size_t)M * F * 4;
    const size_t cb = (size_t)M * F, sb = (size_t)M * (F / 32) * 4;
    if (qk::overlaps(h, hb, gu, gb) || qk::overlaps(codes, cb, gu, gb) || qk::overlaps(scales, sb, gu, gb) ||
        qk::overlaps(h, hb, codes, cb) || qk::overlaps(h, hb, scales, sb) || qk::overlaps(codes, cb, scales, sb))
        return QK_E_ALIAS;
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    int s;
    if ((s = carveout_once(swiglu_q8_1_kernel, g_carve[dev][5])) != QK_OK) return s;
    const int64_t gx = (F / 4 + kThreads - 1) / kThreads;
    return qk::launch(swiglu_q8_1_kernel, dim3((unsigned)gx, (unsigned)M), dim3(kThreads), 0, (cudaStream_t)stream,
                      (flags & QK_LAUNCH_PDL) != 0, gu, ldgu, (int)F, h, codes,
                      reinterpret_cast<__half2 *>(scales));
}
