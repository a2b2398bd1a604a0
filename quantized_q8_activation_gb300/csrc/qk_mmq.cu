// qk_mmq.cu -- prefill contraction Y[M][N] = X_q8 . W_q4k^T (+ R).
//
// Integer-exact tensor-core MMQ: the raw 4-bit Q4_K codes and the int8 q8_1
// codes are the MMA operands; each 32-value sub-block's int32 products are
// scaled by d_a * d * sc and the min term d_a * sum(q_a) * dmin * m is
// subtracted, in binary32, outside the integer accumulation (minfer
// "15 . The CUDA backend" sec. 2.3: weights stay quantized, raw block bytes
// are staged to shared memory and decoded in registers next to the
// mma.m16n8k32 int8 instruction, float scales folded outside the integer
// loop).
//
// Tile: 64 activation rows x 128 weight rows per CTA (8 warps, 2 x 4, each
// 32 x 32), one 256-value superblock per pipeline stage, two stages of
// cp.async staging.  The weight tile is staged straight from the repacked
// planes (two 64-byte runs of codes and the 16-byte scale record per row).
#include "qk_common.cuh"

#include <atomic>

namespace {

constexpr int BM = 64, BN = 128, kThreads = 256;
constexpr int A_STRIDE = 272;                 // 256 codes + 16 pad: conflict-free fragment reads
constexpr int W_STRIDE = 144;                 // 128 codes + 16 meta
constexpr int A_BYTES = BM * A_STRIDE;        // 17408
constexpr int W_BYTES = BN * W_STRIDE;        // 18432
constexpr int STAGE = A_BYTES + W_BYTES;      // 35840
constexpr int SIDE_W = BN * 8 * 8;            // float2 {d*sc, dmin*m} per (row, sub-block)
constexpr int SIDE_A = BM * 8 * 8;            // float2 {d_a, d_a*sum q_a} per (row, sub-block)
constexpr int SMEM = 2 * STAGE + SIDE_W + SIDE_A;

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *g, int bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void mma_s8(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// issue the cp.async copies of superblock sb into stage buffer `st`
__device__ __forceinline__ void load_stage(uint8_t *smem, int st, const uint8_t *__restrict__ w,
                                           const int8_t *__restrict__ codes, int64_t M, int64_t N, int64_t K,
                                           int64_t m0, int64_t n0, int sb)
{
    const int B = (int)(K >> 8);
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem + st * STAGE);
    // activation: 64 rows x 256 bytes = 1024 chunks
    for (int i = threadIdx.x; i < BM * 16; i += kThreads) {
        const int r = i >> 4, c = i & 15;
        const int64_t m = m0 + r;
        const bool ok = m < M;
        const int8_t *src = codes + (ok ? m : 0) * K + (int64_t)sb * 256 + 16 * c;
        cp_async16(sbase + r * A_STRIDE + 16 * c, src, ok ? 16 : 0);
    }
    // weights: 128 rows x (4 half-0 chunks, 4 half-1 chunks, 1 meta chunk)
    const int s = sb >> 3, nsb = min(8, B - 8 * s), G = 4 * nsb, loc = sb - 8 * s;
    for (int i = threadIdx.x; i < BN * 9; i += kThreads) {
        const int r = i / 9, c = i - 9 * r;
        const int64_t n = n0 + r;
        const bool ok = n < N;
        const int64_t nn = ok ? n : 0;
        const uint8_t *src;
        if (c < 4)
            src = w + nn * B * 128 + 1024 * s + 16 * (4 * loc + c);
        else if (c < 8)
            src = w + nn * B * 128 + 1024 * s + 16 * G + 16 * (4 * loc + c - 4);
        else
            src = w + N * (int64_t)B * 128 + (nn * B + sb) * 16;
        cp_async16(sbase + A_BYTES + r * W_STRIDE + 16 * c, src, ok ? 16 : 0);
    }
}

__global__ void __launch_bounds__(kThreads) mmq_q4k_kernel(const uint8_t *__restrict__ w,
                                                           const int8_t *__restrict__ codes,
                                                           const __half2 *__restrict__ scales, int64_t M,
                                                           int64_t N, int64_t K, const float *residual, float *y)
{
    extern __shared__ __align__(16) uint8_t smem[];
    float2 *side_w = reinterpret_cast<float2 *>(smem + 2 * STAGE);
    float2 *side_a = reinterpret_cast<float2 *>(smem + 2 * STAGE + SIDE_W);
    const int B = (int)(K >> 8);
    const int64_t n0 = (int64_t)blockIdx.x * BN, m0 = (int64_t)blockIdx.y * BM;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wm = warp >> 2, wn = warp & 3;     // warp tile origin: rows 32*wm, cols 32*wn
    const int g = lane >> 2, t = lane & 3;

    qk::pdl_wait();
    qk::pdl_launch_dependents();

    float facc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; i++)
#pragma unroll
        for (int j = 0; j < 4; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) facc[i][j][e] = 0.0f;

    load_stage(smem, 0, w, codes, M, N, K, m0, n0, 0);
    cp_commit();
    for (int sb = 0; sb < B; sb++) {
        const int st = sb & 1;
        if (sb + 1 < B) load_stage(smem, st ^ 1, w, codes, M, N, K, m0, n0, sb + 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const uint8_t *sa = smem + st * STAGE;
        const uint8_t *sw = sa + A_BYTES;
        // side data of this superblock
        for (int i = threadIdx.x; i < BN * 8; i += kThreads) {
            const int r = i >> 3, j = i & 7;
            const uint32_t *mt = reinterpret_cast<const uint32_t *>(sw + r * W_STRIDE + 128);
            const float d = __half2float(__ushort_as_half((unsigned short)(mt[0] & 0xffffu)));
            const float dmin = __half2float(__ushort_as_half((unsigned short)(mt[0] >> 16)));
            const uint8_t *rb = sw + r * W_STRIDE + 128 + 4 + 3 * (j >> 1);
            const uint32_t rec = (uint32_t)rb[0] | ((uint32_t)rb[1] << 8) | ((uint32_t)rb[2] << 16);
            const uint32_t sc = (j & 1) ? (rec >> 6) & 63u : rec & 63u;
            const uint32_t mn = (j & 1) ? (rec >> 18) & 63u : (rec >> 12) & 63u;
            side_w[i] = make_float2(d * (float)sc, dmin * (float)mn);
        }
        for (int i = threadIdx.x; i < BM * 8; i += kThreads) {
            const int r = i >> 3, j = i & 7;
            const int64_t m = m0 + r;
            float d = 0.0f, S = 0.0f;
            if (m < M) {
                const uint32_t *q = reinterpret_cast<const uint32_t *>(sa + r * A_STRIDE + 32 * j);
                int s = 0;
#pragma unroll
                for (int k = 0; k < 8; k++) s = qk::dp4a_ss(q[k], 0x01010101u, s);
                d = __low2float(scales[m * (K >> 5) + (int64_t)sb * 8 + j]);
                S = d * (float)s;
            }
            side_a[i] = make_float2(d, S);
        }
        __syncthreads();

#pragma unroll
        for (int gq = 0; gq < 4; gq++) {
            // weight fragments for both sub-blocks of group gq: column g of each n8 tile
            uint32_t blo[4][2], bhi[4][2];
#pragma unroll
            for (int nt = 0; nt < 4; nt++) {
                const uint8_t *row = sw + (32 * wn + 8 * nt + g) * W_STRIDE;
                const uint32_t h0 = *reinterpret_cast<const uint32_t *>(row + 16 * gq + 4 * t);
                const uint32_t h1 = *reinterpret_cast<const uint32_t *>(row + 64 + 16 * gq + 4 * t);
                blo[nt][0] = h0 & 0x0F0F0F0Fu, blo[nt][1] = h1 & 0x0F0F0F0Fu;
                bhi[nt][0] = (h0 >> 4) & 0x0F0F0F0Fu, bhi[nt][1] = (h1 >> 4) & 0x0F0F0F0Fu;
            }
#pragma unroll
            for (int hs = 0; hs < 2; hs++) {
                const int j = 2 * gq + hs;
#pragma unroll
                for (int mt = 0; mt < 2; mt++) {
                    const uint8_t *ar = sa + (32 * wm + 16 * mt + g) * A_STRIDE + 32 * j + 4 * t;
                    const uint32_t a0 = *reinterpret_cast<const uint32_t *>(ar);
                    const uint32_t a1 = *reinterpret_cast<const uint32_t *>(ar + 8 * A_STRIDE);
                    const uint32_t a2 = *reinterpret_cast<const uint32_t *>(ar + 16);
                    const uint32_t a3 = *reinterpret_cast<const uint32_t *>(ar + 8 * A_STRIDE + 16);
                    const float2 sa0 = side_a[(32 * wm + 16 * mt + g) * 8 + j];
                    const float2 sa1 = side_a[(32 * wm + 16 * mt + g + 8) * 8 + j];
#pragma unroll
                    for (int nt = 0; nt < 4; nt++) {
                        int c[4] = {0, 0, 0, 0};
                        if (hs == 0)
                            mma_s8(c, a0, a1, a2, a3, blo[nt][0], blo[nt][1]);
                        else
                            mma_s8(c, a0, a1, a2, a3, bhi[nt][0], bhi[nt][1]);
                        const float2 w0 = side_w[(32 * wn + 8 * nt + 2 * t) * 8 + j];
                        const float2 w1 = side_w[(32 * wn + 8 * nt + 2 * t + 1) * 8 + j];
                        float *f = facc[mt][nt];
                        f[0] = fmaf(sa0.x * w0.x, (float)c[0], f[0]);
                        f[0] = fmaf(-sa0.y, w0.y, f[0]);
                        f[1] = fmaf(sa0.x * w1.x, (float)c[1], f[1]);
                        f[1] = fmaf(-sa0.y, w1.y, f[1]);
                        f[2] = fmaf(sa1.x * w0.x, (float)c[2], f[2]);
                        f[2] = fmaf(-sa1.y, w0.y, f[2]);
                        f[3] = fmaf(sa1.x * w1.x, (float)c[3], f[3]);
                        f[3] = fmaf(-sa1.y, w1.y, f[3]);
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_wait<0>();

#pragma unroll
    for (int mt = 0; mt < 2; mt++)
#pragma unroll
        for (int nt = 0; nt < 4; nt++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int64_t m = m0 + 32 * wm + 16 * mt + g + (e >> 1) * 8;
                const int64_t n = n0 + 32 * wn + 8 * nt + 2 * t + (e & 1);
                if (m < M && n < N) {
                    const size_t o = (size_t)m * N + n;
                    const float v = facc[mt][nt][e];
                    y[o] = residual ? __fadd_rn(v, residual[o]) : v;
                }
            }
}

}  // namespace

extern "C" int qk_mmq_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes)
{
    if (!bytes) return QK_E_NULL;
    if (M < 0 || N < 1 || K < 256 || K % 256 != 0) return QK_E_SHAPE;
    *bytes = 0;
    return QK_OK;
}

extern "C" int qk_mmq_q4k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N, int64_t K,
                          const float *residual, float *y, void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream)
{
    (void)workspace;
    (void)workspace_bytes;
    if (M < 0 || N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || M > 0x7fffffffLL) return QK_E_SHAPE;
    if (M == 0) return QK_OK;
    if (!w || !codes || !scales || !y) return QK_E_NULL;
    if (!qk::aligned(w, 16) || !qk::aligned(codes, 16) || !qk::aligned(scales, 16) || !qk::aligned(y, 4) ||
        (residual && !qk::aligned(residual, 4)))
        return QK_E_ALIGN;
    size_t wbytes = 0;
    qk_repacked_bytes(QK_TYPE_Q4_K, N, K, &wbytes);
    const size_t ybytes = (size_t)M * N * 4, cbytes = (size_t)M * K, sbytes = (size_t)M * (K / 32) * 4;
    if (qk::overlaps(y, ybytes, w, wbytes) || qk::overlaps(y, ybytes, codes, cbytes) ||
        qk::overlaps(y, ybytes, scales, sbytes) || (residual != y && qk::overlaps(y, ybytes, residual, ybytes)))
        return QK_E_ALIAS;
    static std::atomic<int> smem_set{0};
    if (!smem_set.load()) {
        if (cudaFuncSetAttribute(mmq_q4k_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess ||
            qk::max_carveout(mmq_q4k_kernel) != cudaSuccess)
            return QK_E_CUDA;
        smem_set.store(1);
    }
    const int64_t gx = (N + BN - 1) / BN, gy = (M + BM - 1) / BM;
    if (gy > 65535) return QK_E_SHAPE;
    return qk::launch(mmq_q4k_kernel, dim3((unsigned)gx, (unsigned)gy), dim3(kThreads), SMEM, (cudaStream_t)stream,
                      (flags & QK_LAUNCH_PDL) != 0, static_cast<const uint8_t *>(w), codes,
                      static_cast<const __half2 *>(scales), M, N, K, residual, y);
}
