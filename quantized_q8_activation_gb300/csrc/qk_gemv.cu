// qk_gemv.cu -- decode GEMV y = x_q8 . W^T (+ r) for M = 1..8 activation rows
// over a repacked Q4_K or Q6_K weight.
//
// Design (GB300, HBM-bound):
//  - Persistent grid, one CTA of 16 warps per SM.  Warp w of the grid owns
//    output rows w, w + W, w + 2W, ... and walks each row in steps of up to
//    8 superblocks; in a step every lane reads 16-byte chunks so a warp load
//    covers 512 contiguous bytes of the repacked code plane (qk.h layout).
//  - Weight loads for the next two steps are in flight while the current
//    step is computed (ld.global.nc, L1 no-allocate).  With QK_LAUNCH_PDL the
//    first two steps are issued before griddepcontrol.wait, so weight
//    streaming overlaps the tail of the previous kernel.
//  - The q8_1 activation (M x K codes) is staged once per CTA in shared
//    memory with a 16-byte-chunk XOR swizzle that keeps the lanes' 16-byte
//    reads conflict free; per 32-value block the CTA also stores d_a and the
//    exact d_a * sum(q_a) (Q4_K) or the 16-value code sums (Q6_K).
//  - Integer dots with dp4a (int32, exact per block), weight scales decoded
//    in registers, binary32 fold per 32-value (Q4_K) / 16-value (Q6_K)
//    block, per-lane accumulators combined by a fixed xor-shuffle tree, the
//    residual added in binary32 as the row is written.
// Prior art: minfer "15 . The CUDA backend" sec. 3.2.5 (MMVQ, dp4a over q8
// activations; multi-token in-block loop), leone-cuda "CUDA kernel design"
// (four warps per row, 16 lanes per superblock, fixed reduction order),
// cajeta.dev "xpu walkthrough" sec. 4.2 (one pass over a weight row serves
// the batch's activation columns).
#include "qk_common.cuh"

#include <atomic>

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

// 16-byte chunk c of an activation row lives at chunk position swz(c)
__device__ __forceinline__ int swz(int c) { return c ^ ((c >> 2) & 7); }

__device__ __forceinline__ uint4 lds16(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// --------------------------------------------------------------- staging

// Q4_K side data per (m, 32-block): {d_a, d_a * sum(q_a)}; both exact in f32
template <int M>
__device__ void stage_act_q4k(const int8_t *__restrict__ codes, const __half2 *__restrict__ scales, int K,
                              uint8_t *s_codes, float2 *s_sc)
{
    const int nchunk = K >> 4;
    for (int i = threadIdx.x; i < M * nchunk; i += kThreads) {
        const int m = i / nchunk, c = i - m * nchunk;
        const uint4 v = *reinterpret_cast<const uint4 *>(codes + (size_t)m * K + 16 * c);
        *reinterpret_cast<uint4 *>(s_codes + (size_t)m * K + 16 * swz(c)) = v;
    }
    const int nb = K >> 5;
    for (int i = threadIdx.x; i < M * nb; i += kThreads) {
        const int m = i / nb, b = i - m * nb;
        const uint4 *p = reinterpret_cast<const uint4 *>(codes + (size_t)m * K + 32 * b);
        const uint4 a = p[0], c = p[1];
        int s = 0;
        s = qk::dp4a_ss(a.x, 0x01010101u, s), s = qk::dp4a_ss(a.y, 0x01010101u, s);
        s = qk::dp4a_ss(a.z, 0x01010101u, s), s = qk::dp4a_ss(a.w, 0x01010101u, s);
        s = qk::dp4a_ss(c.x, 0x01010101u, s), s = qk::dp4a_ss(c.y, 0x01010101u, s);
        s = qk::dp4a_ss(c.z, 0x01010101u, s), s = qk::dp4a_ss(c.w, 0x01010101u, s);
        const float d = __low2float(scales[(size_t)m * nb + b]);
        s_sc[m * nb + b] = make_float2(d, d * (float)s);
    }
}

// Q6_K side data: d_a per (m, 32-block) and 32 * sum(q_a) per (m, 16-block)
template <int M>
__device__ void stage_act_q6k(const int8_t *__restrict__ codes, const __half2 *__restrict__ scales, int K,
                              uint8_t *s_codes, float *s_d, float *s_s16)
{
    const int nchunk = K >> 4;
    for (int i = threadIdx.x; i < M * nchunk; i += kThreads) {
        const int m = i / nchunk, c = i - m * nchunk;
        const uint4 v = *reinterpret_cast<const uint4 *>(codes + (size_t)m * K + 16 * c);
        *reinterpret_cast<uint4 *>(s_codes + (size_t)m * K + 16 * swz(c)) = v;
        int s = 0;
        s = qk::dp4a_ss(v.x, 0x01010101u, s), s = qk::dp4a_ss(v.y, 0x01010101u, s);
        s = qk::dp4a_ss(v.z, 0x01010101u, s), s = qk::dp4a_ss(v.w, 0x01010101u, s);
        s_s16[i] = (float)(32 * s);
    }
    const int nb = K >> 5;
    for (int i = threadIdx.x; i < M * nb; i += kThreads) s_d[i] = __low2float(scales[i]);
}

// ------------------------------------------------------------ row reduce

template <int M>
__device__ __forceinline__ void finish_row(float (&acc)[M], int lane, int64_t n, int64_t N,
                                           const float *__restrict__ residual, float *__restrict__ y)
{
#pragma unroll
    for (int m = 0; m < M; m++) {
        float v = acc[m];
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        if (lane == m) {
            const size_t o = (size_t)m * N + n;
            y[o] = residual ? __fadd_rn(v, residual[o]) : v;
        }
        acc[m] = 0.0f;
    }
}

// ------------------------------------------------------------------ Q4_K

struct Q4Item {
    uint4 c0, c1, mt;
};

__device__ __forceinline__ void q4_load(Q4Item &it, const uint8_t *__restrict__ w, int64_t N, int B,
                                        int64_t n, int s, int lane)
{
    const int nsb = min(8, B - 8 * s), G = 4 * nsb;
    if (n < N && lane < G) {
        const uint8_t *base = w + n * (int64_t)B * 128 + 1024 * s;
        it.c0 = qk::ldg_stream16(base + 16 * lane);
        it.c1 = qk::ldg_stream16(base + 16 * G + 16 * lane);
        it.mt = qk::ldg_stream16(w + N * (int64_t)B * 128 + (n * B + 8 * s + (lane >> 2)) * 16);
    } else {
        it.c0 = it.c1 = it.mt = make_uint4(0, 0, 0, 0);
    }
}

template <int M>
__device__ __forceinline__ void q4_compute(const Q4Item &it, int s, int lane, int K, uint32_t selA, uint32_t selB,
                                           const uint8_t *s_codes, const float2 *s_sc, float (&acc)[M])
{
    // scales: d, dmin and this lane's group record (sc0 | sc1<<6 | m0<<12 | m1<<18)
    const float d = __half2float(__ushort_as_half((unsigned short)(it.mt.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(it.mt.x >> 16)));
    const uint32_t rec = __byte_perm(__byte_perm(it.mt.y, it.mt.z, selA), it.mt.w, selB);
    const float dsc0 = d * (float)(rec & 63u);
    const float dsc1 = d * (float)((rec >> 6) & 63u) * 0.0625f;      // high nibbles are read as 16*q
    const float dmm0 = dmin * (float)((rec >> 12) & 63u);
    const float dmm1 = dmin * (float)((rec >> 18) & 63u);
    const uint32_t lo[8] = {it.c0.x & 0x0F0F0F0Fu, it.c0.y & 0x0F0F0F0Fu, it.c0.z & 0x0F0F0F0Fu,
                            it.c0.w & 0x0F0F0F0Fu, it.c1.x & 0x0F0F0F0Fu, it.c1.y & 0x0F0F0F0Fu,
                            it.c1.z & 0x0F0F0F0Fu, it.c1.w & 0x0F0F0F0Fu};
    const uint32_t hi[8] = {it.c0.x & 0xF0F0F0F0u, it.c0.y & 0xF0F0F0F0u, it.c0.z & 0xF0F0F0F0u,
                            it.c0.w & 0xF0F0F0F0u, it.c1.x & 0xF0F0F0F0u, it.c1.y & 0xF0F0F0F0u,
                            it.c1.z & 0xF0F0F0F0u, it.c1.w & 0xF0F0F0F0u};
    const int c0 = 128 * s + 4 * lane;          // first activation chunk of this lane's group
    const int kb0 = 64 * s + 2 * lane;          // its first 32-value block
    const int nb = K >> 5;
#pragma unroll
    for (int m = 0; m < M; m++) {
        const uint8_t *arow = s_codes + (size_t)m * K;
        const uint4 a0 = lds16(arow + 16 * swz(c0 + 0));     // sub-block 2g, values 0..15
        const uint4 a1 = lds16(arow + 16 * swz(c0 + 1));     // sub-block 2g, values 16..31
        const uint4 a2 = lds16(arow + 16 * swz(c0 + 2));     // sub-block 2g+1, values 0..15
        const uint4 a3 = lds16(arow + 16 * swz(c0 + 3));     // sub-block 2g+1, values 16..31
        int il = 0, ih = 0;
        il = qk::dp4a_ss(lo[0], a0.x, il), il = qk::dp4a_ss(lo[1], a0.y, il);
        il = qk::dp4a_ss(lo[2], a0.z, il), il = qk::dp4a_ss(lo[3], a0.w, il);
        il = qk::dp4a_ss(lo[4], a1.x, il), il = qk::dp4a_ss(lo[5], a1.y, il);
        il = qk::dp4a_ss(lo[6], a1.z, il), il = qk::dp4a_ss(lo[7], a1.w, il);
        ih = qk::dp4a_us(hi[0], a2.x, ih), ih = qk::dp4a_us(hi[1], a2.y, ih);
        ih = qk::dp4a_us(hi[2], a2.z, ih), ih = qk::dp4a_us(hi[3], a2.w, ih);
        ih = qk::dp4a_us(hi[4], a3.x, ih), ih = qk::dp4a_us(hi[5], a3.y, ih);
        ih = qk::dp4a_us(hi[6], a3.z, ih), ih = qk::dp4a_us(hi[7], a3.w, ih);
        const float4 sc = *reinterpret_cast<const float4 *>(s_sc + (size_t)m * nb + kb0);  // d0 S0 d1 S1
        float a = acc[m];
        a = fmaf(sc.x, dsc0 * (float)il, a);
        a = fmaf(sc.z, dsc1 * (float)ih, a);
        a = fmaf(-dmm0, sc.y, a);
        a = fmaf(-dmm1, sc.w, a);
        acc[m] = a;
    }
}

template <int M>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_q4k_kernel(const uint8_t *__restrict__ w, const int8_t *__restrict__ codes,
                    const __half2 *__restrict__ scales, int64_t N, int K, const float *residual, float *y)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *s_codes = smem;
    float2 *s_sc = reinterpret_cast<float2 *>(smem + (size_t)M * K);
    const int B = K >> 8, nsteps = (B + 7) >> 3;
    const int lane = threadIdx.x & 31;
    const int64_t W = (int64_t)gridDim.x * kWarps;
    const int g = lane & 3;
    const uint32_t selA = g == 0 ? 0x3210u : g == 1 ? 0x6543u : 0x7676u;
    const uint32_t selB = g == 0 ? 0x3210u : g == 1 ? 0x3210u : g == 2 ? 0x3410u : 0x3765u;

    // item = (row n, step s); items of this warp: rows n0, n0+W, ..., each steps 0..nsteps-1
    int64_t n_cur = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    int s_cur = 0;
    int64_t n1 = n_cur, n2;
    int s1 = 0, s2;
    if (++s1 == nsteps) s1 = 0, n1 += W;
    n2 = n1, s2 = s1;
    if (++s2 == nsteps) s2 = 0, n2 += W;

    Q4Item cur, nx1, nx2;
    q4_load(cur, w, N, B, n_cur, s_cur, lane);    // weights never depend on the previous kernel
    q4_load(nx1, w, N, B, n1, s1, lane);

    qk::pdl_wait();
    stage_act_q4k<M>(codes, scales, K, s_codes, s_sc);
    __syncthreads();
    qk::pdl_launch_dependents();

    float acc[M];
#pragma unroll
    for (int m = 0; m < M; m++) acc[m] = 0.0f;

    while (n_cur < N) {
        q4_load(nx2, w, N, B, n2, s2, lane);
        if (lane < 4 * min(8, B - 8 * s_cur)) q4_compute<M>(cur, s_cur, lane, K, selA, selB, s_codes, s_sc, acc);
        if (s_cur == nsteps - 1) finish_row<M>(acc, lane, n_cur, N, residual, y);
        cur = nx1, nx1 = nx2;
        n_cur = n1, s_cur = s1, n1 = n2, s1 = s2;
        if (++s2 == nsteps) s2 = 0, n2 += W;
    }
}

// ------------------------------------------------------------------ Q6_K

struct Q6Item {
    uint4 a, b, h;
    uint32_t sc;
    uint32_t d;
};

__device__ __forceinline__ void q6_load(Q6Item &it, const uint8_t *__restrict__ w, int64_t N, int B, int64_t n,
                                        int s, int lane)
{
    const int nsb = min(8, B - 8 * s), L = 4 * nsb;
    if (n < N && lane < L) {
        const int64_t NB = N * (int64_t)B;
        const int64_t sb0 = n * B + 8 * s;                       // first superblock of the step
        const uint8_t *base = w + n * (int64_t)B * 128 + 1024 * s;
        it.a = qk::ldg_stream16(base + 16 * lane);
        it.b = qk::ldg_stream16(base + 16 * L + 16 * lane);
        it.h = qk::ldg_stream16(w + NB * 128 + sb0 * 64 + 16 * lane);
        it.sc = qk::ldg_stream4(w + NB * 192 + sb0 * 16 + 4 * lane);
        it.d = qk::ldg_stream2(w + NB * 208 + (sb0 + (lane >> 2)) * 2);
    } else {
        it.a = it.b = it.h = make_uint4(0, 0, 0, 0);
        it.sc = it.d = 0;
    }
}

template <int M>
__device__ __forceinline__ void q6_compute(const Q6Item &it, int s, int lane, int K, const uint8_t *s_codes,
                                           const float *s_d, const float *s_s16, float (&acc)[M])
{
    const float d = __half2float(__ushort_as_half((unsigned short)it.d));
    float dsc[4];
#pragma unroll
    for (int t = 0; t < 4; t++) dsc[t] = d * (float)(int)(int8_t)(it.sc >> (8 * t));
    // 6-bit codes u = low4 | high2 << 4 in [0, 63]; the -32 offset is applied with the block sums
    const uint32_t aw[4] = {it.a.x, it.a.y, it.a.z, it.a.w};
    const uint32_t bw[4] = {it.b.x, it.b.y, it.b.z, it.b.w};
    const uint32_t hw[4] = {it.h.x, it.h.y, it.h.z, it.h.w};
    uint32_t u[4][4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        u[0][j] = (aw[j] & 0x0F0F0F0Fu) | ((hw[j] << 4) & 0x30303030u);
        u[1][j] = (bw[j] & 0x0F0F0F0Fu) | ((hw[j] << 2) & 0x30303030u);
        u[2][j] = ((aw[j] >> 4) & 0x0F0F0F0Fu) | (hw[j] & 0x30303030u);
        u[3][j] = ((bw[j] >> 4) & 0x0F0F0F0Fu) | ((hw[j] >> 2) & 0x30303030u);
    }
    const int p = lane & 3, h = p >> 1, e = p & 1;
    const int cbase = 128 * s + 16 * (lane >> 2) + 8 * h + e;    // activation chunk of quarter t: cbase + 2t
    const int nb = K >> 5, nc = K >> 4;
#pragma unroll
    for (int m = 0; m < M; m++) {
        const uint8_t *arow = s_codes + (size_t)m * K;
        float a = acc[m];
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const int c = cbase + 2 * t;
            const uint4 av = lds16(arow + 16 * swz(c));
            int dot = 0;
            dot = qk::dp4a_ss(u[t][0], av.x, dot), dot = qk::dp4a_ss(u[t][1], av.y, dot);
            dot = qk::dp4a_ss(u[t][2], av.z, dot), dot = qk::dp4a_ss(u[t][3], av.w, dot);
            const float da = s_d[m * nb + (c >> 1)];
            const float f = (float)dot - s_s16[m * nc + c];          // exact: sum of (u - 32) * q_a
            a = fmaf(da * dsc[t], f, a);
        }
        acc[m] = a;
    }
}

template <int M>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_q6k_kernel(const uint8_t *__restrict__ w, const int8_t *__restrict__ codes,
                    const __half2 *__restrict__ scales, int64_t N, int K, const float *residual, float *y)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *s_codes = smem;
    float *s_s16 = reinterpret_cast<float *>(smem + (size_t)M * K);
    float *s_d = s_s16 + (size_t)M * (K >> 4);
    const int B = K >> 8, nsteps = (B + 7) >> 3;
    const int lane = threadIdx.x & 31;
    const int64_t W = (int64_t)gridDim.x * kWarps;

    int64_t n_cur = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    int s_cur = 0;
    int64_t n1 = n_cur, n2;
    int s1 = 0, s2;
    if (++s1 == nsteps) s1 = 0, n1 += W;
    n2 = n1, s2 = s1;
    if (++s2 == nsteps) s2 = 0, n2 += W;

    Q6Item cur, nx1, nx2;
    q6_load(cur, w, N, B, n_cur, s_cur, lane);
    q6_load(nx1, w, N, B, n1, s1, lane);

    qk::pdl_wait();
    stage_act_q6k<M>(codes, scales, K, s_codes, s_d, s_s16);
    __syncthreads();
    qk::pdl_launch_dependents();

    float acc[M];
#pragma unroll
    for (int m = 0; m < M; m++) acc[m] = 0.0f;

    while (n_cur < N) {
        q6_load(nx2, w, N, B, n2, s2, lane);
        if (lane < 4 * min(8, B - 8 * s_cur)) q6_compute<M>(cur, s_cur, lane, K, s_codes, s_d, s_s16, acc);
        if (s_cur == nsteps - 1) finish_row<M>(acc, lane, n_cur, N, residual, y);
        cur = nx1, nx1 = nx2;
        n_cur = n1, s_cur = s1, n1 = n2, s1 = s2;
        if (++s2 == nsteps) s2 = 0, n2 += W;
    }
}

// ------------------------------------------------------------------ host

// per (qtype, M) kernel: largest dynamic shared memory opted in so far (per process)
std::atomic<int> g_smem_set[2][8];

template <typename Kern>
int set_smem(Kern kern, std::atomic<int> &done, size_t smem)
{
    // opt in to more than 48 KB of dynamic shared memory; repeated only when a larger size is needed
    if ((int)smem <= done.load(std::memory_order_relaxed)) return QK_OK;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return QK_E_CUDA;
    int prev = done.load(std::memory_order_relaxed);
    while ((int)smem > prev && !done.compare_exchange_weak(prev, (int)smem)) {
    }
    return QK_OK;
}

typedef void (*gemv_fn)(const uint8_t *, const int8_t *, const __half2 *, int64_t, int, const float *, float *);

gemv_fn pick(int qtype, int M)
{
    static const gemv_fn q4[8] = {gemv_q4k_kernel<1>, gemv_q4k_kernel<2>, gemv_q4k_kernel<3>, gemv_q4k_kernel<4>,
                                  gemv_q4k_kernel<5>, gemv_q4k_kernel<6>, gemv_q4k_kernel<7>, gemv_q4k_kernel<8>};
    static const gemv_fn q6[8] = {gemv_q6k_kernel<1>, gemv_q6k_kernel<2>, gemv_q6k_kernel<3>, gemv_q6k_kernel<4>,
                                  gemv_q6k_kernel<5>, gemv_q6k_kernel<6>, gemv_q6k_kernel<7>, gemv_q6k_kernel<8>};
    return qtype == QK_TYPE_Q4_K ? q4[M - 1] : q6[M - 1];
}

int gemv(int qtype, const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N, int64_t K,
         const float *residual, float *y, unsigned flags, void *stream)
{
    if (M < 1 || M > 8 || N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || M * K > 163840)
        return QK_E_SHAPE;
    if (!w || !codes || !scales || !y) return QK_E_NULL;
    if (!qk::aligned(w, 16) || !qk::aligned(codes, 16) || !qk::aligned(scales, 16) || !qk::aligned(y, 4) ||
        (residual && !qk::aligned(residual, 4)))
        return QK_E_ALIGN;
    size_t wbytes = 0;
    qk_repacked_bytes(qtype, N, K, &wbytes);
    const size_t ybytes = (size_t)M * N * 4, cbytes = (size_t)M * K, sbytes = (size_t)M * (K / 32) * 4;
    if (qk::overlaps(y, ybytes, w, wbytes) || qk::overlaps(y, ybytes, codes, cbytes) ||
        qk::overlaps(y, ybytes, scales, sbytes) || (residual != y && qk::overlaps(y, ybytes, residual, ybytes)))
        return QK_E_ALIAS;
    const size_t smem = qtype == QK_TYPE_Q4_K ? (size_t)M * K + (size_t)M * (K / 32) * 8
                                              : (size_t)M * K + (size_t)M * (K / 16) * 4 + (size_t)M * (K / 32) * 4;
    gemv_fn kern = pick(qtype, (int)M);
    int st = set_smem(kern, g_smem_set[qtype == QK_TYPE_Q4_K ? 0 : 1][M - 1], smem);
    if (st != QK_OK) return st;
    const int64_t warps_needed = N;
    int64_t grid = qk::sm_count();
    const int64_t max_useful = (warps_needed + kWarps - 1) / kWarps;
    if (grid > max_useful) grid = max_useful;
    return qk::launch(kern, dim3((unsigned)grid), dim3(kThreads), smem, (cudaStream_t)stream,
                      (flags & QK_LAUNCH_PDL) != 0, static_cast<const uint8_t *>(w), codes,
                      static_cast<const __half2 *>(scales), N, (int)K, residual, y);
}

}  // namespace

extern "C" int qk_gemv_q4k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q4_K, w, codes, scales, M, N, K, residual, y, flags, stream);
}

extern "C" int qk_gemv_q6k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q6_K, w, codes, scales, M, N, K, residual, y, flags, stream);
}
