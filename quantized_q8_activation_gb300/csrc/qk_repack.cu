// qk_repack.cu -- load-time lossless repack of GGUF Q4_K / Q5_K / Q6_K superblocks and Q8_0 blocks
// into the device layout documented in qk.h.
//
// Why: the GEMV and MMQ kernels stream weights with aligned 16-byte loads in
// which 32 lanes read 512 contiguous bytes.  GGUF interleaves a 16-byte header
// with the Q4_K codes and uses a 210-byte Q6_K stride that is not a multiple of
// 16 (minfer "15 . The CUDA backend" sec. 3.2.2: the raw 210-byte stride forced
// byte loads and capped decode; leone-cuda "CUDA kernel design" splits Q4_K
// codes from metadata).  Here the codes become planes ordered by the lanes
// that read them, the 6-bit Q4_K scales become one 24-bit record per lane,
// and Q6_K is split into four planes with no padding.
//
// One thread per superblock; runs once per weight, off the timed path.
#include "qk_common.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void copy16(uint8_t *dst, const uint8_t *src)
{
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
}

// GGUF 6-bit scale (sc) and min (m) of sub-block j from the 12 packed bytes.
__device__ __forceinline__ void q4k_unpack_scale(const uint8_t *q, int j, uint32_t &sc, uint32_t &m)
{
    if (j < 4) {
        sc = q[j] & 63u;
        m = q[j + 4] & 63u;
    } else {
        sc = (q[j + 4] & 15u) | ((uint32_t)(q[j - 4] >> 6) << 4);
        m = (uint32_t)(q[j + 4] >> 4) | ((uint32_t)(q[j] >> 6) << 4);
    }
}

__global__ void __launch_bounds__(kThreads) repack_q4k_kernel(const uint8_t *__restrict__ src, int64_t N, int B,
                                                              uint8_t *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;   // superblock id
    if (i >= N * B) return;
    const int64_t n = i / B;
    const int b = (int)(i - n * B);
    const uint8_t *blk = src + i * 144;
    uint8_t hdr[16];
    *reinterpret_cast<uint4 *>(hdr) = *reinterpret_cast<const uint4 *>(blk);

    const int s = b >> 3, nsb = min(8, B - 8 * s), G = 4 * nsb;
    uint8_t *step = dst + n * (int64_t)B * 128 + 1024 * s;
    for (int g = 0; g < 4; g++) {
        const int u = 4 * (b - 8 * s) + g;
        copy16(step + 16 * u, blk + 16 + 32 * g);
        copy16(step + 16 * G + 16 * u, blk + 16 + 32 * g + 16);
    }
    uint8_t meta[16];
    meta[0] = hdr[0], meta[1] = hdr[1], meta[2] = hdr[2], meta[3] = hdr[3];
    for (int g = 0; g < 4; g++) {
        uint32_t sc0, m0, sc1, m1;
        q4k_unpack_scale(hdr + 4, 2 * g, sc0, m0);
        q4k_unpack_scale(hdr + 4, 2 * g + 1, sc1, m1);
        const uint32_t rec = sc0 | (sc1 << 6) | (m0 << 12) | (m1 << 18);
        meta[4 + 3 * g] = (uint8_t)rec;
        meta[5 + 3 * g] = (uint8_t)(rec >> 8);
        meta[6 + 3 * g] = (uint8_t)(rec >> 16);
    }
    *reinterpret_cast<uint4 *>(dst + N * (int64_t)B * 128 + i * 16) = *reinterpret_cast<const uint4 *>(meta);
}

// Q5_K: the Q4_K planes (codes, metadata) plus the fifth-bit plane (two words per group)
__global__ void __launch_bounds__(kThreads) repack_q5k_kernel(const uint8_t *__restrict__ src, int64_t N, int B,
                                                              uint8_t *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;   // superblock id
    if (i >= N * B) return;
    const int64_t n = i / B;
    const int b = (int)(i - n * B);
    const uint8_t *blk = src + i * 176;                              // 176 = 11 x 16: aligned
    uint8_t hdr[16];
    *reinterpret_cast<uint4 *>(hdr) = *reinterpret_cast<const uint4 *>(blk);
    __align__(16) uint8_t qh[32];
    *reinterpret_cast<uint4 *>(qh) = *reinterpret_cast<const uint4 *>(blk + 16);
    *reinterpret_cast<uint4 *>(qh + 16) = *reinterpret_cast<const uint4 *>(blk + 32);
    const int64_t NB = N * (int64_t)B;

    const int s = b >> 3, nsb = min(8, B - 8 * s), G = 4 * nsb;
    uint8_t *step = dst + n * (int64_t)B * 128 + 1024 * s;
    __align__(16) uint32_t fb[8];
    for (int g = 0; g < 4; g++) {
        const int u = 4 * (b - 8 * s) + g;
        copy16(step + 16 * u, blk + 48 + 32 * g);
        copy16(step + 16 * G + 16 * u, blk + 48 + 32 * g + 16);
        uint32_t rlo = 0, rhi = 0;
        for (int l = 0; l < 32; l++) {
            const int sh = 8 * (l & 3) + (l >> 2);
            rlo |= (uint32_t)((qh[l] >> (2 * g)) & 1) << sh;
            rhi |= (uint32_t)((qh[l] >> (2 * g + 1)) & 1) << sh;
        }
        fb[2 * g] = rlo;
        fb[2 * g + 1] = rhi;
    }
    copy16(dst + NB * 128 + i * 32, reinterpret_cast<const uint8_t *>(fb));
    copy16(dst + NB * 128 + i * 32 + 16, reinterpret_cast<const uint8_t *>(fb + 4));
    uint8_t meta[16];
    meta[0] = hdr[0], meta[1] = hdr[1], meta[2] = hdr[2], meta[3] = hdr[3];
    for (int g = 0; g < 4; g++) {
        uint32_t sc0, m0, sc1, m1;
        q4k_unpack_scale(hdr + 4, 2 * g, sc0, m0);
        q4k_unpack_scale(hdr + 4, 2 * g + 1, sc1, m1);
        const uint32_t rec = sc0 | (sc1 << 6) | (m0 << 12) | (m1 << 18);
        meta[4 + 3 * g] = (uint8_t)rec;
        meta[5 + 3 * g] = (uint8_t)(rec >> 8);
        meta[6 + 3 * g] = (uint8_t)(rec >> 16);
    }
    *reinterpret_cast<uint4 *>(dst + NB * 160 + i * 16) = *reinterpret_cast<const uint4 *>(meta);
}

// Q8_0: one thread per 34-byte block (2-byte aligned): codes to the codes plane, d to the d plane.
// B here counts 32-value blocks per row.
__global__ void __launch_bounds__(kThreads) repack_q80_kernel(const uint8_t *__restrict__ src, int64_t N, int B,
                                                              uint8_t *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;   // block id
    if (i >= N * B) return;
    __align__(16) uint16_t blk[17];
    const uint16_t *s16 = reinterpret_cast<const uint16_t *>(src + i * 34);
    for (int k = 0; k < 17; k++) blk[k] = s16[k];
    __align__(16) uint8_t codes[32];
    for (int k = 0; k < 32; k++) codes[k] = reinterpret_cast<const uint8_t *>(blk)[2 + k];
    copy16(dst + i * 32, codes);
    copy16(dst + i * 32 + 16, codes + 16);
    *reinterpret_cast<uint16_t *>(dst + N * (int64_t)B * 32 + i * 2) = blk[0];
}

// Q2_K (84-byte blocks, 4-byte aligned) and Q3_K (110-byte blocks, 2-byte aligned): one thread per
// superblock, staged through registers; codes in the lane order of the step, scale records in lane
// order (Q3_K: the 6-bit scales unpacked to int8 minus 32), then the per-type planes
__device__ __forceinline__ void q23_codes(const uint8_t *qs, int64_t n, int b, int B, uint8_t *dst)
{
    const int s = b >> 3;
    uint8_t *step = dst + n * (int64_t)B * 64 + 512 * s;
    for (int p = 0; p < 4; p++) {
        const int hn = p >> 1, e = p & 1, u = 4 * (b - 8 * s) + p;
        __align__(16) uint8_t c[16];
        for (int k = 0; k < 16; k++) c[k] = qs[32 * hn + 16 * e + k];
        copy16(step + 16 * u, c);
    }
}

__global__ void __launch_bounds__(kThreads) repack_q2k_kernel(const uint8_t *__restrict__ src, int64_t N, int B,
                                                              uint8_t *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= N * B) return;
    const int64_t n = i / B;
    const int b = (int)(i - n * B);
    __align__(16) uint32_t blk[21];
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(src + i * 84);
    for (int k = 0; k < 21; k++) blk[k] = s32[k];
    const uint8_t *bb = reinterpret_cast<const uint8_t *>(blk);
    const int64_t NB = N * (int64_t)B;
    q23_codes(bb + 16, n, b, B, dst);
    __align__(16) uint8_t sc[16];
    for (int p = 0; p < 4; p++)
        for (int t = 0; t < 4; t++) sc[4 * p + t] = bb[8 * (p >> 1) + 2 * t + (p & 1)];
    copy16(dst + NB * 64 + i * 16, sc);
    *reinterpret_cast<uint32_t *>(dst + NB * 80 + i * 4) = blk[20];
}

__device__ __forceinline__ int q3k_scale(const uint8_t *sc12, int s)
{
    const int lo = s < 8 ? (sc12[s] & 15) : (sc12[s - 8] >> 4);
    const int hi = (sc12[8 + (s & 3)] >> (2 * (s >> 2))) & 3;
    return (lo | (hi << 4)) - 32;
}

__global__ void __launch_bounds__(kThreads) repack_q3k_kernel(const uint8_t *__restrict__ src, int64_t N, int B,
                                                              uint8_t *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= N * B) return;
    const int64_t n = i / B;
    const int b = (int)(i - n * B);
    __align__(16) uint16_t blk[56];
    const uint16_t *s16 = reinterpret_cast<const uint16_t *>(src + i * 110);
    for (int k = 0; k < 55; k++) blk[k] = s16[k];
    const uint8_t *bb = reinterpret_cast<const uint8_t *>(blk);
    const int64_t NB = N * (int64_t)B;
    q23_codes(bb + 32, n, b, B, dst);
    copy16(dst + NB * 64 + i * 32, bb);
    copy16(dst + NB * 64 + i * 32 + 16, bb + 16);
    __align__(16) uint8_t sc[16];
    for (int p = 0; p < 4; p++)
        for (int t = 0; t < 4; t++) sc[4 * p + t] = (uint8_t)(int8_t)q3k_scale(bb + 96, 8 * (p >> 1) + 2 * t + (p & 1));
    copy16(dst + NB * 96 + i * 16, sc);
    *reinterpret_cast<uint16_t *>(dst + NB * 112 + i * 2) = blk[54];
}

__global__ void __launch_bounds__(kThreads) repack_q6k_kernel(const uint8_t *__restrict__ src, int64_t N, int B,
                                                              uint8_t *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= N * B) return;
    const int64_t n = i / B;
    const int b = (int)(i - n * B);
    // 210-byte blocks are only 2-byte aligned: stage through registers
    __align__(16) uint8_t blk[224];
    const uint16_t *s16 = reinterpret_cast<const uint16_t *>(src + i * 210);
    for (int k = 0; k < 105; k++) reinterpret_cast<uint16_t *>(blk)[k] = s16[k];

    const int s = b >> 3, nsb = min(8, B - 8 * s), L = 4 * nsb;
    const int64_t NB = N * (int64_t)B;
    uint8_t *step = dst + n * (int64_t)B * 128 + 1024 * s;
    __align__(16) uint8_t sc[16];
    for (int p = 0; p < 4; p++) {
        const int h = p >> 1, e = p & 1, u = 4 * (b - 8 * s) + p;
        copy16(step + 16 * u, blk + 64 * h + 16 * e);
        copy16(step + 16 * L + 16 * u, blk + 64 * h + 32 + 16 * e);
        for (int t = 0; t < 4; t++) sc[4 * p + t] = blk[192 + 8 * h + e + 2 * t];
    }
    for (int k = 0; k < 4; k++) copy16(dst + NB * 128 + i * 64 + 16 * k, blk + 128 + 16 * k);
    copy16(dst + NB * 192 + i * 16, sc);
    *reinterpret_cast<uint16_t *>(dst + NB * 208 + i * 2) = *reinterpret_cast<const uint16_t *>(blk + 208);
}

}  // namespace

extern "C" int qk_repacked_bytes(int qtype, int64_t N, int64_t K, size_t *bytes)
{
    if (!bytes) return QK_E_NULL;
    if (qtype < QK_TYPE_Q4_K || qtype > QK_TYPE_Q3_K) return QK_E_TYPE;
    if (N < 1 || K < 256 || K % 256 != 0) return QK_E_SHAPE;
    static const size_t per[7] = {0, 144, 210, 176, 272, 84, 114};     // device bytes per 256 weights
    const size_t per256 = per[qtype];
    *bytes = (size_t)N * (size_t)(K / 256) * per256;
    return QK_OK;
}

extern "C" int qk_repack(int qtype, const void *gguf, int64_t N, int64_t K, void *dst, void *stream)
{
    if (qtype < QK_TYPE_Q4_K || qtype > QK_TYPE_Q3_K) return QK_E_TYPE;
    if (N < 1 || K < 256 || K % 256 != 0 || K / 256 > (1 << 24)) return QK_E_SHAPE;
    if (!gguf || !dst) return QK_E_NULL;
    if (!qk::aligned(gguf, 16) || !qk::aligned(dst, 16)) return QK_E_ALIGN;
    size_t bytes = 0;
    qk_repacked_bytes(qtype, N, K, &bytes);
    const size_t gguf_bytes = qtype == QK_TYPE_Q3_K ? (size_t)N * (size_t)(K / 256) * 110 : bytes;
    if (qk::overlaps(gguf, gguf_bytes, dst, bytes)) return QK_E_ALIAS;
    const int B = (int)(K / (qtype == QK_TYPE_Q8_0 ? 32 : 256));     // repack units per row
    const int64_t nsb = N * B;
    const int64_t grid = (nsb + kThreads - 1) / kThreads;
    if (grid > 0x7fffffffLL) return QK_E_SHAPE;
    auto kern = qtype == QK_TYPE_Q4_K   ? repack_q4k_kernel
                : qtype == QK_TYPE_Q5_K ? repack_q5k_kernel
                : qtype == QK_TYPE_Q8_0 ? repack_q80_kernel
                : qtype == QK_TYPE_Q2_K ? repack_q2k_kernel
                : qtype == QK_TYPE_Q3_K ? repack_q3k_kernel
                                        : repack_q6k_kernel;
    return qk::launch(kern, dim3((unsigned)grid), dim3(kThreads), 0, (cudaStream_t)stream, false,
                      static_cast<const uint8_t *>(gguf), N, B, static_cast<uint8_t *>(dst));
}
