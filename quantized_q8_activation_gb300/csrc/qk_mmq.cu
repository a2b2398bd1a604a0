// qk_mmq.cu -- prefill contraction Y[M][N] = Xq8 . W_q4k^T (+ R) on the
// sm_103a tensor cores (tcgen05, accumulator in tensor memory).
//
// Method (minfer "15 . The CUDA backend" sec. 2.3 / 3.2.6: quantized weight
// bytes go straight to the tensor cores; the activation is quantized to q8_1
// once per matmul input).  This part runs integer MMA far below its f16 rate,
// so both operands enter kind::f16 MMAs as pairs of f16 values:
//   A[m][k] = d_a * q_a = A_hi + A_lo   exactly (d_a has 11 significant bits
//             and q_a 7, so the product needs 18 <= 2 x 11 bits);
//   W[n][k] = 256 * (d_b sc_j q_w - dmin_b m_j) = W_hi + W_lo, the Q4_K weight
//             scaled by 2^8 (so that W_lo stays in the normal f16 range for
//             the weights of LLM layers), split to 2^-21 relative;
//   Y = A_hi W_hi + A_hi W_lo + A_lo W_hi   (A_lo W_lo is below 2^-21 of each
//             product and dropped), accumulated in binary32 over all of K in
//             tensor memory;  y = Y / 256 (+ R).
// The Q4_K bytes are dequantized tile by tile in shared memory right before
// the MMAs that use them; they are read from memory in their quantized form.
//
// Two kernels per call:
//  1. mmq_prep_kernel expands the q8_1 activation once per 128-row M-tile into
//     the caller's workspace, already in the tensor core's shared-memory
//     layout: per 32-value K stage a 16 KB block (A_hi and A_lo tiles, K-major
//     SWIZZLE_64B).  Every N-tile then copies these blocks instead of
//     converting the activation again.
//  2. mmq_q4k_kernel, one CTA (20 warps) per 128 x 256 output tile and per SM
//     (256 TMEM columns hold the accumulator):
//       warp 0      TMEM allocation; lane 0 issues every MMA and commit
//       warp 2      lane 0 streams the raw Q4_K bytes with 2D TMA tensor copies
//                   into a ring, per superblock: the two 64-byte runs of code
//                   bytes (256 x 64 B each: first and second 16-byte halves of
//                   its four groups) and the metadata records (256 x 16 B)
//       warps 4-19  converters: per K stage they copy the stage's A block from
//                   the workspace (cp.async, 32 bytes per thread) and, two
//                   threads per weight row, expand the Q4_K codes, scales and
//                   mins into (W_hi, W_lo) in the SWIZZLE_64B layout.  Warps
//                   4-7 then run the epilogue (TMEM lane quadrant = warp % 4)
// Stages are handed over with mbarriers (full: converters -> MMA; empty: MMA
// commit -> converters; raw: TMA bytes -> converters ->
// producer; done: last MMA commit -> epilogue).  Every wait is bounded; a wait
// that gives up sets a device error flag (qk_error_flags), and once it is set
// the other waits return after a few polls, so the kernel runs to its end.
// Before the CTA releases its tensor memory and exits, the MMA thread waits
// for its last MMAs and the producers for their last copies (bounded too), so
// nothing is left in flight.
#include "qk_common.cuh"
#include "qk_tc.cuh"

#include <cuda.h>

#include <atomic>

#ifndef QK_MMQ_NST
#define QK_MMQ_NST 3        // operand stages
#endif
#ifndef QK_MMQ_RAW
#define QK_MMQ_RAW 2        // raw weight superblocks (eight K stages each) in flight
#endif
#ifndef QK_MMQ_SBRAW
#define QK_MMQ_SBRAW 2      // raw metadata superblocks in flight
#endif
#ifndef QK_MMQ_STCS
#define QK_MMQ_STCS 0       // 1: outputs stored with the streaming (evict-first) cache operator
#endif

__device__ unsigned g_qk_errors;

namespace {

using namespace qk::tc;

constexpr int BM = 128, BN = 256, BK = 32;      // BK: one Q4_K sub-block
constexpr int NST = QK_MMQ_NST, NRAW = QK_MMQ_RAW, NSB = QK_MMQ_SBRAW;
constexpr int kThreads = 640;
constexpr int kEpiWarp0 = 4, kConvWarp0 = 4;                 // warps 4-7 convert, then run the epilogue
constexpr int kConv = 512, kConvWarps = kConv / 32;   // two converter threads per weight row
static_assert(kConv == 2 * BN && kConvWarp0 * 32 + kConv == kThreads, "two converter threads per weight row");
constexpr float kWScale = 256.0f, kWUnscale = 1.0f / 256.0f;

constexpr int ATILE = BM * BK * 2;              // 8 KB: 128 rows x 32 f16 (64 B rows), SWIZZLE_64B K-major
constexpr int WTILE = BN * BK * 2;              // 16 KB: 256 rows x 32 f16
constexpr int STAGE = 2 * ATILE + 2 * WTILE;    // A_hi | A_lo | W_hi | W_lo
constexpr int ABLOCK = 2 * ATILE;               // workspace block of one M-tile and K stage: A_hi | A_lo
// raw weight superblock: code bytes, first halves of its 4 groups 256 x 64 B | second halves 256 x 64 B
constexpr int RAW_H0 = 0, RAW_H1 = BN * 64, RAW = 2 * BN * 64;
constexpr int SBR = BN * 16;                    // raw metadata records of one superblock
constexpr int OFF_RAW = NST * STAGE;
constexpr int OFF_SBR = OFF_RAW + NRAW * RAW;
constexpr int OFF_BAR = OFF_SBR + NSB * SBR;
enum {
    B_FULL = 0,
    B_EMPTY = B_FULL + NST,
    B_RFULL = B_EMPTY + NST,
    B_REMPTY = B_RFULL + NRAW,
    B_SFULL = B_REMPTY + NRAW,
    B_SEMPTY = B_SFULL + NSB,
    B_DONE = B_SEMPTY + NSB,       // every MMA of the CTA has completed
    NBAR = B_DONE + 1
};
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_TMEM + 16 + 1024;      // + slack to align the base to 1024
static_assert(SMEM <= 232448, "shared memory plan exceeds the per-block opt-in limit");
static_assert(STAGE % 1024 == 0 && OFF_RAW % 1024 == 0 && RAW % 1024 == 0 && SBR % 1024 == 0,
              "copy destinations and swizzle atoms stay aligned");
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

// byte offset of 16-byte chunk c (< 4) of row r in a SWIZZLE_64B K-major tile (rows of 64 bytes)
__host__ __device__ constexpr uint32_t sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity) { mbar_wait(bar, parity, &g_qk_errors); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

struct MmqArgs {
    const uint8_t *wsA;     // workspace: [M-tiles][K/32] A blocks
    int64_t M, N, K;
    const float *residual;
    float *y;
};

struct MmqMaps {
    CUtensorMap wcodes;     // uint8  [N][B*128]      box 64 x 256  (code plane of the repacked weight)
    CUtensorMap meta;       // uint8  [N][B*16]       box 16 x 256  (metadata plane)
};

// 4 int8 codes -> (A_hi, A_lo) f16 pairs with A_hi + A_lo = d * q exactly
__device__ __forceinline__ void conv_a(uint32_t w4, __half2 d2, uint32_t &hi01, uint32_t &lo01, uint32_t &hi23,
                                       uint32_t &lo23)
{
    // each byte to 1024 + (q + 128) in an f16 lane, then subtract 1152
    const uint32_t x = w4 ^ 0x80808080u;
    const __half2 k1152 = u2h(0x64806480u);
    const __half2 q01 = __hsub2(u2h(__byte_perm(x, 0x64646464u, 0x5140)), k1152);
    const __half2 q23 = __hsub2(u2h(__byte_perm(x, 0x64646464u, 0x7362)), k1152);
    const __half2 h01 = __hmul2(q01, d2), h23 = __hmul2(q23, d2);
    hi01 = h2u(h01);
    hi23 = h2u(h23);
    lo01 = h2u(__hfma2(q01, d2, __hneg2(h01)));    // exact remainder d*q - hi
    lo23 = h2u(__hfma2(q23, d2, __hneg2(h23)));
}

// 4 nibbles (one per byte of x, already masked to 0..15) -> 4 weights w = q*dsc - dmm as
// (hi, lo) f16 pairs.  hi is w with its 13 low mantissa bits cleared (11 significant bits,
// exactly an f16), lo = w - hi exactly in binary32 and then rounded to f16, so hi + lo
// equals w to 2^-21 relative.
__device__ __forceinline__ void conv_w(uint32_t x, float2 dsc2, float2 ndmm2, uint32_t &hi01, uint32_t &hi23,
                                       uint32_t &lo01, uint32_t &lo23)
{
    // byte t of x as the low bits of 2^23 + q (exact), minus 2^23
    const float2 k23 = make_float2(-8388608.0f, -8388608.0f), neg1 = make_float2(-1.0f, -1.0f);
    float2 q01 = make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u)),
                             __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7441u)));
    float2 q23 = make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7442u)),
                             __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7443u)));
    q01 = __fadd2_rn(q01, k23);
    q23 = __fadd2_rn(q23, k23);
    const float2 w01 = __ffma2_rn(q01, dsc2, ndmm2), w23 = __ffma2_rn(q23, dsc2, ndmm2);
    const float2 h01 = make_float2(__uint_as_float(__float_as_uint(w01.x) & 0xFFFFE000u),
                                   __uint_as_float(__float_as_uint(w01.y) & 0xFFFFE000u));
    const float2 h23 = make_float2(__uint_as_float(__float_as_uint(w23.x) & 0xFFFFE000u),
                                   __uint_as_float(__float_as_uint(w23.y) & 0xFFFFE000u));
    const float2 l01 = __ffma2_rn(h01, neg1, w01), l23 = __ffma2_rn(h23, neg1, w23);   // exact differences
    hi01 = h2u(__floats2half2_rn(h01.x, h01.y));
    hi23 = h2u(__floats2half2_rn(h23.x, h23.y));
    lo01 = h2u(__floats2half2_rn(l01.x, l01.y));
    lo23 = h2u(__floats2half2_rn(l23.x, l23.y));
}

__device__ __forceinline__ void sts128(uint8_t *base, uint32_t off, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    *reinterpret_cast<uint4 *>(base + off) = make_uint4(x, y, z, w);
}

// ------------------------------------------------------------- prep kernel
// CTA (superblock sb, M-tile mt), 256 threads, 4 items each: item (row, j) is
// the 32-value q8_1 block j of superblock sb of activation row 128 mt + row.
// It writes the block's 32 (A_hi, A_lo) pairs into row `row` of the stage
// block of K stage 8 sb + j; rows past M are written as zeros.
__global__ void __launch_bounds__(256) mmq_prep_kernel(const int8_t *__restrict__ codes,
                                                       const __half2 *__restrict__ scales, int64_t M, int64_t K,
                                                       uint8_t *__restrict__ wsA)
{
    qk::pdl_launch_dependents();
    qk::pdl_wait();                              // codes may come from the previous kernel
    const int sb = blockIdx.x, mt = blockIdx.y;
    const int nit = (int)(K >> 5);
#pragma unroll 1
    for (int i = 0; i < 4; i++) {
        const int q = threadIdx.x + 256 * i;
        const int row = q >> 3, j = q & 7;
        const int64_t m = (int64_t)mt * BM + row;
        uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
        uint32_t dbits = 0;
        if (m < M) {
            const int8_t *src = codes + m * K + sb * 256 + 32 * j;
            a0 = *reinterpret_cast<const uint4 *>(src);
            a1 = *reinterpret_cast<const uint4 *>(src + 16);
            dbits = *reinterpret_cast<const uint32_t *>(scales + m * (K >> 5) + 8 * sb + j) & 0xffffu;
        }
        const __half dah = __ushort_as_half((unsigned short)dbits);
        const __half2 d2 = __halves2half2(dah, dah);
        const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        uint8_t *tA = wsA + ((size_t)mt * nit + 8 * sb + j) * ABLOCK;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            uint32_t hi[4], lo[4];
            conv_a(aw[2 * c], d2, hi[0], lo[0], hi[1], lo[1]);
            conv_a(aw[2 * c + 1], d2, hi[2], lo[2], hi[3], lo[3]);
            sts128(tA, sw64(row, c), hi[0], hi[1], hi[2], hi[3]);
            sts128(tA + ATILE, sw64(row, c), lo[0], lo[1], lo[2], lo[3]);
        }
    }
}

// ------------------------------------------------------------- main kernel

// Converter state of one half row across K stages: its 16 code bytes of the current
// 64-value group and the row's metadata record of the current superblock.
struct ConvState {
    uint4 c, mt;
};

// one converter thread's share of K stage `it` (operand stage st = it % NST): the 16 weights of
// half h of sub-block j = it % 8 of row `row` as (W_hi, W_lo) chunks 2h and 2h+1, then the
// stage is signalled full
__device__ __forceinline__ void convert_stage(uint8_t *smem, uint64_t *bar, ConvState &cs, const uint8_t *srcA,
                                              int it, int row, int h, int st)
{
    const int j = it & 7, sb = it >> 3, g = j >> 1, nib = j & 1;
    const int rs = sb % NRAW, ss = sb % NSB;
    if (j == 0) {
        wait_bar(&bar[B_SFULL + ss], (sb / NSB) & 1);
        cs.mt = *reinterpret_cast<const uint4 *>(smem + OFF_SBR + ss * SBR + row * 16);
        wait_bar(&bar[B_RFULL + rs], (sb / NRAW) & 1);
    }
    if (nib == 0)
        cs.c = *reinterpret_cast<const uint4 *>(smem + OFF_RAW + rs * RAW + (h ? RAW_H1 : RAW_H0) + row * 64 + 16 * g);
    if (it >= NST) wait_bar(&bar[B_EMPTY + st], ((it / NST) + 1) & 1);
    uint8_t *s0 = smem + st * STAGE;
    // the stage's activation block (A_hi | A_lo, 16 KB): 32 bytes per converter thread, in flight
    // while the weights are converted
    {
        const int ct = threadIdx.x - kConvWarp0 * 32;
        const uint8_t *src = srcA + (size_t)it * ABLOCK + 32 * ct;
        qk::cp_async16(s0 + 32 * ct, src);
        qk::cp_async16(s0 + 32 * ct + 16, src + 16);
        qk::cp_async_commit();
    }
    // this group's record: sc0 | sc1<<6 | m0<<12 | m1<<18 (sub-blocks 2g and 2g+1)
    const uint4 mt = cs.mt;
    const uint32_t rec = __byte_perm(__byte_perm(mt.y, mt.z, g == 0 ? 0x3210u : g == 1 ? 0x6543u : 0x7676u), mt.w,
                                     g == 0 ? 0x3210u : g == 1 ? 0x3210u : g == 2 ? 0x3410u : 0x3765u);
    const int sc = nib ? (int)((rec >> 6) & 63u) : (int)(rec & 63u);
    const int mm = nib ? (int)((rec >> 18) & 63u) : (int)((rec >> 12) & 63u);
    const float d = __half2float(__ushort_as_half((unsigned short)(mt.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(mt.x >> 16)));
    const float dsc = d * (float)sc * kWScale, dmm = dmin * (float)mm * kWScale;   // exact products
    const float2 dsc2 = make_float2(dsc, dsc), ndmm2 = make_float2(-dmm, -dmm);
    const uint32_t cw[4] = {cs.c.x, cs.c.y, cs.c.z, cs.c.w};
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
        uint32_t hi[4], lo[4];
        const uint32_t x0 = nib ? (cw[2 * cc] >> 4) & 0x0F0F0F0Fu : cw[2 * cc] & 0x0F0F0F0Fu;
        const uint32_t x1 = nib ? (cw[2 * cc + 1] >> 4) & 0x0F0F0F0Fu : cw[2 * cc + 1] & 0x0F0F0F0Fu;
        conv_w(x0, dsc2, ndmm2, hi[0], hi[1], lo[0], lo[1]);
        conv_w(x1, dsc2, ndmm2, hi[2], hi[3], lo[2], lo[3]);
        sts128(s0 + 2 * ATILE, sw64(row, 2 * h + cc), hi[0], hi[1], hi[2], hi[3]);
        sts128(s0 + 2 * ATILE + WTILE, sw64(row, 2 * h + cc), lo[0], lo[1], lo[2], lo[3]);
    }
    // Each lane waits for its activation copy and makes its own stores visible to the tensor
    // core (async proxy); after the warp has synchronised, one lane arrives for the whole warp.
    // A raw slot is released only after the values read from it have been consumed by the
    // arithmetic above, so no shared load can still be pending when the producer lets the next
    // TMA copy overwrite it.
    qk::cp_async_wait<0>();
    fence_proxy_async();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (j == 6) mbar_arrive(&bar[B_REMPTY + rs]);           // last read of this superblock's codes
        if (j == 0) mbar_arrive(&bar[B_SEMPTY + ss]);
        mbar_arrive(&bar[B_FULL + st]);
    }
}

__global__ void __launch_bounds__(kThreads, 1) mmq_q4k_kernel(const MmqArgs a, const __grid_constant__ MmqMaps maps)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtile = blockIdx.x;
    const int m0 = mtile * BM, n0 = blockIdx.y * BN;
    const int B = (int)(a.K >> 8), nit = 8 * B;

    qk::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; i++) mbar_init(&bar[B_FULL + i], kConvWarps), mbar_init(&bar[B_EMPTY + i], 1);
        for (int i = 0; i < NRAW; i++) mbar_init(&bar[B_RFULL + i], 1), mbar_init(&bar[B_REMPTY + i], kConvWarps);
        for (int i = 0; i < NSB; i++) mbar_init(&bar[B_SFULL + i], 1), mbar_init(&bar[B_SEMPTY + i], kConvWarps);
        mbar_init(&bar[B_DONE], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tmem_ptr, TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_ptr;
    qk::pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t sbase = smem_u32(smem);
            for (int it = 0; it < nit; it++) {
                const int st = it % NST;
                wait_bar(&bar[B_FULL + st], (it / NST) & 1);
                fence_after_sync();
                const uint32_t s0 = sbase + st * STAGE;
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {
                    const uint64_t ahi = smem_desc(s0 + 32 * kk, 16, 512, kLayoutSw64);
                    const uint64_t alo = smem_desc(s0 + ATILE + 32 * kk, 16, 512, kLayoutSw64);
                    const uint64_t whi = smem_desc(s0 + 2 * ATILE + 32 * kk, 16, 512, kLayoutSw64);
                    const uint64_t wlo = smem_desc(s0 + 2 * ATILE + WTILE + 32 * kk, 16, 512, kLayoutSw64);
                    mma_f16(tmem, ahi, whi, IDESC, (it | kk) != 0);
                    mma_f16(tmem, ahi, wlo, IDESC, 1);
                    mma_f16(tmem, alo, whi, IDESC, 1);
                }
                mma_commit(&bar[B_EMPTY + st]);
            }
            // the epilogue starts once every MMA has completed; the CTA's TMEM is released after it
            mma_commit(&bar[B_DONE]);
            wait_bar(&bar[B_DONE], 0);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ raw weight TMA producer
        if (lane == 0) {
            prefetch_tmap(&maps.wcodes);
            prefetch_tmap(&maps.meta);
            for (int sb = 0; sb < B; sb++) {
                const int ss = sb % NSB;
                if (sb >= NSB) wait_bar(&bar[B_SEMPTY + ss], ((sb / NSB) + 1) & 1);
                mbar_arrive_expect_tx(&bar[B_SFULL + ss], SBR);
                tma_load_2d(smem + OFF_SBR + ss * SBR, &maps.meta, 16 * sb, n0, &bar[B_SFULL + ss]);
                const int rs = sb % NRAW;
                if (sb >= NRAW) wait_bar(&bar[B_REMPTY + rs], ((sb / NRAW) + 1) & 1);
                uint8_t *d = smem + OFF_RAW + rs * RAW;
                // the superblock's 4 groups: first halves at 16u (u = 4 (sb - 8 s) .. +3), second at 16 G + 16u
                const int s = sb >> 3, G = 4 * min(8, B - 8 * s), u = 4 * (sb - 8 * s);
                mbar_arrive_expect_tx(&bar[B_RFULL + rs], RAW);
                tma_load_2d(d + RAW_H0, &maps.wcodes, 1024 * s + 16 * u, n0, &bar[B_RFULL + rs]);
                tma_load_2d(d + RAW_H1, &maps.wcodes, 1024 * s + 16 * G + 16 * u, n0, &bar[B_RFULL + rs]);
            }
            // teardown: every copy this thread issued has landed (normally long since consumed)
            for (int sb = B - NRAW < 0 ? 0 : B - NRAW; sb < B; sb++) wait_bar(&bar[B_RFULL + sb % NRAW], (sb / NRAW) & 1);
            for (int sb = B - NSB < 0 ? 0 : B - NSB; sb < B; sb++) wait_bar(&bar[B_SFULL + sb % NSB], (sb / NSB) & 1);
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        // --------------------------------------------------------- converters
        // Lanes 0-15 of a warp take 16 consecutive rows of half 0, lanes 16-31 the same rows of
        // half 1; a quarter warp stores 8 consecutive rows, which the 64-byte swizzle spreads over
        // all 32 banks.  Unrolled by the stage count, so the operand stage index is static.
        const int cwarp = warp - kConvWarp0;                      // 0..15
        const int row = 16 * cwarp + (lane & 15), h = lane >> 4;
        const uint8_t *srcA = a.wsA + (size_t)mtile * nit * ABLOCK;
        ConvState cs;
        cs.c = cs.mt = make_uint4(0, 0, 0, 0);
        for (int it = 0; it < nit; it += NST) {
#pragma unroll
            for (int k = 0; k < NST; k++)
                if (it + k < nit) convert_stage(smem, bar, cs, srcA, it + k, row, h, k);
        }
        if (warp < kEpiWarp0 + 4) {
            // ---------------------------------------------------------- epilogue
            // y = Y / 256 (+ R), one 32 x 32 block per pass: a thread holds row (32q + lane) of the
            // block; the block is transposed through shared memory (operand stage 0, idle once
            // every MMA has completed) so that each store writes 32 consecutive columns of one row
            wait_bar(&bar[B_DONE], 0);
            fence_after_sync();
            const uint32_t lq = (uint32_t)((warp & 3) * 32) << 16;   // TMEM lane quadrant of this warp
            float *tb_s = reinterpret_cast<float *>(smem) + (warp - kEpiWarp0) * (32 * 33);
            const int q0 = (warp & 3) * 32;
#pragma unroll 1
            for (int c = 0; c < BN / 32; c++) {
                float v[32];
                tmem_ld32(tmem + lq + 32 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; jj++) tb_s[lane * 33 + jj] = v[jj] * kWUnscale;
                __syncwarp();
                const int64_t n = n0 + 32 * c + lane;
                if (n < a.N) {
#pragma unroll 4
                    for (int r = 0; r < 32; r++) {
                        const int64_t m = m0 + q0 + r;
                        if (m < a.M) {
                            const float val = tb_s[r * 33 + lane];
                            const size_t o = (size_t)m * a.N + n;
                            const float out = a.residual ? __fadd_rn(val, a.residual[o]) : val;
                            if (QK_MMQ_STCS) __stcs(a.y + o, out);
                            else a.y[o] = out;
                        }
                    }
                }
                __syncwarp();
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static std::atomic<void *> fn{nullptr};
    void *p = fn.load();
    if (!p) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return nullptr;
        fn.store(p);
    }
    return reinterpret_cast<EncodeTiledFn>(p);
}

// 2D row-major tensor [rows][cols] of elements of the map's type, row pitch `pitch` bytes; box bx x by
bool make_map(EncodeTiledFn enc, CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t cols,
              uint64_t rows, uint64_t pitch, uint32_t bx, uint32_t by)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {bx, by};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// workspace bytes for an M x K activation: one A block per M-tile and 32-value K stage
size_t ws_bytes(int64_t M, int64_t K)
{
    const size_t mt = (size_t)((M + BM - 1) / BM);
    return mt * (size_t)(K / BK) * ABLOCK;
}

}  // namespace

extern "C" int qk_error_flags(unsigned *flags, int clear)
{
    if (!flags) return QK_E_NULL;
    if (cudaMemcpyFromSymbol(flags, g_qk_errors, sizeof(unsigned)) != cudaSuccess) return QK_E_CUDA;
    if (clear) {
        const unsigned z = 0;
        if (cudaMemcpyToSymbol(g_qk_errors, &z, sizeof(unsigned)) != cudaSuccess) return QK_E_CUDA;
    }
    return QK_OK;
}

extern "C" int qk_mmq_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes)
{
    if (!bytes) return QK_E_NULL;
    if (M < 0 || N < 1 || K < 256 || K % 256 != 0) return QK_E_SHAPE;
    *bytes = ws_bytes(M, K);
    return QK_OK;
}

extern "C" int qk_mmq_q4k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N, int64_t K,
                          const float *residual, float *y, void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream)
{
    // TMA coordinates are signed 32-bit: rows and bytes of a row stay below 2^31
    if (M < 0 || N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || M > 0x7fffffffLL || K > 0x7fffffffLL)
        return QK_E_SHAPE;
    if (M == 0) return QK_OK;
    if (!w || !codes || !scales || !y || !workspace) return QK_E_NULL;
    if (!qk::aligned(w, 16) || !qk::aligned(codes, 16) || !qk::aligned(scales, 16) || !qk::aligned(y, 4) ||
        (residual && !qk::aligned(residual, 4)) || !qk::aligned(workspace, 256))
        return QK_E_ALIGN;
    const size_t need = ws_bytes(M, K);
    if (workspace_bytes < need) return QK_E_WORKSPACE;
    size_t wbytes = 0;
    qk_repacked_bytes(QK_TYPE_Q4_K, N, K, &wbytes);
    const size_t ybytes = (size_t)M * N * 4, cbytes = (size_t)M * K, sbytes = (size_t)M * (K / 32) * 4;
    if (qk::overlaps(y, ybytes, w, wbytes) || qk::overlaps(y, ybytes, codes, cbytes) ||
        qk::overlaps(y, ybytes, scales, sbytes) || (residual != y && qk::overlaps(y, ybytes, residual, ybytes)) ||
        qk::overlaps(workspace, need, w, wbytes) || qk::overlaps(workspace, need, codes, cbytes) ||
        qk::overlaps(workspace, need, scales, sbytes) || qk::overlaps(workspace, need, y, ybytes) ||
        (residual && qk::overlaps(workspace, need, residual, ybytes)))
        return QK_E_ALIAS;
    const int64_t gx = (M + BM - 1) / BM, gy = (N + BN - 1) / BN;
    if (gx > 65535 || gy > 65535) return QK_E_SHAPE;
    if ((size_t)SMEM > qk::max_smem_optin()) return QK_E_CUDA;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return QK_E_CUDA;
    const int64_t B = K / 256;
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    MmqMaps maps;
    if (!make_map(enc, &maps.wcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb, B * 128, N, B * 128, 64, BN) ||
        !make_map(enc, &maps.meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb + N * B * 128, B * 16, N, B * 16, 16, BN))
        return QK_E_CUDA;
    static std::atomic<int> attr_set{0};
    if (!attr_set.load()) {
        if (cudaFuncSetAttribute(mmq_q4k_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess ||
            qk::max_carveout(mmq_q4k_kernel) != cudaSuccess)
            return QK_E_CUDA;
        attr_set.store(1);
    }
    uint8_t *wsA = static_cast<uint8_t *>(workspace);
    int st = qk::launch(mmq_prep_kernel, dim3((unsigned)B, (unsigned)gx), dim3(256), 0, (cudaStream_t)stream,
                        (flags & QK_LAUNCH_PDL) != 0, codes, static_cast<const __half2 *>(scales), M, K, wsA);
    if (st != QK_OK) return st;
    MmqArgs args{wsA, M, N, K, residual, y};
    return qk::launch(mmq_q4k_kernel, dim3((unsigned)gx, (unsigned)gy), dim3(kThreads), SMEM, (cudaStream_t)stream,
                      true, args, maps);
}
