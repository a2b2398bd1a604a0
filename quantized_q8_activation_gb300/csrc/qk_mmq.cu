// qk_mmq.cu -- prefill contraction Y[M][N] = Xq8 . W_q4k^T (+ R) on the
// sm_103a tensor cores (tcgen05, accumulators in tensor memory).
//
// Method (minfer "15 . The CUDA backend" sec. 2.3 / 3.2.6: quantized weight
// bytes go straight to the tensor cores, float scales are folded outside the
// integer accumulation).  This part runs integer MMA far below its f16 rate,
// so the contraction uses kind::f16 with operands that are exact:
//   B[n][k] = sc_j * q_w        an integer <= 945, exact in f16;
//   A[m][k] = d_a * q_a = A_hi + A_lo, two f16 values whose sum is exact
//             (d_a has 11 significant bits and q_a 7, so the product needs
//             18 <= 2 x 11 bits);
// the products and their binary32 sums over one 256-value superblock are
// accumulated by the tensor core into T (tensor memory), then folded with the
// superblock scale:  Y += d_b[n] * T.  The min term
//   - sum_b,j dmin_b m_j d_a sum(q_a)  = - S . Mw^T,
//   S[m][b,j] = d_a sum(q_a) / 16,   Mw[n][b,j] = 16 dmin_b m_j
// (the power-of-two factors keep both in f16 range) is a second contraction
// with K/32 terms on the tensor core too: each superblock adds K = 16 MMAs
// (8 values + 8 zeros) of S (hi/lo) against Mw (hi/lo) into U.  The result is
// Y - U (+ R).
//
// Two kernels per call:
//  1. mmq_prep_kernel expands the q8_1 activation once per 128-row M-tile into
//     the caller's workspace, already in the tensor core's shared-memory
//     layout: per 64-value K stage a 32 KB block (A_hi and A_lo tiles, K-major
//     SWIZZLE_128B), per superblock an 8 KB block (S_hi and S_lo tiles,
//     K-major SWIZZLE_32B, zero padded).  Every N-tile then copies these
//     blocks instead of converting the activation again.
//  2. mmq_q4k_kernel, one CTA (16 warps) per 128 x 128 output tile and per SM
//     (all 512 TMEM columns: Y | T0 | T1 | U):
//       warp 0      TMEM allocation; lane 0 issues every MMA and commit
//       warp 1      lane 0 copies the A stage blocks (and the S block of each
//                   superblock) from the workspace straight into the operand
//                   stages with cp.async.bulk
//       warp 2      lane 0 streams the raw Q4_K bytes with 2D TMA tensor
//                   copies into a ring: per K stage the two 16-byte halves of
//                   the code bytes (128 x 16 B each), per superblock the
//                   metadata records (128 x 16 B)
//       warps 4-7   fold T into Y per superblock, then the epilogue (TMEM lane
//                   quadrant = warp % 4)
//       warps 8-15  weight converters: Q4_K codes + scales -> B per K stage in
//                   the SWIZZLE_128B layout, and the Mw entries
// Stages are handed over with mbarriers (full: converters + copy bytes -> MMA;
// empty: MMA commit -> copy and converters; raw: TMA bytes -> converters ->
// producer; T buffers: MMA commit -> fold, fold -> MMA).  Every wait is
// bounded; a wait that gives up sets a device error flag (qk_error_flags), and
// once it is set the other waits return after a few polls, so the kernel runs
// to its end.  Before the CTA releases its tensor memory and exits, the MMA
// thread waits for its last MMAs and the producers wait for their last copies
// (bounded too), so nothing is left in flight.
#include "qk_common.cuh"
#include "qk_tc.cuh"

#include <cuda.h>

#include <atomic>

#ifndef QK_MMQ_NST
#define QK_MMQ_NST 3        // operand stages
#endif
#ifndef QK_MMQ_RAW
#define QK_MMQ_RAW 8        // raw weight K stages in flight
#endif
#ifndef QK_MMQ_SBRAW
#define QK_MMQ_SBRAW 4      // raw metadata superblocks in flight
#endif

__device__ unsigned g_qk_errors;

namespace {

using namespace qk::tc;

constexpr int BM = 128, BN = 128, BK = 64;      // BK: one Q4_K group = two 32-value sub-blocks
constexpr int NST = QK_MMQ_NST, NRAW = QK_MMQ_RAW, NSB = QK_MMQ_SBRAW;
constexpr int kThreads = 512;
constexpr int kFoldWarp0 = 4, kConvWarp0 = 8;
constexpr int kConv = 256, kFold = 128;
constexpr int kConvWarps = kConv / 32, kFoldWarps = kFold / 32;   // barrier arrivals: one per warp

constexpr int TILE = BM * BK * 2;               // 16 KB: 128 rows x 64 f16, SWIZZLE_128B K-major
constexpr int STAGE = 3 * TILE;                 // A_hi | A_lo | B
constexpr int ABLOCK = 2 * TILE;                // workspace block of one M-tile and K stage: A_hi | A_lo
constexpr int MTILE = 128 * 16 * 2;             // 4 KB: 128 rows x 16 f16, SWIZZLE_32B K-major
constexpr int MSET = 4 * MTILE;                 // S_hi | S_lo | Mw_hi | Mw_lo
constexpr int SBLOCK = 2 * MTILE;               // workspace block of one M-tile and superblock: S_hi | S_lo
// raw weight K stage: code bytes, first halves 128 x 16 B | second halves 128 x 16 B
constexpr int RAW_B0 = 0, RAW_B1 = BN * 16, RAW = 2 * BN * 16;
constexpr int SBR = BN * 16;                    // raw metadata records of one superblock
constexpr int OFF_MIN = NST * STAGE;
constexpr int OFF_RAW = OFF_MIN + 2 * MSET;
constexpr int OFF_SBR = OFF_RAW + NRAW * RAW;
constexpr int OFF_DB = OFF_SBR + NSB * SBR;     // fold: d_b of the tile's columns, 2 x 128 floats
constexpr int OFF_BAR = OFF_DB + 2 * 128 * 4;
enum {
    B_FULL = 0,
    B_EMPTY = B_FULL + NST,
    B_MINEMPTY = B_EMPTY + NST,
    B_TFULL = B_MINEMPTY + 2,
    B_TEMPTY = B_TFULL + 2,
    B_RFULL = B_TEMPTY + 2,
    B_REMPTY = B_RFULL + NRAW,
    B_SFULL = B_REMPTY + NRAW,
    B_SEMPTY = B_SFULL + NSB,
    B_DONE = B_SEMPTY + NSB,       // every MMA of the CTA has completed
    NBAR = B_DONE + 1
};
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_TMEM + 16 + 1024;      // + slack to align the base to 1024
static_assert(SMEM <= 232448, "shared memory plan exceeds the per-block opt-in limit");
static_assert(OFF_RAW % 1024 == 0 && OFF_SBR % 1024 == 0 && RAW % 1024 == 0, "copy destinations stay aligned");
constexpr uint32_t COL_Y = 0, COL_T0 = 128, COL_U = 384, TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

// byte offset of 16-byte chunk c of row r in a SWIZZLE_128B K-major tile (rows of 128 bytes)
__host__ __device__ constexpr uint32_t sw128(int r, int c) { return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4); }
// byte offset of element j (< 8, first 16-byte chunk) of row r in a SWIZZLE_32B K-major tile (rows of 32 bytes)
__host__ __device__ constexpr uint32_t sw32(int r, int j) { return (r >> 3) * 256 + (r & 7) * 32 + (((r >> 2) & 1) << 4) + 2 * j; }
// byte offset of the second (always zero) 16-byte chunk of row r in a SWIZZLE_32B K-major tile
__host__ __device__ constexpr uint32_t sw32_pad(int r) { return (r >> 3) * 256 + (r & 7) * 32 + ((((r >> 2) & 1) ^ 1) << 4); }

__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity) { mbar_wait(bar, parity, &g_qk_errors); }

__device__ __forceinline__ void bar_fold() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

struct MmqArgs {
    const uint8_t *w;       // repacked Q4_K weight (the fold reads d_b from its metadata)
    const uint8_t *wsA;     // workspace: [M-tiles][K/64] A blocks
    const uint8_t *wsS;     //            [M-tiles][K/256] S blocks
    int64_t M, N, K;
    const float *residual;
    float *y;
};

struct MmqMaps {
    CUtensorMap wcodes;     // uint8  [N][B*128]      box 16 x 128  (code plane of the repacked weight)
    CUtensorMap meta;       // uint8  [N][B*16]       box 16 x 128  (metadata plane)
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

// 4 code bytes -> (low nibble * sc_lo) and (high nibble * sc_hi) as f16 pairs (exact integers)
__device__ __forceinline__ void conv_b(uint32_t w4, __half2 sl, __half2 sl1024, __half2 sh, __half2 sh64,
                                       uint32_t &l01, uint32_t &l23, uint32_t &h01, uint32_t &h23)
{
    const uint32_t p01 = __byte_perm(w4, 0, 0x4140), p23 = __byte_perm(w4, 0, 0x4342);
    // 1024 + q (low nibble) and 64 + q (high nibble, which sits 16x in its byte)
    l01 = h2u(__hfma2(u2h((p01 & 0x000F000Fu) | 0x64006400u), sl, sl1024));
    l23 = h2u(__hfma2(u2h((p23 & 0x000F000Fu) | 0x64006400u), sl, sl1024));
    h01 = h2u(__hfma2(u2h((p01 & 0x00F000F0u) | 0x54005400u), sh, sh64));
    h23 = h2u(__hfma2(u2h((p23 & 0x00F000F0u) | 0x54005400u), sh, sh64));
}

__device__ __forceinline__ void sts128(uint8_t *base, uint32_t off, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    *reinterpret_cast<uint4 *>(base + off) = make_uint4(x, y, z, w);
}

__device__ __forceinline__ void split_f16(float v, __half &hi, __half &lo)
{
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));
}

// ------------------------------------------------------------- prep kernel
// CTA (superblock sb, M-tile mt), 256 threads, 4 items each: item (row, j) is
// the 32-value q8_1 block j of superblock sb of activation row 128 mt + row.
// It writes the block's 32 (A_hi, A_lo) pairs into the stage block of K stage
// 4 sb + j/2 (chunks 4 (j&1) .. +3) and the S entry j of its row; rows past M
// are written as zeros.
__global__ void __launch_bounds__(256) mmq_prep_kernel(const int8_t *__restrict__ codes,
                                                       const __half2 *__restrict__ scales, int64_t M, int64_t K,
                                                       uint8_t *__restrict__ wsA, uint8_t *__restrict__ wsS)
{
    qk::pdl_launch_dependents();
    qk::pdl_wait();                              // codes may come from the previous kernel
    const int sb = blockIdx.x, mt = blockIdx.y;
    const int B = (int)(K >> 8), nstage = (int)(K >> 6);
#pragma unroll 1
    for (int i = 0; i < 4; i++) {
        const int q = threadIdx.x + 256 * i;
        const int row = q >> 3, j = q & 7, h = j & 1;
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
        uint8_t *tA = wsA + ((size_t)mt * nstage + 4 * sb + (j >> 1)) * ABLOCK;
        int qsum = 0;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            uint32_t hi[4], lo[4];
            conv_a(aw[2 * c], d2, hi[0], lo[0], hi[1], lo[1]);
            conv_a(aw[2 * c + 1], d2, hi[2], lo[2], hi[3], lo[3]);
            sts128(tA, sw128(row, 4 * h + c), hi[0], hi[1], hi[2], hi[3]);
            sts128(tA + TILE, sw128(row, 4 * h + c), lo[0], lo[1], lo[2], lo[3]);
            qsum = qk::dp4a_ss(aw[2 * c], 0x01010101u, qsum);
            qsum = qk::dp4a_ss(aw[2 * c + 1], 0x01010101u, qsum);
        }
        uint8_t *tS = wsS + ((size_t)mt * B + sb) * SBLOCK;
        __half shi, slo;
        split_f16(__half2float(dah) * (float)qsum * 0.0625f, shi, slo);
        *reinterpret_cast<__half *>(tS + sw32(row, j)) = shi;
        *reinterpret_cast<__half *>(tS + MTILE + sw32(row, j)) = slo;
        if (j < 2) *reinterpret_cast<uint4 *>(tS + j * MTILE + sw32_pad(row)) = make_uint4(0, 0, 0, 0);
    }
}

// ------------------------------------------------------------- main kernel

// one converter thread's share of K stage `it` (operand stage st = it % NST): reads its raw weight
// bytes from the TMA ring, writes four B chunks of tile row `row` (half h of group g) and the Mw
// entry j = 2g + h, releases the raw slots and signals the stage full
__device__ __forceinline__ void convert_stage(uint8_t *smem, uint64_t *bar, int it, int row, int h, int st)
{
    const int sb = it >> 2, g = it & 3, tb = sb & 1;
    const int rs = it % NRAW, ss = sb % NSB;
    wait_bar(&bar[B_RFULL + rs], (it / NRAW) & 1);
    if (g == 0) wait_bar(&bar[B_SFULL + ss], (sb / NSB) & 1);
    const uint4 bq = *reinterpret_cast<const uint4 *>(smem + OFF_RAW + rs * RAW + (h ? RAW_B1 : RAW_B0) + row * 16);
    const uint4 mt = *reinterpret_cast<const uint4 *>(smem + OFF_SBR + ss * SBR + row * 16);

    if (it >= NST) wait_bar(&bar[B_EMPTY + st], ((it / NST) + 1) & 1);
    if (g == 0 && sb >= 2) wait_bar(&bar[B_MINEMPTY + tb], ((sb - 2) >> 1) & 1);
    uint8_t *s0 = smem + st * STAGE;
    // ---- B: this half of group g; low nibbles = sub-block 2g at stage k 16h .. 16h+15,
    //      high nibbles = sub-block 2g+1 at stage k 32+16h .. 32+16h+15
    const uint32_t rec = __byte_perm(__byte_perm(mt.y, mt.z, g == 0 ? 0x3210u : g == 1 ? 0x6543u : 0x7676u), mt.w,
                                     g == 0 ? 0x3210u : g == 1 ? 0x3210u : g == 2 ? 0x3410u : 0x3765u);
    const int sc0 = rec & 63u, sc1 = (rec >> 6) & 63u, mn0 = (rec >> 12) & 63u, mn1 = (rec >> 18) & 63u;
    const __half2 sl = __half2half2(__int2half_rn(sc0)), sh = __half2half2(__int2half_rn(sc1));
    const __half2 sl1024 = __half2half2(__int2half_rn(-1024 * sc0));
    const __half2 sh64 = __half2half2(__int2half_rn(-64 * sc1));
    const uint32_t bw[4] = {bq.x, bq.y, bq.z, bq.w};
    uint32_t L[8], H[8];
#pragma unroll
    for (int q = 0; q < 4; q++) conv_b(bw[q], sl, sl1024, sh, sh64, L[2 * q], L[2 * q + 1], H[2 * q], H[2 * q + 1]);
    sts128(s0 + 2 * TILE, sw128(row, 2 * h), L[0], L[1], L[2], L[3]);
    sts128(s0 + 2 * TILE, sw128(row, 2 * h + 1), L[4], L[5], L[6], L[7]);
    sts128(s0 + 2 * TILE, sw128(row, 4 + 2 * h), H[0], H[1], H[2], H[3]);
    sts128(s0 + 2 * TILE, sw128(row, 4 + 2 * h + 1), H[4], H[5], H[6], H[7]);
    // ---- min term entry j = 2g + h: Mw = 16 dmin m_j
    uint8_t *ms = smem + OFF_MIN + tb * MSET;
    const int j = 2 * g + h;
    __half whi, wlo;
    const float dmin = __half2float(__ushort_as_half((unsigned short)(mt.x >> 16)));
    split_f16(dmin * (float)(h ? mn1 : mn0) * 16.0f, whi, wlo);
    *reinterpret_cast<__half *>(ms + 2 * MTILE + sw32(row, j)) = whi;
    *reinterpret_cast<__half *>(ms + 3 * MTILE + sw32(row, j)) = wlo;
    // Each lane makes its own stores visible to the tensor core (async proxy); after the warp
    // has synchronised, one lane arrives for the whole warp.  The raw slots are released only
    // now: every value read from them has been consumed by the arithmetic above, so no shared
    // load can still be pending when the producer lets the next TMA copy overwrite the slot.
    fence_proxy_async();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        mbar_arrive(&bar[B_REMPTY + rs]);
        if (g == 3) mbar_arrive(&bar[B_SEMPTY + ss]);
        mbar_arrive(&bar[B_FULL + st]);
    }
}

__global__ void __launch_bounds__(kThreads, 1) mmq_q4k_kernel(const MmqArgs a, const __grid_constant__ MmqMaps maps)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    float *dB = reinterpret_cast<float *>(smem + OFF_DB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtile = blockIdx.x;
    const int m0 = mtile * BM, n0 = blockIdx.y * BN;
    const int B = (int)(a.K >> 8), nit = 4 * B;

    qk::pdl_launch_dependents();
    // setup: barriers, zero padding of the Mw tiles, TMEM allocation
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; i++) mbar_init(&bar[B_FULL + i], kConvWarps + 1), mbar_init(&bar[B_EMPTY + i], 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar[B_MINEMPTY + i], 1);
            mbar_init(&bar[B_TFULL + i], 1);
            mbar_init(&bar[B_TEMPTY + i], kFoldWarps);
        }
        for (int i = 0; i < NRAW; i++) mbar_init(&bar[B_RFULL + i], 1), mbar_init(&bar[B_REMPTY + i], kConvWarps);
        for (int i = 0; i < NSB; i++) mbar_init(&bar[B_SFULL + i], 1), mbar_init(&bar[B_SEMPTY + i], kConvWarps);
        mbar_init(&bar[B_DONE], 1);
        mbar_init_fence();
    }
    for (int i = threadIdx.x; i < 2 * (SBLOCK / 16); i += kThreads) {
        const int set = i / (SBLOCK / 16), k = i % (SBLOCK / 16);
        reinterpret_cast<uint4 *>(smem + OFF_MIN + set * MSET + SBLOCK)[k] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();                         // the zero padding is read by the tensor core
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
            for (int sb = 0; sb < B; sb++) {
                const int tb = sb & 1;
                if (sb >= 2) wait_bar(&bar[B_TEMPTY + tb], ((sb - 2) >> 1) & 1);
                fence_after_sync();
                const uint32_t dT = tmem + COL_T0 + 128 * tb;
                for (int g = 0; g < 4; g++) {
                    const int it = 4 * sb + g, st = it % NST;
                    wait_bar(&bar[B_FULL + st], (it / NST) & 1);
                    fence_after_sync();
                    const uint32_t s0 = sbase + st * STAGE;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++) {
                        const uint64_t ahi = smem_desc(s0 + 32 * kk, 16, 1024, kLayoutSw128);
                        const uint64_t alo = smem_desc(s0 + TILE + 32 * kk, 16, 1024, kLayoutSw128);
                        const uint64_t bd = smem_desc(s0 + 2 * TILE + 32 * kk, 16, 1024, kLayoutSw128);
                        mma_f16(dT, ahi, bd, IDESC, (g | kk) != 0);
                        mma_f16(dT, alo, bd, IDESC, 1);
                    }
                    mma_commit(&bar[B_EMPTY + st]);
                }
                const uint32_t ms = sbase + OFF_MIN + tb * MSET;
                const uint64_t shi = smem_desc(ms, 16, 256, kLayoutSw32);
                const uint64_t slo = smem_desc(ms + MTILE, 16, 256, kLayoutSw32);
                const uint64_t whi = smem_desc(ms + 2 * MTILE, 16, 256, kLayoutSw32);
                const uint64_t wlo = smem_desc(ms + 3 * MTILE, 16, 256, kLayoutSw32);
                mma_f16(tmem + COL_U, shi, whi, IDESC, sb != 0);
                mma_f16(tmem + COL_U, shi, wlo, IDESC, 1);
                mma_f16(tmem + COL_U, slo, whi, IDESC, 1);
                mma_commit(&bar[B_MINEMPTY + tb]);
                mma_commit(&bar[B_TFULL + tb]);
            }
            // teardown: no MMA may still be running when the TMEM is released
            mma_commit(&bar[B_DONE]);
            wait_bar(&bar[B_DONE], 0);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ activation stage copies
        if (lane == 0) {
            const int nstage = nit;
            const uint8_t *srcA = a.wsA + (size_t)mtile * nstage * ABLOCK;
            const uint8_t *srcS = a.wsS + (size_t)mtile * B * SBLOCK;
            for (int it = 0; it < nit; it++) {
                const int sb = it >> 2, g = it & 3, st = it % NST, tb = sb & 1;
                if (it >= NST) wait_bar(&bar[B_EMPTY + st], ((it / NST) + 1) & 1);
                if (g == 0 && sb >= 2) wait_bar(&bar[B_MINEMPTY + tb], ((sb - 2) >> 1) & 1);
                mbar_arrive_expect_tx(&bar[B_FULL + st], ABLOCK + (g == 0 ? SBLOCK : 0));
                bulk_copy_g2s(smem + st * STAGE, srcA + (size_t)it * ABLOCK, ABLOCK, &bar[B_FULL + st]);
                if (g == 0)
                    bulk_copy_g2s(smem + OFF_MIN + tb * MSET, srcS + (size_t)sb * SBLOCK, SBLOCK, &bar[B_FULL + st]);
            }
            // teardown: every copy this thread issued has landed (normally long since consumed)
            for (int it = nit - NST < 0 ? 0 : nit - NST; it < nit; it++)
                wait_bar(&bar[B_FULL + it % NST], (it / NST) & 1);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ raw weight TMA producer
        if (lane == 0) {
            prefetch_tmap(&maps.wcodes);
            prefetch_tmap(&maps.meta);
            for (int it = 0; it < nit; it++) {
                const int sb = it >> 2, g = it & 3;
                if (g == 0) {
                    const int ss = sb % NSB;
                    if (sb >= NSB) wait_bar(&bar[B_SEMPTY + ss], ((sb / NSB) + 1) & 1);
                    mbar_arrive_expect_tx(&bar[B_SFULL + ss], SBR);
                    tma_load_2d(smem + OFF_SBR + ss * SBR, &maps.meta, 16 * sb, n0, &bar[B_SFULL + ss]);
                }
                const int rs = it % NRAW;
                if (it >= NRAW) wait_bar(&bar[B_REMPTY + rs], ((it / NRAW) + 1) & 1);
                uint8_t *d = smem + OFF_RAW + rs * RAW;
                const int s = sb >> 3, G = 4 * min(8, B - 8 * s), u = 4 * (sb - 8 * s) + g;
                mbar_arrive_expect_tx(&bar[B_RFULL + rs], RAW);
                tma_load_2d(d + RAW_B0, &maps.wcodes, 1024 * s + 16 * u, n0, &bar[B_RFULL + rs]);
                tma_load_2d(d + RAW_B1, &maps.wcodes, 1024 * s + 16 * G + 16 * u, n0, &bar[B_RFULL + rs]);
            }
            // teardown: every copy this thread issued has landed (normally long since consumed)
            for (int it = nit - NRAW < 0 ? 0 : nit - NRAW; it < nit; it++)
                wait_bar(&bar[B_RFULL + it % NRAW], (it / NRAW) & 1);
            for (int sb = B - NSB < 0 ? 0 : B - NSB; sb < B; sb++) wait_bar(&bar[B_SFULL + sb % NSB], (sb / NSB) & 1);
        }
        __syncwarp();
    } else if (warp >= kFoldWarp0 && warp < kConvWarp0) {
        // -------------------------------------------------------------- fold
        const int ft = threadIdx.x - kFoldWarp0 * 32;            // 0..127: the column whose d_b it loads
        const uint32_t lq = (uint32_t)((warp & 3) * 32) << 16;   // TMEM lane quadrant of this warp
        const int64_t nd = n0 + ft;
        const uint8_t *dsrc = a.w + a.N * (int64_t)B * 128 + nd * B * 16;
        float dnext = nd < a.N ? __half2float(__ushort_as_half(qk::ldg_stream2(dsrc))) : 0.0f;
        for (int sb = 0; sb < B; sb++) {
            const int tb = sb & 1;
            dB[tb * 128 + ft] = dnext;
            bar_fold();
            if (sb + 1 < B && nd < a.N) dnext = __half2float(__ushort_as_half(qk::ldg_stream2(dsrc + 16 * (sb + 1))));
            wait_bar(&bar[B_TFULL + tb], (sb >> 1) & 1);
            fence_after_sync();
            const float *d = dB + tb * 128;
#pragma unroll 1
            for (int c = 0; c < 4; c++) {
                float t[32], yv[32];
                tmem_ld32(tmem + lq + COL_T0 + 128 * tb + 32 * c, t);
                if (sb > 0) tmem_ld32(tmem + lq + COL_Y + 32 * c, yv);
                tmem_wait_ld();
                if (sb > 0) {
#pragma unroll
                    for (int j = 0; j < 32; j++) yv[j] = fmaf(d[32 * c + j], t[j], yv[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j++) yv[j] = d[32 * c + j] * t[j];
                }
                tmem_st32(tmem + lq + COL_Y + 32 * c, yv);
            }
            tmem_wait_st();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_TEMPTY + tb]);
        }
        // epilogue: Y - U (+ R), one 32 x 32 block per pass: a thread holds row (32q + lane) of the
        // block; the block is transposed through shared memory (operand stage 0, idle once the last
        // TFULL has been observed) so that each store writes 32 consecutive columns of one row
        float *tb_s = reinterpret_cast<float *>(smem) + (warp - kFoldWarp0) * (32 * 33);
        const int q0 = (warp & 3) * 32;
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
            float yv[32], uv[32];
            tmem_ld32(tmem + lq + COL_Y + 32 * c, yv);
            tmem_ld32(tmem + lq + COL_U + 32 * c, uv);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j++) tb_s[lane * 33 + j] = yv[j] - uv[j];
            __syncwarp();
            const int64_t n = n0 + 32 * c + lane;
            if (n < a.N) {
#pragma unroll 4
                for (int r = 0; r < 32; r++) {
                    const int64_t m = m0 + q0 + r;
                    if (m < a.M) {
                        const float v = tb_s[r * 33 + lane];
                        const size_t o = (size_t)m * a.N + n;
                        a.y[o] = a.residual ? __fadd_rn(v, a.residual[o]) : v;
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp >= kConvWarp0) {
        // --------------------------------------------------------- converters
        // Lanes 0-15 of a warp take 16 consecutive rows of half 0, lanes 16-31 the same rows of
        // half 1, so every quarter warp stores to 8 distinct 16-byte bank groups.  Unrolled by the
        // stage count, so the operand stage index is static.
        const int ct = threadIdx.x - kConvWarp0 * 32;             // 0..255
        const int row = (ct & 15) + 16 * (ct >> 5), h = (ct >> 4) & 1;
        for (int it = 0; it < nit; it += NST) {
#pragma unroll
            for (int k = 0; k < NST; k++)
                if (it + k < nit) convert_stage(smem, bar, it + k, row, h, k);
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

// workspace bytes for an M x K activation: A blocks, then S blocks
size_t ws_bytes(int64_t M, int64_t K)
{
    const size_t mt = (size_t)((M + BM - 1) / BM);
    return mt * (size_t)(K / 64) * ABLOCK + mt * (size_t)(K / 256) * SBLOCK;
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
    if (!make_map(enc, &maps.wcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb, B * 128, N, B * 128, 16, BN) ||
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
    uint8_t *wsS = wsA + (size_t)gx * (size_t)(K / 64) * ABLOCK;
    int st = qk::launch(mmq_prep_kernel, dim3((unsigned)B, (unsigned)gx), dim3(256), 0, (cudaStream_t)stream,
                        (flags & QK_LAUNCH_PDL) != 0, codes, static_cast<const __half2 *>(scales), M, K, wsA, wsS);
    if (st != QK_OK) return st;
    MmqArgs args{wb, wsA, wsS, M, N, K, residual, y};
    return qk::launch(mmq_q4k_kernel, dim3((unsigned)gx, (unsigned)gy), dim3(kThreads), SMEM, (cudaStream_t)stream,
                      true, args, maps);
}
