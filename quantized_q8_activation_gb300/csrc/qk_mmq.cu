// qk_mmq.cu -- prefill contraction Y[M][N] = Xq8 . W^T (+ R), W a Q4_K or a
// Q6_K weight, on the sm_103a tensor cores (tcgen05, accumulator in tensor
// memory).
//
// Method (minfer "15 . The CUDA backend" sec. 2.3 / 3.2.6: quantized weight
// bytes go straight to the tensor cores; the activation is quantized to q8_1
// once per matmul input).  This part runs integer MMA far below its f16 rate,
// so the operands enter kind::f16 MMAs as f16 values, split where one f16 is
// not exact:
//   A[m][k] = d_a * q_a = A_hi + A_lo   exactly (d_a has 11 significant bits
//             and q_a 7, so the product needs 18 <= 2 x 11 bits).
//   Q4_K (mmq_q4k_kernel): the contraction is regrouped by superblock b and
//             sub-block j as  y = sum_b d_b (A . sc q)_b - sum_j dmin m_j S_j
//             (S_j = d_a sum q_a of the sub-block): sc q < 1024 is one exact
//             f16, so a K stage takes two MMAs (A_hi, A_lo) against one weight
//             tile; each superblock accumulates on its own and the epilogue
//             folds it into a register tile with d_b; the min term is a short
//             contraction of the sums S (split to 2^-22) with dmin m (split
//             exactly).
//   Q6_K (mmq_kernel): W[n][k] = 256 * d_b sc_j (q_w - 32) = W_hi + W_lo to
//             2^-21 relative (sc (q - 32) reaches 4096, not exact in one f16;
//             scaled by 2^8 so that W_lo stays a normal f16 for the weights of
//             LLM layers); Y = A_hi W_hi + A_hi W_lo + A_lo W_hi (A_lo W_lo is
//             below 2^-21 of each product and dropped), accumulated in binary32
//             over all of K in tensor memory; y = Y / 256 (+ R).
// The k-quant bytes are dequantized tile by tile in shared memory right before
// the MMAs that use them; they are read from memory in their quantized form.
//
// Two kernels per call:
//  1. mmq_prep_kernel expands the q8_1 activation once per 128-row M-tile into
//     the caller's workspace, already in the tensor core's shared-memory
//     layout: per 32-value K stage a 16 KB block (A_hi and A_lo tiles, K-major
//     SWIZZLE_64B), and for Q4_K per pair of superblocks an 8 KB tile of the
//     sub-block sums (S_hi | S_lo).  Every N-tile then copies these blocks
//     instead of converting the activation again.
//  2. the main kernel: a persistent grid, one CTA per SM, each CTA taking
//     128 x BN output tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...
//     (M-tile fastest).  Warp 0 lane 0 issues every MMA and commit, warp 3
//     (the sync warp) waits for each stage's operands and accumulator buffer
//     and hands the stage to warp 0 through a named barrier, warp 1 lane 0
//     copies each stage's activation block from the workspace with one bulk
//     copy, warp 2 lane 0 streams the raw weight bytes with 2D TMA tensor
//     copies into a ring (the code runs of a superblock and its per-row
//     records), epilogue warps read the accumulators, and converter warps
//     expand each K stage's codes and scales into f16 tiles in the
//     SWIZZLE_64B layout.  The roles of each kernel are listed above it.
// Stages are handed over with mbarriers (full: converters and the activation
// copy's bytes -> sync warp -> MMA; empty: MMA commit -> converters and
// activation copier; raw: TMA bytes -> converters -> producer; accumulator
// full / empty: MMA commit -> epilogue -> sync warp -> MMA; done: last MMA
// commit -> teardown).  The MMA thread itself never polls an mbarrier between
// MMAs: a shared-memory poll there idles the tensor pipe (about 150 ns a
// stage, measured), while a named barrier (bar.sync) does not.  Every
// mbarrier wait is bounded; a wait that gives up sets a device error flag
// (qk_error_flags), and once it is set the other waits return after a few
// polls, so the kernel runs to its end (the sync warp still releases every
// stage, so the MMA warp's named barriers always complete).
// Before the CTA releases its tensor memory and exits, the MMA thread waits
// for its last MMAs and the producers for their last copies (bounded too), so
// nothing is left in flight.
#include "qk_common.cuh"
#include "qk_tc.cuh"

#include <cuda.h>

#include <atomic>
#include <cstring>

#ifndef QK_MMQ_EPI_UNROLL
#define QK_MMQ_EPI_UNROLL 8  // output rows whose residual values are loaded together
#endif
#ifndef QK_MMQ_NST
#define QK_MMQ_NST 3        // operand stages
#endif
#ifndef QK_MMQ_RAW
#define QK_MMQ_RAW 2        // raw weight superblocks (eight K stages each) in flight
#endif
#ifndef QK_MMQ_SBRAW
#define QK_MMQ_SBRAW 2      // raw metadata superblocks in flight
#endif


__device__ unsigned g_qk_errors;

// an operand of the contraction would leave the binary16 range: flag it (one atomic per warp)
__device__ __forceinline__ void flag_range(bool bad)
{
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&g_qk_errors, QK_ERR_RANGE);
}

namespace {

using namespace qk::tc;

constexpr int kEpiUnroll = QK_MMQ_EPI_UNROLL;
constexpr int BM = 128, BK = 32;                // BK: one Q4_K / Q6_K 32-value sub-block
constexpr int NST = QK_MMQ_NST, NRAW = QK_MMQ_RAW, NSB = QK_MMQ_SBRAW;
constexpr int kEpiWarp0 = 4, kEpiWarps = 4, kConvWarp0 = 8;  // epilogue warps 4-7, converters from warp 8
constexpr float kWScale = 256.0f, kWUnscale = 1.0f / 256.0f;

constexpr int ATILE = BM * BK * 2;              // 8 KB: 128 rows x 32 f16 (64 B rows), SWIZZLE_64B K-major
constexpr int ABLOCK = 2 * ATILE;               // workspace block of one M-tile and K stage: A_hi | A_lo
constexpr int EPI_LD = 17;                      // epilogue transpose buffer: 32 rows x 16 columns, padded
// Q4_K split-scale kernel: the sums tile of one min stage, 128 rows x (S_hi 16 | S_lo 16) f16, SWIZZLE_64B
constexpr int SBLK = BM * 64;
constexpr float kSScale = 0.0625f;              // S' = S / 16
constexpr float kMScale = 1024.0f;              // Mw' = 1024 dmin m
constexpr float kMinUndo = -1.0f / 64.0f;       // -sum S Mw = -(sum S' Mw') / 64
enum {
    B_FULL = 0,
    B_EMPTY = B_FULL + NST,
    B_RFULL = B_EMPTY + NST,
    B_REMPTY = B_RFULL + NRAW,
    B_SFULL = B_REMPTY + NRAW,
    B_SEMPTY = B_SFULL + NSB,
    B_ACCFULL = B_SEMPTY + NSB,    // accumulator buffer holds a finished tile
    B_ACCEMPTY = B_ACCFULL + 2,    // the epilogue has read the accumulator buffer
    B_DONE = B_ACCEMPTY + 2,       // every MMA of the CTA has completed
    NBAR = B_DONE + 1
};
// Tile width and shared-memory plan of mmq_kernel<QT, BN> (QT = Q6_K): output tiles of 128 x BN
// (BN = 256, or 128 where 256-wide tiles leave a costly partial last wave on the SMs), two converter
// threads per weight row.
template <int QT, int BN_>
struct Plan {
    static_assert(QT == QK_TYPE_Q6_K, "Q4_K runs on mmq_q4k_kernel");
    static constexpr int BN = BN_;
    static constexpr int kConv = 2 * BN, kConvWarps = kConv / 32, kThreads = kConvWarp0 * 32 + kConv;
    static constexpr int WTILE = BN * BK * 2;              // BN rows x 32 f16
    static constexpr int STAGE = 2 * ATILE + 2 * WTILE;    // A_hi | A_lo | W_hi | W_lo
    // raw unit, half a superblock: ql first-chunk run BN x 32 B | ql second-chunk run BN x 32 B | qh
    // BN x 32 B
    static constexpr int RAW_QL0 = 0, RAW_QL1 = BN * 32, RAW_QH = 2 * BN * 32, RAW = 3 * BN * 32;
    static constexpr int SBR = BN * 16;                    // per-superblock scale records
    static constexpr uint32_t TMEM_COLS = 2 * BN;          // two accumulators: one accumulates while one drains
    static constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
    static constexpr int OFF_RAW = NST * STAGE;
    static constexpr int OFF_SBR = OFF_RAW + NRAW * RAW;
    static constexpr int OFF_EPI = OFF_SBR + NSB * SBR;
    static constexpr int OFF_BAR = OFF_EPI + kEpiWarps * 32 * EPI_LD * 4;
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_TMEM + 16 + 1024;   // + slack to align the base to 1024
    static_assert(SMEM <= 232448, "shared memory plan exceeds the per-block opt-in limit");
    static_assert(STAGE % 1024 == 0 && OFF_RAW % 1024 == 0 && RAW % 1024 == 0 && SBR % 1024 == 0,
                  "copy destinations and swizzle atoms stay aligned");
};

// byte offset of 16-byte chunk c (< 4) of row r in a SWIZZLE_64B K-major tile (rows of 64 bytes)
__host__ __device__ constexpr uint32_t sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }
// byte offset of 16-byte chunk c (< 2) of row r in a SWIZZLE_32B tile (rows of 32 bytes)
__host__ __device__ constexpr uint32_t sw32(int r, int c) { return r * 32 + ((c ^ ((r >> 2) & 1)) << 4); }

__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity) { mbar_wait(bar, parity, &g_qk_errors); }

// named barriers kStageBar0 + stage slot, 64 threads: the sync warp (warp 3) arrives, the MMA warp syncs
constexpr int kStageBar0 = 2;
__device__ __forceinline__ void stage_arrive(int id) { asm volatile("bar.arrive %0, 64;" ::"r"(id) : "memory"); }
__device__ __forceinline__ void stage_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

constexpr int kMaxSplit = 2;
struct MmqArgs {
    const uint8_t *wsA;     // workspace: [M-tiles][K/32] A blocks
    const uint8_t *wsS;     // Q4_K: [M-tiles][ceil(K/512)] sums tiles (after all A blocks)
    const uint16_t *dq;     // Q6_K: the d plane of the repacked weight, binary16 [N][K/256]
    int64_t M, N, K;
    const float *residual;
    float *y;
    int mtiles, ntiles;     // tile t covers M-tile t % mtiles, N-tile t / mtiles
    // Q4_K split of the K range: tiles [0, nfull) are work units of their own; each tile from nfull on
    // is split over two units (segment 0: superblocks [0, mid) and the min term; segment 1: [mid,
    // K/256)), each leaving its partial tile in part[], the second of the two to finish (cnt[]) adding
    // the partials and writing y.
    int split;              // 1: no split tiles (nfull = all tiles); 2: tiles from nfull on are split
    int nfull;
    int mid;
    float *part;            // [2 (tiles - nfull)][128][BN]
    unsigned *cnt;          // [tiles - nfull], zeroed by the prep kernel
};

// One 32 x 16 chunk of an output tile, staged in a warp's transpose buffer (row r at r * EPI_LD),
// to y: lane l stores column n (its own) of rows mb + 2 rr (rr < 16), mb = the chunk's first row
// + l / 16, adding the residual where there is one.  The residual may be y itself, so each group
// of kEpiUnroll rows has all its residual values loaded before any of its outputs is stored;
// grouped, the loads of a group are in flight together.
__device__ __forceinline__ void store_chunk(const MmqArgs &a, const float *tb_s, int64_t mb, int64_t n, int lane)
{
    const int tc = lane & 15, tr = lane >> 4;
    if (!a.residual) {
#pragma unroll
        for (int rr = 0; rr < 16; rr++) {
            const int64_t m = mb + 2 * rr;
            if (m < a.M) a.y[(size_t)m * a.N + n] = tb_s[(2 * rr + tr) * EPI_LD + tc];
        }
        return;
    }
    const size_t ob = (size_t)mb * a.N + n, st2 = 2 * (size_t)a.N;
#pragma unroll
    for (int h = 0; h < 16 / kEpiUnroll; h++) {
        float rv[kEpiUnroll];
#pragma unroll
        for (int i = 0; i < kEpiUnroll; i++) {
            const int rr = kEpiUnroll * h + i;
            rv[i] = mb + 2 * rr < a.M ? __ldcg(a.residual + ob + rr * st2) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kEpiUnroll; i++) {
            const int rr = kEpiUnroll * h + i;
            if (mb + 2 * rr < a.M) a.y[ob + rr * st2] = __fadd_rn(tb_s[(2 * rr + tr) * EPI_LD + tc], rv[i]);
        }
    }
}

struct MmqMaps {
    CUtensorMap wcodes;     // uint8  [N][B*128]  Q4_K code plane, box 32 x BN (32-byte swizzle); Q6_K ql plane
    CUtensorMap meta;       // uint8  [N][B*16]   Q4_K metadata plane / Q6_K scale plane, box 16 x BN
    CUtensorMap qh;         // uint8  [N][B*64]   Q6_K qh plane, box 32 x BN (unused for Q4_K)
    CUtensorMap plane;      // uint8  [N][nmin*64] Q4_K min-operand plane, box 64 x BN (64-byte swizzle; plane calls)
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
// Grid (K/32, M-tiles): CTA (bc, mt) takes 32-value block column bc (K stage bc) of the M-tile's
// 128 rows, eight lanes a row (four codes each), four passes of 32 rows; every load of the four
// passes is issued before the first conversion.  Each lane writes its four (A_hi, A_lo) pairs into
// row `row` of the stage block; rows past M are written as zeros.
__global__ void __launch_bounds__(256) mmq_prep_kernel(const int8_t *__restrict__ codes,
                                                       const __half2 *__restrict__ scales, int64_t M, int64_t K,
                                                       uint8_t *__restrict__ wsA, uint8_t *__restrict__ wsS,
                                                       unsigned *__restrict__ cnt, int ncnt)
{
    qk::pdl_launch_dependents();
    const int bc = blockIdx.x, mt = blockIdx.y, sb = bc >> 3, j = bc & 7;
    const int sub = threadIdx.x & 7;
    const int nit = (int)(K >> 5), B = (int)(K >> 8), nmin = (B + 1) >> 1;
    qk::pdl_wait();                              // codes may come from the previous kernel
    if (bc == 0 && mt == 0)                      // the split-K tile counters of this call start at zero
        for (int i = threadIdx.x; i < ncnt; i += 256) cnt[i] = 0;
    uint32_t rc[4], rd[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int64_t m = (int64_t)mt * BM + ((threadIdx.x + 256 * i) >> 3);
        rc[i] = rd[i] = 0;
        if (m < M) {
            rc[i] = *reinterpret_cast<const uint32_t *>(codes + m * K + 32 * bc + 4 * sub);
            rd[i] = *reinterpret_cast<const uint32_t *>(scales + m * (K >> 5) + bc) & 0xffffu;
        }
    }
    uint8_t *tA = wsA + ((size_t)mt * nit + bc) * ABLOCK;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int row = (threadIdx.x + 256 * i) >> 3;
        const __half dah = __ushort_as_half((unsigned short)rd[i]);
        const __half2 d2 = __halves2half2(dah, dah);
        // value limits of the f16 operands: d_a * 127 (the block's largest |x|) at most 32000 when the
        // sums S / 16 are built (Q4_K), 65000 otherwise (Q6_K); beyond them the result is undefined
        flag_range(__half2float(dah) * 127.0f > (wsS ? 32000.0f : 65000.0f));
        uint32_t hi01, lo01, hi23, lo23;
        conv_a(rc[i], d2, hi01, lo01, hi23, lo23);
        // values 4 sub .. 4 sub + 3 of the stage: half (sub & 1) of 16-byte chunk sub / 2 of the row
        const uint32_t off = sw64(row, sub >> 1) + 8 * (sub & 1);
        *reinterpret_cast<uint2 *>(tA + off) = make_uint2(hi01, hi23);
        *reinterpret_cast<uint2 *>(tA + ATILE + off) = make_uint2(lo01, lo23);
        if (wsS) {
            // the block's source sum S = d_a * sum(q_a), exact in binary32 (11 x 13 significant bits),
            // scaled by 2^-4 and split into f16 S_hi + S_lo (to 2^-22 of S): sub-block j of superblock
            // sb is column 8 (sb % 2) + j (S_hi) and 16 + 8 (sb % 2) + j (S_lo) of row `row` of the
            // sums tile sb / 2
            int sum = __dp4a((int)rc[i], 0x01010101, 0);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            if (sub == 0) {
                const float S = __half2float(dah) * (float)sum * kSScale;
                const __half sh = __float2half_rn(S);
                const __half sl = __float2half_rn(S - __half2float(sh));
                uint8_t *tS = wsS + ((size_t)mt * nmin + (sb >> 1)) * SBLK;
                const int e = sb & 1;
                *reinterpret_cast<__half *>(tS + sw64(row, e) + 2 * j) = sh;
                *reinterpret_cast<__half *>(tS + sw64(row, 2 + e) + 2 * j) = sl;
                if (e == 0 && sb + 1 == B) {     // odd B: the last tile's second superblock does not exist
                    *reinterpret_cast<__half *>(tS + sw64(row, 1) + 2 * j) = __ushort_as_half(0);
                    *reinterpret_cast<__half *>(tS + sw64(row, 3) + 2 * j) = __ushort_as_half(0);
                }
            }
        }
    }
}

// The prep of the f32 entry points (qk_mmq_q4k_f32, qk_mmq_q6k_f32): the f32 activation is quantized
// to q8_1 on the way, by the library's block quantizer (the codes and binary16 scales of
// qk_quantize_q8_1, bit for bit; they are not stored), and expanded as mmq_prep_kernel does.  Grid
// (K/32, M-tiles): CTA (bc, mt) takes 32-value block column bc (K stage bc) of the M-tile's 128 rows,
// eight lanes a row and four values a lane, four passes of 32 rows.
__global__ void __launch_bounds__(256) mmq_prep_f32_kernel(const float *__restrict__ x, int64_t ldx, int64_t M,
                                                           int64_t K, uint8_t *__restrict__ wsA,
                                                           uint8_t *__restrict__ wsS, unsigned *__restrict__ cnt,
                                                           int ncnt)
{
    qk::pdl_launch_dependents();
    const int bc = blockIdx.x, mt = blockIdx.y, sb = bc >> 3, j = bc & 7;
    const int sub = threadIdx.x & 7;
    const int nit = (int)(K >> 5), B = (int)(K >> 8), nmin = (B + 1) >> 1;
    qk::pdl_wait();                              // x may come from the previous kernel
    if (bc == 0 && mt == 0)                      // the split-K tile counters of this call start at zero
        for (int i = threadIdx.x; i < ncnt; i += 256) cnt[i] = 0;
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int64_t m = (int64_t)mt * BM + ((threadIdx.x + 256 * i) >> 3);
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < M) v[i] = *reinterpret_cast<const float4 *>(x + m * ldx + 32 * bc + 4 * sub);
    }
    uint8_t *tA = wsA + ((size_t)mt * nit + bc) * ABLOCK;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int row = (threadIdx.x + 256 * i) >> 3;
        float d;
        int sum;
        const uint32_t packed = qk::q81_quant8(v[i], d, sum);      // rows past M: d = 0, codes 0
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        const __half dah = qk::f16_sat(d);                         // the stored q8_1 scale
        const __half2 d2 = __halves2half2(dah, dah);
        flag_range(__half2float(dah) * 127.0f > (wsS ? 32000.0f : 65000.0f));
        uint32_t hi01, lo01, hi23, lo23;
        conv_a(packed, d2, hi01, lo01, hi23, lo23);
        // values 4 sub .. 4 sub + 3 of the stage: half (sub & 1) of 16-byte chunk sub / 2 of the row
        const uint32_t off = sw64(row, sub >> 1) + 8 * (sub & 1);
        *reinterpret_cast<uint2 *>(tA + off) = make_uint2(hi01, hi23);
        *reinterpret_cast<uint2 *>(tA + ATILE + off) = make_uint2(lo01, lo23);
        if (wsS && sub == 0) {
            // the block's source sum S = d_a * sum(q_a) / 16 as S_hi + S_lo, placed as mmq_prep_kernel does
            const float S = __half2float(dah) * (float)sum * kSScale;
            const __half sh = __float2half_rn(S);
            const __half sl = __float2half_rn(S - __half2float(sh));
            uint8_t *tS = wsS + ((size_t)mt * nmin + (sb >> 1)) * SBLK;
            const int e = sb & 1;
            *reinterpret_cast<__half *>(tS + sw64(row, e) + 2 * j) = sh;
            *reinterpret_cast<__half *>(tS + sw64(row, 2 + e) + 2 * j) = sl;
            if (e == 0 && sb + 1 == B) {         // odd B: the last tile's second superblock does not exist
                *reinterpret_cast<__half *>(tS + sw64(row, 1) + 2 * j) = __ushort_as_half(0);
                *reinterpret_cast<__half *>(tS + sw64(row, 3) + 2 * j) = __ushort_as_half(0);
            }
        }
    }
}

// ------------------------------------------------------------- main kernel

// Converter state of one half row across K stages.  Q4_K: its 16 code bytes of the current
// 64-value group (c) and the row's metadata record of the current superblock (mt).  Q6_K: its 16
// bytes of each ql chunk (c, c2) and of qh (qh) of the current half superblock, the row's scale
// record of the current superblock (mt), and the superblock's d (binary16 bits) with the next
// superblock's d already requested (dn).
struct ConvState {
    uint4 c, mt, c2, qh;
    uint32_t d, dn;
};

// Q6_K: the d of superblock sb of tile t for this converter's weight row (0 past the last row)
template <int BN>
__device__ __forceinline__ uint32_t q6_d(const MmqArgs &a, int t, int sb, int row)
{
    const int64_t n = (int64_t)(t / a.mtiles) * BN + row;
    return n < a.N ? (uint32_t)__ldg(a.dq + n * (a.K >> 8) + sb) : 0u;
}

// Q6_K share of one converter thread in K stage `it` (sub-block j = it % 8 of superblock it / 8:
// half hs = j / 4 of the superblock, quarter q = j % 4): the 16 weights l = 16h .. 16h+15 of the
// sub-block,
//   w = 256 d sc (u - 32),  u = ql nibble | qh bit pair << 4,
// with the ql byte from the first chunk run (q even) or the second (q odd), its low (q < 2) or high
// nibble, the qh bits 2q, 2q+1, and scale byte 4 (2 hs + h) + q of the record.  Stored as
// (W_hi, W_lo) chunks 2h and 2h+1, then the stage is signalled full.
// gsb: superblock counted over all tiles of this CTA; t: the tile (for the d prefetch)
template <class L>
__device__ __forceinline__ void convert_stage_q6(uint8_t *smem, uint64_t *bar, ConvState &cs, const MmqArgs &a,
                                                 int t, int it, int gs, int gsb, int row, int h, int st)
{
    const int j = it & 7, hs = j >> 2, q = j & 3;
    const int gu = 2 * gsb + hs;                              // raw unit: half superblock
    const int rs = gu % NRAW, ss = gsb % NSB;
    if (j == 0) {
        wait_bar(&bar[B_SFULL + ss], (gsb / NSB) & 1);
        cs.mt = *reinterpret_cast<const uint4 *>(smem + L::OFF_SBR + ss * L::SBR + row * 16);
        // this superblock's d was requested one superblock ago; request the next one's
        const int B = (int)(a.K >> 8), sb = it >> 3;
        cs.d = cs.dn;
        if (sb + 1 < B) cs.dn = q6_d<L::BN>(a, t, sb + 1, row);
        else if (t + (int)gridDim.x < a.mtiles * a.ntiles) cs.dn = q6_d<L::BN>(a, t + gridDim.x, 0, row);
        // value limit |w| < 255: |w| <= 32 |d sc| over the codes of a sub-block; checked once per
        // superblock with its largest |sc| (flags every sub-block that can reach 255)
        const uint32_t am = __vmaxu4(__vmaxu4(__vabsss4(cs.mt.x), __vabsss4(cs.mt.y)),
                                     __vmaxu4(__vabsss4(cs.mt.z), __vabsss4(cs.mt.w)));
        const uint32_t am2 = __vmaxu4(am, am >> 16), amax = max(am2 & 0xffu, (am2 >> 8) & 0xffu);
        flag_range(32.0f * fabsf(__half2float(__ushort_as_half((unsigned short)cs.d))) * (float)amax >= 255.0f);
    }
    if (q == 0) {
        wait_bar(&bar[B_RFULL + rs], (gu / NRAW) & 1);
        const uint8_t *r0 = smem + L::OFF_RAW + rs * L::RAW + row * 32 + 16 * h;
        cs.c = *reinterpret_cast<const uint4 *>(r0 + L::RAW_QL0);
        cs.c2 = *reinterpret_cast<const uint4 *>(r0 + L::RAW_QL1);
        cs.qh = *reinterpret_cast<const uint4 *>(r0 + L::RAW_QH);
    }
    if (gs >= NST) wait_bar(&bar[B_EMPTY + st], ((gs / NST) + 1) & 1);
    uint8_t *s0 = smem + st * L::STAGE;
    const int p = 2 * hs + h;                                 // record bytes 4p .. 4p+3: quarters 0..3
    const uint32_t scw = p == 0 ? cs.mt.x : p == 1 ? cs.mt.y : p == 2 ? cs.mt.z : cs.mt.w;
    const int sc = (int)(int8_t)(scw >> (8 * q));
    const float d = __half2float(__ushort_as_half((unsigned short)cs.d));
    const float dsc = d * (float)sc * kWScale;               // exact: 11 + 8 significant bits, times 2^8
    const float2 dsc2 = make_float2(dsc, dsc), ndmm2 = make_float2(-32.0f * dsc, -32.0f * dsc);
    const uint4 lq = (q & 1) ? cs.c2 : cs.c;
    const uint32_t lw[4] = {lq.x, lq.y, lq.z, lq.w};
    const uint32_t hw[4] = {cs.qh.x, cs.qh.y, cs.qh.z, cs.qh.w};
    const int ls = (q >> 1) * 4, hsft = 2 * q;
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
        uint32_t hi[4], lo[4];
        const uint32_t x0 = ((lw[2 * cc] >> ls) & 0x0F0F0F0Fu) | (((hw[2 * cc] >> hsft) & 0x03030303u) << 4);
        const uint32_t x1 = ((lw[2 * cc + 1] >> ls) & 0x0F0F0F0Fu) | (((hw[2 * cc + 1] >> hsft) & 0x03030303u) << 4);
        conv_w(x0, dsc2, ndmm2, hi[0], hi[1], lo[0], lo[1]);
        conv_w(x1, dsc2, ndmm2, hi[2], hi[3], lo[2], lo[3]);
        sts128(s0 + 2 * ATILE, sw64(row, 2 * h + cc), hi[0], hi[1], hi[2], hi[3]);
        sts128(s0 + 2 * ATILE + L::WTILE, sw64(row, 2 * h + cc), lo[0], lo[1], lo[2], lo[3]);
    }
    // as for Q4_K: the stores are made visible to the async proxy, and a ring slot is released only
    // after every value loaded from it has been used by the arithmetic (the second ql chunk is
    // first used in quarter 1)
    fence_proxy_async();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (q == 1) mbar_arrive(&bar[B_REMPTY + rs]);
        if (j == 0) mbar_arrive(&bar[B_SEMPTY + ss]);
        mbar_arrive(&bar[B_FULL + st]);
    }
}

// Q6_K main kernel, one CTA (8 + 2 BN / 32 warps) per SM:
//   warp 0      TMEM allocation (two BN-column accumulators: one tile accumulates while the previous
//               one is written out); lane 0 issues every MMA and commit
//   warp 1      lane 0: one bulk copy per K stage of its 16 KB activation block
//   warp 2      lane 0: per half superblock the 32-byte runs of the two ql chunks and of qh (BN x 32 B
//               each), per superblock the scale records (BN x 16 B); the d plane (2 bytes per
//               superblock) is read by the converters themselves, one superblock ahead
//   warps 4-7   the epilogue of the previous tile (TMEM lane quadrant = warp % 4)
//   warps 8..   converters: two threads per weight row expand each K stage into (W_hi, W_lo)
template <int QT, int BN_>
__global__ void __launch_bounds__(Plan<QT, BN_>::kThreads, 1)
    mmq_kernel(const MmqArgs a, const __grid_constant__ MmqMaps maps)
{
    using L = Plan<QT, BN_>;
    constexpr int BN = L::BN;
    static_assert(kStageBar0 + NST <= 16, "a named barrier per stage slot");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + L::OFF_TMEM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = (int)(a.K >> 8), nit = 8 * B;
    const int ntiles = a.mtiles * a.ntiles;
    // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ... (M-tile fastest, so the CTAs running
    // at the same time share their activation and weight tiles in L2)

    qk::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; i++)
            mbar_init(&bar[B_FULL + i], L::kConvWarps + 1), mbar_init(&bar[B_EMPTY + i], 1);
        for (int i = 0; i < NRAW; i++) mbar_init(&bar[B_RFULL + i], 1), mbar_init(&bar[B_REMPTY + i], L::kConvWarps);
        for (int i = 0; i < NSB; i++) mbar_init(&bar[B_SFULL + i], 1), mbar_init(&bar[B_SEMPTY + i], L::kConvWarps);
        for (int i = 0; i < 2; i++) mbar_init(&bar[B_ACCFULL + i], 1), mbar_init(&bar[B_ACCEMPTY + i], kEpiWarps);
        mbar_init(&bar[B_DONE], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tmem_ptr, L::TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_ptr;
    qk::pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        // the warp takes each stage from the sync warp (warp 3) through a named barrier; lane 0 issues
        const uint32_t sbase = smem_u32(smem);
        int kt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, kt++) {
            const int acc = kt & 1;
            const uint32_t dacc = tmem + acc * BN;
            for (int it = 0; it < nit; it++) {
                const int gs = kt * nit + it, st = gs % NST;
                stage_sync(kStageBar0 + st);
                if (lane == 0) {
                    fence_after_sync();
                    const uint32_t s0 = sbase + st * L::STAGE;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++) {
                        const uint64_t ahi = smem_desc(s0 + 32 * kk, 16, 512, kLayoutSw64);
                        const uint64_t alo = smem_desc(s0 + ATILE + 32 * kk, 16, 512, kLayoutSw64);
                        const uint64_t whi = smem_desc(s0 + 2 * ATILE + 32 * kk, 16, 512, kLayoutSw64);
                        const uint64_t wlo = smem_desc(s0 + 2 * ATILE + L::WTILE + 32 * kk, 16, 512, kLayoutSw64);
                        mma_f16(dacc, ahi, whi, L::IDESC, (it | kk) != 0);
                        mma_f16(dacc, ahi, wlo, L::IDESC, 1);
                        mma_f16(dacc, alo, whi, L::IDESC, 1);
                    }
                    mma_commit(&bar[B_EMPTY + st]);
                    if (it == nit - 1) mma_commit(&bar[B_ACCFULL + acc]);
                }
                __syncwarp();
            }
        }
        // teardown: no MMA may still be running when the TMEM is released
        if (lane == 0) {
            mma_commit(&bar[B_DONE]);
            wait_bar(&bar[B_DONE], 0);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------------ sync warp
        // per stage: wait (bounded) for its operands and, at a tile's first stage, for the accumulator
        // buffer; then hand the stage to the MMA warp (it arrives even after a wait gave up)
        int kt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, kt++) {
            const int acc = kt & 1;
            if (kt >= 2) wait_bar(&bar[B_ACCEMPTY + acc], ((kt >> 1) + 1) & 1);
            for (int it = 0; it < nit; it++) {
                const int gs = kt * nit + it, st = gs % NST;
                wait_bar(&bar[B_FULL + st], (gs / NST) & 1);
                stage_arrive(kStageBar0 + st);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ activation block copier
        // one bulk copy per K stage of the stage's 16 KB activation block, issued as soon as the
        // MMAs have released the stage slot; it completes on the stage's full barrier
        if (lane == 0) {
            int kt = 0;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, kt++) {
                const uint8_t *srcA = a.wsA + (size_t)(t % a.mtiles) * nit * ABLOCK;
                for (int it = 0; it < nit; it++) {
                    const int gs = kt * nit + it, st = gs % NST;
                    if (gs >= NST) wait_bar(&bar[B_EMPTY + st], ((gs / NST) + 1) & 1);
                    mbar_arrive_expect_tx(&bar[B_FULL + st], ABLOCK);
                    bulk_copy_g2s(smem + st * L::STAGE, srcA + (size_t)it * ABLOCK, ABLOCK, &bar[B_FULL + st]);
                }
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ raw weight TMA producer
        if (lane == 0) {
            prefetch_tmap(&maps.wcodes);
            prefetch_tmap(&maps.meta);
            prefetch_tmap(&maps.qh);
            int gsb = 0, gu = 0;                                  // superblocks and raw units issued
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
                const int n0 = (t / a.mtiles) * BN;
                for (int sb = 0; sb < B; sb++, gsb++) {
                    const int ss = gsb % NSB;
                    if (gsb >= NSB) wait_bar(&bar[B_SEMPTY + ss], ((gsb / NSB) + 1) & 1);
                    mbar_arrive_expect_tx(&bar[B_SFULL + ss], L::SBR);
                    tma_load_2d(smem + L::OFF_SBR + ss * L::SBR, &maps.meta, 16 * sb, n0, &bar[B_SFULL + ss]);
                    // the superblock's lanes u = 4 (sb - 8 s) .. +3 of its step s: first 16-byte chunks at 16u,
                    // second chunks at 16 G + 16u
                    const int s = sb >> 3, G = 4 * min(8, B - 8 * s), u = 4 * (sb - 8 * s);
                    // two raw units: superblock half hs holds lanes u + 2hs, u + 2hs + 1 of each ql run and qh
                    // bytes 32hs .. 32hs+31
                    for (int hs = 0; hs < 2; hs++, gu++) {
                        const int rs = gu % NRAW;
                        if (gu >= NRAW) wait_bar(&bar[B_REMPTY + rs], ((gu / NRAW) + 1) & 1);
                        uint8_t *d = smem + L::OFF_RAW + rs * L::RAW;
                        mbar_arrive_expect_tx(&bar[B_RFULL + rs], L::RAW);
                        tma_load_2d(d + L::RAW_QL0, &maps.wcodes, 1024 * s + 16 * u + 32 * hs, n0, &bar[B_RFULL + rs]);
                        tma_load_2d(d + L::RAW_QL1, &maps.wcodes, 1024 * s + 16 * G + 16 * u + 32 * hs, n0,
                                    &bar[B_RFULL + rs]);
                        tma_load_2d(d + L::RAW_QH, &maps.qh, 64 * sb + 32 * hs, n0, &bar[B_RFULL + rs]);
                    }
                }
            }
            // teardown: every copy this thread issued has landed (normally long since consumed)
            for (int g = gu - NRAW < 0 ? 0 : gu - NRAW; g < gu; g++) wait_bar(&bar[B_RFULL + g % NRAW], (g / NRAW) & 1);
            for (int g = gsb - NSB < 0 ? 0 : gsb - NSB; g < gsb; g++) wait_bar(&bar[B_SFULL + g % NSB], (g / NSB) & 1);
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
        // -------------------------------------------------------------- epilogue
        // y = Y / 256 (+ R) per finished tile, 16 columns per pass: a thread holds row (32q + lane)
        // of the block; the block is transposed through shared memory so that each store covers 16
        // consecutive columns of two rows
        const uint32_t lq = (uint32_t)((warp & 3) * 32) << 16;   // TMEM lane quadrant of this warp
        float *tb_s = reinterpret_cast<float *>(smem + L::OFF_EPI) + (warp - kEpiWarp0) * (32 * EPI_LD);
        const int q0 = (warp & 3) * 32;
        int kt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, kt++) {
            const int acc = kt & 1;
            const int64_t m0 = (int64_t)(t % a.mtiles) * BM, n0 = (int64_t)(t / a.mtiles) * BN;
            wait_bar(&bar[B_ACCFULL + acc], (kt >> 1) & 1);
            fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < BN / 16; c++) {
                float v[16];
                tmem_ld16(tmem + lq + acc * BN + 16 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 16; jj++) tb_s[lane * EPI_LD + jj] = v[jj] * kWUnscale;
                __syncwarp();
                const int64_t n = n0 + 16 * c + (lane & 15);
                if (n < a.N) {
                    store_chunk(a, tb_s, m0 + q0 + (lane >> 4), n, lane);
                }
                __syncwarp();
            }
            // the accumulator buffer may be overwritten once every lane's loads have completed
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_ACCEMPTY + acc]);
        }
    } else if (warp >= kConvWarp0) {
        // --------------------------------------------------------- converters
        // Lanes 0-15 of a warp take 16 consecutive rows of half 0, lanes 16-31 the same rows of
        // half 1; a quarter warp stores 8 consecutive rows, which the 64-byte swizzle spreads over
        // all 32 banks.
        const int cwarp = warp - kConvWarp0;                      // 0..15
        const int row = 16 * cwarp + (lane & 15), h = lane >> 4;
        ConvState cs;
        cs.c = cs.mt = cs.c2 = cs.qh = make_uint4(0, 0, 0, 0);
        cs.d = 0;
        cs.dn = q6_d<BN>(a, blockIdx.x, 0, row);
        int kt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, kt++) {
            const int gs0 = kt * nit;
            // the stage slot of K stage it is (gs0 + it) % NST: unroll so that it is static
            static_assert(NST == 3, "the slot prologue below handles three stages");
            int it = 0;
            auto conv = [&](int itk, int gs, int st) {
                convert_stage_q6<L>(smem, bar, cs, a, t, itk, gs, kt * B + (itk >> 3), row, h, st);
            };
            while (it < nit && (gs0 + it) % NST != 0) {
                const int gs = gs0 + it;
                if (gs % NST == 1) conv(it, gs, 1);
                else conv(it, gs, 2);
                it++;
            }
            for (; it < nit; it += NST) {
#pragma unroll
                for (int k = 0; k < NST; k++)
                    if (it + k < nit) conv(it + k, gs0 + it + k, k);
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ------------------------------------------------ Q4_K split-scale kernel
// For Q4_K the tile's contraction is regrouped so that every weight operand is
// exact in one f16 (Q4_K / q8_1 decomposition of minfer "15 . The CUDA
// backend" sec. 3.2.6: the sub-block scale times the code dot, the min times
// the source sum):
//   y[m][n] = sum_b d_b[n] * (sum_{k in b} A[m][k] sc[n][k/32] q[n][k])
//             - sum_j (dmin m)[n][j] S[m][j]
// with A = d_a q_a = A_hi + A_lo (exact), S[m][j] = d_a sum(q_a) of sub-block
// j.  W'[n][k] = sc q is an integer below 1024, so a K stage needs two MMAs
// (A_hi W', A_lo W') and one f16 weight tile; each superblock b accumulates in
// a tensor-memory buffer of its own, and the epilogue warps fold it into a
// register copy of the output tile with the superblock scale d_b (an f16, so
// the product is one binary32 rounding).  The min term is its own short
// contraction over the K/32 sub-blocks, issued first for each tile: sums
// tiles (S_hi | S_lo, built by the prep kernel) against (Mw_hi | Mw_lo),
// Mw = 1024 dmin m (17 significant bits, split exactly down to 2^-8), three MMAs per 16
// sub-blocks; its accumulator seeds the register tile.
// Warps: 0 MMA, 1 activation copier, 2 TMA producer, 3 sync warp, 4-11 epilogue
// (TMEM lane quadrant warp % 4, column half (warp - 4) / 4), 12.. converters
// (one thread per weight row).  With 256- and 192-wide tiles the epilogue warps
// hold 128 or 96 accumulator columns each and take registers from the other
// warps (setmaxnreg); the split stays within the launch's registers (640 x 96
// or 576 x 96).  BN = 192 keeps two 192-column accumulators in a
// 512-column tensor-memory allocation.
template <int BN_>
struct Plan4 {
    static constexpr int BN = BN_;
    static constexpr int kEpiW0 = 4, kEpiW = 8, kConvW0 = 12, kConvW = BN / 32;
    // setmaxnreg acts on whole warpgroups (4 warps), so the launch rounds the converter warps up to a
    // multiple of 4; the extra warps (BN = 192: two) only give their registers back and wait at the end
    static constexpr int kConvWL = (kConvW + 3) / 4 * 4;
    static constexpr int kThreads = (kConvW0 + kConvWL) * 32;
    static constexpr int CPT = BN / 2;                     // output columns per epilogue thread
    static constexpr int WTILE = BN * 64;                  // BN rows x 32 f16
    static constexpr int STAGE = 2 * ATILE + WTILE;        // A_hi | A_lo (or the sums tile) | W' (or Mw)
    // raw unit: half a superblock's code bytes, first 16-byte halves of its 2 groups | second halves
    static constexpr int RAW_H1 = BN * 32, RAW = 2 * BN * 32;
    static constexpr int SBR = BN * 16;
    static_assert(BN == 128 || BN == 192 || BN == 256, "tile widths 128, 192, 256");
    static constexpr int NST = BN == 128 ? 6 : 4, NRAW = 3, NSB = 4, ND = 4;
    static constexpr uint32_t TMEM_COLS = BN == 128 ? 256 : 512;   // a power of two holding both accumulators
    static constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
    static constexpr int OFF_RAW = NST * STAGE;
    static constexpr int OFF_SBR = OFF_RAW + NRAW * RAW;
    static constexpr int OFF_D = OFF_SBR + NSB * SBR;          // superblock scales d_b, binary32 [ND][BN]
    static constexpr int OFF_EPI = OFF_D + ND * BN * 4;
    static constexpr int OFF_BAR = OFF_EPI + kEpiW * 32 * EPI_LD * 4;
    enum {
        FULL = 0,
        EMPTY = FULL + NST,
        RFULL = EMPTY + NST,
        REMPTY = RFULL + NRAW,
        SFULL = REMPTY + NRAW,
        SEMPTY = SFULL + NSB,
        DFULL = SEMPTY + NSB,
        DEMPTY = DFULL + ND,
        ACCFULL = DEMPTY + ND,
        ACCEMPTY = ACCFULL + 2,
        DONE = ACCEMPTY + 2,
        NBAR = DONE + 1
    };
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_TMEM + 16 + 1024;
    static constexpr bool kSplitRegs = BN >= 192;
#ifndef QK_MMQ4_RMISC
#define QK_MMQ4_RMISC 48
#endif
#ifndef QK_MMQ4_REPI
#define QK_MMQ4_REPI 168
#endif
#ifndef QK_MMQ4_RCONV
#define QK_MMQ4_RCONV 48
#endif
    // registers per thread: the least a launch may have (the split's total over the threads, rounded up to
    // the allocation unit of 8), then warps 0-3, epilogue warps, converters
    static constexpr int kRegMisc = QK_MMQ4_RMISC, kRegConv = QK_MMQ4_RCONV;
    static constexpr int kRegEpi = QK_MMQ4_REPI;
    static constexpr int kRegLaunch =
        ((4 * kRegMisc + kEpiW * kRegEpi + kConvWL * kRegConv) * 32 / kThreads + 7) / 8 * 8;
    static_assert(SMEM <= 232448, "shared memory plan exceeds the per-block opt-in limit");
    static_assert(STAGE % 1024 == 0 && OFF_RAW % 1024 == 0 && RAW % 1024 == 0 && OFF_SBR % 1024 == 0,
                  "copy destinations and swizzle atoms stay aligned");
    static_assert(!kSplitRegs || (4 * kRegMisc + kEpiW * kRegEpi + kConvWL * kRegConv) * 32 <= kThreads * kRegLaunch,
                  "the register split must fit in the launch's registers");
    static_assert(kThreads % 128 == 0 && kEpiW0 % 4 == 0 && kEpiW % 4 == 0 && kConvW0 % 4 == 0,
                  "every setmaxnreg warpgroup is whole");
    static_assert(!kSplitRegs || kRegLaunch * kThreads <= 65536, "the launch's registers fit one SM");
};

template <int N> __device__ __forceinline__ void reg_alloc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N> __device__ __forceinline__ void reg_dealloc() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// the 24-bit record of group g (sub-blocks 2g, 2g+1) of a Q4_K metadata record:
// sc[2g] | sc[2g+1] << 6 | m[2g] << 12 | m[2g+1] << 18
__device__ __forceinline__ uint32_t q4_group(const uint4 &mt, int g)
{
    return __byte_perm(__byte_perm(mt.y, mt.z, g == 0 ? 0x3210u : g == 1 ? 0x6543u : 0x7676u), mt.w,
                       g == 0 ? 0x3210u : g == 1 ? 0x3210u : g == 2 ? 0x3410u : 0x3765u);
}

// the f16 pairs (sc, sc) and (-1024 sc, -1024 sc) of a sub-block scale sc < 64 (both exact)
struct ScPair {
    __half2 s, n;
};
__device__ __forceinline__ ScPair sc_pair(uint32_t sc)
{
    const __half2 s2 = __half2half2(__ushort2half_rn((unsigned short)sc));
    return ScPair{s2, __hmul2(s2, u2h(0xE400E400u))};              // x (-1024), exact
}

// 4 nibbles (one per byte of x, masked to 0..15) times the sub-block scale sc as two f16 pairs,
// exactly: each byte goes to a 16-bit lane under 0x64 (the f16 1024 + q), and one fused multiply-add
// gives (1024 + q) sc - 1024 sc = sc q, an integer below 1024 that the single rounding leaves exact
__device__ __forceinline__ void w_sc(uint32_t x, const ScPair &k, uint32_t &p01, uint32_t &p23)
{
    p01 = h2u(__hfma2(u2h(__byte_perm(x, 0x64646464u, 0x4140u)), k.s, k.n));
    p23 = h2u(__hfma2(u2h(__byte_perm(x, 0x64646464u, 0x4342u)), k.s, k.n));
}

// the 8 min products Mw' = 1024 dmin m_j of one superblock record as f16 pairs hi (11 significant
// bits: the binary32 value with its 13 low mantissa bits cleared) and lo (the remaining at most 6
// bits), exact down to Mw' = 2^-8 (below it lo's last bit falls under the f16 subnormal step);
// word i holds sub-blocks 2i, 2i+1
__device__ __forceinline__ void mins_hilo(const uint4 &mt, uint32_t (&hi)[4], uint32_t (&lo)[4], bool &bad)
{
    const float dmin = __half2float(__ushort_as_half((unsigned short)(mt.x >> 16))) * kMScale;
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const uint32_t r = q4_group(mt, g);
        const float w0 = dmin * (float)((r >> 12) & 63u), w1 = dmin * (float)((r >> 18) & 63u);   // exact
        bad |= fmaxf(w0, w1) >= 63.0f * kMScale;                  // value limit dmin * m < 63
        const float h0 = __uint_as_float(__float_as_uint(w0) & 0xFFFFE000u);
        const float h1 = __uint_as_float(__float_as_uint(w1) & 0xFFFFE000u);
        hi[g] = h2u(__floats2half2_rn(h0, h1));
        lo[g] = h2u(__floats2half2_rn(w0 - h0, w1 - h1));
    }
}

// Load-time min-operand plane of a repacked Q4_K weight (qk_q4k_min_plane): for row n and pair i of
// superblocks (2i, 2i+1), the 64 bytes a min stage's converter builds from their metadata records,
// in the order it stores them: the Mw_hi words of superblock 2i, those of 2i+1, then the Mw_lo words
// of each (a missing superblock 2i+1 gives zeros).  One thread per (n, i).
__global__ void __launch_bounds__(256) q4k_min_plane_kernel(const uint4 *__restrict__ meta, int64_t N, int B,
                                                            uint4 *__restrict__ plane)
{
    const int nmin = (B + 1) >> 1;
    const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
    bool bad = false;
    if (idx < N * nmin) {
        const int64_t n = idx / nmin;
        const int i = (int)(idx - n * nmin);
        const uint4 *rec = meta + n * B + 2 * i;
        const uint4 r0 = __ldg(rec);
        const uint4 r1 = 2 * i + 1 < B ? __ldg(rec + 1) : make_uint4(0, 0, 0, 0);
        uint32_t h0[4], l0[4], h1[4], l1[4];
        mins_hilo(r0, h0, l0, bad);
        mins_hilo(r1, h1, l1, bad);
        uint4 *o = plane + 4 * idx;
        o[0] = make_uint4(h0[0], h0[1], h0[2], h0[3]);
        o[1] = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        o[2] = make_uint4(l0[0], l0[1], l0[2], l0[3]);
        o[3] = make_uint4(l1[0], l1[1], l1[2], l1[3]);
    }
    flag_range(bad);
}

// work unit u: its tile, its segment of the tile's K range and the number of segments of that tile
struct Unit {
    int t, seg, ns;
};
__device__ __forceinline__ Unit unit_of(const MmqArgs &a, int u)
{
    if (u < a.nfull) return Unit{u, 0, 1};
    const int v = u - a.nfull;
    return Unit{a.nfull + (v >> 1), v & 1, 2};
}
// superblock range [seg_lo, seg_hi) of a unit
__device__ __forceinline__ int seg_lo(const MmqArgs &a, const Unit &un) { return un.seg == 0 ? 0 : a.mid; }
__device__ __forceinline__ int seg_hi(const MmqArgs &a, const Unit &un, int B) { return un.seg == 0 && un.ns > 1 ? a.mid : B; }

// named barrier 1 over the epilogue warps only
template <int NW>
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory"); }


template <int BN_, bool PL>
__global__ void __launch_bounds__(Plan4<BN_>::kThreads, 1)
    mmq_q4k_kernel(const MmqArgs a, const __grid_constant__ MmqMaps maps)
{
    using L = Plan4<BN_>;
    constexpr int BN = L::BN, NS = L::NST, NR = L::NRAW, NB = L::NSB, ND = L::ND;
    static_assert(kStageBar0 + NS <= 16, "a named barrier per stage slot");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + L::OFF_TMEM);
    float *dring = reinterpret_cast<float *>(smem + L::OFF_D);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = (int)(a.K >> 8), nmin = (B + 1) >> 1;
    const int ntiles = a.mtiles * a.ntiles, nunits = ntiles + (a.split > 1 ? ntiles - a.nfull : 0);

    qk::pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) mbar_init(&bar[L::FULL + i], L::kConvW + 1), mbar_init(&bar[L::EMPTY + i], 1);
        for (int i = 0; i < NR; i++) mbar_init(&bar[L::RFULL + i], 1), mbar_init(&bar[L::REMPTY + i], L::kConvW);
        for (int i = 0; i < NB; i++) mbar_init(&bar[L::SFULL + i], 1), mbar_init(&bar[L::SEMPTY + i], L::kConvW);
        for (int i = 0; i < ND; i++) mbar_init(&bar[L::DFULL + i], L::kConvW), mbar_init(&bar[L::DEMPTY + i], L::kEpiW);
        for (int i = 0; i < 2; i++) mbar_init(&bar[L::ACCFULL + i], 1), mbar_init(&bar[L::ACCEMPTY + i], L::kEpiW);
        mbar_init(&bar[L::DONE], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tmem_ptr, L::TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_ptr;
    qk::pdl_wait();
    const bool epi = warp >= L::kEpiW0 && warp < L::kEpiW0 + L::kEpiW;

    // each warpgroup sets its register count first thing in its own branch
    if (warp < L::kEpiW0) {
    if constexpr (L::kSplitRegs) reg_dealloc<L::kRegMisc>();
    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        // accumulator events in order: per tile the min term, then one per superblock.  The warp takes
        // each stage from the sync warp (warp 3) through a named barrier and lane 0 issues its MMAs: the
        // issuing thread never polls shared memory between MMAs (a poll there leaves the tensor pipe
        // idle for about 150 ns a stage)
        const uint32_t sbase = smem_u32(smem);
        int gs = 0, ge = 0;
        for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
            const Unit un = unit_of(a, u);
            const int nsb = seg_hi(a, un, B) - seg_lo(a, un);
            // events: the min term (segment 0 only), then one per superblock of the segment
            for (int ev = un.seg == 0 ? 0 : 1; ev <= nsb; ev++, ge++) {
                const int acc = ge & 1;
                const uint32_t dacc = tmem + acc * BN;
                const int nst = ev == 0 ? nmin : 8;
                for (int i = 0; i < nst; i++, gs++) {
                    const int st = gs % NS;
                    stage_sync(kStageBar0 + st);
                    if (lane == 0) {
                        fence_after_sync();
                        const uint32_t s0 = sbase + st * L::STAGE, w0 = s0 + 2 * ATILE;
                        if (ev == 0) {
                            const uint64_t shi = smem_desc(s0, 16, 512, kLayoutSw64);
                            const uint64_t slo = smem_desc(s0 + 32, 16, 512, kLayoutSw64);
                            const uint64_t mhi = smem_desc(w0, 16, 512, kLayoutSw64);
                            const uint64_t mlo = smem_desc(w0 + 32, 16, 512, kLayoutSw64);
                            mma_f16(dacc, shi, mhi, L::IDESC, i != 0);
                            mma_f16(dacc, shi, mlo, L::IDESC, 1);
                            mma_f16(dacc, slo, mhi, L::IDESC, 1);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < BK / 16; kk++) {
                                const uint64_t ahi = smem_desc(s0 + 32 * kk, 16, 512, kLayoutSw64);
                                const uint64_t alo = smem_desc(s0 + ATILE + 32 * kk, 16, 512, kLayoutSw64);
                                const uint64_t wd = smem_desc(w0 + 32 * kk, 16, 512, kLayoutSw64);
                                mma_f16(dacc, ahi, wd, L::IDESC, (i | kk) != 0);
                                mma_f16(dacc, alo, wd, L::IDESC, 1);
                            }
                        }
                        mma_commit(&bar[L::EMPTY + st]);
                        if (i == nst - 1) mma_commit(&bar[L::ACCFULL + acc]);
                    }
                    __syncwarp();
                }
            }
        }
        // teardown: no MMA may still be running when the TMEM is released
        if (lane == 0) {
            mma_commit(&bar[L::DONE]);
            wait_bar(&bar[L::DONE], 0);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------------ sync warp
        // the issuer's loop again: per stage, wait (bounded) for its operands and, at the first stage of
        // an event, for the accumulator buffer, then hand the stage to the MMA warp.  It arrives for every
        // stage even after a wait gave up, so the issuer's barrier always completes.  A stage barrier is
        // reused only after the issuer has passed it: the stage's next operands need its MMAs' commit.
        int gs = 0, ge = 0;
        for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
            const Unit un = unit_of(a, u);
            const int nsb = seg_hi(a, un, B) - seg_lo(a, un);
            for (int ev = un.seg == 0 ? 0 : 1; ev <= nsb; ev++, ge++) {
                const int acc = ge & 1;
                if (ge >= 2) wait_bar(&bar[L::ACCEMPTY + acc], ((ge >> 1) + 1) & 1);
                const int nst = ev == 0 ? nmin : 8;
                for (int i = 0; i < nst; i++, gs++) {
                    const int st = gs % NS;
                    wait_bar(&bar[L::FULL + st], (gs / NS) & 1);
                    stage_arrive(kStageBar0 + st);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ activation block copier
        // per tile the sums tiles of its min stages (8 KB each), then the A blocks (16 KB)
        if (lane == 0) {
            int gs = 0;
            for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
                const Unit un = unit_of(a, u);
                const int t = un.t, seg = un.seg, mt = t % a.mtiles;
                const uint8_t *srcS = a.wsS + (size_t)mt * nmin * SBLK;
                const uint8_t *srcA = a.wsA + (size_t)mt * (8 * B) * ABLOCK;
                // the sums tiles of the min stages (segment 0), then the A blocks of the segment's superblocks
                const int i0 = seg == 0 ? 0 : nmin + 8 * seg_lo(a, un), i1 = nmin + 8 * seg_hi(a, un, B);
                for (int i = i0; i < i1; i++, gs++) {
                    const int st = gs % NS;
                    if (gs >= NS) wait_bar(&bar[L::EMPTY + st], ((gs / NS) + 1) & 1);
                    const bool mn = i < nmin;
                    const uint32_t bytes = mn ? SBLK : ABLOCK;
                    mbar_arrive_expect_tx(&bar[L::FULL + st], bytes);
                    bulk_copy_g2s(smem + st * L::STAGE, mn ? srcS + (size_t)i * SBLK : srcA + (size_t)(i - nmin) * ABLOCK,
                                  bytes, &bar[L::FULL + st]);
                }
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ raw weight TMA producer
        // per tile: the metadata records of every superblock (min stages; with a min-operand plane, its
        // tiles instead, through the raw ring), then per superblock its record again and its code bytes
        if (lane == 0) {
            prefetch_tmap(&maps.wcodes);
            prefetch_tmap(&maps.meta);
            if (PL) prefetch_tmap(&maps.plane);
            int gsb = 0, gu = 0;
            for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
                const Unit un = unit_of(a, u);
                const int t = un.t, seg = un.seg;
                const int n0 = (t / a.mtiles) * BN;
                if (PL && seg == 0)
                    for (int i = 0; i < nmin; i++, gu++) {
                        const int rs = gu % NR;
                        if (gu >= NR) wait_bar(&bar[L::REMPTY + rs], ((gu / NR) + 1) & 1);
                        mbar_arrive_expect_tx(&bar[L::RFULL + rs], L::RAW);
                        tma_load_2d(smem + L::OFF_RAW + rs * L::RAW, &maps.plane, 64 * i, n0, &bar[L::RFULL + rs]);
                    }
                // pass 0 (segment 0, no plane): every superblock's record for the min stages; pass 1: the
                // segment's superblocks, record and code bytes
                for (int pass = seg == 0 && !PL ? 0 : 1; pass < 2; pass++) {
                    for (int sb = pass == 0 ? 0 : seg_lo(a, un); sb < (pass == 0 ? B : seg_hi(a, un, B)); sb++, gsb++) {
                        const int ss = gsb % NB;
                        if (gsb >= NB) wait_bar(&bar[L::SEMPTY + ss], ((gsb / NB) + 1) & 1);
                        mbar_arrive_expect_tx(&bar[L::SFULL + ss], L::SBR);
                        tma_load_2d(smem + L::OFF_SBR + ss * L::SBR, &maps.meta, 16 * sb, n0, &bar[L::SFULL + ss]);
                        if (pass == 0) continue;
                        // the superblock's groups u = 4 (sb - 8 s) .. +3 of its step s: first 16-byte halves
                        // at 16u, second halves at 16 G + 16u; one raw unit per pair of groups
                        const int s = sb >> 3, G = 4 * min(8, B - 8 * s), u = 4 * (sb - 8 * s);
                        for (int hs = 0; hs < 2; hs++, gu++) {
                            const int rs = gu % NR;
                            if (gu >= NR) wait_bar(&bar[L::REMPTY + rs], ((gu / NR) + 1) & 1);
                            uint8_t *d = smem + L::OFF_RAW + rs * L::RAW;
                            mbar_arrive_expect_tx(&bar[L::RFULL + rs], L::RAW);
                            tma_load_2d(d, &maps.wcodes, 1024 * s + 16 * (u + 2 * hs), n0, &bar[L::RFULL + rs]);
                            tma_load_2d(d + L::RAW_H1, &maps.wcodes, 1024 * s + 16 * G + 16 * (u + 2 * hs), n0,
                                        &bar[L::RFULL + rs]);
                        }
                    }
                }
            }
            // teardown: every copy this thread issued has landed (normally long since consumed)
            for (int g = gu - NR < 0 ? 0 : gu - NR; g < gu; g++) wait_bar(&bar[L::RFULL + g % NR], (g / NR) & 1);
            for (int g = gsb - NB < 0 ? 0 : gsb - NB; g < gsb; g++) wait_bar(&bar[L::SFULL + g % NB], (g / NB) & 1);
        }
        __syncwarp();
    }
    } else if (epi) {
        if constexpr (L::kSplitRegs) reg_alloc<L::kRegEpi>();
        // -------------------------------------------------------------- epilogue
        // thread: row (32 quad + lane) of the tile, columns ch CPT .. +CPT, in registers across the
        // tile's accumulator events; then y = R (+ residual), transposed through shared memory 16
        // columns at a time so that each store covers 16 consecutive columns of two rows
        const int ew = warp - L::kEpiW0, quad = warp & 3, ch = ew >> 2;
        const uint32_t lq = (uint32_t)(quad * 32) << 16;
        float *tb_s = reinterpret_cast<float *>(smem + L::OFF_EPI) + ew * (32 * EPI_LD);
        float R[L::CPT];
        int ge = 0, gd = 0;
        for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
            const Unit un = unit_of(a, u);
            const int t = un.t, seg = un.seg;
            const int64_t m0 = (int64_t)(t % a.mtiles) * BM, n0 = (int64_t)(t / a.mtiles) * BN;
            if (seg != 0) {
#pragma unroll
                for (int i = 0; i < L::CPT; i++) R[i] = 0.0f;
            } else {
                const int acc = ge & 1;
                wait_bar(&bar[L::ACCFULL + acc], (ge >> 1) & 1);
                fence_after_sync();
                const uint32_t tb = tmem + lq + acc * BN + ch * L::CPT;
#pragma unroll
                for (int c = 0; c < L::CPT / 16; c++) {
                    float v[16];
                    tmem_ld16(tb + 16 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; i++) R[16 * c + i] = v[i] * kMinUndo;
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::ACCEMPTY + acc]);
                ge++;
            }
#pragma unroll 1
            for (int sb = seg_lo(a, un); sb < seg_hi(a, un, B); sb++, ge++, gd++) {
                const int acc = ge & 1, ds = gd % ND;
                wait_bar(&bar[L::DFULL + ds], (gd / ND) & 1);
                wait_bar(&bar[L::ACCFULL + acc], (ge >> 1) & 1);
                fence_after_sync();
                const uint32_t tb = tmem + lq + acc * BN + ch * L::CPT;
                const float4 *dv = reinterpret_cast<const float4 *>(dring + ds * BN + ch * L::CPT);
#pragma unroll
                for (int c = 0; c < L::CPT / 8; c++) {
                    float v[8];
                    tmem_ld8(tb + 8 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 2; q++) {
                        const float4 d4 = dv[2 * c + q];
                        R[8 * c + 4 * q + 0] = __fmaf_rn(d4.x, v[4 * q + 0], R[8 * c + 4 * q + 0]);
                        R[8 * c + 4 * q + 1] = __fmaf_rn(d4.y, v[4 * q + 1], R[8 * c + 4 * q + 1]);
                        R[8 * c + 4 * q + 2] = __fmaf_rn(d4.z, v[4 * q + 2], R[8 * c + 4 * q + 2]);
                        R[8 * c + 4 * q + 3] = __fmaf_rn(d4.w, v[4 * q + 3], R[8 * c + 4 * q + 3]);
                    }
                }
                // the buffer may be overwritten once every lane's loads have completed; the scales
                // were consumed above
                fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[L::ACCEMPTY + acc]);
                    mbar_arrive(&bar[L::DEMPTY + ds]);
                }
            }
            if (un.ns > 1) {
                const int v = u - a.nfull;                 // this split unit's partial-tile slot
                // this segment's partial tile: row (32 quad + lane), columns ch CPT .. +CPT, contiguous
                const size_t poff = ((size_t)(quad * 32 + lane)) * BN + ch * L::CPT;
                float4 *mine = reinterpret_cast<float4 *>(a.part + (size_t)v * BM * BN + poff);
#pragma unroll
                for (int c = 0; c < L::CPT / 4; c++) mine[c] = make_float4(R[4 * c], R[4 * c + 1], R[4 * c + 2], R[4 * c + 3]);
                __threadfence();
                epi_sync<L::kEpiW>();
                unsigned *flag = reinterpret_cast<unsigned *>(smem + L::OFF_TMEM + 8);
                if (ew == 0 && lane == 0) {
                    const unsigned prev = atomicAdd(&a.cnt[t - a.nfull], 1u);
                    const bool last = prev == 1u;
                    if (last) {
                        __threadfence();
                        a.cnt[t - a.nfull] = 0;            // ready for the next call on this workspace
                    }
                    *flag = last ? 1u : 0u;
                }
                epi_sync<L::kEpiW>();
                const bool last = *flag != 0;
                epi_sync<L::kEpiW>();                      // the flag is read before the next unit rewrites it
                if (!last) continue;
                // the last of the two segments to finish: y = P_0 + P_1, the same bits whichever it is
                // (binary32 addition is commutative)
                const float4 *other =
                    reinterpret_cast<const float4 *>(a.part + (size_t)(v ^ 1) * BM * BN + poff);
#pragma unroll
                for (int c = 0; c < L::CPT / 4; c++) {
                    const float4 w = __ldcg(other + c);
                    R[4 * c] = __fadd_rn(R[4 * c], w.x);
                    R[4 * c + 1] = __fadd_rn(R[4 * c + 1], w.y);
                    R[4 * c + 2] = __fadd_rn(R[4 * c + 2], w.z);
                    R[4 * c + 3] = __fadd_rn(R[4 * c + 3], w.w);
                }
            }
#pragma unroll
            for (int c = 0; c < L::CPT / 16; c++) {
#pragma unroll
                for (int i = 0; i < 16; i++) tb_s[lane * EPI_LD + i] = R[16 * c + i];
                __syncwarp();
                const int64_t n = n0 + ch * L::CPT + 16 * c + (lane & 15);
                if (n < a.N) {
                    store_chunk(a, tb_s, m0 + quad * 32 + (lane >> 4), n, lane);
                }
                __syncwarp();
            }
        }
    } else {
        // one setmaxnreg for the whole warpgroup, the padding warps (no rows) included
        if constexpr (L::kSplitRegs) reg_dealloc<L::kRegConv>();
        if (warp < L::kConvW0 + L::kConvW) {
        // --------------------------------------------------------- converters
        // one thread per weight row; a quarter warp stores 8 consecutive rows, which the 64-byte
        // swizzle spreads over all 32 banks
        const int row = 32 * (warp - L::kConvW0) + lane;
        int gs = 0, gsb = 0, gu = 0, gd = 0;
        for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
            const Unit un = unit_of(a, u);
            const int seg = un.seg;
            // min stages (segment 0): sub-blocks of superblocks 2i and 2i+1 -> (Mw_hi | Mw_lo)
#pragma unroll 1
            for (int i = 0; i < (seg == 0 ? nmin : 0); i++, gs++) {
                const int st = gs % NS;
                if constexpr (PL) {
                    // the stage's operand row, built at load time: copied from the raw ring as it is
                    const int rs = gu % NR;
                    wait_bar(&bar[L::RFULL + rs], (gu / NR) & 1);
                    const uint8_t *raw = smem + L::OFF_RAW + rs * L::RAW;
                    uint4 q[4];
#pragma unroll
                    for (int c = 0; c < 4; c++) q[c] = *reinterpret_cast<const uint4 *>(raw + sw64(row, c));
                    if (gs >= NS) wait_bar(&bar[L::EMPTY + st], ((gs / NS) + 1) & 1);
                    uint8_t *w0 = smem + st * L::STAGE + 2 * ATILE;
#pragma unroll
                    for (int c = 0; c < 4; c++) sts128(w0, sw64(row, c), q[c].x, q[c].y, q[c].z, q[c].w);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bar[L::REMPTY + rs]);     // its values were stored above
                        mbar_arrive(&bar[L::FULL + st]);
                    }
                    gu++;
                    continue;
                }
                const bool two = 2 * i + 1 < B;
                const int ss0 = gsb % NB, ss1 = (gsb + 1) % NB;
                wait_bar(&bar[L::SFULL + ss0], (gsb / NB) & 1);
                const uint4 r0 = *reinterpret_cast<const uint4 *>(smem + L::OFF_SBR + ss0 * L::SBR + row * 16);
                uint4 r1 = make_uint4(0, 0, 0, 0);
                if (two) {
                    wait_bar(&bar[L::SFULL + ss1], ((gsb + 1) / NB) & 1);
                    r1 = *reinterpret_cast<const uint4 *>(smem + L::OFF_SBR + ss1 * L::SBR + row * 16);
                }
                uint32_t h0[4], l0[4], h1[4], l1[4];
                bool bad = false;
                mins_hilo(r0, h0, l0, bad);
                mins_hilo(r1, h1, l1, bad);
                flag_range(bad);
                if (gs >= NS) wait_bar(&bar[L::EMPTY + st], ((gs / NS) + 1) & 1);
                uint8_t *w0 = smem + st * L::STAGE + 2 * ATILE;
                sts128(w0, sw64(row, 0), h0[0], h0[1], h0[2], h0[3]);
                sts128(w0, sw64(row, 1), h1[0], h1[1], h1[2], h1[3]);
                sts128(w0, sw64(row, 2), l0[0], l0[1], l0[2], l0[3]);
                sts128(w0, sw64(row, 3), l1[0], l1[1], l1[2], l1[3]);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[L::SEMPTY + ss0]);
                    if (two) mbar_arrive(&bar[L::SEMPTY + ss1]);
                    mbar_arrive(&bar[L::FULL + st]);
                }
                gsb += two ? 2 : 1;
            }
            // main stages: per superblock its scale d into the scale ring, then sub-block j -> W' = sc q
#pragma unroll 1
            for (int sb = seg_lo(a, un); sb < seg_hi(a, un, B); sb++, gsb++, gd++) {
                const int ss = gsb % NB, ds = gd % ND;
                wait_bar(&bar[L::SFULL + ss], (gsb / NB) & 1);
                const uint4 mt = *reinterpret_cast<const uint4 *>(smem + L::OFF_SBR + ss * L::SBR + row * 16);
                if (gd >= ND) wait_bar(&bar[L::DEMPTY + ds], ((gd / ND) + 1) & 1);
                dring[ds * BN + row] = __half2float(__ushort_as_half((unsigned short)(mt.x & 0xffffu)));
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[L::DFULL + ds]);
                // sub-blocks 2g and 2g+1 (the low and high nibbles of group g's code bytes) are converted
                // together: one proxy fence and one warp handoff for both stages
                int rs = 0;
#pragma unroll
                for (int g = 0; g < 4; g++, gs += 2) {
                    const int st0 = gs % NS, st1 = (gs + 1) % NS;
                    if ((g & 1) == 0) {
                        rs = gu % NR;
                        wait_bar(&bar[L::RFULL + rs], (gu / NR) & 1);
                    }
                    const uint8_t *raw = smem + L::OFF_RAW + rs * L::RAW;
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(raw + sw32(row, g & 1));
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(raw + L::RAW_H1 + sw32(row, g & 1));
                    const uint32_t rec = q4_group(mt, g);
                    const ScPair k0 = sc_pair(rec & 63u), k1 = sc_pair((rec >> 6) & 63u);
                    if (gs >= NS) wait_bar(&bar[L::EMPTY + st0], ((gs / NS) + 1) & 1);
                    if (gs + 1 >= NS) wait_bar(&bar[L::EMPTY + st1], (((gs + 1) / NS) + 1) & 1);
                    uint8_t *w0 = smem + st0 * L::STAGE + 2 * ATILE;
                    uint8_t *w1 = smem + st1 * L::STAGE + 2 * ATILE;
                    const uint32_t x[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int cc = 0; cc < 4; cc++) {
                        uint32_t p0, p1, p2, p3;
                        w_sc(x[2 * cc] & 0x0F0F0F0Fu, k0, p0, p1);
                        w_sc(x[2 * cc + 1] & 0x0F0F0F0Fu, k0, p2, p3);
                        sts128(w0, sw64(row, cc), p0, p1, p2, p3);
                        w_sc((x[2 * cc] >> 4) & 0x0F0F0F0Fu, k1, p0, p1);
                        w_sc((x[2 * cc + 1] >> 4) & 0x0F0F0F0Fu, k1, p2, p3);
                        sts128(w1, sw64(row, cc), p0, p1, p2, p3);
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        if (g & 1) mbar_arrive(&bar[L::REMPTY + rs]);        // last read of this raw unit
                        if (g == 0) mbar_arrive(&bar[L::SEMPTY + ss]);
                        mbar_arrive(&bar[L::FULL + st0]);
                        mbar_arrive(&bar[L::FULL + st1]);
                    }
                    if (g & 1) gu++;
                }
            }
        }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tmem, L::TMEM_COLS);
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
              uint64_t rows, uint64_t pitch, uint32_t bx, uint32_t by,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {bx, by};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// workspace bytes for an M x K activation: one A block per M-tile and 32-value K stage, then one
// sums tile per M-tile and pair of superblocks
size_t ws_a_bytes(int64_t M, int64_t K)
{
    const size_t mt = (size_t)((M + BM - 1) / BM);
    return mt * (size_t)(K / BK) * ABLOCK;
}
size_t ws_bytes(int64_t M, int64_t K)
{
    const size_t mt = (size_t)((M + BM - 1) / BM);
    return ws_a_bytes(M, K) + mt * (size_t)((K / 256 + 1) / 2) * SBLK;
}

// Split of each tile's K range over two work units (Q4_K, QK_MMQ_SPLIT_K): each unit needs kMinSegSb
// superblocks or more.  Segment 0 covers superblocks [0, mid) and the min term, segment 1 [mid, K/256).
constexpr int kMinSegSb = 24;

// first superblock of segment 1: the two segments' MMA work balanced, segment 0 also carrying the min term
int split_mid(int B)
{
    const double c = 3.0 * ((B + 1) / 2) / 32.0;                // the min term in superblock units
    int b = (int)((B + c) / 2 - c + 0.5);
    return b < 1 ? 1 : b > B - 1 ? B - 1 : b;
}

// tile width and split of a Q4_K call on `sms` SMs
struct Q4Plan {
    int BN, split;
    int64_t tiles;
    int64_t tail;           // split == 2: the tiles split in two (the last `tail` ones)
};

// Time of one work unit: a fixed part (the tile's pipeline start and its output) and a part per K
// stage, measured per tile width on the Qwen2-7B prefill GEMMs (K = 3584 and 18944, split-scale kernel
// with the sync warp and the min-operand plane): 256: 40 us + 0.43 us a stage, 192: 26 + 0.48,
// 128: 14 + 0.424.  A unit of a split tile adds 40 us (its partial tile out and back, its own
// pipeline start; measured with every down tile split: 648 us for three waves of half tiles).
double unit_us(int BN, int64_t stages, int split)
{
    const double a = BN == 256 ? 40.0 : BN == 192 ? 26.0 : 14.0, b = BN == 256 ? 0.43 : BN == 192 ? 0.48 : 0.424;
    return a + b * (double)stages + (split > 1 ? 40.0 : 0.0);
}

// The width, and whether to split the tiles of a poorly filled last wave, whose waves of work units
// over the SMs should finish first.  A forced width (QK_MMQ_TILE_*) is taken as it is; QK_MMQ_SPLIT_K
// splits every tile.  A split needs K of at least 2 kMinSegSb superblocks; the tail split takes the
// last wave's tiles (fewer than half the SMs) as two units each, so that the tail runs as one wave
// of half tiles: Qwen2-7B down, 224 tiles of 256 on 152 SMs, 152 whole tiles then 144 half tiles.
Q4Plan q4_plan(int64_t M, int64_t N, int64_t K, unsigned flags, int sms, int max_split = kMaxSplit)
{
    if (sms < 1) sms = 1;
    const int forced = (flags & QK_MMQ_TILE_256) ? 256 : (flags & QK_MMQ_TILE_192) ? 192
                     : (flags & QK_MMQ_TILE_128) ? 128 : 0;
    const int widths[3] = {256, 192, 128};
    const int64_t gx = (M + BM - 1) / BM, B = K / 256, stages = 8 * B + (B + 1) / 2;
    const bool can_split = max_split >= 2 && B >= 2 * kMinSegSb;
    Q4Plan best{256, 1, gx * ((N + 255) / 256), 0};
    double bc = 1e300;
    for (int wi = 0; wi < 3; wi++) {
        const int BN = widths[wi];
        if (forced && BN != forced) continue;
        const int64_t tiles = gx * ((N + BN - 1) / BN);
        if (can_split && (flags & QK_MMQ_SPLIT_K)) {                   // every tile split
            best = Q4Plan{BN, 2, tiles, tiles};
            bc = 0.0;
            continue;
        }
        const double c = (double)((tiles + sms - 1) / sms) * unit_us(BN, stages, 1);
        if (c < bc * (1.0 - 1e-9)) bc = c, best = Q4Plan{BN, 1, tiles, 0};
        const int64_t tail = tiles % sms;
        if (can_split && tail > 0 && 2 * tail <= sms) {
            const double ct = (double)(tiles / sms) * unit_us(BN, stages, 1) + unit_us(BN, stages / 2, 2);
            if (ct < bc * (1.0 - 1e-9)) bc = ct, best = Q4Plan{BN, 2, tiles, tail};
        }
    }
    return best;
}

// scratch of a split call after the base workspace: two partial tiles per split tile, then one
// counter per split tile
size_t split_bytes(const Q4Plan &p)
{
    if (p.split <= 1) return 0;
    return (size_t)p.tail * 2 * BM * p.BN * 4 + (size_t)p.tail * 4;
}

// The register-split kernel must be launched with at least the registers its setmaxnreg split hands
// out: with fewer, the epilogue warps' increase could never be granted.  Checked once per kernel,
// before its first launch.
template <int BN, bool PL>
int set_attrs_q4()
{
    static std::atomic<int> done_dev[qk::kMaxDevices];
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    std::atomic<int> &done = done_dev[dev];
    if (done.load()) return QK_OK;
    if (cudaFuncSetAttribute(mmq_q4k_kernel<BN, PL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Plan4<BN>::SMEM) != cudaSuccess ||
        qk::max_carveout(mmq_q4k_kernel<BN, PL>) != cudaSuccess)
        return QK_E_CUDA;
    if (Plan4<BN>::kSplitRegs) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, mmq_q4k_kernel<BN, PL>) != cudaSuccess || fa.numRegs < Plan4<BN>::kRegLaunch)
            return QK_E_CUDA;
    }
    done.store(1);
    return QK_OK;
}

template <int BN, bool PL>
int launch_mmq_q4(const MmqArgs &args, const MmqMaps &maps, int64_t tiles, cudaStream_t stream)
{
    const int st = set_attrs_q4<BN, PL>();
    if (st != QK_OK) return st;
    const int64_t grid = tiles < qk::sm_count() ? tiles : qk::sm_count();
    return qk::launch(mmq_q4k_kernel<BN, PL>, dim3((unsigned)grid), dim3(Plan4<BN>::kThreads), Plan4<BN>::SMEM,
                      stream, true, args, maps);
}

template <int QT, int BN>
int set_attrs()
{
    static std::atomic<int> done_dev[qk::kMaxDevices];
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    std::atomic<int> &done = done_dev[dev];
    if (done.load()) return QK_OK;
    if (cudaFuncSetAttribute(mmq_kernel<QT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Plan<QT, BN>::SMEM) != cudaSuccess ||
        qk::max_carveout(mmq_kernel<QT, BN>) != cudaSuccess)
        return QK_E_CUDA;
    done.store(1);
    return QK_OK;
}

// Tile width for an M x N problem on `sms` SMs.  A CTA takes ceil(tiles / sms) tiles one after the
// other.  A 128-wide tile takes about 0.7 of a 256-wide one (measured on the prefill shapes: the
// activation operand, the MMA issue and the epilogue do not halve with the tile), so 128 is taken
// only where ceil(tiles_128 / sms) * 0.7 < ceil(tiles_256 / sms): in practice single-wave problems.
int pick_bn(int64_t M, int64_t N, int sms)
{
    if (sms < 1) sms = 1;
    const int64_t gx = (M + BM - 1) / BM;
    const int64_t w256 = (gx * ((N + 255) / 256) + sms - 1) / sms, w128 = (gx * ((N + 127) / 128) + sms - 1) / sms;
    return w128 * 7 < w256 * 10 ? 128 : 256;
}

template <int QT, int BN>
int launch_mmq(const MmqArgs &args, const MmqMaps &maps, int64_t tiles, cudaStream_t stream)
{
    const int st = set_attrs<QT, BN>();
    if (st != QK_OK) return st;
    const int64_t grid = tiles < qk::sm_count() ? tiles : qk::sm_count();
    return qk::launch(mmq_kernel<QT, BN>, dim3((unsigned)grid), dim3(Plan<QT, BN>::kThreads), Plan<QT, BN>::SMEM,
                      stream, true, args, maps);
}

// bytes of the Q4_K min-operand plane of an N x K weight: 64 per row and pair of superblocks
size_t plane_bytes(int64_t N, int64_t K) { return (size_t)N * (size_t)((K / 256 + 1) / 2) * 64; }

// The activation comes as q8_1 (codes, scales) or, for the f32 entry points, as f32 rows x with row
// pitch ldx (quantized inside the prep kernel; codes and scales are then null).
int mmq(int qt, const void *w, const void *plane, const int8_t *codes, const void *scales, const float *x,
        int64_t ldx, int64_t M, int64_t N, int64_t K, const float *residual, float *y, void *workspace,
        size_t workspace_bytes, unsigned flags, void *stream)
{
    // TMA coordinates are signed 32-bit: rows and bytes of a row stay below 2^31
    if (M < 0 || N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || M > 0x7fffffffLL || K > 0x7fffffffLL)
        return QK_E_SHAPE;
    if (x && (ldx < K || ldx > ((int64_t)1 << 40))) return QK_E_SHAPE;
    if (M == 0) return QK_OK;
    if (!w || (!x && (!codes || !scales)) || !y || !workspace) return QK_E_NULL;
    if (!qk::aligned(w, 16) || !qk::aligned(codes, 16) || !qk::aligned(scales, 16) || !qk::aligned(y, 4) ||
        (residual && !qk::aligned(residual, 4)) || !qk::aligned(workspace, 256) || !qk::aligned(plane, 16) ||
        !qk::aligned(x, 16) || (x && ldx % 4 != 0))
        return QK_E_ALIGN;
    const size_t need = ws_bytes(M, K);
    if (workspace_bytes < need) return QK_E_WORKSPACE;
    const unsigned tf = flags & (QK_MMQ_TILE_256 | QK_MMQ_TILE_192 | QK_MMQ_TILE_128);
    if (tf & (tf - 1)) return QK_E_SHAPE;                               // more than one width forced
    const int sms = qk::sm_count();
    Q4Plan plan;
    if (qt == QK_TYPE_Q6_K) {
        if (tf == QK_MMQ_TILE_192) return QK_E_SHAPE;                   // Q6_K tiles are 128 or 256 wide
        plan.BN = tf == QK_MMQ_TILE_256 ? 256 : tf == QK_MMQ_TILE_128 ? 128 : pick_bn(M, N, sms);
        plan.split = 1;
        plan.tiles = ((M + BM - 1) / BM) * ((N + plan.BN - 1) / plan.BN);
        plan.tail = 0;
    } else {
        plan = q4_plan(M, N, K, flags, sms);
        if (workspace_bytes < need + split_bytes(plan)) plan = q4_plan(M, N, K, flags, sms, 1);  // no scratch
    }
    const size_t used = need + split_bytes(plan);                     // the workspace bytes this call writes
    size_t wbytes = 0;
    qk_repacked_bytes(qt, N, K, &wbytes);
    const size_t ybytes = (size_t)M * N * 4, cbytes = (size_t)M * K, sbytes = (size_t)M * (K / 32) * 4;
    const size_t xbytes = x ? ((size_t)(M - 1) * (size_t)ldx + (size_t)K) * 4 : 0;
    if (x && (qk::overlaps(y, ybytes, x, xbytes) || qk::overlaps(workspace, used, x, xbytes)))
        return QK_E_ALIAS;
    if (qk::overlaps(y, ybytes, w, wbytes) || qk::overlaps(y, ybytes, codes, cbytes) ||
        qk::overlaps(y, ybytes, scales, sbytes) || (residual != y && qk::overlaps(y, ybytes, residual, ybytes)) ||
        qk::overlaps(workspace, used, w, wbytes) || qk::overlaps(workspace, used, codes, cbytes) ||
        qk::overlaps(workspace, used, scales, sbytes) || qk::overlaps(workspace, used, y, ybytes) ||
        (residual && qk::overlaps(workspace, used, residual, ybytes)) ||
        (plane && (qk::overlaps(y, ybytes, plane, plane_bytes(N, K)) ||
                   qk::overlaps(workspace, used, plane, plane_bytes(N, K)))))
        return QK_E_ALIAS;
    const int BN = plan.BN;
    const int64_t gx = (M + BM - 1) / BM, gy = (N + BN - 1) / BN;
    if (gx > 65535 || gy > 65535 || gx * gy > 0x7fffffffLL) return QK_E_SHAPE;
    const bool q6 = qt == QK_TYPE_Q6_K;
    const size_t smem = q6 ? (size_t)Plan<QK_TYPE_Q6_K, 256>::SMEM : (size_t)Plan4<256>::SMEM;
    if (smem > qk::max_smem_optin()) return QK_E_CUDA;     // the larger plan of each weight type
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return QK_E_CUDA;
    const int64_t B = K / 256;
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    MmqMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!q6) {
        if (!make_map(enc, &maps.wcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb, B * 128, N, B * 128, 32, (uint32_t)BN,
                      CU_TENSOR_MAP_SWIZZLE_32B) ||
            !make_map(enc, &maps.meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb + N * B * 128, B * 16, N, B * 16, 16,
                      (uint32_t)BN))
            return QK_E_CUDA;
        const uint64_t prow = (uint64_t)((B + 1) / 2) * 64;
        if (plane && !make_map(enc, &maps.plane, CU_TENSOR_MAP_DATA_TYPE_UINT8, plane, prow, N, prow, 64,
                               (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_64B))
            return QK_E_CUDA;
    } else {
        if (!make_map(enc, &maps.wcodes, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb, B * 128, N, B * 128, 32, (uint32_t)BN) ||
            !make_map(enc, &maps.qh, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb + N * B * 128, B * 64, N, B * 64, 32,
                      (uint32_t)BN) ||
            !make_map(enc, &maps.meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, wb + N * B * 192, B * 16, N, B * 16, 16,
                      (uint32_t)BN))
            return QK_E_CUDA;
    }
    uint8_t *wsA = static_cast<uint8_t *>(workspace);
    uint8_t *wsS = q6 ? nullptr : wsA + ws_a_bytes(M, K);
    const int64_t tiles = gx * gy;
    cudaStream_t cs = (cudaStream_t)stream;
    if (!q6) {
        // validate the main kernel's launch configuration before anything is launched
        const int sa = plane ? (BN == 128 ? set_attrs_q4<128, true>() : BN == 192 ? set_attrs_q4<192, true>()
                                                                       : set_attrs_q4<256, true>())
                             : (BN == 128 ? set_attrs_q4<128, false>() : BN == 192 ? set_attrs_q4<192, false>()
                                                                       : set_attrs_q4<256, false>());
        if (sa != QK_OK) return sa;
    }
    float *part = nullptr;
    unsigned *cnt = nullptr;
    if (plan.split > 1) {
        part = reinterpret_cast<float *>(wsA + need);
        cnt = reinterpret_cast<unsigned *>(wsA + need + (size_t)plan.tail * 2 * BM * BN * 4);
    }
    const int ncnt = plan.split > 1 ? (int)plan.tail : 0;
    int st = x ? qk::launch(mmq_prep_f32_kernel, dim3((unsigned)(K / 32), (unsigned)gx), dim3(256), 0, cs,
                            (flags & QK_LAUNCH_PDL) != 0, x, ldx, M, K, wsA, wsS, cnt, ncnt)
               : qk::launch(mmq_prep_kernel, dim3((unsigned)(K / 32), (unsigned)gx), dim3(256), 0, cs,
                            (flags & QK_LAUNCH_PDL) != 0, codes, static_cast<const __half2 *>(scales), M, K, wsA,
                            wsS, cnt, ncnt);
    if (st != QK_OK) return st;
    MmqArgs args{};
    args.wsA = wsA;
    args.wsS = wsS;
    args.dq = q6 ? reinterpret_cast<const uint16_t *>(wb + N * B * 208) : nullptr;
    args.M = M;
    args.N = N;
    args.K = K;
    args.residual = residual;
    args.y = y;
    args.mtiles = (int)gx;
    args.ntiles = (int)gy;
    args.split = plan.split;
    args.nfull = (int)(plan.split > 1 ? tiles - plan.tail : tiles);
    args.mid = plan.split > 1 ? split_mid((int)B) : (int)B;
    args.part = part;
    args.cnt = cnt;
    if (q6) return BN == 128 ? launch_mmq<QK_TYPE_Q6_K, 128>(args, maps, tiles, cs)
                             : launch_mmq<QK_TYPE_Q6_K, 256>(args, maps, tiles, cs);
    const int64_t units = tiles + (plan.split > 1 ? plan.tail : 0);
    if (plane)
        return BN == 128   ? launch_mmq_q4<128, true>(args, maps, units, cs)
               : BN == 192 ? launch_mmq_q4<192, true>(args, maps, units, cs)
                           : launch_mmq_q4<256, true>(args, maps, units, cs);
    return BN == 128   ? launch_mmq_q4<128, false>(args, maps, units, cs)
           : BN == 192 ? launch_mmq_q4<192, false>(args, maps, units, cs)
                       : launch_mmq_q4<256, false>(args, maps, units, cs);
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
    // the scratch of the tail split the call would take on this device (QK_MMQ_SPLIT_K's is the
    // caller's to add)
    *bytes = ws_bytes(M, K) + (M > 0 ? split_bytes(q4_plan(M, N, K, 0, qk::sm_count())) : 0);
    return QK_OK;
}

namespace qk {
// the workspace a call needs without the split scratch (a workspace of this size runs unsplit)
size_t mmq_base_workspace_bytes(int64_t M, int64_t K) { return ws_bytes(M, K); }
}  // namespace qk

extern "C" int qk_mmq_q4k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N, int64_t K,
                          const float *residual, float *y, void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream)
{
    return mmq(QK_TYPE_Q4_K, w, nullptr, codes, scales, nullptr, 0, M, N, K, residual, y, workspace,
               workspace_bytes, flags, stream);
}

extern "C" int qk_q4k_min_plane_bytes(int64_t N, int64_t K, size_t *bytes)
{
    if (!bytes) return QK_E_NULL;
    if (N < 1 || K < 256 || K % 256 != 0) return QK_E_SHAPE;
    *bytes = plane_bytes(N, K);
    return QK_OK;
}

extern "C" int qk_q4k_min_plane(const void *w, int64_t N, int64_t K, void *plane, size_t bytes, void *stream)
{
    if (N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || K > 0x7fffffffLL) return QK_E_SHAPE;
    if (!w || !plane) return QK_E_NULL;
    if (!qk::aligned(w, 16) || !qk::aligned(plane, 16)) return QK_E_ALIGN;
    const size_t need = plane_bytes(N, K);
    if (bytes < need) return QK_E_WORKSPACE;
    size_t wbytes = 0;
    qk_repacked_bytes(QK_TYPE_Q4_K, N, K, &wbytes);
    if (qk::overlaps(plane, need, w, wbytes)) return QK_E_ALIAS;
    const int B = (int)(K / 256);
    const int64_t threads = N * ((B + 1) / 2), blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return QK_E_SHAPE;
    const uint4 *meta = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(w) + (size_t)N * B * 128);
    return qk::launch(q4k_min_plane_kernel, dim3((unsigned)blocks), dim3(256), 0, (cudaStream_t)stream, false, meta,
                      N, B, static_cast<uint4 *>(plane));
}

extern "C" int qk_mmq_q4k_plane(const void *w, const void *plane, const int8_t *codes, const void *scales, int64_t M,
                                int64_t N, int64_t K, const float *residual, float *y, void *workspace,
                                size_t workspace_bytes, unsigned flags, void *stream)
{
    if (M > 0 && !plane) return QK_E_NULL;
    return mmq(QK_TYPE_Q4_K, w, plane, codes, scales, nullptr, 0, M, N, K, residual, y, workspace, workspace_bytes,
               flags, stream);
}

extern "C" int qk_mmq_q4k_f32(const void *w, const void *plane, const float *x, int64_t ldx, int64_t M, int64_t N,
                              int64_t K, const float *residual, float *y, void *workspace, size_t workspace_bytes,
                              unsigned flags, void *stream)
{
    if (M > 0 && !x) return QK_E_NULL;
    return mmq(QK_TYPE_Q4_K, w, plane, nullptr, nullptr, x, ldx, M, N, K, residual, y, workspace, workspace_bytes,
               flags, stream);
}

extern "C" int qk_mmq_q6k_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                              const float *residual, float *y, void *workspace, size_t workspace_bytes,
                              unsigned flags, void *stream)
{
    if (M > 0 && !x) return QK_E_NULL;
    return mmq(QK_TYPE_Q6_K, w, nullptr, nullptr, nullptr, x, ldx, M, N, K, residual, y, workspace, workspace_bytes,
               flags, stream);
}

extern "C" int qk_mmq_q6k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N, int64_t K,
                          const float *residual, float *y, void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream)
{
    return mmq(QK_TYPE_Q6_K, w, nullptr, codes, scales, nullptr, 0, M, N, K, residual, y, workspace,
               workspace_bytes, flags, stream);
}
