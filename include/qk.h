/*
 * qk.h -- C ABI of the GB300 (sm_103a) k-quant x q8_1 contraction library.
 *
 * The library computes the hot path of Q4_K_M LLM inference:
 *   1. quantize f32 activations to q8_1 blocks          (qk_quantize_q8_1)
 *   2. once, at load time, repack GGUF Q4_K / Q6_K weights into the device
 *      layout below                                       (qk_repack)
 *   3. y = x_q8 . W^T (+ r) for a few activation rows     (qk_gemv_q4k, qk_gemv_q6k)
 *   4. the same for many rows (prefill)                   (qk_mmq_q4k)
 * with y[m][n] = sum_k w[n][k] * xhat[m][k] (+ r[m][n]), xhat = d_a * q_a the
 * dequantized q8_1 activation and w the dequantized weight.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must be device memory of the current
 *    CUDA device (or managed memory); host pointers are never accepted in
 *    their place.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *  - The caller owns all memory.  No call allocates, frees or keeps a
 *    pointer after it returns; every compute call is asynchronous on
 *    `stream`.  The library keeps no per-call state.
 *  - Arguments are validated on the host before anything is launched.  On
 *    a validation error nothing is launched and a negative QK_E_* status is
 *    returned.  QK_E_CUDA means a CUDA runtime call failed (the launch
 *    itself, or a kernel attribute call); errors of earlier asynchronous
 *    work on the stream can also surface there.
 *  - Matrices are row-major.  N = output rows of W, K = reduction length,
 *    M = activation rows (tokens).  K must be a positive multiple of 256.
 *  - Floating point is IEEE: no fast-math; reductions run in a fixed order,
 *    so results are identical from run to run on the same device.
 */
#ifndef QK_H
#define QK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define QK_OK 0
#define QK_E_NULL (-1)      /* a required pointer is NULL                     */
#define QK_E_SHAPE (-2)     /* M, N or K out of range, or K % 256 != 0        */
#define QK_E_ALIGN (-3)     /* a pointer or leading dimension is misaligned   */
#define QK_E_ALIAS (-4)     /* an output overlaps an input it may not overlap */
#define QK_E_TYPE (-5)      /* unknown quantization type                      */
#define QK_E_WORKSPACE (-6) /* workspace too small                            */
#define QK_E_CUDA (-7)      /* a CUDA runtime call failed                     */

/* quantization types for qk_repacked_bytes / qk_repack */
#define QK_TYPE_Q4_K 1
#define QK_TYPE_Q6_K 2
#define QK_TYPE_Q5_K 3
#define QK_TYPE_Q8_0 4
#define QK_TYPE_Q2_K 5
#define QK_TYPE_Q3_K 6

/* flags for the compute calls */
#define QK_LAUNCH_PDL 1u
/*
 * QK_LAUNCH_PDL: launch with programmatic dependent launch, so the kernel
 * can start while the previous kernel on the stream is still running.  The
 * kernel waits for that kernel (and so for everything before it) to finish
 * before it reads any activation, scale or residual or writes any output.
 * A GEMV or MMQ launched this way may read its weight buffer `w` EARLY: the
 * caller guarantees that no work still in flight on the stream writes `w`
 * (e.g. qk_repack must have completed, or have been followed by another
 * launch, before the first PDL launch that reads its output).  Without the
 * flag every call is ordinary stream-ordered work.
 *
 * QK_MMQ_TILE_256 / QK_MMQ_TILE_192 / QK_MMQ_TILE_128 (MMQ only): force
 * output tiles 256, 192 (Q4_K only) or 128 weight rows wide.  By default the
 * MMQ picks per call the width whose waves of tiles over the SMs should
 * finish first, from a per-width model of a tile's time (a fixed part and a
 * part per 32-value K stage, measured on the prefill shapes): in practice
 * 128 for problems that fit in one wave, 192 for short K where 256-wide tiles
 * leave a second wave half empty, 256 otherwise.  Results are the same
 * within the stated bound either way; the flags exist for tests and tuning.
 * Setting more than one, or QK_MMQ_TILE_192 for Q6_K, is QK_E_SHAPE.
 *
 * QK_MMQ_SPLIT_K (Q4_K MMQ only): split every output tile's K range over two
 * work units, the second to finish adding the two partial tiles (binary32,
 * the same bits either way).  Taken only when K has at least 48 superblocks
 * and the workspace also holds the split scratch (see qk_mmq_q4k); otherwise
 * ignored.  By default only the tiles of a poorly filled last wave are
 * split (qk_mmq_q4k); splitting every tile measured slower.
 */
#define QK_MMQ_TILE_256 2u
#define QK_MMQ_TILE_128 4u
#define QK_MMQ_TILE_192 8u
#define QK_MMQ_SPLIT_K 16u

/*
 * QK_GEMV_ROWS4 / QK_GEMV_ROWS2 (Q4_K and Q6_K GEMV, M >= 3): force items of
 * four or of two weight rows.  An item is the slice of weight rows a warp
 * takes through its shared-memory ring; with four rows one read of the
 * staged activation serves four rows instead of two, which halves the
 * activation traffic per weight byte where several activation rows make the
 * GEMV bound by instruction issue and shared-memory reads.  By default four
 * rows are taken for Q4_K when the groups of four rows still give every warp
 * of the grid one group (N >= 4 * 12 warps * SMs) and the ring and the
 * activation fit in shared memory; QK_GEMV_ROWS4 drops the first condition
 * and also applies to Q6_K (measured slower there at M = 4: its four-row
 * kernel runs 12 warps instead of 16).
 * Results are the same within the stated bound either way (the reduction
 * order is fixed for a given choice).  Setting both is QK_E_SHAPE for any
 * GEMV call; the other GEMV formats and the MMQ calls ignore them otherwise.
 */
#define QK_GEMV_ROWS4 32u
#define QK_GEMV_ROWS2 64u

/* Library version (major*10000 + minor*100 + patch). */
int qk_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *qk_status_string(int status);

/* ==================================================================== q8_1
 * q8_1 activation blocks (leone-cuda "CUDA kernel design": each q8_1 block
 * stores 32 signed codes, an f16 scale and an f16 source sum; minfer
 * "15 . The CUDA backend" sec. 2.3 quantizes the activations once per
 * matmul in a small prepass).
 *
 * Layout of a quantized M x K activation (two caller buffers):
 *   codes:  int8   [M][K]      row-major, row stride K
 *   scales: half2  [M][K/32]   (.x = d, .y = s) as IEEE binary16
 * For block b of row m (values x[32b .. 32b+31]):
 *   amax = max |x_i| (binary32), d = amax / 127 (binary32 division),
 *   q_i  = roundf(x_i / d) in [-127, 127] (ties away from zero; 0 if d == 0),
 *   s    = d * sum_i q_i (binary32),
 *   stored d and s are binary16, round to nearest even, saturating at
 *   +-65504.
 */

/* Sizes of the two q8_1 buffers for an M x K activation. */
int qk_q8_1_bytes(int64_t M, int64_t K, size_t *codes_bytes, size_t *scales_bytes);

/*
 * x:      device, float [M][ldx], 16-byte aligned, ldx % 4 == 0, ldx >= K.
 * codes:  device, int8 [M][K], 16-byte aligned.
 * scales: device, half2 [M][K/32], 16-byte aligned.
 * M >= 0 (0 launches nothing), K % 32 == 0 and K > 0.  Outputs must not
 * overlap x.  Codes and scales match the definition above bit for bit.
 */
int qk_quantize_q8_1(const float *x, int64_t ldx, int64_t M, int64_t K,
                     int8_t *codes, void *scales, unsigned flags, void *stream);

/* =============================================================== producers
 * The producers of GEMV / MMQ inputs with the q8_1 pack fused into their
 * write-out, so that no standalone quantization runs before the next
 * contraction (leone-cuda "CUDA kernel design": RMSNorm and SwiGLU write
 * their dense output and its q8_1 blocks in one kernel; minfer "15 . The
 * CUDA backend" sec. 3.2.5: decode producers fuse an int8 quantize epilogue
 * so the following MMVQ skips its quantize launch).  The codes and scales
 * are exactly those qk_quantize_q8_1 gives for the binary32 output the kernel
 * computes, whether or not that output is also written.
 *
 * qk_rmsnorm_q8_1: per row m, s = x[m] (+ r[m], binary32 add),
 *   y = (s * inv) * g with inv = 1 / sqrtf(sum(s^2) / K + eps), all IEEE
 *   binary32; the square sum is taken in a fixed order (reruns give the same
 *   bits), sqrtf is the IEEE square root (leone-cuda: not the approximate
 *   reciprocal square root).
 *   x:      device float [M][ldx], 16-byte aligned, ldx % 4 == 0, ldx >= K.
 *   r:      device float [M][K] or NULL (the residual-stream variant: left +
 *           right is normalized), 16-byte aligned.
 *   g:      device float [K], the norm weight, 16-byte aligned.
 *   eps:    >= 0 and finite.
 *   h_out:  device float [M][K] or NULL; receives s (with r: the updated
 *           residual stream x + r).
 *   y:      device float [M][K] or NULL; receives the normalized row.
 *   codes, scales: q8_1 of y, laid out as qk_quantize_q8_1's outputs.
 *   M >= 0 (0 launches nothing), K % 32 == 0.  Outputs are 16-byte aligned
 *   and overlap neither the inputs nor each other.
 */
int qk_rmsnorm_q8_1(const float *x, int64_t ldx, const float *r, const float *g, float eps,
                    int64_t M, int64_t K, float *h_out, float *y,
                    int8_t *codes, void *scales, unsigned flags, void *stream);

/*
 * qk_swiglu_q8_1: per row m, h = silu(gate) * up = (g / (1 + expf(-g))) * u
 *   in binary32 (expf: the CUDA math library's accurate exponential, IEEE
 *   division and multiply), gate = gu[m][0 .. F), up = gu[m][F .. 2F): the
 *   output row of the concatenated gate||up GEMV.
 *   gu:     device float [M][ldgu], 16-byte aligned, ldgu % 4 == 0,
 *           ldgu >= 2F.
 *   h:      device float [M][F] or NULL; receives silu(gate) * up.
 *   codes, scales: q8_1 of h ([M][F] and [M][F/32]).
 *   0 <= M <= 65535, F % 32 == 0.  Outputs are 16-byte aligned and overlap
 *   neither gu nor each other.
 */
int qk_swiglu_q8_1(const float *gu, int64_t ldgu, int64_t M, int64_t F, float *h,
                   int8_t *codes, void *scales, unsigned flags, void *stream);

/* ================================================================== repack
 * Load-time lossless repack of GGUF k-quant weights into the device layout
 * that the GEMV and MMQ kernels stream with aligned 16-byte loads (leone-cuda
 * "CUDA kernel design" splits Q4_K codes from metadata; minfer "15 . The CUDA
 * backend" sec. 3.2.2 pads Q6_K's 210-byte blocks for aligned loads -- this
 * layout splits Q6_K into planes instead and adds no padding).
 *
 * GGUF input: row-major [N][K/256] superblocks;
 *   Q4_K 144 B: f16 d, f16 dmin, 12 B packed 6-bit scales/mins, 128 B codes;
 *   Q6_K 210 B: 128 B low 4 bits, 64 B high 2 bits, 16 int8 scales, f16 d.
 *   Q5_K 176 B: f16 d, f16 dmin, 12 B 6-bit scales/mins packed as for Q4_K,
 *     32 B qh (value 64g+l takes bit 2g of qh[l] as its fifth bit, value
 *     64g+32+l bit 2g+1), 128 B qs (low / high nibbles as for Q4_K).
 *   Q8_0 34 B per 32 values: f16 d, 32 int8 codes (w = d * q).
 *   Q2_K 84 B: scales[16] (low nibble scale, high nibble min of each 16
 *     values), qs[64] (2-bit codes), f16 d, f16 dmin; value 128n+32j+l takes
 *     bits 2j of qs[32n+l] and the scale byte of sub-block 8n+2j+(l>=16):
 *     w = d*sc*q - dmin*m.
 *   Q3_K 110 B: hmask[32], qs[64], 12 B of sixteen 6-bit scales, f16 d;
 *     w = d*(S-32)*(q - 4 + 4h), h = bit 4n+j of hmask[l] (q, S as for Q2_K;
 *     scale s: low nibble in byte s (s < 8) or the high nibble of byte s-8,
 *     high two bits at bits 2*(s/4) of byte 8 + s%4).
 * Output (B = K/256 superblocks per row, same total byte count):
 *   Q4_K: codes plane [0, N*B*128): row n at n*B*128, cut into steps of up
 *           to 8 superblocks at 1024*s; step s holds G = 4*nsb groups
 *           (nsb = min(8, B-8s)); group u is code bytes 32g..32g+31 (g = u%4)
 *           of superblock 8s+u/4, its first 16 bytes at 16u and its last 16
 *           at 16G+16u.
 *         meta plane [N*B*128, N*B*144): 16 B per superblock: d, dmin
 *           (binary16, as in GGUF), then for g = 0..3 a 24-bit little-endian
 *           record at bytes 4+3g: sc[2g] | sc[2g+1]<<6 | m[2g]<<12 | m[2g+1]<<18.
 *   Q6_K: ql plane [0, N*B*128): row n at n*B*128, steps of up to 8
 *           superblocks at 1024*s with L = 4*nsb lanes; lane u is superblock
 *           8s+u/4 with p = u%4, h = p/2, e = p%2; GGUF ql[64h+16e ..+16] at
 *           16u and ql[64h+32+16e ..+16] at 16L+16u.
 *         qh plane [N*B*128, N*B*192): GGUF qh, 64 B per superblock.
 *         scale plane [N*B*192, N*B*208): 16 B per superblock, byte 4p+t =
 *           GGUF sc[8h + e + 2t] (p = 2h+e).
 *         d plane [N*B*208, N*B*210): binary16 d per superblock.
 *   Q5_K: codes plane [0, N*B*128): the qs bytes, ordered exactly as the
 *           Q4_K codes plane.
 *         fifth-bit plane [N*B*128, N*B*160): 32 B per superblock, 8 B per
 *           group g: little-endian words R_lo then R_hi; bit 8b+w of R_lo is
 *           bit 2g of GGUF qh[4w+b] (the low nibble of code byte 4w+b of the
 *           group), bit 8b+w of R_hi is bit 2g+1 (its high nibble).
 *         meta plane [N*B*160, N*B*176): as for Q4_K.
 *   Q8_0: codes plane [0, N*K): int8 codes row-major [N][K]; d plane
 *           [N*K, N*K*34/32): binary16 d per block, row-major [N][K/32].
 *           (K % 256 == 0 here too.)
 *   Q2_K: codes plane [0, N*B*64): row n at n*B*64, steps of up to 8
 *           superblocks at 512*s; lane u of a step is superblock 8s+u/4 with
 *           p = u%4 = 2n'+e and holds GGUF qs[32n'+16e ..+16] at 16u.
 *         scale plane [N*B*64, N*B*80): 16 B per superblock, byte 4p+t = GGUF
 *           scales[8n'+2t+e].
 *         d plane [N*B*80, N*B*84): d, dmin (binary16) per superblock.
 *   Q3_K (114 B per superblock: 4 B more than GGUF, the scales unpacked):
 *         codes plane as for Q2_K; hmask plane [N*B*64, N*B*96): GGUF hmask;
 *         scale plane [N*B*96, N*B*112): int8 S-32 in Q2_K's lane order;
 *         d plane [N*B*112, N*B*114).
 */

/* Bytes of the repacked weight (== GGUF bytes: N*K/256 * 144, 176, 210 or 84;
 * N*K/32 * 34 for Q8_0; N*K/256 * 114 for Q3_K, 4 B per superblock more than
 * its 110-byte GGUF block). */
int qk_repacked_bytes(int qtype, int64_t N, int64_t K, size_t *bytes);

/*
 * gguf: device, GGUF superblocks as above, 16-byte aligned.
 * dst:  device, qk_repacked_bytes() bytes, 16-byte aligned, must not
 *       overlap gguf.  N >= 1, K % 256 == 0.  Never launched with PDL.
 */
int qk_repack(int qtype, const void *gguf, int64_t N, int64_t K, void *dst, void *stream);

/* ==================================================================== GEMV
 * Decode GEMV, M = 1..8 activation rows sharing one pass over the weight
 * (minfer "15 . The CUDA backend" sec. 3.2.5 multi-token MMVQ; cajeta.dev
 * "xpu walkthrough" sec. 4.2 batched Cols kernels: one pass over a weight
 * row serves every sequence).  The integer dot of each 32-value q8_1 block
 * with the weight codes is exact; the weight scales (d*sc, dmin*m for Q4_K,
 * d*sc for Q6_K) and the activation scale are applied in binary32 per
 * 32-value block (per 16-value block for Q6_K), the Q4_K min term using the
 * exact integer sum of the block's codes (leone-cuda "CUDA kernel design":
 * the minimum correction comes from the same codes).  Per-lane partial sums
 * are combined by a fixed shuffle tree.
 *
 * w:        device, qk_repack() output for this qtype, 16-byte aligned.
 * codes:    device, int8 [M][K] q8_1 codes, 16-byte aligned.
 * scales:   device, half2 [M][K/32] q8_1 (d, s), 16-byte aligned (only d
 *           is read).
 * residual: device float [M][N] or NULL; may be equal to y (in-place
 *           accumulate: y += W x).  Added in binary32 when the row is written
 *           (leone-cuda "CUDA kernel design": the GEMV can add a residual as
 *           it writes an output row).
 * y:        device float [M][N], 4-byte aligned; must not overlap w, codes,
 *           scales, or residual unless residual == y.
 * Ranges: 1 <= M <= 8, 1 <= N <= 2^31-1, K % 256 == 0, 256 <= K, and
 * M*K <= 81920 for Q4_K, M*K <= 40960 for Q6_K (the q8_1 activation is
 * staged in shared memory next to the weight streaming buffers).
 */
int qk_gemv_q4k(const void *w, const int8_t *codes, const void *scales,
                int64_t M, int64_t N, int64_t K,
                const float *residual, float *y, unsigned flags, void *stream);

int qk_gemv_q6k(const void *w, const int8_t *codes, const void *scales,
                int64_t M, int64_t N, int64_t K,
                const float *residual, float *y, unsigned flags, void *stream);

/*
 * The same GEMV over a Q5_K weight (qk_repack output for QK_TYPE_Q5_K):
 * minfer "15 . The CUDA backend" sec. 2.2 and cajeta.dev "xpu walkthrough"
 * sec. 4.2 serve Q5_K beside Q4_K and Q6_K.  The fold is that of Q4_K with
 * 5-bit codes (q = nibble + 16 * fifth bit): d*sc and dmin*m per 32 values,
 * the min term from the exact integer code sum of the activation block.
 * Arguments as for qk_gemv_q4k; M*K <= 65536.
 */
int qk_gemv_q5k(const void *w, const int8_t *codes, const void *scales,
                int64_t M, int64_t N, int64_t K,
                const float *residual, float *y, unsigned flags, void *stream);

/*
 * The same GEMV over a Q8_0 weight (qk_repack output for QK_TYPE_Q8_0):
 * cajeta.dev "xpu walkthrough" sec. 4.2 serves Q8_0 in its batched decode.
 * Per 32-value block the int8 x int8 dot is exact and is folded with
 * d_w * d_a in binary32.  Arguments as for qk_gemv_q4k; K % 256 == 0 and
 * M*K <= 65536.
 */
int qk_gemv_q8_0(const void *w, const int8_t *codes, const void *scales,
                 int64_t M, int64_t N, int64_t K,
                 const float *residual, float *y, unsigned flags, void *stream);

/*
 * The same GEMV over Q2_K and Q3_K weights (qk_repack output for
 * QK_TYPE_Q2_K / QK_TYPE_Q3_K; cajeta.dev "xpu walkthrough" sec. 4.2 serves
 * both).  Per 16 values the integer dot of the codes with the q8_1 codes is
 * exact; it is folded with d*sc (Q2_K, the min term from the exact integer
 * code sum of the activation) or d*(S-32) (Q3_K, its -4 offset likewise).
 * Arguments as for qk_gemv_q4k; M*K <= 81920.
 */
int qk_gemv_q2k(const void *w, const int8_t *codes, const void *scales,
                int64_t M, int64_t N, int64_t K,
                const float *residual, float *y, unsigned flags, void *stream);

int qk_gemv_q3k(const void *w, const int8_t *codes, const void *scales,
                int64_t M, int64_t N, int64_t K,
                const float *residual, float *y, unsigned flags, void *stream);

/*
 * Same GEMVs with the q8_1 quantization of the activation done inside the
 * kernel (every CTA quantizes x into shared memory with the same arithmetic
 * as qk_quantize_q8_1, so the codes are bit-identical).  For decode, where an
 * activation of a few thousand values feeds one GEMV, this removes the
 * quantize kernel and its grid boundary from the chain (leone-cuda "CUDA
 * kernel design" fuses the q8_1 pack into the producers of GEMV inputs for
 * the same reason; here the consumer does it).
 *
 * x:          device float [M][ldx], 16-byte aligned, ldx % 4 == 0, ldx >= K.
 * codes_out,  NULL, or device buffers laid out as qk_quantize_q8_1's outputs
 * scales_out: (16-byte aligned) that receive the q8_1 codes and scales the
 *             kernel computed; both NULL or both non-NULL.
 * w, residual, y, M, N, K, flags: as for qk_gemv_q4k / qk_gemv_q6k.  y must
 * not overlap x; codes_out / scales_out must not overlap any other argument.
 */
int qk_gemv_q4k_f32(const void *w, const float *x, int64_t ldx,
                    int64_t M, int64_t N, int64_t K,
                    const float *residual, float *y,
                    int8_t *codes_out, void *scales_out, unsigned flags, void *stream);

int qk_gemv_q6k_f32(const void *w, const float *x, int64_t ldx,
                    int64_t M, int64_t N, int64_t K,
                    const float *residual, float *y,
                    int8_t *codes_out, void *scales_out, unsigned flags, void *stream);

int qk_gemv_q5k_f32(const void *w, const float *x, int64_t ldx,
                    int64_t M, int64_t N, int64_t K,
                    const float *residual, float *y,
                    int8_t *codes_out, void *scales_out, unsigned flags, void *stream);

int qk_gemv_q8_0_f32(const void *w, const float *x, int64_t ldx,
                     int64_t M, int64_t N, int64_t K,
                     const float *residual, float *y,
                     int8_t *codes_out, void *scales_out, unsigned flags, void *stream);

int qk_gemv_q2k_f32(const void *w, const float *x, int64_t ldx,
                    int64_t M, int64_t N, int64_t K,
                    const float *residual, float *y,
                    int8_t *codes_out, void *scales_out, unsigned flags, void *stream);

int qk_gemv_q3k_f32(const void *w, const float *x, int64_t ldx,
                    int64_t M, int64_t N, int64_t K,
                    const float *residual, float *y,
                    int8_t *codes_out, void *scales_out, unsigned flags, void *stream);

/* ===================================================================== MMQ
 * Prefill contraction of many activation rows with a Q4_K weight: the
 * quantized weight bytes are streamed to the SMs in their Q4_K form and
 * expanded tile by tile right before the tensor-core MMAs (minfer "15 . The
 * CUDA backend" sec. 2.3 and 3.2.6).  The contraction is regrouped as
 *   y = sum_b d_b * (sum_{k in b} (d_a q_a) * (sc q)) - sum_j dmin m_j * S_j
 * (b: superblocks, j: 32-value sub-blocks, S_j = d_a * sum q_a): the
 * activation enters f16 MMAs exactly as A_hi + A_lo, the integer sc*q (< 1024)
 * exactly as one f16, each superblock accumulates on its own and is scaled by
 * d_b in binary32, and the min term is a contraction over the K/32
 * sub-blocks of S (split to 2^-22) with dmin*m (split exactly down to
 * 1024*dmin*m = 2^-8, to 2^-25 absolute below).  The binary32
 * result is within 1e-4 * sum_k |w * xhat| of the exact contraction (in
 * practice ~1e-7).
 *
 * w, codes, scales, residual, y: as for qk_gemv_q4k.
 * Ranges: M >= 1, N >= 1, K % 256 == 0, K >= 256, ceil(M/128) <= 65535 and
 * ceil(N/256) <= 65535.  (M == 0 is a no-op.)
 * Value limits: max |x| <= 32000 per 32-value block (the f16 operands
 * d_a * q_a and S_j / 16 must not overflow) and dmin * m < 63 for every
 * sub-block (the operand 1024 * dmin * m is an f16); LLM layers are far
 * inside both.  A call outside them sets QK_ERR_RANGE (qk_error_flags).
 * workspace: device scratch of at least qk_mmq_workspace_bytes(M, N, K)
 *   bytes, 256-byte aligned, not overlapping any other argument.  The call
 *   writes it (the q8_1 activation expanded once per 128-row tile into the
 *   tensor-core operand layout, then its sub-block sums S) before reading it;
 *   nothing needs to be initialised.  Its contents are consumed by kernels of
 *   this call that run after the call returns, so the workspace must not be
 *   reused by work that is not ordered after this call on `stream`.  Size:
 *   at least the base ceil(M/128) * (K * 512 + ceil(K/512) * 8192) bytes
 *   (M = 2048, K = 18944: 160,038,912 bytes).  After it, a Q4_K call whose
 *   tiles are split in two along K keeps scratch: 1024 * BN bytes of partial
 *   tiles and 4 bytes of counter per split tile, BN the tile width it picks.
 *   By default the Q4_K MMQ splits the tiles of a poorly filled last wave
 *   when K has at least 48 superblocks (Qwen2-7B down, M = 2048: 72 of 224
 *   tiles of 256 on 152 SMs, 18,874,656 bytes); QK_MMQ_SPLIT_K splits every
 *   tile.  qk_mmq_workspace_bytes returns the base size plus the default
 *   plan's scratch on the current device (QK_MMQ_SPLIT_K's is the caller's
 *   to add: 224 tiles, 58,721,152 bytes).  A workspace without room for the
 *   scratch runs the call unsplit.  Split and unsplit results differ only
 *   in rounding, within the same bound, and each is reproducible (the two
 *   partial tiles are added in binary32 by the second unit to finish).
 * Returns QK_E_WORKSPACE if workspace_bytes is below the base size.
 */
int qk_mmq_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes);

int qk_mmq_q4k(const void *w, const int8_t *codes, const void *scales,
               int64_t M, int64_t N, int64_t K,
               const float *residual, float *y,
               void *workspace, size_t workspace_bytes,
               unsigned flags, void *stream);

/*
 * The same prefill contraction with a Q6_K weight (qk_repack output for
 * QK_TYPE_Q6_K).  Q4_K_M models keep some tensors in Q6_K: minfer "15 .
 * The CUDA backend" sec. 2.2 sends Q4_K, Q5_K and Q6_K weights to the same
 * MMQ, and in cajeta.dev "xpu walkthrough" step 3 (prefill) the Q6_K value
 * and down projections of 16 layers run on their own tiles.  Each weight
 * enters the tensor cores as
 * 256 * d * sc * (q - 32) = W_hi + W_lo (to about 2^-22 relative; sc * (q - 32)
 * reaches 4096 and is not exact in one f16), against A_hi + A_lo; the bound,
 * the workspace (same size, qk_mmq_workspace_bytes; the sums S are not
 * used) and every other argument rule are those of qk_mmq_q4k.  Value
 * limits: max |x| <= 65000 per 32-value block and |w| < 255 for every
 * dequantized weight (the weight operand is scaled by 256); a call outside
 * them sets QK_ERR_RANGE (qk_error_flags).
 */
int qk_mmq_q6k(const void *w, const int8_t *codes, const void *scales,
               int64_t M, int64_t N, int64_t K,
               const float *residual, float *y,
               void *workspace, size_t workspace_bytes,
               unsigned flags, void *stream);

/* ======================================= Q4_K MMQ with a min-operand plane
 * The load-time scale plane of minfer "15 . The CUDA backend" sec. 3.2.6
 * (the W_dsc plane: scale pairs computed once when the weights are loaded,
 * so that the MMQ's hot loop does not decode the packed sub-block fields),
 * restated for this library's Q4_K MMQ.  Its min term needs, per weight row
 * and sub-block, the operand 1024 * dmin * m split exactly into two f16
 * (hi: 11 significant bits, lo: the rest); without a plane every CTA builds
 * them from the 6-bit fields for every tile.  The plane holds them ready:
 *   qk_q4k_min_plane_bytes: N * ceil(K/512) * 64 bytes.
 *   qk_q4k_min_plane: builds the plane of a repacked Q4_K weight w (N x K,
 *     qk_repack output) into `plane` (device, 16-byte aligned, `bytes` >=
 *     qk_q4k_min_plane_bytes, not overlapping w).  Layout: [N][ceil(K/512)]
 *     records of 64 bytes, record (n, i) = the 8 hi f16 pairs of superblocks
 *     2i and 2i+1 (sub-blocks 0-7 of each, two per 4-byte word) then their
 *     8 lo pairs; an odd last superblock leaves its partner's words zero.
 *     Asynchronous on `stream`; a weight with dmin * m >= 63 sets
 *     QK_ERR_RANGE (qk_error_flags), as the MMQ would.
 *   qk_mmq_q4k_plane: qk_mmq_q4k reading the min operands from the plane
 *     (built from the same w; not checked) instead of building them.  Same
 *     arguments otherwise, and the same result bit for bit: the operands are
 *     the same words.
 * Returns as qk_mmq_q4k; QK_E_NULL for a NULL plane, QK_E_ALIGN for a plane
 * not 16-byte aligned, QK_E_ALIAS if it overlaps y or the workspace, and
 * QK_E_WORKSPACE from qk_q4k_min_plane for too small a plane.
 */
int qk_q4k_min_plane_bytes(int64_t N, int64_t K, size_t *bytes);

int qk_q4k_min_plane(const void *w, int64_t N, int64_t K, void *plane, size_t bytes, void *stream);

int qk_mmq_q4k_plane(const void *w, const void *plane, const int8_t *codes, const void *scales,
                     int64_t M, int64_t N, int64_t K,
                     const float *residual, float *y,
                     void *workspace, size_t workspace_bytes,
                     unsigned flags, void *stream);

/* ============================================== MMQ from f32 activations
 * The prefill contraction with the q8_1 quantization of the activation done
 * inside the call (the GEMV's _f32 entry points do the same for decode): the
 * activation is quantized once per call, as minfer "15 . The CUDA backend"
 * sec. 2.3 prescribes, by the kernel that expands it into the workspace, so
 * the separate quantize launch and the q8_1 round trip through memory go.
 * The codes and binary16 scales are those of qk_quantize_q8_1, bit for bit
 * (the same block quantizer); they are not stored.  The results are
 * therefore bit-identical to qk_quantize_q8_1 followed by qk_mmq_q4k /
 * qk_mmq_q4k_plane / qk_mmq_q6k on the same arguments.
 *   x: device f32 activation rows, row i at x + i * ldx, ldx >= K, 16-byte
 *      aligned with ldx % 4 == 0; must not overlap y or the workspace.
 *   plane (qk_mmq_q4k_f32 only): a min-operand plane (qk_q4k_min_plane) or
 *      NULL for none.
 * Everything else (shapes, value limits, workspace, flags, errors) as for
 * qk_mmq_q4k / qk_mmq_q6k; QK_E_NULL for a NULL x.
 */
int qk_mmq_q4k_f32(const void *w, const void *plane, const float *x, int64_t ldx,
                   int64_t M, int64_t N, int64_t K,
                   const float *residual, float *y,
                   void *workspace, size_t workspace_bytes,
                   unsigned flags, void *stream);

int qk_mmq_q6k_f32(const void *w, const float *x, int64_t ldx,
                   int64_t M, int64_t N, int64_t K,
                   const float *residual, float *y,
                   void *workspace, size_t workspace_bytes,
                   unsigned flags, void *stream);

/* ================================================ MMQ without a workspace
 * The pages have no counterpart of this entry point: it is a convenience of
 * this library for callers that cannot supply a device workspace (a host
 * without its own device allocator, or a steady-state loop that must not
 * call cudaMalloc).  Same arguments and results as qk_mmq_q4k, but the
 * workspace is a statically allocated device array of
 * QK_MMQ_STATIC_WS_BYTES bytes inside the library; the call allocates and
 * frees nothing.
 *  - Problems whose base workspace size (qk_mmq_q4k) exceeds
 *    QK_MMQ_STATIC_WS_BYTES return QK_E_WORKSPACE (nothing launched).
 *    Example: M = 2048, K = 3584 needs 30,277,632 bytes and fits; K = 18944
 *    does not.  Where the array cannot also hold the split-K scratch, the
 *    call runs unsplit.
 *  - The array needs no initialisation (each call writes what it reads).
 *  - All calls on a device share the array: calls that may run concurrently
 *    (other streams, unordered host threads) race on it.
 *  - The first call on each device looks the array's address up with
 *    cudaGetSymbolAddress; make that first call outside stream capture.
 */
#define QK_MMQ_STATIC_WS_BYTES (32u << 20)
int qk_mmq_q4k_noalloc(const void *w, const int8_t *codes, const void *scales,
                       int64_t M, int64_t N, int64_t K,
                       const float *residual, float *y,
                       unsigned flags, void *stream);

/* ========================================================== error flags
 * A device-wide flag word that the MMQ kernels set when something went wrong
 * that the host could not see before the launch (invariant violations are
 * reported, never passed over silently: minfer "15 . The CUDA backend"
 * sec. 3.4).  Bits:
 *  QK_ERR_TIMEOUT  a bounded mbarrier wait gave up -- which only happens if
 *                  the hardware or the kernel misbehaves; the kernel then
 *                  skips its remaining waits and returns.
 *  QK_ERR_RANGE    an input is outside the MMQ's value limits, so an f16
 *                  operand would overflow: a q8_1 block with d_a * 127 >
 *                  32000 (qk_mmq_q4k) or > 65000 (qk_mmq_q6k), a Q4_K
 *                  sub-block with dmin * m >= 63, or a Q6_K superblock whose
 *                  largest |d * sc| * 32 is >= 255 (a weight can reach
 *                  |w| >= 255).  The GEMVs have no such limits.
 * With either bit set the output of the call is undefined.  qk_error_flags
 * copies the word to *flags (synchronously, on the current device) and, when
 * `clear` is non-zero, resets it to 0.  The word is not cleared by the
 * kernels: it collects every call since the last clear.
 * Returns QK_E_NULL if flags is NULL, QK_E_CUDA if the copy fails.
 */
#define QK_ERR_TIMEOUT 1u
#define QK_ERR_RANGE 2u
int qk_error_flags(unsigned *flags, int clear);

#ifdef __cplusplus
}
#endif

#endif /* QK_H */
