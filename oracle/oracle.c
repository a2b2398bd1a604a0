/*
 * oracle.c -- CPU oracle for the k-quant x q8_1 contraction.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this file: only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py use it.  It shares no code,
 * header, table or constant with the CUDA library under
 * quantized_q8_activation_gb300/csrc.
 *
 * Plain C99, no CUDA headers, one thread.  Floating point is IEEE binary64
 * except where the method fixes binary32 (the q8_1 quantizer, whose codes
 * must match bit for bit) or binary16 (stored scales).  Build with
 * -ffp-contract=off so that no multiply-add is fused behind our back.
 *
 * What each function follows (citations name the web page and section):
 *
 *  - orc_f16_*:      IEEE 754 binary16, written from the format definition
 *                    (1 sign bit, 5 exponent bits biased by 15, 10 fraction
 *                    bits, subnormals at 2^-24 spacing).  Encoding rounds to
 *                    nearest, ties to even, and saturates finite overflow at
 *                    +-65504 (reading: the pages store f16 scales but never
 *                    say how overflow is treated).
 *  - orc_quantize_q8_1: leone-cuda "CUDA kernel design" (q8_1 block = 32
 *                    signed codes, an f16 scale and an f16 source sum), with
 *                    the scale d = amax/127 and the sum s = d*sum(q) of the
 *                    benchmark definition.  Readings: q = roundf(x/d) (ties
 *                    away from zero), division in binary32 by the binary32 d,
 *                    amax == 0 gives d = s = 0 and all-zero codes.
 *  - orc_q4k_*:      GGUF Q4_K superblock (256 values, 144 bytes: f16 d, f16
 *                    dmin, 12 bytes of packed 6-bit scales and mins, 128
 *                    bytes of 4-bit codes); value = d*sc*q - dmin*m (minfer
 *                    "15 . The CUDA backend", sec. 2.3, block_q4_K nibbles,
 *                    sub-scales and mins).  The bit layout is the public GGUF
 *                    one; the pages name the fields but do not print it.
 *  - orc_q5k_*:      GGUF Q5_K superblock (256 values, 176 bytes: f16 d, f16
 *                    dmin, 12 bytes of 6-bit scales and mins packed as for
 *                    Q4_K, 32 bytes qh of fifth bits, 128 bytes qs of low
 *                    nibbles); value = d*sc*q - dmin*m with q = nibble + 16 *
 *                    fifth bit (minfer "15 . The CUDA backend" sec. 2.2 and
 *                    cajeta.dev "xpu walkthrough" sec. 4.2 name Q5_K among
 *                    the k-quants they serve).  The layout is the public GGUF
 *                    one (group g: low nibbles of qs[32g..] with qh bit 2g,
 *                    high nibbles with qh bit 2g+1); the pages do not print it.
 *  - orc_q80_*:      GGUF Q8_0 blocks (32 values, 34 bytes: f16 d, 32 int8
 *                    codes); value = d*q (cajeta.dev "xpu walkthrough" sec.
 *                    4.2 serves Q8_0 beside the k-quants).  Handled in runs of
 *                    8 blocks (256 values, 272 bytes) so that rows walk the
 *                    same 256-value units as the k-quants.
 *  - orc_q2k_*:      GGUF Q2_K superblock (256 values, 84 bytes: 16 scale bytes
 *                    (low nibble the scale, high nibble the min of each
 *                    16-value sub-block), 64 bytes of 2-bit codes, f16 d, f16
 *                    dmin); value = d*sc*q - dmin*m.
 *  - orc_q3k_*:      GGUF Q3_K superblock (256 values, 110 bytes: 32 bytes
 *                    hmask, 64 bytes of 2-bit codes, 12 bytes of sixteen 6-bit
 *                    scales, f16 d); value = d*(S - 32)*(q - 4*(1 - h)) with h
 *                    the hmask bit.  For both: value 128n + 32j + l takes code
 *                    bits 2j of qs[32n + l] and the scale of sub-block
 *                    8n + 2j + (l >= 16); Q3_K's h is bit 4n + j of hmask[l].
 *                    The 12 Q3_K scale bytes hold the low nibbles of scales
 *                    0-7 and 8-15 in bytes 0-7 (low, high nibble) and the high
 *                    two bits of scale s in byte 8 + s%4, bits 2*(s/4).  (The
 *                    pages name Q2_K and Q3_K among the served formats --
 *                    cajeta.dev "xpu walkthrough" sec. 4.2 -- but print no
 *                    layout; this is the public GGUF one.)
 *  - orc_q6k_*:      GGUF Q6_K superblock (256 values, 210 bytes: 128 bytes
 *                    of low 4 bits, 64 bytes of high 2 bits, 16 int8 scales,
 *                    f16 d); value = d*sc*(q - 32) (minfer sec. 3.2.2, "raw
 *                    210-byte block stride").  Same caveat on the layout.
 *  - orc_gemm_rows:  y[m][n] = sum_k w[n][k] * (d_a * q_a[m][k]) (+ r[m][n]),
 *                    the dequantize-then-dot definition, in binary64, plus
 *                    the per-output tolerance scale sum_k |w * xhat|.
 *  - orc_rmsnorm:    RMSNorm of a row, s = x (+ r), y = s / sqrt(mean(s^2) +
 *                    eps) * g (leone-cuda "CUDA kernel design", RMSNorm
 *                    paragraphs: the residual variant normalizes left +
 *                    right).  s is the binary32 sum the residual stream holds;
 *                    the rest is binary64.
 *  - orc_swiglu:     h = silu(gate) * up = gate / (1 + exp(-gate)) * up, in
 *                    binary64, gate and up being the two halves of a gate||up
 *                    row (leone-cuda "CUDA kernel design", SwiGLU paragraph).
 *  - orc_repack_*:   the device weight layout this project defines for its
 *                    GPU kernels (a lossless byte permutation; leone-cuda
 *                    "CUDA kernel design" repacks Q4_K into a code part and a
 *                    metadata part; minfer sec. 3.2.2 pads Q6_K for aligned
 *                    16-byte loads).  Written from the layout specification,
 *                    not from the GPU code.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORC_QK 256          /* values per k-quant superblock */
#define ORC_Q81 32          /* values per q8_1 block */
#define ORC_Q4K_BYTES 144
#define ORC_Q6K_BYTES 210
#define ORC_Q5K_BYTES 176
#define ORC_Q80_BYTES 272       /* 8 Q8_0 blocks of 34 bytes: one 256-value unit */
#define ORC_Q2K_BYTES 84
#define ORC_Q3K_BYTES 110

enum { ORC_Q4_K = 1, ORC_Q6_K = 2, ORC_Q5_K = 3, ORC_Q8_0 = 4, ORC_Q2_K = 5, ORC_Q3_K = 6 };

int orc_block_bytes(int qtype)
{
    if (qtype == ORC_Q4_K) return ORC_Q4K_BYTES;
    if (qtype == ORC_Q6_K) return ORC_Q6K_BYTES;
    if (qtype == ORC_Q5_K) return ORC_Q5K_BYTES;
    if (qtype == ORC_Q8_0) return ORC_Q80_BYTES;
    if (qtype == ORC_Q2_K) return ORC_Q2K_BYTES;
    if (qtype == ORC_Q3_K) return ORC_Q3K_BYTES;
    return -1;
}

/* ---------------------------------------------------------------- binary16 */

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* round x / 2^sh to the nearest integer, ties to even (x >= 0, sh >= 0) */
static uint64_t rne_shift(uint64_t x, int sh)
{
    if (sh <= 0) return x;
    if (sh >= 63) return 0;
    uint64_t q = x >> sh;
    uint64_t r = x & ((1ull << sh) - 1);
    uint64_t half = 1ull << (sh - 1);
    if (r > half || (r == half && (q & 1))) q++;
    return q;
}

uint16_t orc_f32_to_f16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t ex = (u >> 23) & 0xff;
    uint32_t fr = u & 0x7fffffu;
    if (ex == 0xff)                                /* inf saturates, NaN stays NaN */
        return fr ? (uint16_t)(sign | 0x7e00u) : (uint16_t)(sign | 0x7bffu);
    if (ex == 0)                                   /* binary32 zero/subnormal < 2^-126 */
        return sign;
    uint64_t sig = (1ull << 23) | fr;              /* value = sig * 2^(ex-150) */
    int e = (int)ex - 127;                         /* unbiased exponent */
    if (e >= -14) {                                /* binary16 normal range */
        uint64_t m = rne_shift(sig, 13);           /* 11-bit significand, maybe 2048 */
        int E = e + 15;
        if (m == 2048) { m = 1024; E++; }
        if (E >= 31) return (uint16_t)(sign | 0x7bffu);
        return (uint16_t)(sign | (E << 10) | (uint16_t)(m - 1024));
    }
    /* binary16 subnormal: count units of 2^-24; sig * 2^(ex-150) / 2^-24 */
    uint64_t q = rne_shift(sig, 126 - (int)ex);
    return (uint16_t)(sign | (uint16_t)q);         /* q == 1024 encodes 2^-14 */
}

/* ------------------------------------------------------------------- q8_1 */

/* codes: [M][K] int8, d and s: [M][K/32] binary16 bit patterns */
int orc_quantize_q8_1(const float *x, int64_t ldx, int64_t M, int64_t K,
                      int8_t *codes, uint16_t *d_out, uint16_t *s_out)
{
    if (K % ORC_Q81 != 0 || M < 0 || ldx < K) return -1;
    int64_t nb = K / ORC_Q81;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t b = 0; b < nb; b++) {
            const float *xb = x + m * ldx + b * ORC_Q81;
            float amax = 0.0f;
            for (int i = 0; i < ORC_Q81; i++) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int i = 0; i < ORC_Q81; i++) {
                int q = 0;
                if (d > 0.0f) q = (int)roundf(xb[i] / d);
                codes[m * K + b * ORC_Q81 + i] = (int8_t)q;
                sum += q;
            }
            float s = d * (float)sum;
            d_out[m * nb + b] = orc_f32_to_f16(d);
            s_out[m * nb + b] = orc_f32_to_f16(s);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------- Q4_K */

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes */
void orc_q4k_scale_min(const uint8_t *q12, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = q12[j] & 63;
        *mn = q12[j + 4] & 63;
    } else {
        *sc = (q12[j + 4] & 0x0f) | ((q12[j - 4] >> 6) << 4);
        *mn = (q12[j + 4] >> 4) | ((q12[j] >> 6) << 4);
    }
}

/* one 144-byte superblock -> 256 binary64 weights */
void orc_q4k_dequant(const uint8_t *blk, double *out)
{
    double d = orc_f16_to_f64(rd16(blk));
    double dmin = orc_f16_to_f64(rd16(blk + 2));
    const uint8_t *q12 = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int g = 0; g < 4; g++) {             /* 32 code bytes per group */
        int sc0, m0, sc1, m1;
        orc_q4k_scale_min(q12, 2 * g, &sc0, &m0);
        orc_q4k_scale_min(q12, 2 * g + 1, &sc1, &m1);
        for (int l = 0; l < 32; l++) {
            int lo = qs[32 * g + l] & 0x0f;
            int hi = qs[32 * g + l] >> 4;
            out[64 * g + l] = d * sc0 * lo - dmin * m0;
            out[64 * g + 32 + l] = d * sc1 * hi - dmin * m1;
        }
    }
}

/* ------------------------------------------------------------------- Q5_K */

/* one 176-byte superblock -> 256 binary64 weights */
void orc_q5k_dequant(const uint8_t *blk, double *out)
{
    double d = orc_f16_to_f64(rd16(blk));
    double dmin = orc_f16_to_f64(rd16(blk + 2));
    const uint8_t *q12 = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    for (int g = 0; g < 4; g++) {
        int sc0, m0, sc1, m1;
        orc_q4k_scale_min(q12, 2 * g, &sc0, &m0);
        orc_q4k_scale_min(q12, 2 * g + 1, &sc1, &m1);
        for (int l = 0; l < 32; l++) {
            int lo = (qs[32 * g + l] & 0x0f) | (((qh[l] >> (2 * g)) & 1) << 4);
            int hi = (qs[32 * g + l] >> 4) | (((qh[l] >> (2 * g + 1)) & 1) << 4);
            out[64 * g + l] = d * sc0 * lo - dmin * m0;
            out[64 * g + 32 + l] = d * sc1 * hi - dmin * m1;
        }
    }
}

/* ------------------------------------------------------------------- Q8_0 */

/* eight consecutive 34-byte blocks -> 256 binary64 weights */
void orc_q80_dequant(const uint8_t *blk, double *out)
{
    for (int b = 0; b < 8; b++) {
        const uint8_t *p = blk + 34 * b;
        double d = orc_f16_to_f64(rd16(p));
        for (int l = 0; l < 32; l++) out[32 * b + l] = d * (double)(int8_t)p[2 + l];
    }
}

/* ------------------------------------------------------------- Q2_K, Q3_K */

void orc_q2k_dequant(const uint8_t *blk, double *out)
{
    const uint8_t *sc = blk, *qs = blk + 16;
    double d = orc_f16_to_f64(rd16(blk + 80));
    double dmin = orc_f16_to_f64(rd16(blk + 82));
    for (int n = 0; n < 2; n++)
        for (int j = 0; j < 4; j++)
            for (int l = 0; l < 32; l++) {
                int q = (qs[32 * n + l] >> (2 * j)) & 3;
                int s = sc[8 * n + 2 * j + (l >= 16)];
                out[128 * n + 32 * j + l] = d * (s & 15) * q - dmin * (s >> 4);
            }
}

/* signed 6-bit scale s (0..15) of a Q3_K superblock, minus 32 */
int orc_q3k_scale(const uint8_t *sc12, int s)
{
    int lo = s < 8 ? (sc12[s] & 15) : (sc12[s - 8] >> 4);
    int hi = (sc12[8 + (s & 3)] >> (2 * (s >> 2))) & 3;
    return (lo | (hi << 4)) - 32;
}

void orc_q3k_dequant(const uint8_t *blk, double *out)
{
    const uint8_t *hm = blk, *qs = blk + 32, *sc12 = blk + 96;
    double d = orc_f16_to_f64(rd16(blk + 108));
    for (int n = 0; n < 2; n++)
        for (int j = 0; j < 4; j++)
            for (int l = 0; l < 32; l++) {
                int q = ((qs[32 * n + l] >> (2 * j)) & 3) - (((hm[l] >> (4 * n + j)) & 1) ? 0 : 4);
                out[128 * n + 32 * j + l] = d * orc_q3k_scale(sc12, 8 * n + 2 * j + (l >= 16)) * q;
            }
}

/* ------------------------------------------------------------------- Q6_K */

void orc_q6k_dequant(const uint8_t *blk, double *out)
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *sc = (const int8_t *)(blk + 192);
    double d = orc_f16_to_f64(rd16(blk + 208));
    for (int h = 0; h < 2; h++) {             /* two halves of 128 values */
        for (int l = 0; l < 32; l++) {
            int is = l / 16;
            int hb = qh[32 * h + l];
            int q0 = ((ql[64 * h + l] & 0x0f) | (((hb >> 0) & 3) << 4)) - 32;
            int q1 = ((ql[64 * h + l + 32] & 0x0f) | (((hb >> 2) & 3) << 4)) - 32;
            int q2 = ((ql[64 * h + l] >> 4) | (((hb >> 4) & 3) << 4)) - 32;
            int q3 = ((ql[64 * h + l + 32] >> 4) | (((hb >> 6) & 3) << 4)) - 32;
            out[128 * h + l] = d * sc[8 * h + is + 0] * q0;
            out[128 * h + l + 32] = d * sc[8 * h + is + 2] * q1;
            out[128 * h + l + 64] = d * sc[8 * h + is + 4] * q2;
            out[128 * h + l + 96] = d * sc[8 * h + is + 6] * q3;
        }
    }
}

/* dequantize a whole row of K/256 superblocks */
int orc_dequant_row(int qtype, const uint8_t *row, int64_t K, double *out)
{
    int bs = orc_block_bytes(qtype);
    if (bs < 0 || K % ORC_QK != 0) return -1;
    for (int64_t b = 0; b < K / ORC_QK; b++) {
        if (qtype == ORC_Q4_K) orc_q4k_dequant(row + b * bs, out + b * ORC_QK);
        else if (qtype == ORC_Q5_K) orc_q5k_dequant(row + b * bs, out + b * ORC_QK);
        else if (qtype == ORC_Q8_0) orc_q80_dequant(row + b * bs, out + b * ORC_QK);
        else if (qtype == ORC_Q2_K) orc_q2k_dequant(row + b * bs, out + b * ORC_QK);
        else if (qtype == ORC_Q3_K) orc_q3k_dequant(row + b * bs, out + b * ORC_QK);
        else orc_q6k_dequant(row + b * bs, out + b * ORC_QK);
    }
    return 0;
}

/* ------------------------------------------------------------ contraction */

/*
 * Rows n0..n1-1 of y = xhat @ W^T (+ r), binary64.
 *   w:      GGUF superblocks, row-major [N][K/256]
 *   codes:  q8_1 codes [M][K]; d_a: q8_1 scales (binary16 bits) [M][K/32]
 *   r:      optional residual [M][N] (binary32), NULL for none
 *   y:      out [M][n1-n0]; absdot: out [M][n1-n0] = sum_k |w*xhat|
 */
int orc_gemm_rows(int qtype, const uint8_t *w, int64_t N, int64_t K,
                  int64_t n0, int64_t n1,
                  const int8_t *codes, const uint16_t *d_a, int64_t M,
                  const float *r, double *y, double *absdot)
{
    int bs = orc_block_bytes(qtype);
    if (bs < 0 || K % ORC_QK != 0 || n0 < 0 || n1 > N || n0 > n1) return -1;
    int64_t nb = K / ORC_Q81;
    int64_t rowbytes = (K / ORC_QK) * bs;
    int64_t nn = n1 - n0;
    double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
    double *xhat = (double *)malloc(sizeof(double) * (size_t)(M * K + 1));
    if (!wrow || !xhat) { free(wrow); free(xhat); return -2; }
    for (int64_t m = 0; m < M; m++)
        for (int64_t k = 0; k < K; k++)
            xhat[m * K + k] = orc_f16_to_f64(d_a[m * nb + k / ORC_Q81]) * codes[m * K + k];
    for (int64_t n = n0; n < n1; n++) {
        orc_dequant_row(qtype, w + n * rowbytes, K, wrow);
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, ab = 0.0;
            const double *xm = xhat + m * K;
            for (int64_t k = 0; k < K; k++) {
                double p = wrow[k] * xm[k];
                acc += p;
                ab += fabs(p);
            }
            if (r) acc += (double)r[m * N + n];
            y[m * nn + (n - n0)] = acc;
            absdot[m * nn + (n - n0)] = ab;
        }
    }
    free(wrow);
    free(xhat);
    return 0;
}

/* ----------------------------------------------------------- device layout */

/*
 * Q4_K device layout for an N x K weight (B = K/256 superblocks per row),
 * N*B*144 bytes in two planes:
 *   codes plane at 0, N*B*128 bytes, row n at n*B*128.  A row is cut into
 *     steps of up to 8 superblocks; step s starts at 1024*s and holds
 *     G = 4*nsb groups (nsb = min(8, B-8s)).  Group u of the step is group
 *     u%4 (code bytes 32g..32g+31) of superblock 8s+u/4; its first 16 code
 *     bytes sit at 16*u and its last 16 at 16*G + 16*u.
 *   meta plane at N*B*128, 16 bytes per superblock in row-major order:
 *     bytes 0-1 d, 2-3 dmin (binary16 as in GGUF), then for g = 0..3 a
 *     24-bit little-endian record at bytes 4+3g..6+3g holding
 *     sc[2g] | sc[2g+1] << 6 | m[2g] << 12 | m[2g+1] << 18.
 */
int orc_repack_q4k(const uint8_t *gguf, int64_t N, int64_t K, uint8_t *out)
{
    if (K % ORC_QK != 0 || N < 0) return -1;
    int64_t B = K / ORC_QK;
    uint8_t *codes = out;
    uint8_t *meta = out + N * B * 128;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t b = 0; b < B; b++) {
            const uint8_t *blk = gguf + (n * B + b) * ORC_Q4K_BYTES;
            int64_t s = b / 8;
            int64_t nsb = (B - 8 * s) < 8 ? (B - 8 * s) : 8;
            int64_t G = 4 * nsb;
            uint8_t *step = codes + n * B * 128 + 1024 * s;
            for (int g = 0; g < 4; g++) {
                int64_t u = 4 * (b - 8 * s) + g;
                memcpy(step + 16 * u, blk + 16 + 32 * g, 16);
                memcpy(step + 16 * G + 16 * u, blk + 16 + 32 * g + 16, 16);
            }
            uint8_t *mt = meta + (n * B + b) * 16;
            memcpy(mt, blk, 4);
            for (int g = 0; g < 4; g++) {
                int sc0, m0, sc1, m1;
                orc_q4k_scale_min(blk + 4, 2 * g, &sc0, &m0);
                orc_q4k_scale_min(blk + 4, 2 * g + 1, &sc1, &m1);
                uint32_t rec = (uint32_t)sc0 | ((uint32_t)sc1 << 6) |
                               ((uint32_t)m0 << 12) | ((uint32_t)m1 << 18);
                mt[4 + 3 * g + 0] = (uint8_t)(rec & 0xff);
                mt[4 + 3 * g + 1] = (uint8_t)((rec >> 8) & 0xff);
                mt[4 + 3 * g + 2] = (uint8_t)((rec >> 16) & 0xff);
            }
        }
    }
    return 0;
}

/*
 * Q5_K device layout for an N x K weight (B = K/256), N*B*176 bytes in three
 * planes:
 *   codes plane at 0, N*B*128 bytes: the GGUF qs bytes in the Q4_K codes
 *     plane order (steps of up to 8 superblocks, group u of a step at 16*u
 *     and 16*G + 16*u).
 *   fifth-bit plane at N*B*128, 32 bytes per superblock, 8 per group g:
 *     two little-endian 32-bit words R_lo (bytes 8g..8g+3) and R_hi
 *     (8g+4..8g+7).  Bit 8b + w of R_lo is the fifth bit of the low-nibble
 *     value of code byte l = 4w + b (w = 0..7, b = 0..3), i.e. GGUF qh[l]
 *     bit 2g; R_hi holds qh[l] bit 2g+1 for the high nibbles the same way.
 *   meta plane at N*B*160, 16 bytes per superblock exactly as for Q4_K.
 */
int orc_repack_q5k(const uint8_t *gguf, int64_t N, int64_t K, uint8_t *out)
{
    if (K % ORC_QK != 0 || N < 0) return -1;
    int64_t B = K / ORC_QK;
    uint8_t *codes = out;
    uint8_t *hb = out + N * B * 128;
    uint8_t *meta = out + N * B * 160;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t b = 0; b < B; b++) {
            const uint8_t *blk = gguf + (n * B + b) * ORC_Q5K_BYTES;
            int64_t s = b / 8;
            int64_t nsb = (B - 8 * s) < 8 ? (B - 8 * s) : 8;
            int64_t G = 4 * nsb;
            uint8_t *step = codes + n * B * 128 + 1024 * s;
            for (int g = 0; g < 4; g++) {
                int64_t u = 4 * (b - 8 * s) + g;
                memcpy(step + 16 * u, blk + 48 + 32 * g, 16);
                memcpy(step + 16 * G + 16 * u, blk + 48 + 32 * g + 16, 16);
                uint32_t rlo = 0, rhi = 0;
                for (int l = 0; l < 32; l++) {
                    int w = l / 4, byte = l % 4;
                    rlo |= (uint32_t)((blk[16 + l] >> (2 * g)) & 1) << (8 * byte + w);
                    rhi |= (uint32_t)((blk[16 + l] >> (2 * g + 1)) & 1) << (8 * byte + w);
                }
                uint8_t *r = hb + (n * B + b) * 32 + 8 * g;
                for (int k = 0; k < 4; k++) {
                    r[k] = (uint8_t)(rlo >> (8 * k));
                    r[4 + k] = (uint8_t)(rhi >> (8 * k));
                }
            }
            uint8_t *mt = meta + (n * B + b) * 16;
            memcpy(mt, blk, 4);
            for (int g = 0; g < 4; g++) {
                int sc0, m0, sc1, m1;
                orc_q4k_scale_min(blk + 4, 2 * g, &sc0, &m0);
                orc_q4k_scale_min(blk + 4, 2 * g + 1, &sc1, &m1);
                uint32_t rec = (uint32_t)sc0 | ((uint32_t)sc1 << 6) |
                               ((uint32_t)m0 << 12) | ((uint32_t)m1 << 18);
                mt[4 + 3 * g + 0] = (uint8_t)(rec & 0xff);
                mt[4 + 3 * g + 1] = (uint8_t)((rec >> 8) & 0xff);
                mt[4 + 3 * g + 2] = (uint8_t)((rec >> 16) & 0xff);
            }
        }
    }
    return 0;
}

/*
 * Q8_0 device layout for an N x K weight, N*K*34/32 bytes in two planes:
 *   codes plane at 0, N*K bytes: the int8 codes, row-major [N][K].
 *   d plane at N*K, the binary16 d of each 32-value block, row-major
 *     [N][K/32].
 */
int orc_repack_q80(const uint8_t *gguf, int64_t N, int64_t K, uint8_t *out)
{
    if (K % ORC_QK != 0 || N < 0) return -1;
    int64_t nb = K / 32;
    uint8_t *codes = out;
    uint8_t *dp = out + N * K;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *p = gguf + (n * nb + b) * 34;
            memcpy(codes + n * K + 32 * b, p + 2, 32);
            memcpy(dp + (n * nb + b) * 2, p, 2);
        }
    return 0;
}

/*
 * Q2_K / Q3_K device layouts (B = K/256).  Both start with a codes plane of
 * N*B*64 bytes, row n at n*B*64, cut into steps of up to 8 superblocks at
 * 512*s; lane u of a step is superblock 8s + u/4 with p = u%4 = 2n' + e and
 * holds GGUF qs[32n' + 16e .. +16] at 16*u.  Scale records are 16 bytes per
 * superblock in lane order: byte 4p + t is the scale of sub-block 8n' + 2t + e.
 *   Q2_K (84 bytes per superblock): codes | scale plane (the GGUF scale bytes,
 *     scale in the low nibble, min in the high) at N*B*64 | d, dmin (binary16)
 *     at N*B*80, 4 bytes per superblock.
 *   Q3_K (114 bytes per superblock, 4 more than GGUF: the sixteen 6-bit scales
 *     are stored unpacked): codes | hmask plane (GGUF hmask, 32 bytes per
 *     superblock) at N*B*64 | scale plane (int8 scale - 32) at N*B*96 | d
 *     (binary16) at N*B*112.
 */
static void q23_codes_and_order(const uint8_t *qs, int64_t n, int64_t b, int64_t B, uint8_t *codes)
{
    int64_t s = b / 8;
    uint8_t *step = codes + n * B * 64 + 512 * s;
    for (int p = 0; p < 4; p++) {
        int hn = p / 2, e = p % 2;
        int64_t u = 4 * (b - 8 * s) + p;
        memcpy(step + 16 * u, qs + 32 * hn + 16 * e, 16);
    }
}

int orc_repack_q2k(const uint8_t *gguf, int64_t N, int64_t K, uint8_t *out)
{
    if (K % ORC_QK != 0 || N < 0) return -1;
    int64_t B = K / ORC_QK, NB = N * B;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < B; b++) {
            const uint8_t *blk = gguf + (n * B + b) * ORC_Q2K_BYTES;
            q23_codes_and_order(blk + 16, n, b, B, out);
            for (int p = 0; p < 4; p++)
                for (int t = 0; t < 4; t++)
                    out[NB * 64 + (n * B + b) * 16 + 4 * p + t] = blk[8 * (p / 2) + 2 * t + (p % 2)];
            memcpy(out + NB * 80 + (n * B + b) * 4, blk + 80, 4);
        }
    return 0;
}

int orc_repack_q3k(const uint8_t *gguf, int64_t N, int64_t K, uint8_t *out)
{
    if (K % ORC_QK != 0 || N < 0) return -1;
    int64_t B = K / ORC_QK, NB = N * B;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < B; b++) {
            const uint8_t *blk = gguf + (n * B + b) * ORC_Q3K_BYTES;
            q23_codes_and_order(blk + 32, n, b, B, out);
            memcpy(out + NB * 64 + (n * B + b) * 32, blk, 32);
            for (int p = 0; p < 4; p++)
                for (int t = 0; t < 4; t++)
                    out[NB * 96 + (n * B + b) * 16 + 4 * p + t] =
                        (uint8_t)(int8_t)orc_q3k_scale(blk + 96, 8 * (p / 2) + 2 * t + (p % 2));
            memcpy(out + NB * 112 + (n * B + b) * 2, blk + 108, 2);
        }
    return 0;
}

/*
 * Q6_K device layout for an N x K weight (B = K/256), N*B*210 bytes in four
 * planes:
 *   ql plane at 0, N*B*128 bytes, row n at n*B*128, steps of up to 8
 *     superblocks at 1024*s with L = 4*nsb lanes.  Lane u of the step is
 *     superblock 8s+u/4 with p = u%4, h = p/2, e = p%2; its chunk A (GGUF
 *     ql[64h+16e .. +16]) sits at 16*u, its chunk B (GGUF ql[64h+32+16e ..
 *     +16]) at 16*L + 16*u.
 *   qh plane at N*B*128, 64 bytes per superblock, GGUF qh in natural order.
 *   scale plane at N*B*192, 16 bytes per superblock; byte 4p+t is GGUF
 *     sc[8h + e + 2t] with p = 2h+e, t = 0..3.
 *   d plane at N*B*208, the binary16 d of each superblock.
 */
int orc_repack_q6k(const uint8_t *gguf, int64_t N, int64_t K, uint8_t *out)
{
    if (K % ORC_QK != 0 || N < 0) return -1;
    int64_t B = K / ORC_QK;
    uint8_t *qlp = out;
    uint8_t *qhp = out + N * B * 128;
    uint8_t *scp = out + N * B * 192;
    uint8_t *dp = out + N * B * 208;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t b = 0; b < B; b++) {
            const uint8_t *blk = gguf + (n * B + b) * ORC_Q6K_BYTES;
            int64_t s = b / 8;
            int64_t nsb = (B - 8 * s) < 8 ? (B - 8 * s) : 8;
            int64_t L = 4 * nsb;
            uint8_t *step = qlp + n * B * 128 + 1024 * s;
            for (int p = 0; p < 4; p++) {
                int h = p / 2, e = p % 2;
                int64_t u = 4 * (b - 8 * s) + p;
                memcpy(step + 16 * u, blk + 64 * h + 16 * e, 16);
                memcpy(step + 16 * L + 16 * u, blk + 64 * h + 32 + 16 * e, 16);
                for (int t = 0; t < 4; t++)
                    scp[(n * B + b) * 16 + 4 * p + t] = blk[192 + 8 * h + e + 2 * t];
            }
            memcpy(qhp + (n * B + b) * 64, blk + 128, 64);
            memcpy(dp + (n * B + b) * 2, blk + 208, 2);
        }
    }
    return 0;
}

/* ------------------------------------------------------------ producers */

/* RMSNorm of M rows of K values: s = x (+ r) (binary32 add, as stored in the
   residual stream), y = s / sqrt(sum(s^2) / K + eps) * g in binary64.  s_out
   (nullable) receives s. */
int orc_rmsnorm(const float *x, int64_t ldx, const float *r, const float *g, double eps, int64_t M,
                int64_t K, float *s_out, double *y)
{
    if (M < 0 || K <= 0 || ldx < K || !(eps >= 0.0)) return -1;
    for (int64_t m = 0; m < M; m++) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; k++) {
            float sk = x[m * ldx + k];
            if (r) sk = sk + r[m * K + k];          /* float + float: one binary32 rounding */
            if (s_out) s_out[m * K + k] = sk;
            ss += (double)sk * (double)sk;
        }
        const double inv = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; k++) {
            float sk = x[m * ldx + k];
            if (r) sk = sk + r[m * K + k];
            y[m * K + k] = (double)sk * inv * (double)g[k];
        }
    }
    return 0;
}

/* h[m][f] = silu(gate) * up with gate = gu[m][f], up = gu[m][F + f], binary64 */
int orc_swiglu(const float *gu, int64_t ld, int64_t M, int64_t F, double *h)
{
    if (M < 0 || F <= 0 || ld < 2 * F) return -1;
    for (int64_t m = 0; m < M; m++)
        for (int64_t f = 0; f < F; f++) {
            const double gv = gu[m * ld + f], uv = gu[m * ld + F + f];
            h[m * F + f] = gv / (1.0 + exp(-gv)) * uv;
        }
    return 0;
}
