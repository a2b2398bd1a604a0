// qk_gemv.cu -- decode GEMV y = x_q8 . W^T (+ r) for M = 1..8 activation rows
// over a repacked k-quant (Q2_K, Q3_K, Q4_K, Q5_K, Q6_K) or Q8_0 weight.
//
// Design (GB300, HBM-bound):
//  - Persistent grid, one CTA of 16 warps per SM (20 for the Q6_K kernels with M <= 2
//    where the ring fits, 12 for four-row items).  Warp w of the grid owns
//    groups of P output rows w, w + W, w + 2W, ... and walks each group in
//    steps of up to 8 superblocks (an "item"); in an item every lane copies
//    16-byte chunks so a warp covers 512 contiguous bytes of the repacked code
//    plane per copy instruction (qk.h layout).  P = 2, or P = 4 for Q4_K with
//    M >= 3 where the groups still fill the grid (12 warps per CTA): one read
//    of the staged activation then serves four weight rows.
//  - Each warp streams its items through a private ring of R shared-memory
//    slots with cp.async (L2 -> SMEM, no register cost), R-1 items in flight
//    while one is computed; no block-wide barrier inside the loop.  With
//    QK_LAUNCH_PDL the first R-1 items are issued before griddepcontrol.wait,
//    so weight streaming overlaps the tail of the previous kernel, and the
//    kernel lets its successor launch at entry.
//  - The q8_1 activation (M x K codes) is staged once per CTA in shared
//    memory with a 16-byte-chunk XOR swizzle that keeps the lanes' 16-byte
//    reads conflict free; per 32-value block the CTA also stores d_a and the
//    exact d_a * sum(q_a) (Q4_K) or per 16 values the -32 bias term (Q6_K).
//    Two front ends: the q8_1 entry points copy caller-quantized codes; the
//    _f32 entry points quantize the f32 activation in every CTA with the
//    library's q8_1 block quantizer (bit-identical codes), which removes the
//    quantize kernel and its grid boundary from the decode chain and lets
//    consecutive GEMVs co-reside under programmatic dependent launch.
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

// tile constants (compile-time; -D overrides exist for tuning sweeps)
#ifndef QK_GEMV_WARPS
#define QK_GEMV_WARPS 16              // warps per CTA for M > 2
#endif
#ifndef QK_GEMV_WARPS_SMALL_M
#define QK_GEMV_WARPS_SMALL_M 16      // warps per CTA for M <= 2
#endif
#ifndef QK_GEMV_CTAS_PER_SM
#define QK_GEMV_CTAS_PER_SM 1
#endif
#ifndef QK_GEMV_Q4_RING
#define QK_GEMV_Q4_RING 3
#endif
#ifndef QK_GEMV_Q6_RING
#define QK_GEMV_Q6_RING 3
#endif
// 0: allow the next kernel to launch at entry; 1: after the activation is staged; 2: at exit
#ifndef QK_GEMV_TRIGGER
#define QK_GEMV_TRIGGER 0
#endif
// warps and CTAs per SM of the f32-input (self-quantizing) kernels for M <= 2
#ifndef QK_GEMV_WARPS_FUSED
#define QK_GEMV_WARPS_FUSED 16
#endif
#ifndef QK_GEMV_MINB_FUSED
#define QK_GEMV_MINB_FUSED 1
#endif
#ifndef QK_GEMV_MINB_SMALL_M
#define QK_GEMV_MINB_SMALL_M 1         // CTAs per SM the q8_1-input kernels for M <= 2 are compiled for
#endif
// warps per CTA of the wide Q6_K kernels for M <= 2, taken where their ring and the activation fit
// in shared memory (their registers leave room for 20 warps; the Q4_K kernels keep 16, which the
// chained decode layer measured faster)
#ifndef QK_GEMV_WARPS_Q6_SMALL_M
#define QK_GEMV_WARPS_Q6_SMALL_M 20
#endif
// four-row items (Q4_K / Q6_K, M >= 3): warps per CTA and ring slots
#ifndef QK_GEMV_P4_WARPS
#define QK_GEMV_P4_WARPS 12
#endif
#ifndef QK_GEMV_P4_Q4_RING
#define QK_GEMV_P4_Q4_RING 3
#endif
#ifndef QK_GEMV_P4_Q6_RING
#define QK_GEMV_P4_Q6_RING 2
#endif
template <int M, bool FUSED>
struct Cfg {
    static constexpr int warps = M > 2 ? QK_GEMV_WARPS : FUSED ? QK_GEMV_WARPS_FUSED : QK_GEMV_WARPS_SMALL_M;
    static constexpr int threads = warps * 32;
    static constexpr int minb = M <= 2 ? (FUSED ? QK_GEMV_MINB_FUSED : QK_GEMV_MINB_SMALL_M) : 1;
};
// launch shape of a kernel whose items hold PR weight rows (WIDE: the 20-warp Q6_K kernels, M <= 2)
template <int M, bool FUSED, int PR, bool WIDE = false>
struct KCfg {
    static constexpr int warps = PR == 4 ? QK_GEMV_P4_WARPS : WIDE ? QK_GEMV_WARPS_Q6_SMALL_M : Cfg<M, FUSED>::warps;
    static constexpr int threads = warps * 32;
    static constexpr int minb = PR == 4 ? 1 : Cfg<M, FUSED>::minb;
};
constexpr int kCtasPerSm = QK_GEMV_CTAS_PER_SM;
constexpr int kRowsPerItem = 2;                                     // rows a lane works on at once (default)
constexpr int Q4_R = QK_GEMV_Q4_RING, Q4_SLOT = kRowsPerItem * (1024 + 128);       // codes + 8 metadata records
constexpr int Q6_R = QK_GEMV_Q6_RING, Q6_SLOT = kRowsPerItem * (1024 + 512 + 128); // ql + qh + scales
constexpr int Q5_R = QK_GEMV_Q4_RING, Q5_SLOT = kRowsPerItem * (1024 + 256 + 128);  // codes + fifth bits + metadata
constexpr int Q80_R = 2, Q80_SLOT = kRowsPerItem * (2048 + 128);                       // int8 codes + block scales
constexpr int Q2_SLOT = kRowsPerItem * (512 + 128), Q3_SLOT = kRowsPerItem * (512 + 256 + 128);  // codes (+ hmask) + scales
static_assert(Q4_R >= 2 && Q6_R >= 2, "ring needs two slots at least");

// kernel arguments (one struct: the q8_1 and the f32 front ends share the kernels)
struct GemvArgs {
    const uint8_t *w;              // repacked weight
    const int8_t *codes;           // q8_1 front end: codes [M][K]
    const __half2 *scales;         //                 scales [M][K/32]
    const float *x;                // f32 front end: activation [M][ldx]
    int64_t ldx;
    int8_t *codes_out;             //                optional copy of the codes it computed
    __half2 *scales_out;           //                and of the scales
    int64_t N;
    int K;
    const float *residual;
    float *y;
};

// 16-byte chunk c of an activation row lives at chunk position swz(c); for
// c = 128*s + c' (c' < 128), swz(c) = 128*s + swz(c')
__device__ __forceinline__ int swz(int c) { return c ^ ((c >> 2) & 7); }

__device__ __forceinline__ uint4 lds16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ float f16lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

__device__ __forceinline__ int sum16(uint4 v)
{
    int s = qk::dp4a_ss(v.x, 0x01010101u, 0);
    s = qk::dp4a_ss(v.y, 0x01010101u, s);
    s = qk::dp4a_ss(v.z, 0x01010101u, s);
    return qk::dp4a_ss(v.w, 0x01010101u, s);
}

// --------------------------------------------------------------- staging
// One pass over the M x K codes in 16-byte chunks: copy to the swizzled
// shared-memory image and reduce the chunk's code sum (exact, dp4a).

// Q4_K side data per (m, 32-block): {d_a, d_a * sum(q_a)}; odd blocks are the
// high-nibble sub-blocks whose codes the kernel reads as 16*q, so their d_a
// is stored divided by 16 (exact).
template <int M, int NT>
__device__ void stage_act_q4k(const int8_t *__restrict__ codes, const __half2 *__restrict__ scales, int K,
                              uint8_t *s_codes, float2 *s_sc)
{
    const int nchunk = K >> 4, total = M * nchunk;        // total is even
    for (int base = 0; base < total; base += NT) {
        const int i = base + threadIdx.x;
        const bool ok = i < total;
        const int m = ok ? i / nchunk : 0, c = ok ? i - m * nchunk : 0;
        uint4 v = make_uint4(0, 0, 0, 0);
        float d = 0.0f;
        if (ok) {                                          // both loads in flight together
            v = *reinterpret_cast<const uint4 *>(codes + (size_t)m * K + 16 * c);
            d = __low2float(scales[(size_t)m * (K >> 5) + (c >> 1)]);
            *reinterpret_cast<uint4 *>(s_codes + (size_t)m * K + 16 * swz(c)) = v;
        }
        int s = sum16(v);
        s += __shfl_xor_sync(0xffffffffu, s, 1);           // the other half of the 32-value block
        if (ok && (c & 1) == 0) {
            const int b = c >> 1;
            s_sc[m * (K >> 5) + b] = make_float2((b & 1) ? d * 0.0625f : d, d * (float)s);
        }
    }
}

// Q6_K side data per (m, 16-value chunk): d_a and -32 * d_a * sum(q_a), the
// activation scale and the offset term of the weight codes' -32 bias (exact),
// kept as two float planes D [M][K/16] and Bias [M][K/16] (Bias after D).
// Within each 128-chunk step the entries are stored in the order the lanes
// read them: chunk 16j + 8h + e + 2t (lane 4j+2h+e, quarter t) at 4*lane + t,
// so a lane fetches its four scales and its four biases with one 16-byte load
// each, 8 lanes covering 128 consecutive bytes (no bank conflict).
__device__ __forceinline__ int q6_side_pos(int c)
{
    const int lo = c & 127;
    return (c & ~127) + ((((lo >> 4) << 2) + (((lo >> 3) & 1) << 1) + (lo & 1)) << 2) + ((lo >> 1) & 3);
}

template <int M, int NT>
__device__ void stage_act_q6k(const int8_t *__restrict__ codes, const __half2 *__restrict__ scales, int K,
                              uint8_t *s_codes, float2 *s_c16)
{
    const int nchunk = K >> 4;
    float *sd = reinterpret_cast<float *>(s_c16), *sb = sd + M * nchunk;
    for (int i = threadIdx.x; i < M * nchunk; i += NT) {
        const int m = i / nchunk, c = i - m * nchunk;
        const uint4 v = *reinterpret_cast<const uint4 *>(codes + (size_t)m * K + 16 * c);
        *reinterpret_cast<uint4 *>(s_codes + (size_t)m * K + 16 * swz(c)) = v;
        const float d = __low2float(scales[(size_t)m * (K >> 5) + (c >> 1)]);
        const int pos = m * nchunk + q6_side_pos(c);
        sd[pos] = d;
        sb[pos] = -32.0f * d * (float)sum16(v);
    }
}

// a lane's four Q6_K side entries of activation row m at step s: d_a and bias of quarters 0..3
template <int M>
__device__ __forceinline__ void q6_side4(const float2 *s_c16, int K, int m, int s, int lane, float4 &dq, float4 &bq)
{
    const int nc = K >> 4;
    const float *sd = reinterpret_cast<const float *>(s_c16) + (size_t)m * nc + 128 * s + 4 * lane;
    dq = *reinterpret_cast<const float4 *>(sd);
    bq = *reinterpret_cast<const float4 *>(sd + (size_t)M * nc);
}

// f32 front end: quantize the activation into the same shared-memory image
// (Q6 selects the Q6_K side data).  8 lanes per 32-value block, 4 values per
// lane; CTA 0 also writes the codes and scales out when asked to.
// U float4 per thread per batch, all of them loaded before any is quantized; the
// batch loop has no early exit, so the U blocks' shuffle and division chains
// interleave (lanes past the end quantize zeros and store nothing)
template <int M, int NT, bool Q6, int U>
__device__ void stage_quant_u(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
{
    const int K = a.K, k4n = K >> 2, total = M * k4n;      // total is a multiple of 8
    const int nb = K >> 5;
    const bool out = a.codes_out != nullptr && blockIdx.x == 0;
    for (int base = 0; base < total; base += NT * U) {
        float4 v[U];
        int idx[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int i = base + u * NT + threadIdx.x;
            idx[u] = -1;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < total) {
                idx[u] = i;
                const int m = i / k4n, k4 = i - m * k4n;
                v[u] = *reinterpret_cast<const float4 *>(a.x + m * a.ldx + 4 * k4);
            }
        }
        float d[U];
        int s4[U];
        uint32_t packed[U];
#pragma unroll
        for (int u = 0; u < U; u++) packed[u] = qk::q81_quant8(v[u], d[u], s4[u]);
#pragma unroll
        for (int u = 0; u < U; u++) {
            int s16 = s4[u] + __shfl_xor_sync(0xffffffffu, s4[u], 1);
            s16 += __shfl_xor_sync(0xffffffffu, s16, 2);                  // 16 values (4 lanes)
            const int s32 = s16 + __shfl_xor_sync(0xffffffffu, s16, 4);   // the 32-value block
            const int i = idx[u];
            if (i >= 0) {
                const int m = i / k4n, k4 = i - m * k4n;
                const int c = k4 >> 2, sub = k4 & 7;
                *reinterpret_cast<uint32_t *>(s_codes + (size_t)m * K + 16 * swz(c) + 4 * (k4 & 3)) = packed[u];
                const __half dh = qk::f16_sat(d[u]);
                const float da = __half2float(dh);                         // the stored scale is what the dot uses
                if (!Q6) {
                    if (sub == 0) {
                        const int b = k4 >> 3;
                        s_side[m * nb + b] = make_float2((b & 1) ? da * 0.0625f : da, da * (float)s32);
                    }
                } else if ((sub & 3) == 0) {
                    float *sd = reinterpret_cast<float *>(s_side);
                    const int pos = m * (K >> 4) + q6_side_pos(c);
                    sd[pos] = da;
                    sd[M * (K >> 4) + pos] = -32.0f * da * (float)s16;
                }
                if (out) {
                    *reinterpret_cast<uint32_t *>(a.codes_out + (size_t)m * K + 4 * k4) = packed[u];
                    if (sub == 0)
                        a.scales_out[(size_t)m * nb + (k4 >> 3)] = __halves2half2(dh, qk::q81_sum_f16(d[u], s32));
                }
            }
        }
    }
}

// quantize the M x K f32 activation into the CTA's shared-memory q8_1 copy, with the
// batch size matched to the float4 count per thread
template <int M, int NT, bool Q6>
__device__ void stage_quant(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
{
    const int per = (M * (a.K >> 2) + NT - 1) / NT;
    if (per <= 1) stage_quant_u<M, NT, Q6, 1>(a, s_codes, s_side);
    else if (per <= 2) stage_quant_u<M, NT, Q6, 2>(a, s_codes, s_side);
    else if (per <= 4) stage_quant_u<M, NT, Q6, 4>(a, s_codes, s_side);
    else stage_quant_u<M, NT, Q6, 8>(a, s_codes, s_side);
}

// ------------------------------------------------------------ row reduce

__device__ __forceinline__ float warp_sum(float v)
{
    v += __shfl_xor_sync(0xffffffffu, v, 16);              // fixed xor tree over the 32 lanes
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

// Fixed-order reduce-scatter of 2^L per-lane values over the warp: at each of the first L xor
// steps (offsets 16, 8, ...) every lane keeps one half of its values and adds its partner's copy
// of that half, then the remaining 5 - L steps add up the one value left.  Lane l ends with the
// warp total of value l >> (5 - L).  Per group of outputs it takes about a third of the shuffles
// and adds of one xor tree per value.
template <int L>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[1 << L], int lane)
{
#pragma unroll
    for (int k = 0; k < L; k++) {
        const int o = 16 >> k, h = (1 << L) >> (k + 1);
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; i++) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 >> L; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

__host__ __device__ constexpr int ceil_log2(int v) { return v <= 1 ? 0 : 1 + ceil_log2((v + 1) / 2); }

// ------------------------------------------------------------ work split
// Rows are taken in groups of P consecutive rows; an item is (group, step s),
// the step-s bytes of the group's rows.  Groups are dealt round robin over
// the W warps of the grid (warp w takes groups w, w+W, ...), so at any time
// the grid streams one contiguous window of the weight; each group is
// finished by one warp, so no partial sums cross warps.  (A split of the
// last round into equal item ranges per CTA, combined in shared memory, was
// measured slower: it breaks the window into per-CTA streams.)
struct ItemSeq {
    int64_t g;                     // current item: group g, step s
    int s;
    int64_t sb;                    // index of the group's first superblock (g * P * B)
    int64_t W, gsb;                // groups per round, superblocks per group
    __device__ __forceinline__ void next(int nsteps)
    {
        if (++s == nsteps) s = 0, g += W, sb += W * gsb;
    }
};

// ------------------------------------------------------------------ Q4_K
// slot: [P][1024] code bytes of the step, then [P][8] 16-byte metadata records

constexpr int Q4_CODES = 1024, Q4_META = 128;

// PR weight rows per item: 2, or 4 for M >= 3 where one activation load then serves four rows
template <int PR>
struct Q4OpsT {
    static constexpr int P = PR;
    static constexpr int R = PR == 2 ? Q4_R : QK_GEMV_P4_Q4_RING, SLOT = PR * (Q4_CODES + Q4_META);
    static_assert(R >= 2, "ring needs two slots at least");
    struct LaneConst {
        uint32_t selA, selB;
        int aoff[4];
    };
    __device__ static LaneConst lane_const(int lane)
    {
        LaneConst c;
        const int g = lane & 3;
        c.selA = g == 0 ? 0x3210u : g == 1 ? 0x6543u : 0x7676u;
        c.selB = g == 0 ? 0x3210u : g == 1 ? 0x3210u : g == 2 ? 0x3410u : 0x3765u;
#pragma unroll
        for (int i = 0; i < 4; i++) c.aoff[i] = 16 * ((4 * lane + i) ^ (lane & 7));
        return c;
    }
    // copy item (group with first superblock sb, first row n, step s) into a ring slot; no register payload
    __device__ static uint32_t issue(uint8_t *slot, const uint8_t *__restrict__ w, int64_t N, int B, int64_t n,
                                     int64_t sb, int s, int lane)
    {
        const int nsb = min(8, B - 8 * s), G = 4 * nsb;
        const uint8_t *src = w + (sb << 7) + 1024 * s;                      // codes plane
        const uint8_t *meta = w + N * (int64_t)B * 128 + ((sb + 8 * s) << 4); // metadata plane
#pragma unroll
        for (int r = 0; r < P; r++) {
            if (n + r < N) {
                uint8_t *dst = slot + r * Q4_CODES;
                if (lane < G) {
                    qk::cp_async16(dst + 16 * lane, src + 16 * lane);
                    qk::cp_async16(dst + 16 * G + 16 * lane, src + 16 * G + 16 * lane);
                }
                if (lane < nsb) qk::cp_async16(slot + P * Q4_CODES + r * Q4_META + 16 * lane, meta + 16 * lane);
            }
            src += (int64_t)B * 128;
            meta += (int64_t)B * 16;
        }
        return 0;
    }
    template <int M>
    __device__ static void compute(const uint8_t *sl, int s, int B, int lane, uint32_t, const LaneConst &lc,
                                   const uint8_t *s_codes, const float2 *s_sc, int K, float (&acc)[P][M])
    {
        const int G = 4 * min(8, B - 8 * s);
        if (lane >= G) return;
        uint4 c0[P], c1[P];
        float d[P], dmin[P], m0[P], m1[P];
        int sc0[P], sc1[P];
#pragma unroll
        for (int r = 0; r < P; r++) {
            c0[r] = lds16(sl + r * Q4_CODES + 16 * lane);
            c1[r] = lds16(sl + r * Q4_CODES + 16 * G + 16 * lane);
            const uint4 mt = lds16(sl + P * Q4_CODES + r * Q4_META + 16 * (lane >> 2));
            d[r] = f16lo(mt.x);
            dmin[r] = f16hi(mt.x);
            // this lane's group record: sc0 | sc1<<6 | m0<<12 | m1<<18
            const uint32_t rec = __byte_perm(__byte_perm(mt.y, mt.z, lc.selA), mt.w, lc.selB);
            sc0[r] = rec & 63u;
            sc1[r] = (rec >> 6) & 63u;
            m0[r] = (float)((rec >> 12) & 63u);
            m1[r] = (float)((rec >> 18) & 63u);
        }
        const uint8_t *abase = s_codes + 2048 * s;             // activation of this step (chunk 128*s)
        const float2 *sbase = s_sc + 64 * s + 2 * lane;       // 32-blocks 8*(8s + lane/4) + 2g, +1
        const int nb = K >> 5;
#pragma unroll
        for (int m = 0; m < M; m++) {
            const uint8_t *ar = abase + (size_t)m * K;
            const uint4 a0 = lds16(ar + lc.aoff[0]), a1 = lds16(ar + lc.aoff[1]);   // sub-block 2g
            const uint4 a2 = lds16(ar + lc.aoff[2]), a3 = lds16(ar + lc.aoff[3]);   // sub-block 2g+1
            const float4 sa = *reinterpret_cast<const float4 *>(sbase + (size_t)m * nb);   // d0 S0 d1/16 S1
#pragma unroll
            for (int r = 0; r < P; r++) {
                const uint4 x0 = c0[r], x1 = c1[r];
                int il = qk::dp4a_ss(x0.x & 0x0F0F0F0Fu, a0.x, 0), ih = qk::dp4a_us(x0.x & 0xF0F0F0F0u, a2.x, 0);
                il = qk::dp4a_ss(x0.y & 0x0F0F0F0Fu, a0.y, il), ih = qk::dp4a_us(x0.y & 0xF0F0F0F0u, a2.y, ih);
                il = qk::dp4a_ss(x0.z & 0x0F0F0F0Fu, a0.z, il), ih = qk::dp4a_us(x0.z & 0xF0F0F0F0u, a2.z, ih);
                il = qk::dp4a_ss(x0.w & 0x0F0F0F0Fu, a0.w, il), ih = qk::dp4a_us(x0.w & 0xF0F0F0F0u, a2.w, ih);
                il = qk::dp4a_ss(x1.x & 0x0F0F0F0Fu, a1.x, il), ih = qk::dp4a_us(x1.x & 0xF0F0F0F0u, a3.x, ih);
                il = qk::dp4a_ss(x1.y & 0x0F0F0F0Fu, a1.y, il), ih = qk::dp4a_us(x1.y & 0xF0F0F0F0u, a3.y, ih);
                il = qk::dp4a_ss(x1.z & 0x0F0F0F0Fu, a1.z, il), ih = qk::dp4a_us(x1.z & 0xF0F0F0F0u, a3.z, ih);
                il = qk::dp4a_ss(x1.w & 0x0F0F0F0Fu, a1.w, il), ih = qk::dp4a_us(x1.w & 0xF0F0F0F0u, a3.w, ih);
                float t = sa.x * (float)(il * sc0[r]);
                t = fmaf(sa.z, (float)(ih * sc1[r]), t);
                const float v = fmaf(m1[r], sa.w, m0[r] * sa.y);
                acc[r][m] = fmaf(d[r], t, fmaf(-dmin[r], v, acc[r][m]));
            }
        }
    }
    template <int M, int NT, bool FUSED>
    __device__ static void stage(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
    {
        if (FUSED) stage_quant<M, NT, false>(a, s_codes, s_side);
        else stage_act_q4k<M, NT>(a.codes, a.scales, a.K, s_codes, s_side);
    }
};
using Q4Ops = Q4OpsT<2>;

// ------------------------------------------------------------------ Q5_K
// slot: [P][1024] code bytes of the step, [P][256] fifth-bit words, [P][8] 16-byte metadata records.
// The codes and metadata are those of Q4_K; each lane adds its group's two fifth-bit words
// (R_lo, R_hi: bit 8b + w is the fifth bit of code byte 4w + b's low / high nibble).

constexpr int Q5_HB = 256;

struct Q5Ops {
    static constexpr int P = kRowsPerItem;
    static constexpr int R = Q5_R, SLOT = Q5_SLOT;
    using LaneConst = Q4Ops::LaneConst;
    __device__ static LaneConst lane_const(int lane) { return Q4Ops::lane_const(lane); }
    __device__ static uint32_t issue(uint8_t *slot, const uint8_t *__restrict__ w, int64_t N, int B, int64_t n,
                                     int64_t sb, int s, int lane)
    {
        const int nsb = min(8, B - 8 * s), G = 4 * nsb;
        const int64_t NB = N * (int64_t)B;
        const uint8_t *src = w + (sb << 7) + 1024 * s;                      // codes plane
        const uint8_t *hb = w + (NB << 7) + ((sb + 8 * s) << 5);            // fifth-bit plane
        const uint8_t *meta = w + NB * 160 + ((sb + 8 * s) << 4);           // metadata plane
#pragma unroll
        for (int r = 0; r < P; r++) {
            if (n + r < N) {
                uint8_t *dst = slot + r * Q4_CODES;
                if (lane < G) {
                    qk::cp_async16(dst + 16 * lane, src + 16 * lane);
                    qk::cp_async16(dst + 16 * G + 16 * lane, src + 16 * G + 16 * lane);
                }
                if (lane < 2 * nsb) qk::cp_async16(slot + P * Q4_CODES + r * Q5_HB + 16 * lane, hb + 16 * lane);
                if (lane < nsb)
                    qk::cp_async16(slot + P * (Q4_CODES + Q5_HB) + r * Q4_META + 16 * lane, meta + 16 * lane);
            }
            src += (int64_t)B * 128;
            hb += (int64_t)B * 32;
            meta += (int64_t)B * 16;
        }
        return 0;
    }
    // fifth bits of code word w (bytes 4w .. 4w+3) moved to bit 4 of each byte
    __device__ __forceinline__ static uint32_t fifth(uint32_t R, int w)
    {
        return (w <= 4 ? R << (4 - w) : R >> (w - 4)) & 0x10101010u;
    }
    template <int M>
    __device__ static void compute(const uint8_t *sl, int s, int B, int lane, uint32_t, const LaneConst &lc,
                                   const uint8_t *s_codes, const float2 *s_sc, int K, float (&acc)[P][M])
    {
        const int G = 4 * min(8, B - 8 * s);
        if (lane >= G) return;
        uint32_t lo5[P][8];                        // low-nibble codes with their fifth bits (0 .. 31)
        uint32_t hn[P][8], hb[P][8];               // high nibbles in place (16 q) and their fifth bits (0 / 1)
        float d[P], dmin[P], m0[P], m1[P];
        int sc0[P], sc1[P];
#pragma unroll
        for (int r = 0; r < P; r++) {
            const uint4 c0 = lds16(sl + r * Q4_CODES + 16 * lane);
            const uint4 c1 = lds16(sl + r * Q4_CODES + 16 * G + 16 * lane);
            const uint2 fb = *reinterpret_cast<const uint2 *>(sl + P * Q4_CODES + r * Q5_HB + 8 * lane);
            const uint4 mt = lds16(sl + P * (Q4_CODES + Q5_HB) + r * Q4_META + 16 * (lane >> 2));
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int i = 0; i < 8; i++) {
                lo5[r][i] = (cw[i] & 0x0F0F0F0Fu) | fifth(fb.x, i);
                hn[r][i] = cw[i] & 0xF0F0F0F0u;
                hb[r][i] = (fb.y >> i) & 0x01010101u;
            }
            d[r] = f16lo(mt.x);
            dmin[r] = f16hi(mt.x);
            const uint32_t rec = __byte_perm(__byte_perm(mt.y, mt.z, lc.selA), mt.w, lc.selB);
            sc0[r] = rec & 63u;
            sc1[r] = (rec >> 6) & 63u;
            m0[r] = (float)((rec >> 12) & 63u);
            m1[r] = (float)((rec >> 18) & 63u);
        }
        const uint8_t *abase = s_codes + 2048 * s;
        const float2 *sbase = s_sc + 64 * s + 2 * lane;
        const int nb = K >> 5;
#pragma unroll
        for (int m = 0; m < M; m++) {
            const uint8_t *ar = abase + (size_t)m * K;
            const uint4 a0 = lds16(ar + lc.aoff[0]), a1 = lds16(ar + lc.aoff[1]);   // sub-block 2g
            const uint4 a2 = lds16(ar + lc.aoff[2]), a3 = lds16(ar + lc.aoff[3]);   // sub-block 2g+1
            const uint32_t al[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t ah[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
            const float4 sa = *reinterpret_cast<const float4 *>(sbase + (size_t)m * nb);   // d0 S0 d1/16 S1
#pragma unroll
            for (int r = 0; r < P; r++) {
                int il = 0, ih = 0, ib = 0;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    il = qk::dp4a_ss(lo5[r][i], al[i], il);
                    ih = qk::dp4a_us(hn[r][i], ah[i], ih);
                    ib = qk::dp4a_ss(hb[r][i], ah[i], ib);
                }
                ih += ib << 8;                     // 16 * (high nibble + 16 * fifth bit)
                float t = sa.x * (float)(il * sc0[r]);
                t = fmaf(sa.z, (float)(ih * sc1[r]), t);
                const float v = fmaf(m1[r], sa.w, m0[r] * sa.y);
                acc[r][m] = fmaf(d[r], t, fmaf(-dmin[r], v, acc[r][m]));
            }
        }
    }
    template <int M, int NT, bool FUSED>
    __device__ static void stage(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
    {
        Q4Ops::stage<M, NT, FUSED>(a, s_codes, s_side);
    }
};

// ------------------------------------------------------------------ Q8_0
// slot: [P][2048] int8 codes of the step (2048 values), then [P][128] binary16 block scales.
// Lane l takes the 16-value chunks l, l + 32, l + 64, l + 96 of the step; its dot with the
// activation chunk (same 32-value block) is folded with d_w * d_a per chunk.

constexpr int Q80_CODES = 2048, Q80_D = 128;

struct Q80Ops {
    static constexpr int P = kRowsPerItem;
    static constexpr int R = Q80_R, SLOT = Q80_SLOT;
    struct LaneConst {
        int aoff[4];
    };
    __device__ static LaneConst lane_const(int lane)
    {
        LaneConst c;
#pragma unroll
        for (int i = 0; i < 4; i++) c.aoff[i] = 16 * swz(lane + 32 * i);
        return c;
    }
    __device__ static uint32_t issue(uint8_t *slot, const uint8_t *__restrict__ w, int64_t N, int B, int64_t n,
                                     int64_t sb, int s, int lane)
    {
        const int nsb = min(8, B - 8 * s), nch = 16 * nsb;
        const uint8_t *src = w + (sb << 8) + 2048 * s;                               // codes plane, row n
        const uint8_t *dsrc = w + ((N * (int64_t)B) << 8) + (sb << 4) + 128 * s;    // d plane, row n
#pragma unroll
        for (int r = 0; r < P; r++) {
            if (n + r < N) {
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int c = lane + 32 * i;
                    if (c < nch) qk::cp_async16(slot + r * Q80_CODES + 16 * c, src + 16 * c);
                }
                if (lane < nsb) qk::cp_async16(slot + P * Q80_CODES + r * Q80_D + 16 * lane, dsrc + 16 * lane);
            }
            src += (int64_t)B << 8;
            dsrc += (int64_t)B << 4;
        }
        return 0;
    }
    template <int M>
    __device__ static void compute(const uint8_t *sl, int s, int B, int lane, uint32_t, const LaneConst &lc,
                                   const uint8_t *s_codes, const float2 *s_sc, int K, float (&acc)[P][M])
    {
        const int nch = 16 * min(8, B - 8 * s);
        if (lane >= nch) return;
        uint4 wc[P][4];
        float dw[P][4];
#pragma unroll
        for (int r = 0; r < P; r++)
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int c = lane + 32 * i;
                wc[r][i] = make_uint4(0, 0, 0, 0);
                dw[r][i] = 0.0f;
                if (c < nch) {
                    wc[r][i] = lds16(sl + r * Q80_CODES + 16 * c);
                    dw[r][i] = __half2float(*reinterpret_cast<const __half *>(sl + P * Q80_CODES + r * Q80_D +
                                                                              2 * (c >> 1)));
                }
            }
        const uint8_t *abase = s_codes + 2048 * s;
        const int nb = K >> 5;
#pragma unroll
        for (int m = 0; m < M; m++) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int c = lane + 32 * i;
                if (c < nch) {
                    const uint4 a = lds16(abase + (size_t)m * K + lc.aoff[i]);
                    // the Q4_K side data holds d_a / 16 for odd 32-value blocks: undo it (exact)
                    const float2 sa = s_sc[(size_t)m * nb + 64 * s + (c >> 1)];
                    const float da = (c & 2) ? sa.x * 16.0f : sa.x;
#pragma unroll
                    for (int r = 0; r < P; r++) {
                        int dot = qk::dp4a_ss(wc[r][i].x, a.x, 0);
                        dot = qk::dp4a_ss(wc[r][i].y, a.y, dot);
                        dot = qk::dp4a_ss(wc[r][i].z, a.z, dot);
                        dot = qk::dp4a_ss(wc[r][i].w, a.w, dot);
                        acc[r][m] = fmaf(dw[r][i] * da, (float)dot, acc[r][m]);
                    }
                }
            }
        }
    }
    template <int M, int NT, bool FUSED>
    __device__ static void stage(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
    {
        Q4Ops::stage<M, NT, FUSED>(a, s_codes, s_side);
    }
};

// ------------------------------------------------------------------ Q6_K
// slot: [P][1024] ql bytes of the step, [P][512] qh bytes, [P][8] 16-byte scale records

constexpr int Q6_QL = 1024, Q6_QH = 512, Q6_SC = 128;

template <int PR>
struct Q6OpsT {
    static constexpr int P = PR;
    static constexpr int R = PR == 2 ? Q6_R : QK_GEMV_P4_Q6_RING, SLOT = PR * (Q6_QL + Q6_QH + Q6_SC);
    static_assert(R >= 2, "ring needs two slots at least");
    struct LaneConst {
        int qoff[4], coff[4];
    };
    __device__ static LaneConst lane_const(int lane)
    {
        // lane (superblock lane/4, p = lane%4 = 2h+e) reads activation chunk
        // 16*(lane/4) + 8h + e + 2t of the step for quarter t
        LaneConst c;
        const int p = lane & 3, h = p >> 1, e = p & 1;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            c.coff[t] = 16 * (lane >> 2) + 8 * h + e + 2 * t;
            c.qoff[t] = 16 * swz(c.coff[t]);
        }
        return c;
    }
    // copy an item into a ring slot; returns this lane's binary16 d register:
    // lane 8r+j (j < nsb) holds d of superblock 8s+j of row r (2-byte records)
    __device__ static uint32_t issue(uint8_t *slot, const uint8_t *__restrict__ w, int64_t N, int B, int64_t n,
                                     int64_t sb, int s, int lane)
    {
        uint32_t dv = 0;
        const int nsb = min(8, B - 8 * s), L = 4 * nsb;
        const int64_t NB = N * (int64_t)B, sbs = sb + 8 * s;
        const uint8_t *ql = w + (sb << 7) + 1024 * s;
        const uint8_t *qh = w + (NB << 7) + (sbs << 6);
        const uint8_t *sc = w + NB * 192 + (sbs << 4);
        const uint8_t *dp = w + NB * 208 + (sbs << 1);
#pragma unroll
        for (int r = 0; r < P; r++) {
            if (n + r < N) {
                uint8_t *dst = slot + r * Q6_QL;
                if (lane < L) {
                    qk::cp_async16(dst + 16 * lane, ql + 16 * lane);
                    qk::cp_async16(dst + 16 * L + 16 * lane, ql + 16 * L + 16 * lane);
                    qk::cp_async16(slot + P * Q6_QL + r * Q6_QH + 16 * lane, qh + 16 * lane);
                }
                if (lane < nsb) qk::cp_async16(slot + P * (Q6_QL + Q6_QH) + r * Q6_SC + 16 * lane, sc + 16 * lane);
                if ((lane >> 3) == r && (lane & 7) < nsb) dv = qk::ldg_stream2(dp + 2 * (lane & 7));
            }
            ql += (int64_t)B * 128;
            qh += (int64_t)B * 64;
            sc += (int64_t)B * 16;
            dp += (int64_t)B * 2;
        }
        return dv;
    }
    template <int M>
    __device__ static void compute(const uint8_t *sl, int s, int B, int lane, uint32_t dreg, const LaneConst &lc,
                                   const uint8_t *s_codes, const float2 *s_c16, int K, float (&acc)[P][M])
    {
        const int L = 4 * min(8, B - 8 * s);
        float d[P];
#pragma unroll
        for (int r = 0; r < P; r++)
            d[r] = __half2float(__ushort_as_half((unsigned short)__shfl_sync(0xffffffffu, dreg, 8 * r + (lane >> 2))));
        if (lane >= L) return;
        uint4 qa[P], qb[P], qhh[P];
        float dsc[P][4];
#pragma unroll
        for (int r = 0; r < P; r++) {
            qa[r] = lds16(sl + r * Q6_QL + 16 * lane);
            qb[r] = lds16(sl + r * Q6_QL + 16 * L + 16 * lane);
            qhh[r] = lds16(sl + P * Q6_QL + r * Q6_QH + 16 * lane);
            const uint32_t scw =
                *reinterpret_cast<const uint32_t *>(sl + P * (Q6_QL + Q6_QH) + r * Q6_SC + 4 * lane);
#pragma unroll
            for (int t = 0; t < 4; t++) dsc[r][t] = d[r] * (float)(int)(int8_t)(scw >> (8 * t));
        }
        const uint8_t *abase = s_codes + 2048 * s;
        if (M <= 2) {
            // u = low4 + 16*high2: each part is dotted with its bits masked in place and the power-of-two
            // factor restored on the integer sums (2 logic ops + 2 dp4a per word, no shifts)
#pragma unroll
            for (int m = 0; m < M; m++) {
                const uint8_t *ar = abase + (size_t)m * K;
                float4 dq, bq;
                q6_side4<M>(s_c16, K, m, s, lane, dq, bq);
                const float2 dc[4] = {make_float2(dq.x, bq.x), make_float2(dq.y, bq.y), make_float2(dq.z, bq.z),
                                      make_float2(dq.w, bq.w)};
                uint4 av[4];
#pragma unroll
                for (int t = 0; t < 4; t++) av[t] = lds16(ar + lc.qoff[t]);
#pragma unroll
                for (int r = 0; r < P; r++) {
                    const uint32_t aw[4] = {qa[r].x, qa[r].y, qa[r].z, qa[r].w};
                    const uint32_t bw[4] = {qb[r].x, qb[r].y, qb[r].z, qb[r].w};
                    const uint32_t hw[4] = {qhh[r].x, qhh[r].y, qhh[r].z, qhh[r].w};
                    int n0 = 0, h0 = 0, n1 = 0, h1 = 0, n2 = 0, h2 = 0, n3 = 0, h3 = 0;
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint32_t x0 = (&av[0].x)[j], x1 = (&av[1].x)[j], x2 = (&av[2].x)[j], x3 = (&av[3].x)[j];
                        n0 = qk::dp4a_ss(aw[j] & 0x0F0F0F0Fu, x0, n0);   // low4 of quarter 0
                        h0 = qk::dp4a_ss(hw[j] & 0x03030303u, x0, h0);   // high2 of quarter 0
                        n1 = qk::dp4a_ss(bw[j] & 0x0F0F0F0Fu, x1, n1);
                        h1 = qk::dp4a_ss(hw[j] & 0x0C0C0C0Cu, x1, h1);   // = 4 * high2
                        n2 = qk::dp4a_us(aw[j] & 0xF0F0F0F0u, x2, n2);   // = 16 * low4
                        h2 = qk::dp4a_ss(hw[j] & 0x30303030u, x2, h2);   // = 16 * high2
                        n3 = qk::dp4a_us(bw[j] & 0xF0F0F0F0u, x3, n3);   // = 16 * low4
                        h3 = qk::dp4a_us(hw[j] & 0xC0C0C0C0u, x3, h3);   // = 64 * high2
                    }
                    const int u0 = n0 + 16 * h0, u1 = n1 + 4 * h1;     // sum of u * q_a
                    const int u2 = n2 + 16 * h2, u3 = n3 + 4 * h3;     // 16 * sum of u * q_a
                    float t = acc[r][m];
                    t = fmaf(dsc[r][0], fmaf(dc[0].x, (float)u0, dc[0].y), t);
                    t = fmaf(dsc[r][1], fmaf(dc[1].x, (float)u1, dc[1].y), t);
                    t = fmaf(dsc[r][2], fmaf(dc[2].x * 0.0625f, (float)u2, dc[2].y), t);
                    t = fmaf(dsc[r][3], fmaf(dc[3].x * 0.0625f, (float)u3, dc[3].y), t);
                    acc[r][m] = t;
                }
            }
        } else {
            // 6-bit codes u = low4 | high2 << 4 in [0, 63] built once and reused for every row m
            uint32_t u[P][4][4];
#pragma unroll
            for (int r = 0; r < P; r++) {
                const uint32_t aw[4] = {qa[r].x, qa[r].y, qa[r].z, qa[r].w};
                const uint32_t bw[4] = {qb[r].x, qb[r].y, qb[r].z, qb[r].w};
                const uint32_t hw[4] = {qhh[r].x, qhh[r].y, qhh[r].z, qhh[r].w};
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    u[r][0][j] = (aw[j] & 0x0F0F0F0Fu) | ((hw[j] << 4) & 0x30303030u);
                    u[r][1][j] = (bw[j] & 0x0F0F0F0Fu) | ((hw[j] << 2) & 0x30303030u);
                    u[r][2][j] = ((aw[j] >> 4) & 0x0F0F0F0Fu) | (hw[j] & 0x30303030u);
                    u[r][3][j] = ((bw[j] >> 4) & 0x0F0F0F0Fu) | ((hw[j] >> 2) & 0x30303030u);
                }
            }
#pragma unroll
            for (int m = 0; m < M; m++) {
                const uint8_t *ar = abase + (size_t)m * K;
                float4 dq, bq;
                q6_side4<M>(s_c16, K, m, s, lane, dq, bq);
                const float2 dc[4] = {make_float2(dq.x, bq.x), make_float2(dq.y, bq.y), make_float2(dq.z, bq.z),
                                      make_float2(dq.w, bq.w)};
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    const uint4 av = lds16(ar + lc.qoff[t]);
#pragma unroll
                    for (int r = 0; r < P; r++) {
                        int dot = qk::dp4a_ss(u[r][t][0], av.x, 0);
                        dot = qk::dp4a_ss(u[r][t][1], av.y, dot);
                        dot = qk::dp4a_ss(u[r][t][2], av.z, dot);
                        dot = qk::dp4a_ss(u[r][t][3], av.w, dot);
                        acc[r][m] = fmaf(dsc[r][t], fmaf(dc[t].x, (float)dot, dc[t].y), acc[r][m]);
                    }
                }
            }
        }
    }
    template <int M, int NT, bool FUSED>
    __device__ static void stage(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
    {
        if (FUSED) stage_quant<M, NT, true>(a, s_codes, s_side);
        else stage_act_q6k<M, NT>(a.codes, a.scales, a.K, s_codes, s_side);
    }
};
using Q6Ops = Q6OpsT<2>;

// ------------------------------------------------------------- Q2_K / Q3_K
// slot: [P][512] 2-bit codes of the step, Q3_K only [P][256] hmask bytes, then [P][128] scale records.
// The lane of superblock j of the step with p = lane % 4 = 2n + e holds code bytes 32n + 16e .. +16
// (four codes each: quarters t = 0..3 at bits 2t) and meets the same activation chunks as the Q6_K
// lanes, so the Q6_K activation staging (d_a and -32 d_a sum(q_a) per 16 values) serves both:
//   Q2_K  w = d sc q - dmin m:       acc += d sc (d_a dot) + dmin m (-32 d_a sum(q_a)) / 32
//   Q3_K  w = d S (q + 4 h - 4):     acc += d S (d_a (dot(q) + 4 dot(h)) + (-32 d_a sum(q_a)) / 8)
// The codes of quarter t are dotted in place (bits 2t, 2t+1 of each byte: 4^t q, at most 192, an
// unsigned byte) and the hmask bits likewise (2^(4n+t) h); the powers of two are undone in the
// binary32 factors, exactly.

template <int QT>
struct Q23Ops {
    static constexpr int P = kRowsPerItem;
    static constexpr bool Q3 = QT == QK_TYPE_Q3_K;
    static constexpr int CODES = 512, HM = Q3 ? 256 : 0, SCR = 128;
    static constexpr int R = Q4_R, SLOT = Q3 ? Q3_SLOT : Q2_SLOT;
    using LaneConst = Q6Ops::LaneConst;
    __device__ static LaneConst lane_const(int lane) { return Q6Ops::lane_const(lane); }
    // copy an item into a ring slot; returns this lane's d record: lane 8r + j (j < nsb) holds the
    // binary16 d (Q3_K) or d | dmin << 16 (Q2_K) of superblock 8s + j of row r
    __device__ static uint32_t issue(uint8_t *slot, const uint8_t *__restrict__ w, int64_t N, int B, int64_t n,
                                     int64_t sb, int s, int lane)
    {
        uint32_t dv = 0;
        const int nsb = min(8, B - 8 * s), L = 4 * nsb;
        const int64_t NB = N * (int64_t)B, sbs = sb + 8 * s;
        const uint8_t *codes = w + (sb << 6) + 512 * s;
        const uint8_t *hm = w + (NB << 6) + (sbs << 5);
        const uint8_t *sc = w + NB * (Q3 ? 96 : 64) + (sbs << 4);
        const uint8_t *dd = w + NB * (Q3 ? 112 : 80) + sbs * (Q3 ? 2 : 4);
#pragma unroll
        for (int r = 0; r < P; r++) {
            if (n + r < N) {
                if (lane < L) qk::cp_async16(slot + r * CODES + 16 * lane, codes + 16 * lane);
                if (Q3 && lane < 2 * nsb) qk::cp_async16(slot + P * CODES + r * HM + 16 * lane, hm + 16 * lane);
                if (lane < nsb) qk::cp_async16(slot + P * (CODES + HM) + r * SCR + 16 * lane, sc + 16 * lane);
                if ((lane >> 3) == r && (lane & 7) < nsb)
                    dv = Q3 ? qk::ldg_stream2(dd + 2 * (lane & 7)) : qk::ldg_stream4(dd + 4 * (lane & 7));
            }
            codes += (int64_t)B * 64;
            hm += (int64_t)B * 32;
            sc += (int64_t)B * 16;
            dd += (int64_t)B * (Q3 ? 2 : 4);
        }
        return dv;
    }
    template <int M>
    __device__ static void compute(const uint8_t *sl, int s, int B, int lane, uint32_t dreg, const LaneConst &lc,
                                   const uint8_t *s_codes, const float2 *s_c16, int K, float (&acc)[P][M])
    {
        const int L = 4 * min(8, B - 8 * s);
        uint32_t dr[P];
#pragma unroll
        for (int r = 0; r < P; r++) dr[r] = __shfl_sync(0xffffffffu, dreg, 8 * r + (lane >> 2));
        if (lane >= L) return;
        const int hsh = 4 * ((lane >> 1) & 1);                // hmask bit 4n + t of this lane's half n
        uint4 cq[P], hq[P];
        float dsl[P][4], dml[P][4];
#pragma unroll
        for (int r = 0; r < P; r++) {
            cq[r] = lds16(sl + r * CODES + 16 * lane);
            hq[r] = Q3 ? lds16(sl + P * CODES + r * HM + 32 * (lane >> 2) + 16 * (lane & 1)) : make_uint4(0, 0, 0, 0);
            const uint32_t scw = *reinterpret_cast<const uint32_t *>(sl + P * (CODES + HM) + r * SCR + 4 * lane);
            const float d = f16lo(dr[r]);
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const float inv4t = 1.0f / (float)(1 << (2 * t));                 // 4^-t, exact
                if (Q3) {
                    dsl[r][t] = d * (float)(int)(int8_t)(scw >> (8 * t));
                    dml[r][t] = 0.0f;
                } else {
                    dsl[r][t] = d * (float)((scw >> (8 * t)) & 15u) * inv4t;
                    dml[r][t] = f16hi(dr[r]) * (float)((scw >> (8 * t + 4)) & 15u) * 0.03125f;   // / 32, exact
                }
            }
        }
        const uint8_t *abase = s_codes + 2048 * s;
#pragma unroll
        for (int m = 0; m < M; m++) {
            float4 dq, bq;
            q6_side4<M>(s_c16, K, m, s, lane, dq, bq);
            const float2 dcs[4] = {make_float2(dq.x, bq.x), make_float2(dq.y, bq.y), make_float2(dq.z, bq.z),
                                   make_float2(dq.w, bq.w)};
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const uint4 av = lds16(abase + (size_t)m * K + lc.qoff[t]);
                const float2 dc = dcs[t];
#pragma unroll
                for (int r = 0; r < P; r++) {
                    const uint32_t xw[4] = {cq[r].x, cq[r].y, cq[r].z, cq[r].w};
                    const uint32_t hw[4] = {hq[r].x, hq[r].y, hq[r].z, hq[r].w};
                    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
                    const uint32_t cmask = 0x03030303u << (2 * t), hmask = 0x01010101u << (hsh + t);
                    int dot = 0, doth = 0;
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        dot = qk::dp4a_us(xw[k] & cmask, aw[k], dot);                 // 4^t q
                        if (Q3) doth = qk::dp4a_us(hw[k] & hmask, aw[k], doth);       // 2^(4n+t) h
                    }
                    if (Q3) {
                        // d_a (q . a + 4 h . a) with q . a = dot / 4^t and h . a = doth / 2^(4n+t)
                        const float qa = fmaf((float)doth, __uint_as_float((uint32_t)(129 - hsh - t) << 23),
                                              (float)dot * (1.0f / (float)(1 << (2 * t))));
                        acc[r][m] = fmaf(dsl[r][t], fmaf(dc.x, qa, dc.y * 0.125f), acc[r][m]);
                    } else {
                        acc[r][m] = fmaf(dsl[r][t], dc.x * (float)dot, fmaf(dml[r][t], dc.y, acc[r][m]));
                    }
                }
            }
        }
    }
    template <int M, int NT, bool FUSED>
    __device__ static void stage(const GemvArgs &a, uint8_t *s_codes, float2 *s_side)
    {
        Q6Ops::stage<M, NT, FUSED>(a, s_codes, s_side);
    }
};

// ---------------------------------------------------------------- driver

// L2 prefetch of the rows this CTA is about to stage: the f32 activation, or the
// q8_1 codes and scales (one prefetch per 128-byte line)
template <int M, int NT, bool FUSED>
__device__ __forceinline__ void prefetch_activation(const GemvArgs &a)
{
    const int K = a.K;
    if (FUSED) {
        const int per_row = K >> 5;                        // 128-byte lines of K floats
        for (int i = threadIdx.x; i < M * per_row; i += NT) {
            const int m = i / per_row, j = i - m * per_row;
            qk::prefetch_l2(a.x + m * a.ldx + 32 * j);
        }
    } else {
        const int code_lines = (M * K) >> 7, scale_lines = (M * K) >> 10;   // K is a multiple of 256
        for (int i = threadIdx.x; i < code_lines + scale_lines; i += NT) {
            if (i < code_lines) qk::prefetch_l2(a.codes + 128 * i);
            else qk::prefetch_l2(reinterpret_cast<const uint8_t *>(a.scales) + 128 * (i - code_lines));
        }
    }
}

template <class Ops, int M, bool FUSED, int kWarps>
__device__ __forceinline__ void gemv_body(const GemvArgs &a, uint8_t *smem)
{
    constexpr int R = Ops::R, P = Ops::P, NT = kWarps * 32;
    if (QK_GEMV_TRIGGER == 0) qk::pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t N = a.N;
    const int K = a.K, B = K >> 8, nsteps = (B + 7) >> 3;
    const uint8_t *__restrict__ w = a.w;
    uint8_t *ring = smem + warp * (R * Ops::SLOT);
    uint8_t *s_codes = smem + kWarps * R * Ops::SLOT;
    float2 *s_side = reinterpret_cast<float2 *>(s_codes + (size_t)M * K);
    const typename Ops::LaneConst lc = Ops::lane_const(lane);

    // this warp's items: groups wg0, wg0+W, ... below NG, each with steps 0..nsteps-1
    const int64_t NG = (N + P - 1) / P;
    const int64_t W = (int64_t)gridDim.x * kWarps, wg0 = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t total = wg0 < NG ? ((NG - 1 - wg0) / W + 1) * nsteps : 0;
    ItemSeq rd;
    rd.W = W;
    rd.gsb = (int64_t)P * B;
    rd.g = wg0;
    rd.s = 0;
    rd.sb = wg0 * rd.gsb;
    ItemSeq wr = rd;

    // weights never depend on the previous kernel: the first R-1 items are
    // requested before waiting for it
    int64_t wi = 0;
    uint32_t reg[R - 1];
#pragma unroll
    for (int j = 0; j < R - 1; j++) {
        reg[j] = 0;
        if (wi < total) reg[j] = Ops::issue(ring + j * Ops::SLOT, w, N, B, P * wr.g, wr.sb, wr.s, lane);
        qk::cp_async_commit();
        wr.next(nsteps);
        ++wi;
    }
    // The activation may be written by the previous kernel, so it is read only after the
    // wait; its lines are requested into L2 now.  L2 is where the producer's stores land,
    // so a line fetched early is updated in place and the reads after the wait see the
    // producer's values; the prefetch only saves the DRAM latency when the activation is
    // not in L2 already.
    prefetch_activation<M, NT, FUSED>(a);
    qk::pdl_wait();
    Ops::template stage<M, NT, FUSED>(a, s_codes, s_side);
    __syncthreads();
    if (QK_GEMV_TRIGGER == 1) qk::pdl_launch_dependents();

    float acc[P][M];
#pragma unroll
    for (int r = 0; r < P; r++)
#pragma unroll
        for (int m = 0; m < M; m++) acc[r][m] = 0.0f;

    int slot = 0, wslot = R - 1;
    for (int64_t k = 0; k < total; k++) {
        uint32_t rnew = 0;
        if (wi < total) rnew = Ops::issue(ring + wslot * Ops::SLOT, w, N, B, P * wr.g, wr.sb, wr.s, lane);
        qk::cp_async_commit();
        wr.next(nsteps);
        ++wi;
        qk::cp_async_wait<R - 1>();
        __syncwarp();
        Ops::template compute<M>(ring + slot * Ops::SLOT, rd.s, B, lane, reg[0], lc, s_codes, s_side, K, acc);
        __syncwarp();
        if (rd.s == nsteps - 1) {
            if constexpr (M >= 3) {
                // the group's P x M sums by a fixed-order reduce-scatter: lane (j << (5 - LV))
                // holds sum j = r M + m and writes output m of row r
                constexpr int V = P * M, LV = ceil_log2(V);
                float v[1 << LV];
#pragma unroll
                for (int j = 0; j < (1 << LV); j++) v[j] = j < V ? acc[j / M][j % M] : 0.0f;
#pragma unroll
                for (int r = 0; r < P; r++)
#pragma unroll
                    for (int m = 0; m < M; m++) acc[r][m] = 0.0f;
                const float t = warp_reduce_scatter<LV>(v, lane);
                const int j = lane >> (5 - LV);
                if ((lane & ((1 << (5 - LV)) - 1)) == 0 && j < V) {
                    const int r = j / M, m = j - r * M;
                    const int64_t n = P * rd.g + r;
                    if (n < N) {
                        const size_t o = (size_t)m * N + n;
                        a.y[o] = a.residual ? __fadd_rn(t, a.residual[o]) : t;
                    }
                }
            } else {
                // fixed xor tree over the lanes, then lane m writes output m of each row of the group
#pragma unroll
                for (int r = 0; r < P; r++)
#pragma unroll
                    for (int m = 0; m < M; m++) {
                        const float v = warp_sum(acc[r][m]);
                        acc[r][m] = 0.0f;
                        const int64_t n = P * rd.g + r;
                        if (lane == m && n < N) {
                            const size_t o = (size_t)m * N + n;
                            a.y[o] = a.residual ? __fadd_rn(v, a.residual[o]) : v;
                        }
                    }
            }
        }
        rd.next(nsteps);
#pragma unroll
        for (int j = 0; j < R - 2; j++) reg[j] = reg[j + 1];
        reg[R - 2] = rnew;
        wslot = slot;
        slot = slot + 1 == R ? 0 : slot + 1;
    }
    qk::cp_async_wait<0>();
    if (QK_GEMV_TRIGGER == 2) qk::pdl_launch_dependents();
}

template <int M, bool FUSED, int PR>
__global__ void __launch_bounds__(KCfg<M, FUSED, PR>::threads, KCfg<M, FUSED, PR>::minb)
    gemv_q4k_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    gemv_body<Q4OpsT<PR>, M, FUSED, KCfg<M, FUSED, PR>::warps>(a, smem);
}

template <int M, bool FUSED, int PR, bool WIDE = false>
__global__ void __launch_bounds__(KCfg<M, FUSED, PR, WIDE>::threads, KCfg<M, FUSED, PR, WIDE>::minb)
    gemv_q6k_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    gemv_body<Q6OpsT<PR>, M, FUSED, KCfg<M, FUSED, PR, WIDE>::warps>(a, smem);
}

template <int M, bool FUSED>
__global__ void __launch_bounds__(Cfg<M, FUSED>::threads, Cfg<M, FUSED>::minb) gemv_q5k_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    gemv_body<Q5Ops, M, FUSED, Cfg<M, FUSED>::warps>(a, smem);
}

template <int M, bool FUSED>
__global__ void __launch_bounds__(Cfg<M, FUSED>::threads, Cfg<M, FUSED>::minb) gemv_q80_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    gemv_body<Q80Ops, M, FUSED, Cfg<M, FUSED>::warps>(a, smem);
}

template <int M, bool FUSED>
__global__ void __launch_bounds__(Cfg<M, FUSED>::threads, Cfg<M, FUSED>::minb) gemv_q2k_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    gemv_body<Q23Ops<QK_TYPE_Q2_K>, M, FUSED, Cfg<M, FUSED>::warps>(a, smem);
}

template <int M, bool FUSED>
__global__ void __launch_bounds__(Cfg<M, FUSED>::threads, Cfg<M, FUSED>::minb) gemv_q3k_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    gemv_body<Q23Ops<QK_TYPE_Q3_K>, M, FUSED, Cfg<M, FUSED>::warps>(a, smem);
}

// ------------------------------------------------------------------ host

typedef void (*gemv_fn)(const GemvArgs);

// per device and kernel: largest dynamic shared memory opted in so far
std::atomic<int> g_smem_set[qk::kMaxDevices][6][2][8][3];

int prepare(gemv_fn kern, std::atomic<int> &done, size_t smem)
{
    // opt in to more than 48 KB of dynamic shared memory; repeated only when a larger size is needed
    if ((int)smem <= done.load(std::memory_order_relaxed)) return QK_OK;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = qk::max_carveout(kern);
    if (e != cudaSuccess) return QK_E_CUDA;
    int prev = done.load(std::memory_order_relaxed);
    while ((int)smem > prev && !done.compare_exchange_weak(prev, (int)smem)) {
    }
    return QK_OK;
}

template <bool FUSED>
gemv_fn pick(int qtype, int M)
{
    static const gemv_fn q4[8] = {gemv_q4k_kernel<1, FUSED, 2>, gemv_q4k_kernel<2, FUSED, 2>, gemv_q4k_kernel<3, FUSED, 2>,
                                  gemv_q4k_kernel<4, FUSED, 2>, gemv_q4k_kernel<5, FUSED, 2>, gemv_q4k_kernel<6, FUSED, 2>,
                                  gemv_q4k_kernel<7, FUSED, 2>, gemv_q4k_kernel<8, FUSED, 2>};
    static const gemv_fn q6[8] = {gemv_q6k_kernel<1, FUSED, 2>, gemv_q6k_kernel<2, FUSED, 2>, gemv_q6k_kernel<3, FUSED, 2>,
                                  gemv_q6k_kernel<4, FUSED, 2>, gemv_q6k_kernel<5, FUSED, 2>, gemv_q6k_kernel<6, FUSED, 2>,
                                  gemv_q6k_kernel<7, FUSED, 2>, gemv_q6k_kernel<8, FUSED, 2>};
    static const gemv_fn q5[8] = {gemv_q5k_kernel<1, FUSED>, gemv_q5k_kernel<2, FUSED>, gemv_q5k_kernel<3, FUSED>,
                                  gemv_q5k_kernel<4, FUSED>, gemv_q5k_kernel<5, FUSED>, gemv_q5k_kernel<6, FUSED>,
                                  gemv_q5k_kernel<7, FUSED>, gemv_q5k_kernel<8, FUSED>};
    static const gemv_fn q80[8] = {gemv_q80_kernel<1, FUSED>, gemv_q80_kernel<2, FUSED>, gemv_q80_kernel<3, FUSED>,
                                   gemv_q80_kernel<4, FUSED>, gemv_q80_kernel<5, FUSED>, gemv_q80_kernel<6, FUSED>,
                                   gemv_q80_kernel<7, FUSED>, gemv_q80_kernel<8, FUSED>};
    static const gemv_fn q2[8] = {gemv_q2k_kernel<1, FUSED>, gemv_q2k_kernel<2, FUSED>, gemv_q2k_kernel<3, FUSED>,
                                  gemv_q2k_kernel<4, FUSED>, gemv_q2k_kernel<5, FUSED>, gemv_q2k_kernel<6, FUSED>,
                                  gemv_q2k_kernel<7, FUSED>, gemv_q2k_kernel<8, FUSED>};
    static const gemv_fn q3[8] = {gemv_q3k_kernel<1, FUSED>, gemv_q3k_kernel<2, FUSED>, gemv_q3k_kernel<3, FUSED>,
                                  gemv_q3k_kernel<4, FUSED>, gemv_q3k_kernel<5, FUSED>, gemv_q3k_kernel<6, FUSED>,
                                  gemv_q3k_kernel<7, FUSED>, gemv_q3k_kernel<8, FUSED>};
    return qtype == QK_TYPE_Q4_K   ? q4[M - 1]
           : qtype == QK_TYPE_Q5_K ? q5[M - 1]
           : qtype == QK_TYPE_Q8_0 ? q80[M - 1]
           : qtype == QK_TYPE_Q2_K ? q2[M - 1]
           : qtype == QK_TYPE_Q3_K ? q3[M - 1]
                                   : q6[M - 1];
}

// four-row kernels (Q4_K / Q6_K, M = 3..8)
template <bool FUSED>
gemv_fn pick4(int qtype, int M)
{
    static const gemv_fn q4[6] = {gemv_q4k_kernel<3, FUSED, 4>, gemv_q4k_kernel<4, FUSED, 4>,
                                  gemv_q4k_kernel<5, FUSED, 4>, gemv_q4k_kernel<6, FUSED, 4>,
                                  gemv_q4k_kernel<7, FUSED, 4>, gemv_q4k_kernel<8, FUSED, 4>};
    static const gemv_fn q6[6] = {gemv_q6k_kernel<3, FUSED, 4>, gemv_q6k_kernel<4, FUSED, 4>,
                                  gemv_q6k_kernel<5, FUSED, 4>, gemv_q6k_kernel<6, FUSED, 4>,
                                  gemv_q6k_kernel<7, FUSED, 4>, gemv_q6k_kernel<8, FUSED, 4>};
    return qtype == QK_TYPE_Q4_K ? q4[M - 3] : q6[M - 3];
}

// the wide (20-warp) Q6_K kernels, M = 1, 2
template <bool FUSED>
gemv_fn pick_q6_wide(int M)
{
    static const gemv_fn q6[2] = {gemv_q6k_kernel<1, FUSED, 2, true>, gemv_q6k_kernel<2, FUSED, 2, true>};
    return q6[M - 1];
}

int warps_for(int M, bool fused)
{
    return M > 2 ? QK_GEMV_WARPS : fused ? QK_GEMV_WARPS_FUSED : QK_GEMV_WARPS_SMALL_M;
}

int gemv(int qtype, bool fused, GemvArgs a, int64_t M, int64_t N, int64_t K, unsigned flags, void *stream)
{
    if (M < 1 || M > 8 || N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 ||
        M * K > (qtype == QK_TYPE_Q4_K || qtype == QK_TYPE_Q2_K || qtype == QK_TYPE_Q3_K ? 81920
                 : qtype == QK_TYPE_Q6_K                                                ? 40960
                                                                                        : 65536))
        return QK_E_SHAPE;
    if (!a.w || !a.y) return QK_E_NULL;
    if (fused ? !a.x : (!a.codes || !a.scales)) return QK_E_NULL;
    if (fused && (a.codes_out == nullptr) != (a.scales_out == nullptr)) return QK_E_NULL;
    if (fused && a.ldx < K) return QK_E_SHAPE;
    if (!qk::aligned(a.w, 16) || !qk::aligned(a.y, 4) || (a.residual && !qk::aligned(a.residual, 4)))
        return QK_E_ALIGN;
    if (!fused && (!qk::aligned(a.codes, 16) || !qk::aligned(a.scales, 16))) return QK_E_ALIGN;
    if (fused && (!qk::aligned(a.x, 16) || a.ldx % 4 != 0 || (a.codes_out && !qk::aligned(a.codes_out, 16)) ||
                  (a.scales_out && !qk::aligned(a.scales_out, 16))))
        return QK_E_ALIGN;
    size_t wbytes = 0;
    qk_repacked_bytes(qtype, N, K, &wbytes);
    const size_t ybytes = (size_t)M * N * 4, cbytes = (size_t)M * K, sbytes = (size_t)M * (K / 32) * 4;
    const size_t xbytes = fused ? ((size_t)(M - 1) * (size_t)a.ldx + (size_t)K) * 4 : 0;
    if (qk::overlaps(a.y, ybytes, a.w, wbytes) || qk::overlaps(a.y, ybytes, a.codes, cbytes) ||
        qk::overlaps(a.y, ybytes, a.scales, sbytes) || qk::overlaps(a.y, ybytes, a.x, xbytes) ||
        (a.residual != a.y && qk::overlaps(a.y, ybytes, a.residual, ybytes)))
        return QK_E_ALIAS;
    if (a.codes_out &&
        (qk::overlaps(a.codes_out, cbytes, a.x, xbytes) || qk::overlaps(a.scales_out, sbytes, a.x, xbytes) ||
         qk::overlaps(a.codes_out, cbytes, a.y, ybytes) || qk::overlaps(a.scales_out, sbytes, a.y, ybytes) ||
         qk::overlaps(a.codes_out, cbytes, a.w, wbytes) || qk::overlaps(a.scales_out, sbytes, a.w, wbytes) ||
         qk::overlaps(a.codes_out, cbytes, a.scales_out, sbytes) ||
         (a.residual && (qk::overlaps(a.codes_out, cbytes, a.residual, ybytes) ||
                         qk::overlaps(a.scales_out, sbytes, a.residual, ybytes)))))
        return QK_E_ALIAS;
    if ((flags & QK_GEMV_ROWS4) && (flags & QK_GEMV_ROWS2)) return QK_E_SHAPE;
    // ring | activation codes | side data
    const bool q6side = qtype == QK_TYPE_Q6_K || qtype == QK_TYPE_Q2_K || qtype == QK_TYPE_Q3_K;
    const size_t act = (size_t)M * K + (size_t)M * (K / 32) * (q6side ? 16 : 8);
    // four-row items: one activation load serves four weight rows (Q4_K / Q6_K, M >= 3).  Taken
    // when the row groups of four still give every warp of the grid one at least, or on request,
    // and only where the ring and the activation fit in shared memory.
    // (by default for Q4_K only: the Q6_K head measured slower with four-row items, 12 warps)
    const bool q46 = qtype == QK_TYPE_Q4_K || (qtype == QK_TYPE_Q6_K && (flags & QK_GEMV_ROWS4));
    const size_t smem4 = (size_t)QK_GEMV_P4_WARPS * (qtype == QK_TYPE_Q4_K ? Q4OpsT<4>::R * Q4OpsT<4>::SLOT
                                                                            : Q6OpsT<4>::R * Q6OpsT<4>::SLOT) +
                         act;
    const int64_t groups4 = (N + 3) / 4;
    const bool p4 = q46 && M >= 3 && !(flags & QK_GEMV_ROWS2) && smem4 <= qk::max_smem_optin() &&
                    ((flags & QK_GEMV_ROWS4) ||
                     groups4 >= (int64_t)QK_GEMV_P4_WARPS * kCtasPerSm * qk::sm_count());
    const int rows = p4 ? 4 : kRowsPerItem;
    // Q6_K with M <= 2: the 20-warp kernel where its ring and the activation fit
    const bool wide = !p4 && qtype == QK_TYPE_Q6_K && M <= 2 &&
                      (size_t)QK_GEMV_WARPS_Q6_SMALL_M * Q6_R * Q6_SLOT + act <= qk::max_smem_optin();
    const int warps = p4 ? QK_GEMV_P4_WARPS : wide ? QK_GEMV_WARPS_Q6_SMALL_M : warps_for((int)M, fused);
    const size_t smem = p4 ? smem4
                           : (size_t)warps * (qtype == QK_TYPE_Q4_K   ? Q4_R * Q4_SLOT
                                              : qtype == QK_TYPE_Q5_K ? Q5_R * Q5_SLOT
                                              : qtype == QK_TYPE_Q8_0 ? Q80_R * Q80_SLOT
                                              : qtype == QK_TYPE_Q2_K ? Q4_R * Q2_SLOT
                                              : qtype == QK_TYPE_Q3_K ? Q4_R * Q3_SLOT
                                                                      : Q6_R * Q6_SLOT) +
                                 act;
    if (smem > qk::max_smem_optin()) return QK_E_SHAPE;
    gemv_fn kern = p4     ? (fused ? pick4<true>(qtype, (int)M) : pick4<false>(qtype, (int)M))
                   : wide ? (fused ? pick_q6_wide<true>((int)M) : pick_q6_wide<false>((int)M))
                          : (fused ? pick<true>(qtype, (int)M) : pick<false>(qtype, (int)M));
    const int dev = qk::device_slot();
    if (dev < 0) return QK_E_CUDA;
    int st = prepare(kern, g_smem_set[dev][qtype - 1][fused ? 1 : 0][M - 1][p4 ? 1 : wide ? 2 : 0], smem);
    if (st != QK_OK) return st;
    int64_t grid = (int64_t)kCtasPerSm * qk::sm_count();
    const int64_t groups = (N + rows - 1) / rows;
    const int64_t need = (groups + warps - 1) / warps;              // CTAs that get a group in the first round
    if (grid > need) grid = need;
    a.N = N;
    a.K = (int)K;
    return qk::launch(kern, dim3((unsigned)grid), dim3(warps * 32), smem, (cudaStream_t)stream,
                      (flags & QK_LAUNCH_PDL) != 0, a);
}

GemvArgs q8_args(const void *w, const int8_t *codes, const void *scales, const float *residual, float *y)
{
    GemvArgs a = {};
    a.w = static_cast<const uint8_t *>(w);
    a.codes = codes;
    a.scales = static_cast<const __half2 *>(scales);
    a.residual = residual;
    a.y = y;
    return a;
}

GemvArgs f32_args(const void *w, const float *x, int64_t ldx, const float *residual, float *y, int8_t *codes_out,
                  void *scales_out)
{
    GemvArgs a = {};
    a.w = static_cast<const uint8_t *>(w);
    a.x = x;
    a.ldx = ldx;
    a.codes_out = codes_out;
    a.scales_out = static_cast<__half2 *>(scales_out);
    a.residual = residual;
    a.y = y;
    return a;
}

}  // namespace

extern "C" int qk_gemv_q4k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q4_K, false, q8_args(w, codes, scales, residual, y), M, N, K, flags, stream);
}

extern "C" int qk_gemv_q6k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q6_K, false, q8_args(w, codes, scales, residual, y), M, N, K, flags, stream);
}

extern "C" int qk_gemv_q5k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q5_K, false, q8_args(w, codes, scales, residual, y), M, N, K, flags, stream);
}

extern "C" int qk_gemv_q5k_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                               const float *residual, float *y, int8_t *codes_out, void *scales_out,
                               unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q5_K, true, f32_args(w, x, ldx, residual, y, codes_out, scales_out), M, N, K, flags,
                stream);
}

extern "C" int qk_gemv_q8_0(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                            int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q8_0, false, q8_args(w, codes, scales, residual, y), M, N, K, flags, stream);
}

extern "C" int qk_gemv_q8_0_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                                const float *residual, float *y, int8_t *codes_out, void *scales_out,
                                unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q8_0, true, f32_args(w, x, ldx, residual, y, codes_out, scales_out), M, N, K, flags,
                stream);
}

extern "C" int qk_gemv_q2k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q2_K, false, q8_args(w, codes, scales, residual, y), M, N, K, flags, stream);
}

extern "C" int qk_gemv_q3k(const void *w, const int8_t *codes, const void *scales, int64_t M, int64_t N,
                           int64_t K, const float *residual, float *y, unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q3_K, false, q8_args(w, codes, scales, residual, y), M, N, K, flags, stream);
}

extern "C" int qk_gemv_q2k_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                               const float *residual, float *y, int8_t *codes_out, void *scales_out,
                               unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q2_K, true, f32_args(w, x, ldx, residual, y, codes_out, scales_out), M, N, K, flags,
                stream);
}

extern "C" int qk_gemv_q3k_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                               const float *residual, float *y, int8_t *codes_out, void *scales_out,
                               unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q3_K, true, f32_args(w, x, ldx, residual, y, codes_out, scales_out), M, N, K, flags,
                stream);
}

extern "C" int qk_gemv_q4k_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                               const float *residual, float *y, int8_t *codes_out, void *scales_out,
                               unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q4_K, true, f32_args(w, x, ldx, residual, y, codes_out, scales_out), M, N, K, flags,
                stream);
}

extern "C" int qk_gemv_q6k_f32(const void *w, const float *x, int64_t ldx, int64_t M, int64_t N, int64_t K,
                               const float *residual, float *y, int8_t *codes_out, void *scales_out,
                               unsigned flags, void *stream)
{
    return gemv(QK_TYPE_Q6_K, true, f32_args(w, x, ldx, residual, y, codes_out, scales_out), M, N, K, flags,
                stream);
}
