// qk_common.cuh -- helpers shared by the library's translation units:
// host-side argument checks, the launch wrapper (optional programmatic
// dependent launch), and small device primitives written as inline PTX.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qk.h"

namespace qk {

// ----------------------------------------------------------------- host side

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [a, a+na) and [b, b+nb) overlap (byte ranges; empty ranges never overlap)
inline bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? QK_OK : QK_E_CUDA; }

// Launch `kern` on `stream`; with pdl the launch carries the programmatic
// stream serialization attribute so the kernel may begin before the
// previous kernel on the stream has finished (it must call pdl_wait()
// before touching anything that kernel could have produced).
template <typename... KArgs, typename... Args>
inline int launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                  bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    return cuda_status(e);
}

// Number of SMs of the current device (queried once per device id).
int sm_count();

// Devices the per-device caches of the library cover (ids 0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

// Id of the host thread's current CUDA device, or -1 if it cannot be read or is
// past kMaxDevices.  Every one-time set-up (kernel attributes, symbol addresses)
// is cached per device id, since each device holds its own copy of the module.
inline int device_slot()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Largest dynamic shared memory a CTA may opt in to on the current device.
size_t max_smem_optin();

// MMQ workspace bytes without the split-K scratch (enough for an unsplit call).
size_t mmq_base_workspace_bytes(int64_t M, int64_t K);

// Every kernel of the library asks for the same (maximal) shared-memory
// carveout, so consecutive kernels never force an L1/shared reconfiguration.
template <typename Kern>
inline cudaError_t max_carveout(Kern kern)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

// ---------------------------------------------------------------- device side

// Wait until the previous grid on the stream has completed and its memory
// is visible (no-op for a launch without the PDL attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid on the stream to start launching.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte read-only streaming load (weights: read once, never written by a
// running kernel).
__device__ __forceinline__ uint4 ldg_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream4(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ldg_stream2(const void *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// dot of four unsigned bytes of a with four signed bytes of b, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// dot of four signed bytes, plus c
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 16-byte asynchronous global -> shared copy (L2 only); `bytes` < 16 zero-fills the rest
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, int bytes = 16)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gsrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// binary32 -> binary16, round to nearest even, saturating at +-65504
__device__ __forceinline__ __half f16_sat(float v) { return __float2half_rn(fminf(fmaxf(v, -65504.0f), 65504.0f)); }

// request the 128-byte line holding p into L2 (no L1 allocation, no register result)
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// RN(a / 127) for every binary32 a >= 0 (zero, subnormal and normal): the
// quotient q0 = RN(a * y) with y = RN(1/127) is corrected once with the exact
// remainder r = a - 127 q0 (one fma), q = RN(q0 + r y) -- division by a
// divisor known in advance (Markstein; Brisebarre, Muller and Raina,
// "Accelerating correctly rounded floating-point division when the divisor
// is known in advance", IEEE TC 2004).  For this divisor the sequence was
// checked against IEEE division on all 2^31 non-negative finite inputs.
__device__ __forceinline__ float div127_rn(float a)
{
    const float y = 0x1.020408p-7f;                         // RN(1/127)
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q0, 127.0f, a);
    return __fmaf_rn(r, y, q0);
}

// approximate reciprocal (PTX rcp.approx.f32: at most 1 ulp of error over the
// whole range, subnormal inputs included)
__device__ __forceinline__ float rcp_approx(float v)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// q8_1 quantization of one 32-value block held by 8 consecutive lanes (lane
// group 8j..8j+7 of the warp, 4 values each, all 32 lanes participating):
// d = amax/127 (binary32 division), q = roundf(x/d) (0 when d == 0).  Returns
// this lane's 4 codes packed little-endian; d is the block's binary32 scale and
// s4 the sum of this lane's 4 codes.  Used by the standalone quantizer and by
// the GEMV kernels that quantize their activation themselves, so both produce
// the same codes bit for bit.
//
// roundf(x/d) is taken from t = x * r with r = 1/d to within 1 ulp: |x/d| is at
// most 127 (1 + 2^-24), so t differs from x/d by at most 1.5 * 2^-23 * 127.01
// < 2.28e-5, and RN(x/d) from x/d by at most 7.6e-6.  Unless t lies within
// 2^-15 = 3.05e-5 of a half-integer, x/d and RN(x/d) are on t's side of it, and
// round-to-nearest-even of t (no tie there) equals roundf(RN(x/d)).  Near a
// half-integer, or when 1/d is not finite, the code is taken from the IEEE
// quotient instead; that path is entered warp-uniformly and only when some
// lane needs it, so the common case has no branches.
__device__ __forceinline__ uint32_t q81_quant8(float4 v, float &d, int &s4)
{
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    d = div127_rn(amax);
    const bool live = d > 0.0f;
    const float r = rcp_approx(d);
    const float x[4] = {v.x, v.y, v.z, v.w};
    int q[4];
    bool near = false;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const float t = __fmul_rn(x[j], r);
        const float tr = rintf(t);
        near |= !(fabsf(t - tr) < 0.5f - 3.0517578125e-05f);     // also true for a non-finite t
        q[j] = __float2int_rz(tr);                                 // tr is an integer (or not finite)
    }
    near = near && live;
    if (__any_sync(0xffffffffu, near)) {
        if (near) {
#pragma unroll
            for (int j = 0; j < 4; j++) q[j] = (int)roundf(__fdiv_rn(x[j], d));
        }
    }
    if (!live) q[0] = q[1] = q[2] = q[3] = 0;
    s4 = q[0] + q[1] + q[2] + q[3];
    return (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) | ((uint32_t)(q[2] & 0xff) << 16) |
           ((uint32_t)(q[3] & 0xff) << 24);
}

// stored binary16 s of a q8_1 block: s = d * sum(q) in binary32, then binary16
__device__ __forceinline__ __half q81_sum_f16(float d, int sum) { return f16_sat(__fmul_rn(d, (float)sum)); }

}  // namespace qk
