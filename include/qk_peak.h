/*
 * qk_peak.h -- measurement entry points of libqk.so: the tensor-core peaks
 * that the prefill MMQ's roofline fractions are divided by.
 *
 * The method's prefill contraction is an int8 x int8 -> int32 product (minfer
 * "15 . The CUDA backend" sec. 2.3: int8 MMA over q8_1 activations).  On
 * sm_103a the int8 tensor path exists only as the warp-level mma.sync
 * (tcgen05 has no int8 kind there), and the library's MMQ instead runs exact
 * f16 operands through tcgen05.mma kind::f16.  These two calls measure both
 * rates on the device they run on, with the same instruction shapes the
 * comparison needs:
 *   qk_peak_mma_s8        mma.sync.m16n8k32 s8 x s8 -> s32, register
 *                         operands, 8 independent accumulators per warp,
 *                         16 warps per SM: int8 ops/s (2 ops per MAC).
 *   qk_peak_tcgen05_f16   tcgen05.mma.cta_group::1.kind::f16, 128 x 256 x 16
 *                         per instruction, f16 operands in shared memory,
 *                         f32 accumulator in tensor memory, one CTA per SM
 *                         issuing back to back: f16 flop/s (2 per MAC).
 * Neither reads or writes global memory in its loop; operand values are
 * zeros (the rate does not depend on them).
 *
 * Both calls are synchronous: they launch one untimed warm-up, then `reps`
 * launches of `iters` instructions per issuing warp between two CUDA events
 * recorded on `stream`, wait for them, and return the achieved rate in
 * units of 10^12 per second in *rate (TOPS / TFLOP/s) and the measured
 * milliseconds in *ms.  iters >= 1, 1 <= reps <= 1000.
 * Returns QK_E_NULL for a NULL output, QK_E_SHAPE for iters/reps out of
 * range, QK_E_CUDA if a CUDA call fails or a bounded in-kernel wait gave up.
 * Not part of the method: they exist so that measurements can be reproduced.
 */
#ifndef QK_PEAK_H
#define QK_PEAK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int qk_peak_mma_s8(int64_t iters, int reps, double *rate, double *ms, void *stream);

int qk_peak_tcgen05_f16(int64_t iters, int reps, double *rate, double *ms, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QK_PEAK_H */
