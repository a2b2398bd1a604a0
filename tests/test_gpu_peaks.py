"""The tensor-core peak micro-benchmarks (include/qk_peak.h) run and give plausible rates.

Their figures are the denominators of the prefill MMQ's roofline fractions, so they are checked
for completing without a timed-out wait and for landing inside a wide band around the part's
nominal rates (GB300: 2.25 PFLOP/s dense f16 nominal; the legacy int8 mma.sync path far below)."""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q8_activation_gb300 as m
    m.build()
    m.lib()
    return m


def test_peak_tcgen05_f16(qk):
    tflops, ms = qk.peak_tcgen05_f16(iters=2048, reps=3)
    assert math.isfinite(tflops) and ms > 0
    assert 300.0 < tflops < 3000.0, tflops


def test_peak_mma_s8(qk):
    tops, ms = qk.peak_mma_s8(iters=4000, reps=3)
    assert math.isfinite(tops) and ms > 0
    assert 10.0 < tops < 3000.0, tops
