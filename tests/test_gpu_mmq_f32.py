"""GPU: the MMQ entry points that take the f32 activation (qk_mmq_q4k_f32, qk_mmq_q6k_f32).

The q8_1 quantization happens inside the call with the library's block quantizer, so the result
must be bit-identical to qk_quantize_q8_1 followed by the q8_1 entry point on the same inputs
(and the q8_1 path itself is checked against the oracle in test_gpu_parity.py).  Also within the
parity bound of the oracle on the ragged last rows, with strided activation rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

qk = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    global qk
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q8_activation_gb300 as m
    m.build()
    m.lib()
    qk = m
    yield


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K,tile,ldx_pad", [(1, 64, 256, None, 0), (130, 300, 4096, None, 32),
                                                (200, 1000, 768, 128, 0), (333, 4608, 3584, None, 4),
                                                (150, 3584, 1280, 192, 0), (64, 512, 2304, 256, 100)])
def test_mmq_f32_bitexact(qt, M, N, K, tile, ldx_pad):
    if qt == "q6k" and tile == 192:
        pytest.skip("Q6_K tiles are 128 or 256 wide")
    w = synth.weights(qt, N, K, seed=M + K)
    wr = qk.repack(1 if qt == "q4k" else 2, dev(w), N, K)
    xs = synth.activations(M, K + ldx_pad, seed=N) * np.float32(2.5)
    xd = dev(xs)[:, :K]                                   # rows K + ldx_pad apart
    r = dev(synth.residual(M, N, seed=K))
    codes, scales = qk.quantize_q8_1(xd)
    qk.error_flags(clear=True)
    if qt == "q4k":
        y0 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, tile=tile)
        y1 = qk.mmq_q4k_f32(wr, xd, N, K, residual=r, tile=tile)
        plane = qk.q4k_min_plane(wr, N, K)
        y2 = qk.mmq_q4k_f32(wr, xd, N, K, residual=r, tile=tile, plane=plane, pdl=True)
    else:
        y0 = qk.mmq_q6k(wr, codes, scales, N, K, residual=r, tile=tile)
        y1 = qk.mmq_q6k_f32(wr, xd, N, K, residual=r, tile=tile)
        y2 = qk.mmq_q6k_f32(wr, xd, N, K, residual=r, tile=tile, pdl=True)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) == 0
    assert torch.equal(y0, y1) and torch.equal(y0, y2)
    c, d = codes.cpu().numpy(), scales.cpu().numpy()[:, :, 0].view(np.uint16).copy()
    r_np = r.cpu().numpy()
    lo, hi = max(0, N - 9), N
    y_ref, ab = oracle.gemm(oracle.Q4_K if qt == "q4k" else oracle.Q6_K, w, N, K, c, d, residual=r_np,
                            rows=(lo, hi))
    err = np.abs(y1.cpu().numpy()[:, lo:hi].astype(np.float64) - y_ref)
    assert np.all(err <= 1e-4 * ab + 2.0 ** -22 * np.abs(r_np[:, lo:hi]))


def test_mmq_f32_tail_split_and_zero_rows():
    """The default plan's tail split (on 152 SMs) and all-zero / tiny activation blocks."""
    M, N, K = 256, 256 * 112, 48 * 256
    w = synth.weights("q4k", N, K, seed=5)
    wr = qk.repack(1, dev(w), N, K)
    x = synth.activations(M, K, seed=6)
    x[3, :64] = 0.0                                       # all-zero blocks: d = 0
    x[7, 32:64] = np.float32(1e-30)                       # a subnormal scale
    xd = dev(x)
    codes, scales = qk.quantize_q8_1(xd)
    ws = torch.empty(qk.mmq_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    y0 = qk.mmq_q4k(wr, codes, scales, N, K, workspace=ws)
    y1 = qk.mmq_q4k_f32(wr, xd, N, K, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


def test_mmq_f32_range_flag():
    """A block past the Q4_K activation limit (d_a * 127 > 32000) sets QK_ERR_RANGE, as it does
    through the q8_1 entry point."""
    M, N, K = 24, 96, 512
    wr = qk.repack(1, dev(synth.weights("q4k", N, K, seed=31)), N, K)
    x = synth.activations(M, K, seed=32)
    x[5, 64:96] *= np.float32(40000.0 / np.abs(x[5, 64:96]).max())
    qk.error_flags(clear=True)
    qk.mmq_q4k_f32(wr, dev(x), N, K)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) & qk.ERR_RANGE
