"""GPU parity of the fused producers (RMSNorm -> q8_1, SwiGLU -> q8_1) through the C ABI.

Bars:
  - the q8_1 codes and scales are bit for bit those the oracle's quantizer gives for the
    binary32 output the kernel computed (the integer decision is taken on the same binary32
    values on both sides);
  - that binary32 output is within the rounding bound of its binary32 arithmetic of the
    oracle's binary64 value: RMSNorm (K/2 + 8) * 2^-24 relative (square sum of K terms,
    halved by the square root, plus the division, root and two products), SwiGLU
    8 * 2^-24 relative (expf within 2 ulp, then an add, a division and a product) plus
    2^-126 absolute where the exponential overflows;
  - the residual stream x + r is the exact binary32 sum;
  - reruns give the same bits.
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


def check_q8(codes, scales, y_gpu):
    c, d, s = oracle.quantize_q8_1(y_gpu)
    sc = scales.cpu().numpy().view(np.uint16)
    assert np.array_equal(codes.cpu().numpy(), c)
    assert np.array_equal(sc[:, :, 0], d) and np.array_equal(sc[:, :, 1], s)


@pytest.mark.parametrize("M,K", [(1, 32), (1, 4096), (3, 3584), (4, 1056), (2, 8192), (1, 14336), (17, 256)])
@pytest.mark.parametrize("with_r", [False, True])
def test_rmsnorm_q8_1(M, K, with_r):
    rng = np.random.default_rng(M * 7 + K)
    x = synth.activations(M, K, seed=K, tag="norm_x") * np.float32(3)
    r = synth.residual(M, K, seed=K, tag="norm_r") if with_r else None
    g = (rng.standard_normal(K) * 0.5 + 1).astype(np.float32)
    eps = 1e-5
    y_ref, s_ref = oracle.rmsnorm(x, g, eps, r=r)
    y = torch.empty((M, K), dtype=torch.float32, device="cuda")
    h = torch.empty((M, K), dtype=torch.float32, device="cuda") if with_r else None
    codes, scales = qk.rmsnorm_q8_1(dev(x), dev(g), eps, r=None if r is None else dev(r), h_out=h, y=y)
    y_gpu = y.cpu().numpy()
    tol = (K / 2 + 8) * 2.0 ** -24 * np.abs(y_ref) + 2.0 ** -126
    assert np.all(np.abs(y_gpu.astype(np.float64) - y_ref) <= tol)
    check_q8(codes, scales, y_gpu)
    if with_r:
        assert np.array_equal(h.cpu().numpy(), s_ref)
    # without the dense output: the same codes; reruns: the same bits
    c2, s2 = qk.rmsnorm_q8_1(dev(x), dev(g), eps, r=None if r is None else dev(r), pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(c2, codes) and torch.equal(s2, scales)


def test_rmsnorm_strided_rows_and_scale():
    M, K, ldx = 5, 2048, 2304
    xs = synth.activations(M, ldx, seed=9, tag="norm_strided") * np.float32(1e3)
    g = np.full(K, 0.25, np.float32)
    xt = dev(xs)[:, :K]
    y = torch.empty((M, K), dtype=torch.float32, device="cuda")
    codes, scales = qk.rmsnorm_q8_1(xt, dev(g), 1e-6, y=y)
    y_ref, _ = oracle.rmsnorm(np.ascontiguousarray(xs[:, :K]), g, 1e-6)
    y_gpu = y.cpu().numpy()
    assert np.all(np.abs(y_gpu - y_ref) <= (K / 2 + 8) * 2.0 ** -24 * np.abs(y_ref) + 2.0 ** -126)
    check_q8(codes, scales, y_gpu)


@pytest.mark.parametrize("M,F", [(1, 32), (1, 14336), (4, 4096), (5, 1056), (2, 18944)])
def test_swiglu_q8_1(M, F):
    gu = synth.activations(M, 2 * F, seed=F, tag="gateup") * np.float32(2)
    h_ref = oracle.swiglu(gu, F)
    h = torch.empty((M, F), dtype=torch.float32, device="cuda")
    codes, scales = qk.swiglu_q8_1(dev(gu), F, h=h)
    h_gpu = h.cpu().numpy()
    assert np.all(np.abs(h_gpu.astype(np.float64) - h_ref) <= 8 * 2.0 ** -24 * np.abs(h_ref) + 2.0 ** -126)
    check_q8(codes, scales, h_gpu)
    c2, s2 = qk.swiglu_q8_1(dev(gu), F, pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(c2, codes) and torch.equal(s2, scales)


def test_swiglu_padded_rows_and_extreme_gates():
    M, F, ld = 3, 256, 640
    gu = synth.activations(M, ld, seed=5, tag="gateup_pad")
    gu[0, :8] = [100.0, -100.0, 88.0, -88.0, 30.0, -30.0, 0.0, 1e-30]
    h_ref = oracle.swiglu(gu, F)
    h = torch.empty((M, F), dtype=torch.float32, device="cuda")
    codes, scales = qk.swiglu_q8_1(dev(gu), F, h=h)
    h_gpu = h.cpu().numpy()
    assert np.all(np.abs(h_gpu.astype(np.float64) - h_ref) <= 8 * 2.0 ** -24 * np.abs(h_ref) + 2.0 ** -126)
    check_q8(codes, scales, h_gpu)


def test_producer_feeds_gemv():
    """RMSNorm -> q8_1 -> Q4_K GEMV -> SwiGLU -> q8_1 -> Q4_K GEMV, chained with PDL on one stream,
    against the oracle run on the same intermediate values."""
    K, F = 1024, 512
    x = synth.activations(1, K, seed=1, tag="chain_x")
    g = np.ones(K, np.float32)
    w1 = synth.weights("q4k", 2 * F, K, seed=2, tag="chain_w1")
    w2 = synth.weights("q4k", K, F, seed=3, tag="chain_w2")
    w1r = qk.repack(qk.Q4_K, dev(w1), 2 * F, K)
    w2r = qk.repack(qk.Q4_K, dev(w2), K, F)
    s = torch.cuda.Stream()
    y = torch.empty((1, K), dtype=torch.float32, device="cuda")
    h = torch.empty((1, F), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        c1, s1 = qk.rmsnorm_q8_1(dev(x), dev(g), 1e-5, y=y, pdl=True, stream=s)
        gu = qk.gemv_q4k(w1r, c1, s1, 2 * F, K, pdl=True, stream=s)
        c2, s2 = qk.swiglu_q8_1(gu, F, h=h, pdl=True, stream=s)
        out = qk.gemv_q4k(w2r, c2, s2, K, F, pdl=True, stream=s)
    torch.cuda.synchronize()
    # each stage against the oracle applied to the previous stage's device output
    q1 = oracle.quantize_q8_1(y.cpu().numpy())
    gu_ref, ab1 = oracle.gemm(oracle.Q4_K, w1, 2 * F, K, q1[0], q1[1])
    assert np.all(np.abs(gu.cpu().numpy().astype(np.float64) - gu_ref) <= 1e-4 * ab1)
    check_q8(c2, s2, h.cpu().numpy())
    q2 = oracle.quantize_q8_1(h.cpu().numpy())
    out_ref, ab2 = oracle.gemm(oracle.Q4_K, w2, K, F, q2[0], q2[1])
    assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - out_ref) <= 1e-4 * ab2)
