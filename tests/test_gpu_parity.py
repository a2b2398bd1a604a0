"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars (set by the method's definition):
  - q8_1 codes and binary16 scales: bit for bit.
  - device weight layout: byte for byte against the oracle's statement of it.
  - GEMV / MMQ outputs: |y_gpu - y_ref| <= 1e-4 * sum_k |w * xhat| per
    output, plus 2^-22 * |r| for the binary32 residual add.
Shapes span several tiles and ragged tails (rows, superblock steps, M).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

qk = None
QT = {"q4k": (1, oracle.Q4_K), "q6k": (2, oracle.Q6_K), "q5k": (3, oracle.Q5_K), "q80": (4, oracle.Q8_0),
      "q2k": (5, oracle.Q2_K), "q3k": (6, oracle.Q3_K)}


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


def weights(qt, N, K, seed):
    w = synth.weights(qt, N, K, seed=seed)
    return w, qk.repack(QT[qt][0], dev(w), N, K)


def q8(x_np):
    codes, scales = qk.quantize_q8_1(dev(x_np))
    return codes, scales


def q8_host(codes, scales):
    c = codes.cpu().numpy()
    d = scales.cpu().numpy()[:, :, 0].view(np.uint16).copy()
    return c, d


def check(y_gpu, y_ref, ab, r=None, what=""):
    y_gpu = np.asarray(y_gpu, np.float64)
    tol = 1e-4 * ab
    if r is not None:
        tol = tol + 2.0 ** -22 * np.abs(np.asarray(r, np.float64))
    err = np.abs(y_gpu - y_ref)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} outputs out of bound; worst err/tol " \
                          f"{np.max(err / np.maximum(tol, 1e-300)):.3g}"


# ---------------------------------------------------------------------- q8_1

@pytest.mark.parametrize("M,K", [(1, 256), (1, 4096), (3, 4096), (2, 14336), (4, 3584), (7, 32 * 13)])
def test_quantize_bitexact(M, K):
    x = synth.activations(M, K, seed=M + K) * np.float32(3.0)
    x[0, :32] = 0.0                                  # an all-zero block
    x[-1, 32:64] = np.float32(1e-30)                 # tiny values (subnormal scale)
    if K >= 128:
        x[0, 64:96] = np.float32(7.25)               # constant block
    codes, scales = q8(x)
    c_ref, d_ref, s_ref = oracle.quantize_q8_1(x)
    c, sc = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    assert np.array_equal(c, c_ref)
    assert np.array_equal(sc[:, :, 0], d_ref)
    assert np.array_equal(sc[:, :, 1], s_ref)


def test_quantize_golden_ties_and_strided_rows():
    x = np.zeros((2, 64), np.float32)
    x[0, :8] = [127.0, -63.5, 0.5, -0.5, 1.5, 2.5, -2.5, 63.49]
    x[1, :] = 0.3
    big = np.zeros((2, 96), np.float32)
    big[:, :64] = x                                   # rows with stride 96
    xt = dev(big)[:, :64]
    codes, scales = qk.quantize_q8_1(xt)
    c_ref, d_ref, s_ref = oracle.quantize_q8_1(x)
    assert codes.cpu().numpy()[0, :8].tolist() == [127, -64, 1, -1, 2, 3, -3, 63]
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    sc = scales.cpu().numpy().view(np.uint16)
    assert np.array_equal(sc[:, :, 0], d_ref) and np.array_equal(sc[:, :, 1], s_ref)
    assert int(sc[1, 0, 0]) == 0x18D6 and int(sc[1, 0, 1]) == 0x48CD


def test_quantize_saturates_large_blocks():
    x = np.full((1, 32), 1.0e7, np.float32)
    codes, scales = q8(x)
    c_ref, d_ref, s_ref = oracle.quantize_q8_1(x)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    sc = scales.cpu().numpy().view(np.uint16)
    assert int(sc[0, 0, 0]) == int(d_ref[0, 0]) == 0x7BFF
    assert int(sc[0, 0, 1]) == int(s_ref[0, 0]) == 0x7BFF


# -------------------------------------------------------------------- repack

@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
@pytest.mark.parametrize("N,K", [(1, 256), (3, 2304), (5, 4096), (2, 256 * 17), (9, 256 * 8)])
def test_repack_bitexact(qt, N, K):
    w, wr = weights(qt, N, K, seed=N * 7 + K)
    assert np.array_equal(wr.cpu().numpy(), oracle.repack(QT[qt][1], w, N, K))


# ---------------------------------------------------------------------- GEMV

def gemv(qt, *a, **kw):
    return {"q4k": qk.gemv_q4k, "q5k": qk.gemv_q5k, "q6k": qk.gemv_q6k, "q80": qk.gemv_q8_0,
            "q2k": qk.gemv_q2k, "q3k": qk.gemv_q3k}[qt](*a, **kw)


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 256), (37, 2304), (300, 4096), (130, 256 * 11)])
def test_gemv_parity(qt, M, N, K):
    w, wr = weights(qt, N, K, seed=M + N + K)
    x = synth.activations(M, K, seed=N)
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    y = gemv(qt, wr, codes, scales, N, K).cpu().numpy()
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what=f"{qt} M={M} N={N} K={K}")


# Row counts that leave a partial last round of row pairs on the persistent grid
# (152 SMs x 16 warps: a pair per warp per round), with 2 to 16 superblock steps
# per pair and a ragged last pair.  Every output row is checked.
@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
@pytest.mark.parametrize("K,frac", [(4096, 8), (8192, 8), (32768, 10), (32768, 20)])
@pytest.mark.parametrize("front", ["q8", "f32"])
def test_gemv_partial_last_round(qt, K, frac, front):
    W = torch.cuda.get_device_properties(0).multi_processor_count * 16
    N = 2 * (W + W // frac) - 1
    M = 1 if K > 8192 else 3
    w, wr = weights(qt, N, K, seed=N + K)
    x = synth.activations(M, K, seed=K + 7)
    if front == "q8":
        codes, scales = q8(x)
        c, d = q8_host(codes, scales)
        y = gemv(qt, wr, codes, scales, N, K).cpu().numpy()
    else:
        codes, scales = qk.empty_q8_1(M, K)
        y = gemv_f32(qt, wr, dev(x), N, K, codes_out=codes, scales_out=scales).cpu().numpy()
        c, d = q8_host(codes, scales)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what=f"{qt} {front} M={M} N={N} K={K}")


# Items of four weight rows (Q4_K / Q6_K, M >= 3), forced at small shapes: a ragged last
# group (N not a multiple of 4), one to eleven superblocks per row, both front ends, with a
# residual added in place.  The same call with two-row items forced must also be within the
# bound, and each choice must give the same bits on a second run.
@pytest.mark.parametrize("qt", ["q4k", "q6k"])
@pytest.mark.parametrize("M", [3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 256), (7, 2304), (301, 4096), (130, 256 * 11)])
@pytest.mark.parametrize("front", ["q8", "f32"])
def test_gemv_rows4_parity(qt, M, N, K, front):
    if M * K > {"q4k": 81920, "q6k": 40960}[qt]:
        pytest.skip("activation larger than the GEMV's staging limit")
    w, wr = weights(qt, N, K, seed=3 * M + N + K)
    x = synth.activations(M, K, seed=N + 5)
    r = synth.residual(M, N, seed=M + 9)
    outs = {}
    for rows in (4, 2, 4):
        rt = dev(r)
        if front == "q8":
            codes, scales = q8(x)
            y = gemv(qt, wr, codes, scales, N, K, residual=rt, y=rt, rows=rows)
        else:
            codes, scales = qk.empty_q8_1(M, K)
            f = qk.gemv_q4k_f32 if qt == "q4k" else qk.gemv_q6k_f32
            y = f(wr, dev(x), N, K, residual=rt, y=rt, codes_out=codes, scales_out=scales, rows=rows)
        c, d = q8_host(codes, scales)
        y = y.cpu().numpy()
        if rows in outs:
            assert np.array_equal(outs[rows], y), f"{qt} rows={rows}: second run differs"
        else:
            y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d, residual=r)
            check(y, y_ref, ab, r, what=f"{qt} {front} rows={rows} M={M} N={N} K={K}")
            outs[rows] = y


# The default choice takes four-row items once the groups of four fill every warp: a shape
# just past that point, with a partial last round and a ragged last group, every row checked.
@pytest.mark.parametrize("qt", ["q4k", "q6k"])
@pytest.mark.parametrize("front", ["q8", "f32"])
def test_gemv_rows4_default_partial_round(qt, front):
    W4 = torch.cuda.get_device_properties(0).multi_processor_count * 12
    N = 4 * (W4 + W4 // 8) - 3
    M, K = 4, 4096
    w, wr = weights(qt, N, K, seed=N + 1)
    x = synth.activations(M, K, seed=N + 2)
    if front == "q8":
        codes, scales = q8(x)
        y = gemv(qt, wr, codes, scales, N, K).cpu().numpy()
    else:
        codes, scales = qk.empty_q8_1(M, K)
        f = qk.gemv_q4k_f32 if qt == "q4k" else qk.gemv_q6k_f32
        y = f(wr, dev(x), N, K, codes_out=codes, scales_out=scales).cpu().numpy()
    c, d = q8_host(codes, scales)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what=f"{qt} {front} default rows M={M} N={N}")


def test_gemv_rows_flags_exclusive():
    M, N, K = 4, 64, 256
    w, wr = weights("q4k", N, K, seed=1)
    codes, scales = q8(synth.activations(M, K, seed=2))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = qk.lib().qk_gemv_q4k(wr.data_ptr(), codes.data_ptr(), scales.data_ptr(), M, N, K, None, y.data_ptr(),
                              qk.GEMV_ROWS4 | qk.GEMV_ROWS2, None)
    assert qk.STATUS[st] == "QK_E_SHAPE"


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
@pytest.mark.parametrize("mode", ["separate", "inplace", "pdl"])
def test_gemv_residual(qt, mode):
    M, N, K = 4, 515, 4096
    w, wr = weights(qt, N, K, seed=11)
    x = synth.activations(M, K, seed=12)
    r = synth.residual(M, N, seed=13)
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    rt = dev(r)
    if mode == "inplace":
        y = gemv(qt, wr, codes, scales, N, K, residual=rt, y=rt)
    else:
        y = gemv(qt, wr, codes, scales, N, K, residual=rt, pdl=(mode == "pdl"))
    torch.cuda.synchronize()
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d, residual=r)
    check(y.cpu().numpy(), y_ref, ab, r, what=f"{qt} residual {mode}")


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
def test_gemv_edges(qt):
    # zero activation gives the residual exactly; one-hot activation gives a scaled column
    N, K = 33, 512
    w, wr = weights(qt, N, K, seed=21)
    r = synth.residual(1, N, seed=22)
    codes, scales = q8(np.zeros((1, K), np.float32))
    y = gemv(qt, wr, codes, scales, N, K, residual=dev(r)).cpu().numpy()
    assert np.array_equal(y, r)
    x = np.zeros((1, K), np.float32)
    x[0, 300] = 2.0
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    y = gemv(qt, wr, codes, scales, N, K).cpu().numpy()
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what="one-hot")


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
def test_gemv_max_activation(qt):
    M, N = 8, 40
    K = {"q4k": 10240, "q5k": 8192, "q6k": 5120, "q80": 8192, "q2k": 10240, "q3k": 10240}[qt]   # at the limit
    w, wr = weights(qt, N, K, seed=31)
    x = synth.activations(M, K, seed=32)
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    y = gemv(qt, wr, codes, scales, N, K).cpu().numpy()
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what="max M*K")


# Q6_K with M <= 2 runs 20 warps per CTA where the ring and the activation fit in shared memory and
# 16 beyond (M*K over about 21.8K values): both sides of the choice, a partial last round of row
# pairs for 20 warps, both front ends, every row checked.
@pytest.mark.parametrize("M,K", [(1, 4096), (2, 8192), (1, 20480), (1, 40960), (2, 20480)])
@pytest.mark.parametrize("front", ["q8", "f32"])
def test_gemv_q6k_small_m_warp_choice(M, K, front):
    W = torch.cuda.get_device_properties(0).multi_processor_count * 20
    N = 2 * (W + W // 9) - 1 if K <= 8192 else 301
    w, wr = weights("q6k", N, K, seed=N + K + M)
    x = synth.activations(M, K, seed=K + 11)
    r = synth.residual(M, N, seed=M + 12)
    if front == "q8":
        codes, scales = q8(x)
        y = qk.gemv_q6k(wr, codes, scales, N, K, residual=dev(r)).cpu().numpy()
    else:
        codes, scales = qk.empty_q8_1(M, K)
        y = qk.gemv_q6k_f32(wr, dev(x), N, K, residual=dev(r), codes_out=codes, scales_out=scales).cpu().numpy()
    c, d = q8_host(codes, scales)
    y_ref, ab = oracle.gemm(oracle.Q6_K, w, N, K, c, d, residual=r)
    check(y, y_ref, ab, r, what=f"q6k {front} M={M} N={N} K={K}")


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
def test_gemv_deterministic_and_guard_band(qt):
    M, N, K = 3, 1000, 4096
    w, wr = weights(qt, N, K, seed=41)
    codes, scales = q8(synth.activations(M, K, seed=42))
    guard = torch.full((M * N + 1024,), 1234.5, dtype=torch.float32, device="cuda")
    y1 = guard[:M * N].view(M, N)
    gemv(qt, wr, codes, scales, N, K, y=y1)
    y2 = gemv(qt, wr, codes, scales, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.all(guard[M * N:] == 1234.5)


# ----------------------------------------------- GEMV, in-kernel quantization

def gemv_f32(qt, *a, **kw):
    return {"q4k": qk.gemv_q4k_f32, "q5k": qk.gemv_q5k_f32, "q6k": qk.gemv_q6k_f32,
            "q80": qk.gemv_q8_0_f32, "q2k": qk.gemv_q2k_f32, "q3k": qk.gemv_q3k_f32}[qt](*a, **kw)


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("N,K", [(1, 256), (37, 2304), (300, 4096), (130, 256 * 11)])
def test_gemv_f32_parity_and_codes(qt, M, N, K):
    w, wr = weights(qt, N, K, seed=M + 2 * N + K)
    x = synth.activations(M, K, seed=N + 1) * np.float32(2.0)
    x[0, :32] = 0.0
    codes, scales = qk.empty_q8_1(M, K)
    y = gemv_f32(qt, wr, dev(x), N, K, codes_out=codes, scales_out=scales).cpu().numpy()
    c_ref, d_ref, s_ref = oracle.quantize_q8_1(x)
    sc = scales.cpu().numpy().view(np.uint16)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(sc[:, :, 0], d_ref) and np.array_equal(sc[:, :, 1], s_ref)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c_ref, d_ref)
    check(y, y_ref, ab, what=f"{qt} f32 M={M} N={N} K={K}")


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
@pytest.mark.parametrize("mode", ["separate", "inplace", "pdl", "strided"])
def test_gemv_f32_residual(qt, mode):
    M, N, K = 2, 515, 4096
    w, wr = weights(qt, N, K, seed=61)
    x = synth.activations(M, K, seed=62)
    r = synth.residual(M, N, seed=63)
    rt = dev(r)
    if mode == "strided":
        big = np.zeros((M, K + 64), np.float32)
        big[:, :K] = x
        xt = dev(big)[:, :K]
    else:
        xt = dev(x)
    if mode == "inplace":
        y = gemv_f32(qt, wr, xt, N, K, residual=rt, y=rt)
    else:
        y = gemv_f32(qt, wr, xt, N, K, residual=rt, pdl=(mode == "pdl"))
    torch.cuda.synchronize()
    c_ref, d_ref, _ = oracle.quantize_q8_1(x)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c_ref, d_ref, residual=r)
    check(y.cpu().numpy(), y_ref, ab, r, what=f"{qt} f32 residual {mode}")


@pytest.mark.parametrize("qt", ["q4k", "q5k", "q6k", "q80", "q2k", "q3k"])
def test_gemv_f32_matches_q8_path_bitwise(qt):
    # same codes, same kernel body: the two front ends give identical outputs
    M, N, K = 2, 700, 4096
    w, wr = weights(qt, N, K, seed=71)
    x = dev(synth.activations(M, K, seed=72))
    codes, scales = qk.quantize_q8_1(x)
    y1 = gemv(qt, wr, codes, scales, N, K)
    y2 = gemv_f32(qt, wr, x, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


# ----------------------------------------------------------------------- MMQ

def mmq_fn(qt):
    return qk.mmq_q4k if qt == "q4k" else qk.mmq_q6k


@pytest.mark.parametrize("tile", [None, 256, 192, 128])
@pytest.mark.parametrize("qt", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", [(1, 64, 256), (17, 130, 512), (64, 128, 2304), (130, 300, 4096),
                                   (200, 77, 768), (65, 129, 256 * 9), (140, 450, 1024)])
def test_mmq_parity(qt, M, N, K, tile):
    if qt == "q6k" and tile == 192:
        pytest.skip("Q6_K tiles are 128 or 256 wide")
    w, wr = weights(qt, N, K, seed=M * 3 + N + K)
    x = synth.activations(M, K, seed=M)
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    y = mmq_fn(qt)(wr, codes, scales, N, K, tile=tile).cpu().numpy()
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what=f"mmq {qt} M={M} N={N} K={K} tile={tile}")


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_mmq_tile_widths_agree_and_many_tiles_per_cta(qt):
    """More tiles than SMs at both widths (each CTA walks several tiles and both accumulators);
    the two widths agree to the bound."""
    M, N, K = 300, 128 * 160, 256
    w, wr = weights(qt, N, K, seed=77)
    x = synth.activations(M, K, seed=78)
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    rows = (N - 700, N)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d, rows=rows)
    for tile in (256, 192, 128) if qt == "q4k" else (256, 128):
        y = mmq_fn(qt)(wr, codes, scales, N, K, tile=tile).cpu().numpy()
        check(y[:, rows[0]:rows[1]], y_ref, ab, what=f"mmq {qt} tile={tile}")


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_mmq_residual_inplace_deterministic(qt):
    M, N, K = 96, 200, 1024
    w, wr = weights(qt, N, K, seed=51)
    codes, scales = q8(synth.activations(M, K, seed=52))
    c, d = q8_host(codes, scales)
    r = synth.residual(M, N, seed=53)
    rt = dev(r)
    y = mmq_fn(qt)(wr, codes, scales, N, K, residual=rt, y=rt)
    y2 = mmq_fn(qt)(wr, codes, scales, N, K, residual=dev(r), pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d, residual=r)
    check(y.cpu().numpy(), y_ref, ab, r, what=f"mmq {qt} residual")


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
@pytest.mark.parametrize("scale", [1e-3, 30.0, 1000.0])
def test_mmq_activation_magnitudes(qt, scale):
    """Small and large activations (the min-term operands are rescaled by powers of two)."""
    M, N, K = 40, 96, 1024
    w, wr = weights(qt, N, K, seed=61)
    x = synth.activations(M, K, seed=62) * np.float32(scale)
    codes, scales = q8(x)
    c, d = q8_host(codes, scales)
    y = mmq_fn(qt)(wr, codes, scales, N, K).cpu().numpy()
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    check(y, y_ref, ab, what=f"mmq {qt} scale={scale}")


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_mmq_edges_and_error_flags(qt):
    """One row, one column, a ragged 129 x 257 tile grid; no bounded wait gives up."""
    qk.error_flags(clear=True)
    for M, N, K in [(1, 1, 256), (129, 257, 512), (128, 128, 256)]:
        w, wr = weights(qt, N, K, seed=M + N)
        codes, scales = q8(synth.activations(M, K, seed=N))
        c, d = q8_host(codes, scales)
        y = mmq_fn(qt)(wr, codes, scales, N, K).cpu().numpy()
        y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
        check(y, y_ref, ab, what=f"mmq {qt} edge M={M} N={N} K={K}")
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) == 0


def special_scale_weights(qt, N, K, seed):
    """synth weights with per-row cases of the superblock scales edited in the GGUF bytes:
    row n % 5 == 0: d = 0 in every other superblock (Q4_K: only the min term is left there);
    1: dmin = 0 everywhere (Q4_K); 2: a large scale in superblock 1 (Q4_K: dmin = 0.98, so
    dmin * m reaches 61.7, just inside the operand limit of 63; Q6_K: d = 0.2, |w| up to 205);
    3: every scale zero (the row is exactly 0); 4: unchanged."""
    w = synth.weights(qt, N, K, seed=seed).copy()
    blocks = w.reshape(N, K // 256, oracle.BLOCK_BYTES[QT[qt][1]])
    doff = 0 if qt == "q4k" else 208                   # GGUF offset of the f16 d

    def f16(v):
        return np.frombuffer(np.float16(v).tobytes(), np.uint8)

    for n in range(N):
        kind = n % 5
        if kind == 0:
            blocks[n, ::2, doff:doff + 2] = 0
        elif kind == 1 and qt == "q4k":
            blocks[n, :, 2:4] = 0
        elif kind == 2:
            if qt == "q4k":
                blocks[n, 1, 2:4] = f16(0.98)
            else:
                blocks[n, 1, doff:doff + 2] = f16(0.2)
        elif kind == 3:
            blocks[n, :, doff:doff + 2] = 0
            if qt == "q4k":
                blocks[n, :, 2:4] = 0
    return w


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_mmq_superblock_scale_special_cases(qt):
    """Zero superblock scales (the per-superblock fold multiplies by 0, the min term stands
    alone), zero mins, scales at the operand limits, all-zero rows (exactly 0); an odd number
    of superblocks (the last min stage's second half is empty) and ragged tiles."""
    M, N, K = 130, 300, 256 * 7
    w = special_scale_weights(qt, N, K, seed=91)
    wr = qk.repack(QT[qt][0], dev(w), N, K)
    codes, scales = q8(synth.activations(M, K, seed=93))
    c, d = q8_host(codes, scales)
    y_ref, ab = oracle.gemm(QT[qt][1], w, N, K, c, d)
    qk.error_flags(clear=True)
    for tile in (256, 128):
        y = mmq_fn(qt)(wr, codes, scales, N, K, tile=tile).cpu().numpy()
        check(y, y_ref, ab, what=f"mmq {qt} special scales tile={tile}")
        assert np.all(y[:, 3::5] == 0)
    assert qk.error_flags(clear=True) == 0            # inside the value limits: no range flag


@pytest.mark.parametrize("M,N", [(256, 256 * 112), (200, 256 * 112 - 40)])
def test_mmq_q4k_split_k_tail(M, N):
    """224 tiles of 128 x 256 with 48 superblocks of K, QK_MMQ_SPLIT_K: with the split
    scratch in the workspace the Q4_K MMQ splits each tile's K range over two work units (the second
    to finish adds the partial tiles).
    Checked against the oracle on sampled rows, against the same call run unsplit (a base-size
    workspace), for reproducibility, and for the tile counters being left at zero."""
    K = 48 * 256
    w, wr = weights("q4k", N, K, seed=41)
    codes, scales = q8(synth.activations(M, K, seed=42))
    c, d = q8_host(codes, scales)
    r = dev(synth.residual(M, N, seed=43))
    base = 2 * (K * 512 + (K // 512) * 8192)              # two M-tiles: A blocks and sums tiles
    full = base + 224 * 2 * 128 * 256 * 4 + 224 * 4       # with the scratch of a split of 224 256-wide tiles
    assert qk.mmq_workspace_bytes(M, N, K) >= base
    ws = torch.full((full,), 0xAB, dtype=torch.uint8, device="cuda")
    qk.error_flags(clear=True)
    y1 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws, tile=256, split_k=True)
    torch.cuda.synchronize()
    assert int((ws[base:base + 4096] != 0xAB).sum()) > 0          # the split wrote its partial tiles
    y2 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws, pdl=True, tile=256, split_k=True)
    yu = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws[:base], tile=256, split_k=True)
    y9 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws, tile=192)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) == 0
    assert torch.equal(y1, y2)
    counters = ws[full - 224 * 4:].view(torch.int32)
    assert torch.count_nonzero(counters).item() == 0
    r_np = r.cpu().numpy()
    for lo in (0, N // 2 - 20, N - 40):                   # first, middle and last tiles
        hi = lo + 40
        y_ref, ab = oracle.gemm(oracle.Q4_K, w, N, K, c, d, residual=r_np, rows=(lo, hi))
        check(y1.cpu().numpy()[:, lo:hi], y_ref, ab, r_np[:, lo:hi], what=f"split rows {lo}")
        check(yu.cpu().numpy()[:, lo:hi], y_ref, ab, r_np[:, lo:hi], what=f"unsplit rows {lo}")
        check(y9.cpu().numpy()[:, lo:hi], y_ref, ab, r_np[:, lo:hi], what=f"192-wide rows {lo}")


@pytest.mark.parametrize("M,N", [(256, 256 * 112), (200, 256 * 112 - 40)])
def test_mmq_q4k_tail_split(M, N):
    """The default plan on 152 SMs: 224 tiles of 256 with 48 superblocks of K run as 152 whole
    tiles, then the last wave's 72 tiles split in two (144 half tiles).  Checked against the
    oracle on the first and last tiles (a whole tile and a split one), against the same call run
    unsplit, for reproducibility, and for the split scratch being written and its counters left
    at zero."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the tail split is sized for 152 SMs")
    K = 48 * 256
    w, wr = weights("q4k", N, K, seed=44)
    codes, scales = q8(synth.activations(M, K, seed=45))
    c, d = q8_host(codes, scales)
    r = dev(synth.residual(M, N, seed=46))
    base = 2 * (K * 512 + (K // 512) * 8192)
    full = qk.mmq_workspace_bytes(M, N, K)
    assert full == base + 72 * 2 * 128 * 256 * 4 + 72 * 4           # the plan's tail scratch
    ws = torch.full((full,), 0xAB, dtype=torch.uint8, device="cuda")
    qk.error_flags(clear=True)
    y1 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws, tile=256)
    torch.cuda.synchronize()
    assert int((ws[base:base + 4096] != 0xAB).sum()) > 0              # partial tiles written
    y2 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws, tile=256, pdl=True)
    yu = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, workspace=ws[:base], tile=256)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) == 0
    assert torch.equal(y1, y2)
    assert torch.count_nonzero(ws[full - 72 * 4:]).item() == 0
    r_np = r.cpu().numpy()
    for lo in (0, N - 40):
        hi = lo + 40
        y_ref, ab = oracle.gemm(oracle.Q4_K, w, N, K, c, d, residual=r_np, rows=(lo, hi))
        check(y1.cpu().numpy()[:, lo:hi], y_ref, ab, r_np[:, lo:hi], what=f"tail-split rows {lo}")
        check(yu.cpu().numpy()[:, lo:hi], y_ref, ab, r_np[:, lo:hi], what=f"unsplit rows {lo}")


def _f16_bytes(v):
    return np.frombuffer(np.float16(v).tobytes(), np.uint8)


@pytest.mark.parametrize("case", ["q4k_x", "q4k_min", "q6k_x", "q6k_w", "inside"])
def test_mmq_value_limits_set_range_flag(case):
    """An input outside the MMQ's value limits sets QK_ERR_RANGE (the f16 operands would overflow,
    so the output is undefined); the same call inside them leaves the word clear."""
    qt = "q6k" if case.startswith("q6k") else "q4k"
    M, N, K = 24, 96, 512
    w = synth.weights(qt, N, K, seed=31).copy()
    blocks = w.reshape(N, K // 256, oracle.BLOCK_BYTES[QT[qt][1]])
    x = synth.activations(M, K, seed=32)
    if case == "q4k_x":
        x[5, 64:96] *= np.float32(40000.0 / np.abs(x[5, 64:96]).max())          # d_a * 127 = 40000 > 32000
    elif case == "q4k_min":
        blocks[7, 1, 8] = (blocks[7, 1, 8] & 0xC0) | 63                        # m_0 = 63 (GGUF scale byte 4)
        blocks[7, 1, 2:4] = _f16_bytes(70.0 / 63.0)                            # dmin * m_0 = 70 >= 63
    elif case == "q6k_x":
        x[3, 0:32] *= np.float32(70000.0 / np.abs(x[3, 0:32]).max())           # d_a * 127 = 70000 > 65000
    elif case == "q6k_w":
        blocks[11, 0, 192] = np.uint8(0xE0)                                    # sc[0] = -32
        blocks[11, 0, 208:210] = _f16_bytes(0.25)                              # 32 * |d sc| = 256 >= 255
    wr = qk.repack(QT[qt][0], dev(w), N, K)
    codes, scales = q8(x)
    qk.error_flags(clear=True)
    mmq_fn(qt)(wr, codes, scales, N, K)
    torch.cuda.synchronize()
    flags = qk.error_flags(clear=True)
    if case == "inside":
        assert flags == 0
    else:
        assert flags & qk.ERR_RANGE, (case, flags)
        assert not flags & qk.ERR_TIMEOUT
