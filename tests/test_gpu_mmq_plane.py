"""GPU: the Q4_K MMQ with a load-time min-operand plane (qk_q4k_min_plane, qk_mmq_q4k_plane).

The plane holds, per weight row and pair of superblocks, the exact f16 split (hi | lo) of
1024 * dmin * m that the MMQ's min stages otherwise build from the 6-bit fields.  Bars:
  - the plane, byte for byte, against the split computed here from the GGUF blocks (the
    oracle's 6-bit unpack, binary32 product, 13 low mantissa bits cleared for hi);
  - the MMQ with the plane, bit for bit, against the MMQ without it (the operands are the
    same words), and within the parity bound of the oracle on sampled rows.
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


def plane_ref(w, N, K):
    """The expected plane of GGUF Q4_K weight bytes w (N x K), as bytes."""
    B = K // 256
    nmin = (B + 1) // 2
    blk = w.reshape(N, B, 144)
    out = np.zeros((N, nmin, 4, 8), np.float16)
    for n in range(N):
        for b in range(B):
            dmin = np.frombuffer(blk[n, b, 2:4].tobytes(), np.float16)[0].astype(np.float32)
            q12 = bytes(blk[n, b, 4:16])
            i, half = divmod(b, 2)
            for j in range(8):
                m = oracle.q4k_scale_min(q12, j)[1]
                v = np.float32(dmin * np.float32(m)) * np.float32(1024.0)     # exact: 17 significant bits
                hi = np.array([v], np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
                hi = hi.view(np.float32)[0]
                out[n, i, half, j] = np.float16(hi)
                out[n, i, 2 + half, j] = np.float16(np.float32(v - hi))
    return out.view(np.uint8).reshape(-1)


@pytest.mark.parametrize("N,K", [(37, 256), (64, 768), (130, 2048)])
def test_min_plane_bytes(N, K):
    w = synth.weights("q4k", N, K, seed=N + K)
    wr = qk.repack(1, dev(w), N, K)
    assert qk.q4k_min_plane_bytes(N, K) == N * ((K // 256 + 1) // 2) * 64
    qk.error_flags(clear=True)
    plane = qk.q4k_min_plane(wr, N, K)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) == 0
    assert np.array_equal(plane.cpu().numpy(), plane_ref(w, N, K))


@pytest.mark.parametrize("M,N,K,tile", [(200, 1000, 768, None), (256, 512, 1024, 128), (130, 2000, 2560, 256),
                                        (1, 300, 256, None), (333, 4608, 3584, None), (150, 3584, 1280, 192)])
def test_mmq_plane_bitexact(M, N, K, tile):
    w = synth.weights("q4k", N, K, seed=M + N)
    wr = qk.repack(1, dev(w), N, K)
    codes, scales = qk.quantize_q8_1(dev(synth.activations(M, K, seed=K)))
    r = dev(synth.residual(M, N, seed=M))
    plane = qk.q4k_min_plane(wr, N, K)
    qk.error_flags(clear=True)
    y0 = qk.mmq_q4k(wr, codes, scales, N, K, residual=r, tile=tile)
    y1 = qk.mmq_q4k_plane(wr, plane, codes, scales, N, K, residual=r, tile=tile)
    y2 = qk.mmq_q4k_plane(wr, plane, codes, scales, N, K, residual=r, tile=tile, pdl=True)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) == 0
    assert torch.equal(y0, y1) and torch.equal(y1, y2)
    c, d = codes.cpu().numpy(), scales.cpu().numpy()[:, :, 0].view(np.uint16).copy()
    r_np = r.cpu().numpy()
    lo, hi = N - 7, N                                          # the ragged last rows of the last tile
    y_ref, ab = oracle.gemm(oracle.Q4_K, w, N, K, c, d, residual=r_np, rows=(lo, hi))
    err = np.abs(y1.cpu().numpy()[:, lo:hi].astype(np.float64) - y_ref)
    assert np.all(err <= 1e-4 * ab + 2.0 ** -22 * np.abs(r_np[:, lo:hi]))


def test_mmq_plane_split_k():
    """The plane with the K range of each tile split in two (QK_MMQ_SPLIT_K; 224 tiles, 48 superblocks)."""
    M, N, K = 256, 256 * 112, 48 * 256
    w = synth.weights("q4k", N, K, seed=7)
    wr = qk.repack(1, dev(w), N, K)
    codes, scales = qk.quantize_q8_1(dev(synth.activations(M, K, seed=8)))
    plane = qk.q4k_min_plane(wr, N, K)
    ws = torch.empty(2 * (K * 512 + (K // 512) * 8192) + 224 * 2 * 128 * 256 * 4 + 224 * 4, dtype=torch.uint8,
                     device="cuda")                       # with the scratch of a split of 224 256-wide tiles
    y0 = qk.mmq_q4k(wr, codes, scales, N, K, workspace=ws, tile=256, split_k=True)
    y1 = qk.mmq_q4k_plane(wr, plane, codes, scales, N, K, workspace=ws, tile=256, split_k=True)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)


def test_min_plane_range_flag():
    """dmin * m >= 63 makes the plane builder set QK_ERR_RANGE, as the MMQ does."""
    N, K = 96, 512
    w = synth.weights("q4k", N, K, seed=31).copy()
    blocks = w.reshape(N, K // 256, 144)
    blocks[7, 1, 8] = (blocks[7, 1, 8] & 0xC0) | 63                 # m_0 = 63 (GGUF scale byte 4)
    blocks[7, 1, 2:4] = np.frombuffer(np.float16(70.0 / 63.0).tobytes(), np.uint8)   # dmin * m_0 = 70
    wr = qk.repack(1, dev(w), N, K)
    qk.error_flags(clear=True)
    qk.q4k_min_plane(wr, N, K)
    torch.cuda.synchronize()
    assert qk.error_flags(clear=True) & qk.ERR_RANGE


def test_plane_arguments_rejected():
    N, K = 64, 512
    wr = qk.repack(1, dev(synth.weights("q4k", N, K, seed=3)), N, K)
    plane = torch.empty(qk.q4k_min_plane_bytes(N, K), dtype=torch.uint8, device="cuda")
    L = qk.lib()
    assert L.qk_q4k_min_plane(wr.data_ptr(), N, K, plane.data_ptr(), plane.numel() - 1, None) == -6
    assert L.qk_q4k_min_plane(wr.data_ptr(), N, K, plane.data_ptr() + 8, plane.numel(), None) == -3
    assert L.qk_q4k_min_plane(wr.data_ptr(), N, 300, plane.data_ptr(), plane.numel(), None) == -2
    assert L.qk_q4k_min_plane(wr.data_ptr(), N, K, wr.data_ptr(), plane.numel(), None) == -4
    codes, scales = qk.quantize_q8_1(dev(synth.activations(4, K, seed=1)))
    y = torch.empty((4, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(qk.mmq_workspace_bytes(4, N, K), dtype=torch.uint8, device="cuda")
    args = (codes.data_ptr(), scales.data_ptr(), 4, N, K, None, y.data_ptr(), ws.data_ptr(), ws.numel(), 0, None)
    assert L.qk_mmq_q4k_plane(wr.data_ptr(), None, *args) == -1
    assert L.qk_mmq_q4k_plane(wr.data_ptr(), plane.data_ptr() + 4, *args) == -3
    assert L.qk_mmq_q4k_plane(wr.data_ptr(), y.data_ptr(), *args) == -4
