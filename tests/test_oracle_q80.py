"""Pins of the oracle's Q8_0 dequantization and device layout.

Reading (cajeta.dev "xpu walkthrough" sec. 4.2 names Q8_0 among the formats its
batched decode serves; the pages print no layout): the public GGUF block of 34
bytes, f16 d then 32 int8 codes; w = d * q.
"""
import numpy as np

import oracle


def blk(d, codes):
    b = np.zeros(34, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:34] = np.asarray(codes, np.int8).view(np.uint8)
    return b


def test_unit_bytes():
    # eight 34-byte blocks per 256 values
    assert oracle.BLOCK_BYTES[oracle.Q8_0] == 8 * 34


def test_hand_example():
    # block 3 has d = 0.5 and codes -128 .. +127 in steps of 8: w = 0.5 q; the other blocks are zero
    codes = np.arange(-128, 128, 8)
    blocks = [blk(0.0, np.zeros(32)) for _ in range(8)]
    blocks[3] = blk(0.5, codes)
    w = oracle.dequant_block(oracle.Q8_0, np.concatenate(blocks))
    want = np.zeros(256)
    want[96:128] = 0.5 * codes
    assert np.array_equal(w, want)


def test_closed_form_integer_matmul():
    rng = np.random.default_rng(8)
    N, K = 4, 512
    q = rng.integers(-127, 128, (N, K))
    w = np.concatenate([blk(1.0, q[n, 32 * b:32 * b + 32]) for n in range(N) for b in range(K // 32)])
    assert np.array_equal(oracle.dequant_matrix(oracle.Q8_0, w, N, K), q.astype(np.float64))
    codes = rng.integers(-127, 128, (3, K), dtype=np.int8)
    y, ab = oracle.gemm(oracle.Q8_0, w, N, K, codes, np.full((3, K // 32), 0x3C00, np.uint16))
    assert np.array_equal(y, (codes.astype(np.int64) @ q.T).astype(np.float64))
    assert np.array_equal(ab, (np.abs(codes.astype(np.int64)) @ np.abs(q).T).astype(np.float64))


def test_device_layout():
    # codes plane: the codes row-major; d plane: each block's two d bytes in block order
    rng = np.random.default_rng(9)
    N, K = 3, 256 * 3
    raw = rng.integers(0, 256, N * K // 32 * 34, dtype=np.uint8)
    r = oracle.repack(oracle.Q8_0, raw, N, K)
    b = raw.reshape(N * K // 32, 34)
    assert np.array_equal(r[:N * K], b[:, 2:].reshape(-1))
    assert np.array_equal(r[N * K:], b[:, :2].reshape(-1))
