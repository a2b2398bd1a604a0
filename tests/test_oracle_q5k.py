"""Pins of the oracle's Q5_K dequantization and device layout.

Reading (the pages name Q5_K among the served k-quants -- minfer "15 . The CUDA
backend" sec. 2.2, cajeta.dev "xpu walkthrough" sec. 4.2 -- but print no layout):
the public GGUF block of 176 bytes, f16 d, f16 dmin, 12 bytes of 6-bit scales and
mins packed as for Q4_K, qh[32], qs[128]; value 64g + l (l < 32) is the low nibble
of qs[32g + l] plus 16 * bit 2g of qh[l], value 64g + 32 + l the high nibble plus
16 * bit 2g+1; w = d * sc * q - dmin * m.
"""
import numpy as np

import oracle


def block(d=1.0, dmin=0.0, scales=None, qh=None, qs=None):
    b = np.zeros(176, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    if scales is not None:
        b[4:16] = scales
    if qh is not None:
        b[16:48] = qh
    if qs is not None:
        b[48:176] = qs
    return b


def unit_scales():
    # sc = 1 and m = 0 for all eight sub-blocks under the Q4_K packing: bytes 0-3 hold sc 0-3,
    # 4-7 m 0-3, 8-11 the low nibbles of sc 4-7 / m 4-7 (high bits of sc 4-7 live in bytes 0-3)
    q = np.zeros(12, np.uint8)
    q[0:4] = 1
    q[8:12] = 0x01
    return q


def test_block_size():
    assert oracle.BLOCK_BYTES[oracle.Q5_K] == 176


def test_hand_example_fifth_bits():
    # group 2, position 5: qs[64 + 5] = 0x7A (low 10, high 7); qh[5] = 0b0011_0000 sets bit 4 (= 2g,
    # the low nibble's fifth bit) and bit 5 (= 2g+1, the high nibble's)
    qs = np.zeros(128, np.uint8)
    qh = np.zeros(32, np.uint8)
    qs[64 + 5] = 0x7A
    qh[5] = 0b00110000
    w = oracle.dequant_block(oracle.Q5_K, block(scales=unit_scales(), qh=qh, qs=qs))
    want = np.zeros(256)
    want[128 + 5] = 10 + 16
    want[128 + 32 + 5] = 7 + 16
    assert np.array_equal(w, want)


def test_one_hot_probes_over_groups_and_positions():
    for g in range(4):
        for l in (0, 13, 31):
            for lo_bit in (0, 1):
                qs = np.zeros(128, np.uint8)
                qh = np.zeros(32, np.uint8)
                qs[32 * g + l] = 0x35                       # low 5, high 3
                qh[l] = (lo_bit << (2 * g)) | ((1 - lo_bit) << (2 * g + 1))
                w = oracle.dequant_block(oracle.Q5_K, block(scales=unit_scales(), qh=qh, qs=qs))
                nz = np.flatnonzero(w)
                assert set(nz) == {64 * g + l, 64 * g + 32 + l}
                assert w[64 * g + l] == 5 + 16 * lo_bit
                assert w[64 * g + 32 + l] == 3 + 16 * (1 - lo_bit)


def test_scale_and_min_of_a_sub_block():
    # sub-block 3 (group 1, high nibbles): sc = 5, m = 7 (bytes 3 and 7 of the packing); d = 0.5,
    # dmin = 0.25; every high nibble of group 1 is 9 and every fifth bit set -> q = 25
    q12 = np.zeros(12, np.uint8)
    q12[3], q12[7] = 5, 7
    qs = np.zeros(128, np.uint8)
    qs[32:64] = 0x90
    qh = np.full(32, 0b1000, np.uint8)                      # bit 3 = 2*1 + 1
    w = oracle.dequant_block(oracle.Q5_K, block(d=0.5, dmin=0.25, scales=q12, qh=qh, qs=qs))
    assert np.allclose(w[96:128], 0.5 * 5 * 25 - 0.25 * 7, rtol=0, atol=0)
    # sub-block 2 (group 1, low nibbles 0, fifth bit 0, sc = m = 0) is exactly zero
    assert np.all(w[64:96] == 0)


def test_closed_form_integer_matmul():
    rng = np.random.default_rng(5)
    N, K = 3, 512
    blocks = []
    qvals = np.zeros((N, K), np.int64)
    for n in range(N):
        for b in range(K // 256):
            qs = rng.integers(0, 256, 128, dtype=np.uint8)
            qh = rng.integers(0, 256, 32, dtype=np.uint8)
            blocks.append(block(scales=unit_scales(), qh=qh, qs=qs))
            for g in range(4):
                for l in range(32):
                    qvals[n, 256 * b + 64 * g + l] = (qs[32 * g + l] & 15) + 16 * ((qh[l] >> (2 * g)) & 1)
                    qvals[n, 256 * b + 64 * g + 32 + l] = (qs[32 * g + l] >> 4) + 16 * ((qh[l] >> (2 * g + 1)) & 1)
    w = np.concatenate(blocks)
    assert np.array_equal(oracle.dequant_matrix(oracle.Q5_K, w, N, K), qvals.astype(np.float64))
    codes = rng.integers(-127, 128, (2, K), dtype=np.int8)
    d1 = np.full((2, K // 32), 0x3C00, np.uint16)            # d_a = 1.0
    y, ab = oracle.gemm(oracle.Q5_K, w, N, K, codes, d1)
    assert np.array_equal(y, (codes.astype(np.int64) @ qvals.T).astype(np.float64))
    assert np.array_equal(ab, (np.abs(codes.astype(np.int64)) @ qvals.T).astype(np.float64))


def test_device_layout_fifth_bit_positions():
    # one set bit of qh lands at one documented bit of the fifth-bit plane: GGUF qh[l] bit 2g -> R_lo
    # of group g, bit 8 * (l % 4) + l // 4; bit 2g+1 -> R_hi, same bit
    N, K = 1, 256
    for g, l, hi in ((0, 0, 0), (1, 7, 1), (3, 30, 0), (2, 17, 1)):
        qh = np.zeros(32, np.uint8)
        qh[l] = 1 << (2 * g + hi)
        r = oracle.repack(oracle.Q5_K, block(qh=qh), N, K)
        plane = r[128:160]
        bit = 8 * (l % 4) + l // 4
        want = np.zeros(32, np.uint8)
        want[8 * g + 4 * hi + bit // 8] = 1 << (bit % 8)
        assert np.array_equal(plane, want), (g, l, hi)


def test_device_layout_codes_and_meta_match_q4k():
    # the codes and metadata planes are those of a Q4_K block with the same d, dmin, scales and codes
    rng = np.random.default_rng(6)
    N, K = 3, 256 * 9                                        # a full step of 8 and a ragged one
    w5 = []
    w4 = []
    for _ in range(N * K // 256):
        b = rng.integers(0, 256, 176, dtype=np.uint8)
        w5.append(b)
        w4.append(np.concatenate([b[0:16], b[48:176]]))
    r5 = oracle.repack(oracle.Q5_K, np.concatenate(w5), N, K)
    r4 = oracle.repack(oracle.Q4_K, np.concatenate(w4), N, K)
    nb = N * K // 256
    assert np.array_equal(r5[:nb * 128], r4[:nb * 128])
    assert np.array_equal(r5[nb * 160:], r4[nb * 128:])
