"""Pins of the oracle's Q2_K and Q3_K dequantization and device layouts.

Reading (cajeta.dev "xpu walkthrough" sec. 4.2 names Q2_K and Q3_K among the formats its batched
decode serves; the pages print no layout): the public GGUF blocks.
  Q2_K, 84 bytes: scales[16] (low nibble scale, high nibble min per 16 values), qs[64], f16 d,
    f16 dmin; value 128n + 32j + l = d * sc * q - dmin * m with q = bits 2j of qs[32n + l] and the
    scale byte of sub-block 8n + 2j + (l >= 16).
  Q3_K, 110 bytes: hmask[32], qs[64], 12 bytes of sixteen 6-bit scales, f16 d; value 128n + 32j + l
    = d * (S - 32) * (q - 4 (1 - h)), h = bit 4n + j of hmask[l].
"""
import numpy as np

import oracle


def f16(v):
    return np.frombuffer(np.float16(v).tobytes(), np.uint8)


def q2_block(d=1.0, dmin=0.0, scales=None, qs=None):
    b = np.zeros(84, np.uint8)
    if scales is not None:
        b[0:16] = scales
    if qs is not None:
        b[16:80] = qs
    b[80:82], b[82:84] = f16(d), f16(dmin)
    return b


def q3_block(d=1.0, hmask=None, qs=None, sc12=None):
    b = np.zeros(110, np.uint8)
    if hmask is not None:
        b[0:32] = hmask
    if qs is not None:
        b[32:96] = qs
    if sc12 is not None:
        b[96:108] = sc12
    b[108:110] = f16(d)
    return b


def q3_scales_all(v):
    """12 packed bytes that give every one of the 16 scales the 6-bit value v (S - 32 = v - 32)."""
    lo, hi = v & 15, v >> 4
    b = np.zeros(12, np.uint8)
    b[0:8] = lo | (lo << 4)
    b[8:12] = hi | (hi << 2) | (hi << 4) | (hi << 6)
    return b


def test_sizes():
    assert oracle.BLOCK_BYTES[oracle.Q2_K] == 84 and oracle.BLOCK_BYTES[oracle.Q3_K] == 110
    assert oracle.DEVICE_BYTES[oracle.Q3_K] == 114


def test_q2k_hand_example():
    # sub-block 3 = (n 0, j 1, l >= 16): scale byte 0x52 -> sc 2, m 5; d 0.5, dmin 0.25;
    # qs[16 + 3] = 0b0000_1100 puts code 3 at bits 2-3 (j = 1) of position l = 19 -> value 51
    sc = np.zeros(16, np.uint8)
    sc[3] = 0x52
    qs = np.zeros(64, np.uint8)
    qs[19] = 0b00001100
    w = oracle.dequant_block(oracle.Q2_K, q2_block(0.5, 0.25, sc, qs))
    want = np.zeros(256)
    want[48:64] = -0.25 * 5                      # the other 15 values of sub-block 3: min term only
    want[51] = 0.5 * 2 * 3 - 0.25 * 5
    assert np.array_equal(w, want)


def test_q2k_one_hot_code_positions():
    sc = np.full(16, 0x01, np.uint8)             # sc 1, m 0
    for n in range(2):
        for j in range(4):
            for l in (0, 15, 16, 31):
                qs = np.zeros(64, np.uint8)
                qs[32 * n + l] = 2 << (2 * j)
                w = oracle.dequant_block(oracle.Q2_K, q2_block(1.0, 0.0, sc, qs))
                assert list(np.flatnonzero(w)) == [128 * n + 32 * j + l] and w[128 * n + 32 * j + l] == 2


def test_q2k_closed_form_integer_matmul():
    rng = np.random.default_rng(11)
    N, K = 3, 512
    qsb = rng.integers(0, 256, (N * K // 256, 64), dtype=np.uint8)
    w = np.concatenate([q2_block(1.0, 0.0, np.full(16, 1, np.uint8), qsb[i]) for i in range(len(qsb))])
    q = np.zeros((N, K), np.int64)
    for i in range(len(qsb)):
        n, b = divmod(i, K // 256)
        for hn in range(2):
            for j in range(4):
                for l in range(32):
                    q[n, 256 * b + 128 * hn + 32 * j + l] = (qsb[i][32 * hn + l] >> (2 * j)) & 3
    assert np.array_equal(oracle.dequant_matrix(oracle.Q2_K, w, N, K), q.astype(np.float64))
    codes = rng.integers(-127, 128, (2, K), dtype=np.int8)
    y, _ = oracle.gemm(oracle.Q2_K, w, N, K, codes, np.full((2, K // 32), 0x3C00, np.uint16))
    assert np.array_equal(y, (codes.astype(np.int64) @ q.T).astype(np.float64))


def test_q3k_scale_unpacking():
    # scale 13: low nibble = high nibble of byte 5, high bits = bits 6-7 of byte 9 (13 % 4 = 1, 13 / 4 = 3)
    sc12 = np.zeros(12, np.uint8)
    sc12[5] = 0xB0                               # low nibble 11 for scale 13 (and 0 for scale 5)
    sc12[9] = 0b10 << 6                          # high bits 2 for scale 13
    assert oracle.q3k_scale(sc12, 13) == (11 | (2 << 4)) - 32
    assert oracle.q3k_scale(sc12, 5) == -32
    sc12 = np.zeros(12, np.uint8)
    sc12[2] = 0x07                               # scale 2: low 7
    sc12[10] = 0b11                              # scale 2: high bits 3 (2 % 4 = 2, 2 / 4 = 0)
    assert oracle.q3k_scale(sc12, 2) == (7 | (3 << 4)) - 32
    for v in (0, 1, 32, 45, 63):
        assert all(oracle.q3k_scale(q3_scales_all(v), s) == v - 32 for s in range(16))


def test_q3k_hmask_and_code_positions():
    sc12 = q3_scales_all(33)                     # S - 32 = 1 everywhere
    for n in range(2):
        for j in range(4):
            for l in (0, 17, 31):
                for h in (0, 1):
                    qs = np.zeros(64, np.uint8)
                    hm = np.zeros(32, np.uint8)
                    qs[32 * n + l] = 3 << (2 * j)
                    hm[l] = h << (4 * n + j)
                    w = oracle.dequant_block(oracle.Q3_K, q3_block(1.0, hm, qs, sc12))
                    v = 128 * n + 32 * j + l
                    assert w[v] == 3 - 4 * (1 - h)
                    others = np.delete(w, v)
                    assert np.all(others == -4)      # code 0, h 0 -> q = -4


def test_q3k_closed_form_integer_matmul():
    rng = np.random.default_rng(12)
    N, K = 2, 512
    nb = N * K // 256
    qsb = rng.integers(0, 256, (nb, 64), dtype=np.uint8)
    hmb = rng.integers(0, 256, (nb, 32), dtype=np.uint8)
    w = np.concatenate([q3_block(1.0, hmb[i], qsb[i], q3_scales_all(33)) for i in range(nb)])
    q = np.zeros((N, K), np.int64)
    for i in range(nb):
        n, b = divmod(i, K // 256)
        for hn in range(2):
            for j in range(4):
                for l in range(32):
                    c = int((qsb[i][32 * hn + l] >> (2 * j)) & 3)
                    h = int((hmb[i][l] >> (4 * hn + j)) & 1)
                    q[n, 256 * b + 128 * hn + 32 * j + l] = c - 4 * (1 - h)
    assert np.array_equal(oracle.dequant_matrix(oracle.Q3_K, w, N, K), q.astype(np.float64))
    codes = rng.integers(-127, 128, (3, K), dtype=np.int8)
    y, _ = oracle.gemm(oracle.Q3_K, w, N, K, codes, np.full((3, K // 32), 0x3C00, np.uint16))
    assert np.array_equal(y, (codes.astype(np.int64) @ q.T).astype(np.float64))


def test_device_layouts():
    # codes: lane u = 4 sb' + 2n' + e of a step holds qs[32n' + 16e .. +16] at 16u; scale records in
    # lane order (byte 4p + t = sub-block 8n' + 2t + e); then the per-type planes
    rng = np.random.default_rng(13)
    N, K = 2, 256 * 9                            # a full step and a ragged one
    B = K // 256
    for qt, bs, qoff in ((oracle.Q2_K, 84, 16), (oracle.Q3_K, 110, 32)):
        raw = rng.integers(0, 256, N * B * bs, dtype=np.uint8)
        r = oracle.repack(qt, raw, N, K)
        blocks = raw.reshape(N, B, bs)
        for n in range(N):
            for b in (0, 7, 8):
                s, sbp = divmod(b, 8)
                for p in range(4):
                    hn, e = divmod(p, 2)
                    u = 4 * sbp + p
                    got = r[n * B * 64 + 512 * s + 16 * u:][:16]
                    assert np.array_equal(got, blocks[n, b, qoff + 32 * hn + 16 * e:][:16])
                    for t in range(4):
                        sub = 8 * hn + 2 * t + e
                        off = N * B * (64 if qt == oracle.Q2_K else 96) + (n * B + b) * 16 + 4 * p + t
                        if qt == oracle.Q2_K:
                            assert r[off] == blocks[n, b, sub]
                        else:
                            assert np.int8(r[off].view(np.int8)) == oracle.q3k_scale(blocks[n, b, 96:108], sub)
                if qt == oracle.Q2_K:
                    assert np.array_equal(r[N * B * 80 + (n * B + b) * 4:][:4], blocks[n, b, 80:84])
                else:
                    assert np.array_equal(r[N * B * 64 + (n * B + b) * 32:][:32], blocks[n, b, 0:32])
                    assert np.array_equal(r[N * B * 112 + (n * B + b) * 2:][:2], blocks[n, b, 108:110])
