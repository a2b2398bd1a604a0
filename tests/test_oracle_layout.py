"""Pins for the oracle's statement of the device weight layout (no GPU).

The layout is this project's own (a lossless byte permutation of GGUF
blocks, documented in include/qk.h); the expected byte positions below are
worked out by hand from that specification.
"""
import numpy as np

import oracle
import synth


def test_q4k_single_superblock_code_plane():
    blk = np.zeros(144, np.uint8)
    blk[16:] = np.arange(128, dtype=np.uint8)
    out = oracle.repack(oracle.Q4_K, blk, 1, 256)
    want = np.concatenate([np.arange(0, 16), np.arange(32, 48), np.arange(64, 80), np.arange(96, 112),
                           np.arange(16, 32), np.arange(48, 64), np.arange(80, 96), np.arange(112, 128)])
    assert np.array_equal(out[:128], want.astype(np.uint8))


def test_q4k_meta_records():
    blk = np.zeros(144, np.uint8)
    blk[0:4] = [0x11, 0x22, 0x33, 0x44]
    blk[4:16] = [0xC1, 0x42, 0x83, 0x04, 0x45, 0x86, 0xC7, 0x08, 0x9A, 0xBC, 0xDE, 0xF0]
    out = oracle.repack(oracle.Q4_K, blk, 1, 256)
    meta = out[128:144]
    assert meta[:4].tolist() == [0x11, 0x22, 0x33, 0x44]
    # (sc, m) pairs (1,5) (2,6) | (3,7) (4,8) | (58,25) (28,43) | (46,61) (0,15)
    recs = [1 | 2 << 6 | 5 << 12 | 6 << 18, 3 | 4 << 6 | 7 << 12 | 8 << 18,
            58 | 28 << 6 | 25 << 12 | 43 << 18, 46 | 0 << 6 | 61 << 12 | 15 << 18]
    assert recs[0] == 0x185081
    for g, r in enumerate(recs):
        assert meta[4 + 3 * g:7 + 3 * g].tolist() == [r & 0xFF, (r >> 8) & 0xFF, r >> 16]


def test_q4k_ragged_step_position():
    N, K = 2, 256 * 11                    # steps of 8 and 3 superblocks
    w = synth.q4k_weights(N, K, seed=4)
    out = oracle.repack(oracle.Q4_K, w, N, K)
    B = 11
    blocks = w.reshape(N, B, 144)
    row = 1
    base = row * B * 128 + 1024 * 1       # step 1 of row 1
    G = 12                                # 4 groups x 3 superblocks
    u = 4 * 1 + 2                         # superblock 9 is local 1; group 2
    qs = blocks[row, 9, 16:]
    assert np.array_equal(out[base + 16 * u: base + 16 * u + 16], qs[64:80])
    assert np.array_equal(out[base + 16 * G + 16 * u: base + 16 * G + 16 * u + 16], qs[80:96])
    # the code plane is a permutation of all code bytes, the meta plane keeps d/dmin
    assert np.array_equal(np.sort(out[:N * B * 128]), np.sort(blocks[:, :, 16:].reshape(-1)))
    meta = out[N * B * 128:].reshape(N, B, 16)
    assert np.array_equal(meta[:, :, :4], blocks[:, :, :4])


def test_q6k_single_superblock_planes():
    blk = np.zeros(210, np.uint8)
    blk[0:128] = np.arange(128, dtype=np.uint8)
    blk[128:192] = np.arange(200, 264, dtype=np.int64).astype(np.uint8)
    blk[192:208] = np.arange(16, dtype=np.uint8) + 100
    blk[208:210] = [0xAB, 0xCD]
    out = oracle.repack(oracle.Q6_K, blk, 1, 256)
    want_ql = np.concatenate([np.arange(0, 16), np.arange(16, 32), np.arange(64, 80), np.arange(80, 96),
                              np.arange(32, 48), np.arange(48, 64), np.arange(96, 112), np.arange(112, 128)])
    assert np.array_equal(out[:128], want_ql.astype(np.uint8))
    assert np.array_equal(out[128:192], blk[128:192])
    want_sc = [0, 2, 4, 6, 1, 3, 5, 7, 8, 10, 12, 14, 9, 11, 13, 15]
    assert out[192:208].tolist() == [100 + i for i in want_sc]
    assert out[208:210].tolist() == [0xAB, 0xCD]


def test_q6k_ragged_and_permutation():
    N, K = 3, 256 * 9
    w = synth.q6k_weights(N, K, seed=6)
    out = oracle.repack(oracle.Q6_K, w, N, K)
    assert out.size == w.size
    assert np.array_equal(np.sort(out), np.sort(w))
    B = 9
    blocks = w.reshape(N, B, 210)
    # row 2, superblock 8 = step 1, local 0, one lane step (L = 4); lane 3 -> h=1, e=1
    base = 2 * B * 128 + 1024
    assert np.array_equal(out[base + 48: base + 64], blocks[2, 8, 64 + 16:64 + 32])
    assert np.array_equal(out[base + 64 + 48: base + 64 + 64], blocks[2, 8, 64 + 32 + 16:64 + 64])
