"""Pins for the CPU oracle (no GPU).

Every check here ties the oracle to something other than itself: IEEE 754
binary16 values worked out by hand, hand-computed q8_1 blocks, the byte
layout facts of tests/golden/*.json, closed forms (w = q integer case,
d = 0), numpy's independent float16 and integer matmul, and algebraic
invariants (x = 0, one-hot columns, linearity).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ binary16

F16_TABLE = [  # value, bits (IEEE 754 binary16, worked out by hand)
    (0.0, 0x0000), (-0.0, 0x8000), (1.0, 0x3C00), (-2.0, 0xC000), (0.5, 0x3800),
    (65504.0, 0x7BFF), (2.0 ** -14, 0x0400), (2.0 ** -24, 0x0001),
    (2.0 ** -25, 0x0000),            # tie between 0 and 2^-24 -> even (0)
    (3 * 2.0 ** -25, 0x0002),        # tie between 1 and 2 units -> even (2)
    (1.0 + 2.0 ** -11, 0x3C00),      # tie -> even mantissa 0
    (1.0 + 3 * 2.0 ** -11, 0x3C02),  # tie -> even mantissa 2
    (0.1, 0x2E66), (1e-3, 0x1419), (0.3, 0x34CD),
    (65519.0, 0x7BFF),               # rounds down to 65504
    (65520.0, 0x7BFF),               # would round to inf: saturates
    (1e6, 0x7BFF), (-1e6, 0xFBFF),   # saturation
]


@pytest.mark.parametrize("v,bits", F16_TABLE)
def test_f16_encode_table(v, bits):
    assert oracle.f32_to_f16(v) == bits


F16_DECODE = [  # bits, value (IEEE 754 binary16, worked out by hand)
    (0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x0400, 2.0 ** -14),
    (0x7BFF, 65504.0), (0xC000, -2.0), (0x2E66, 0.0999755859375), (0x3C02, 1.0 + 2.0 ** -9),
    (0x8000, -0.0), (0x18D6, 2.0 ** -9 * (1 + 214 / 1024)),
]


@pytest.mark.parametrize("bits,v", F16_DECODE)
def test_f16_decode_table(bits, v):
    assert oracle.f16_to_f64(bits) == v


def test_f16_matches_numpy_in_range():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.uniform(-1, 1, 20000) * 1e-6).astype(np.float32),     # subnormal region
        (rng.uniform(-65000, 65000, 20000)).astype(np.float32),
        np.float32(2.0) ** rng.integers(-30, 15, 5000).astype(np.float32),
    ])
    ours = np.array([oracle.f32_to_f16(v) for v in vals], np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_decode_exhaustive_vs_numpy():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    ours = np.array([oracle.f16_to_f64(int(b)) for b in bits[finite]])
    assert np.array_equal(ours, ref[finite])


# ---------------------------------------------------------------------- q8_1

def _expand(v, n=32):
    if isinstance(v, str):
        count, val = v.split(" x ")
        return [float(val)] * int(count)
    return v


def test_q8_1_golden_blocks():
    for blk in gold("q8_1_blocks.json")["blocks"]:
        x = np.array(_expand(blk["x"]), np.float32)[None, :]
        codes, d, s = oracle.quantize_q8_1(x)
        want = [int(c) for c in _expand(blk["codes"])]
        assert codes[0].tolist() == want, blk["name"]
        assert int(d[0, 0]) == int(blk["d_f16"], 16), blk["name"]
        assert int(s[0, 0]) == int(blk["s_f16"], 16), blk["name"]


def test_q8_1_invariants_random():
    x = synth.activations(7, 4096, seed=3) * np.float32(2.5)
    x[2, :64] = 0.0                      # two all-zero blocks
    codes, d, s = oracle.quantize_q8_1(x)
    assert codes.min() >= -127 and codes.max() <= 127
    xb = x.reshape(7, -1, 32)
    cb = codes.reshape(7, -1, 32).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    dd = d.view(np.float16).astype(np.float64)
    nz = amax > 0
    # every non-zero block reaches |q| = 127 at its largest element
    assert np.all(np.abs(cb).max(axis=2)[nz] == 127)
    assert np.all(cb[~nz] == 0) and np.all(dd[~nz] == 0)
    # d is amax/127 to binary16 precision
    assert np.allclose(dd[nz], amax[nz] / 127.0, rtol=2 ** -10, atol=0)
    # round trip with the binary32 d: |x - d q| <= d/2 (plus binary32 slack)
    d32 = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    err = np.abs(xb - d32[:, :, None] * cb)
    assert np.all(err <= d32[:, :, None] * (0.5 + 1e-6) + 1e-30)
    # s is d*sum(q) to binary16 precision
    ss = s.view(np.float16).astype(np.float64)
    assert np.allclose(ss, d32 * cb.sum(axis=2), rtol=2 ** -10, atol=2 ** -24)


def test_q8_1_sign_symmetry():
    x = synth.activations(3, 1024, seed=11)
    c1, d1, s1 = oracle.quantize_q8_1(x)
    c2, d2, s2 = oracle.quantize_q8_1(-x)
    assert np.array_equal(c1, -c2) and np.array_equal(d1, d2)
    assert np.array_equal(s1 ^ np.uint16(0x8000), s2) or np.all((s1 & 0x7FFF) == 0)


def test_q8_1_scale_invariance_power_of_two():
    x = synth.activations(2, 512, seed=5)
    c1, d1, _ = oracle.quantize_q8_1(x)
    c2, d2, _ = oracle.quantize_q8_1(x * np.float32(4.0))
    assert np.array_equal(c1, c2)
    assert np.allclose(d2.view(np.float16).astype(np.float64), 4 * d1.view(np.float16).astype(np.float64))


# ---------------------------------------------------------------------- Q4_K

def q4k_block(d=0x3C00, dmin=0x0000, scales=None, qs=None):
    b = np.zeros(144, np.uint8)
    b[0:2] = np.array([d & 0xFF, d >> 8], np.uint8)
    b[2:4] = np.array([dmin & 0xFF, dmin >> 8], np.uint8)
    if scales is not None:
        b[4:16] = np.array(scales, np.uint8)
    if qs is not None:
        b[16:144] = np.array(qs, np.uint8)
    return b


def test_q4k_block_size():
    assert oracle.BLOCK_BYTES[oracle.Q4_K] == 144 == gold("q4k_layout.json")["block_bytes"]
    assert synth.q4k_weights(3, 512).size == 3 * 2 * 144


def test_q4k_scale_unpack_golden():
    g = gold("q4k_layout.json")
    q12 = bytes(int(v, 16) for v in g["scale_bytes"])
    for j in range(8):
        assert oracle.q4k_scale_min(q12, j) == (g["scales"][j], g["mins"][j])


def test_q4k_scales_through_dequant():
    # d = 1, dmin = 1, every nibble 1: sub-block j holds sc_j - m_j
    g = gold("q4k_layout.json")
    scales = [int(v, 16) for v in g["scale_bytes"]]
    blk = q4k_block(d=0x3C00, dmin=0x3C00, scales=scales, qs=[0x11] * 128)
    w = oracle.dequant_block(oracle.Q4_K, blk)
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == g["scales"][j] - g["mins"][j])


def test_q4k_nibble_index_golden():
    g = gold("q4k_layout.json")
    unit = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]
    for probe in g["nibble_to_index"]:
        qs = [0] * 128
        qs[probe["byte"]] = 7 if probe["nibble"] == "low" else 7 << 4
        w = oracle.dequant_block(oracle.Q4_K, q4k_block(scales=unit, qs=qs))
        nz = np.nonzero(w)[0].tolist()
        assert nz == [probe["index"]] and w[probe["index"]] == 7.0


def test_q4k_closed_form_integer():
    # d = 1, dmin = 0, sc = 1 -> w equals the raw 4-bit codes
    rng = np.random.default_rng(1)
    qs = rng.integers(0, 256, 128)
    w = oracle.dequant_block(oracle.Q4_K, q4k_block(scales=[1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], qs=qs))
    lo, hi = qs & 15, qs >> 4
    want = np.concatenate([np.concatenate([lo[32 * g:32 * g + 32], hi[32 * g:32 * g + 32]]) for g in range(4)])
    assert np.array_equal(w, want.astype(np.float64))


def test_q4k_closed_form_d_zero():
    # d = 0: w = -dmin * m_j whatever the codes
    g = gold("q4k_layout.json")
    scales = [int(v, 16) for v in g["scale_bytes"]]
    blk = q4k_block(d=0x0000, dmin=0x3800, scales=scales, qs=np.arange(128) % 256)  # dmin = 0.5
    w = oracle.dequant_block(oracle.Q4_K, blk)
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == -0.5 * g["mins"][j])


# ---------------------------------------------------------------------- Q6_K

def q6k_block(d=0x3C00, sc=None, ql=None, qh=None):
    b = np.zeros(210, np.uint8)
    b[0:128] = np.array(ql if ql is not None else [0] * 128, np.uint8)
    b[128:192] = np.array(qh if qh is not None else [0xAA] * 64, np.uint8)
    b[192:208] = np.array(sc if sc is not None else [1] * 16, np.int8).view(np.uint8)
    b[208:210] = np.array([d & 0xFF, d >> 8], np.uint8)
    return b


def test_q6k_block_size():
    assert oracle.BLOCK_BYTES[oracle.Q6_K] == 210 == gold("q6k_layout.json")["block_bytes"]
    assert synth.q6k_weights(2, 768).size == 2 * 3 * 210


def test_q6k_neutral_code_is_zero():
    rng = np.random.default_rng(2)
    sc = rng.integers(-32, 32, 16)
    w = oracle.dequant_block(oracle.Q6_K, q6k_block(sc=sc))
    assert np.all(w == 0.0)


def test_q6k_ql_index_golden():
    g = gold("q6k_layout.json")
    for probe in g["ql_nibble_to_index"]:
        ql = [0] * 128
        ql[probe["byte"]] = 5 if probe["nibble"] == "low" else 5 << 4
        w = oracle.dequant_block(oracle.Q6_K, q6k_block(ql=ql))
        assert np.nonzero(w)[0].tolist() == [probe["index"]] and w[probe["index"]] == 5.0


def test_q6k_qh_and_scale_golden():
    g = gold("q6k_layout.json")
    p = g["qh_probe"]
    qh = [0xAA] * 64
    qh[p["byte"]] = int(p["value"], 16)
    w = oracle.dequant_block(oracle.Q6_K, q6k_block(qh=qh))
    assert np.nonzero(w)[0].tolist() == [p["index"]] and w[p["index"]] == p["weight"]
    s = g["scale_probe"]
    sc = [1] * 16
    sc[s["scale_index"]] = s["scale"]
    # every code 33 (ql nibble 1, high bits 0b10): w = d * sc
    w = oracle.dequant_block(oracle.Q6_K, q6k_block(sc=sc, ql=[0x11] * 128))
    lo, hi = s["indices"]
    assert np.all(w[lo:hi + 1] == s["scale"])
    mask = np.ones(256, bool)
    mask[lo:hi + 1] = False
    assert np.all(w[mask] == 1.0)


@pytest.mark.parametrize("direction", ["raise", "lower"])
def test_q6k_qh_every_pair_golden(direction):
    # every qh bit pair, in both halves and both 16-value scale groups: one pair moved off the neutral
    # 0b10 must change exactly the value the hand-derived table names, by 16 (or -16) times d * sc of
    # the named scale (distinct scales 1..16, so a wrong scale index shows too)
    g = gold("q6k_layout.json")
    sc = list(range(1, 17))
    pairs = set()
    for p in g["qh_pair_probes"]:
        t = p["pair"]
        qh = [0xAA] * 64
        if direction == "raise":
            qh[p["byte"]] = 0xAA | (1 << (2 * t))                           # 0b10 -> 0b11: code 48
        else:
            qh[p["byte"]] = (0xAA & ~(3 << (2 * t))) | (1 << (2 * t))       # 0b10 -> 0b01: code 16
        w = oracle.dequant_block(oracle.Q6_K, q6k_block(sc=sc, qh=qh))
        want = (16.0 if direction == "raise" else -16.0) * sc[p["scale_index"]]
        assert np.nonzero(w)[0].tolist() == [p["index"]], p
        assert w[p["index"]] == want, p
        pairs.add((p["byte"] // 32, p["byte"] % 32 >= 16, t))
    assert len(pairs) == 16                       # 2 halves x 2 scale groups x 4 bit pairs


def _q6k_int_matrix_numpy(w, N, K):
    """Integer weights q - 32 of unit-scale Q6_K rows, rebuilt with numpy from the GGUF planes:
    value 128h + 32t + l takes ql[64h + 32(t % 2) + l] (low nibble for t < 2, high for t >= 2)
    and bits 2t, 2t+1 of qh[32h + l]."""
    blk = w.reshape(N, K // 256, 210).astype(np.int64)
    ql, qh = blk[:, :, 0:128], blk[:, :, 128:192]
    parts = []
    for h in range(2):
        for t in range(4):
            lo = ql[:, :, 64 * h + 32 * (t % 2):64 * h + 32 * (t % 2) + 32]
            nib = (lo >> 4) if t >= 2 else (lo & 15)
            hb = (qh[:, :, 32 * h:32 * h + 32] >> (2 * t)) & 3
            parts.append((nib | (hb << 4)) - 32)
    return np.concatenate(parts, axis=2).reshape(N, K)


def test_q6k_contraction_integer_case_vs_numpy():
    # d = 1 and every sc = 1: w = q - 32 (integers), so y is an exact integer matmul
    rng = np.random.default_rng(14)
    N, K, M = 5, 768, 3
    w = np.concatenate([q6k_block(sc=[1] * 16, ql=rng.integers(0, 256, 128), qh=rng.integers(0, 256, 64))
                        for _ in range(N * K // 256)])
    codes = rng.integers(-127, 128, (M, K)).astype(np.int8)
    d_a = np.full((M, K // 32), 0x3C00, np.uint16)
    y, ab = oracle.gemm(oracle.Q6_K, w, N, K, codes, d_a)
    Wi = _q6k_int_matrix_numpy(w, N, K)
    assert np.array_equal(y, (codes.astype(np.int64) @ Wi.T).astype(np.float64))
    assert np.array_equal(ab, (np.abs(codes.astype(np.int64)) @ np.abs(Wi).T).astype(np.float64))


def test_q6k_code_range_and_sign():
    # all bits set -> code 63 -> 31; all clear -> -32; negative scale flips sign
    w = oracle.dequant_block(oracle.Q6_K, q6k_block(ql=[0xFF] * 128, qh=[0xFF] * 64, sc=[-2] * 16))
    assert np.all(w == -62.0)
    w = oracle.dequant_block(oracle.Q6_K, q6k_block(ql=[0] * 128, qh=[0] * 64, sc=[3] * 16, d=0x3800))
    assert np.all(w == -48.0)


# --------------------------------------------------------------- contraction

def _unit_q4k_matrix(N, K, rng):
    blocks = []
    for _ in range(N * K // 256):
        blocks.append(q4k_block(scales=[1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], qs=rng.integers(0, 256, 128)))
    return np.concatenate(blocks)


def test_contraction_integer_case_vs_numpy():
    rng = np.random.default_rng(4)
    N, K, M = 6, 512, 3
    w = _unit_q4k_matrix(N, K, rng)
    codes = rng.integers(-127, 128, (M, K)).astype(np.int8)
    d_a = np.full((M, K // 32), 0x3C00, np.uint16)
    y, ab = oracle.gemm(oracle.Q4_K, w, N, K, codes, d_a)
    # w = raw codes: rebuild the integer matrix from the nibbles (layout of the golden file)
    qs = w.reshape(N, K // 256, 144)[:, :, 16:].astype(np.int64)
    Wi = np.concatenate([np.concatenate([qs[:, b, 32 * g:32 * g + 32] & 15, qs[:, b, 32 * g:32 * g + 32] >> 4], axis=1)
                         for b in range(K // 256) for g in range(4)], axis=1)
    want = codes.astype(np.int64) @ Wi.T
    assert np.array_equal(y, want.astype(np.float64))
    assert np.array_equal(ab, (np.abs(codes.astype(np.int64)) @ Wi.T).astype(np.float64))


def test_contraction_min_only_closed_form():
    # d = 0, dmin = 1, all m_j = 1: w = -1 everywhere, y = -sum(xhat)
    N, K, M = 3, 256, 2
    scales = [0, 0, 0, 0, 1, 1, 1, 1, 0x10, 0x10, 0x10, 0x10]   # m_j = 1 for all j, sc_j = 0
    blk = q4k_block(d=0, dmin=0x3C00, scales=scales, qs=np.arange(128))
    w = np.concatenate([blk] * N)
    rng = np.random.default_rng(9)
    codes = rng.integers(-127, 128, (M, K)).astype(np.int8)
    d_a = np.full((M, K // 32), 0x3800, np.uint16)  # 0.5
    y, _ = oracle.gemm(oracle.Q4_K, w, N, K, codes, d_a)
    want = -0.5 * codes.astype(np.float64).sum(axis=1)
    assert np.array_equal(y, np.repeat(want[:, None], N, axis=1))


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_contraction_zero_activation_gives_residual(qt):
    N, K, M = 5, 512, 3
    w = synth.weights(qt, N, K, seed=1)
    r = synth.residual(M, N, seed=1)
    codes = np.zeros((M, K), np.int8)
    d_a = np.zeros((M, K // 32), np.uint16)
    y, ab = oracle.gemm(oracle.Q4_K if qt == "q4k" else oracle.Q6_K, w, N, K, codes, d_a, residual=r)
    assert np.array_equal(y, r.astype(np.float64)) and np.all(ab == 0)


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_contraction_one_hot_is_a_column(qt):
    qtype = oracle.Q4_K if qt == "q4k" else oracle.Q6_K
    N, K = 7, 768
    w = synth.weights(qt, N, K, seed=2)
    W = oracle.dequant_matrix(qtype, w, N, K)
    for k in (0, 31, 32, 255, 256, 700, 767):
        codes = np.zeros((1, K), np.int8)
        codes[0, k] = 127
        d_a = np.full((1, K // 32), 0x3C00, np.uint16)
        y, _ = oracle.gemm(qtype, w, N, K, codes, d_a)
        assert np.array_equal(y[0], 127.0 * W[:, k])


@pytest.mark.parametrize("qt", ["q4k", "q6k"])
def test_contraction_linearity_and_brute_force(qt):
    qtype = oracle.Q4_K if qt == "q4k" else oracle.Q6_K
    rng = np.random.default_rng(12)
    N, K, M = 8, 512, 5
    w = synth.weights(qt, N, K, seed=3)
    c1 = rng.integers(-60, 61, (M, K)).astype(np.int8)
    c2 = rng.integers(-60, 61, (M, K)).astype(np.int8)
    d_a = rng.choice(np.array([0x3C00, 0x3800, 0x2C00, 0x4000], np.uint16), (M, K // 32))
    y1, _ = oracle.gemm(qtype, w, N, K, c1, d_a)
    y2, _ = oracle.gemm(qtype, w, N, K, c2, d_a)
    y12, _ = oracle.gemm(qtype, w, N, K, (c1.astype(np.int16) + c2).astype(np.int8), d_a)
    assert np.allclose(y12, y1 + y2, rtol=1e-12, atol=1e-12)
    # dense binary64 product with the weights dequantized by this test's own loops (not the oracle's
    # dequantizer; numpy's float16 decode and matmul are the library steps)
    W = _dense_dequant(qt, w, N, K)
    xhat = np.repeat(d_a.view(np.float16).astype(np.float64), 32, axis=1) * c1
    assert np.allclose(y1, xhat @ W.T, rtol=1e-12, atol=1e-12)


def _f16(b0, b1):
    return float(np.array([b0 | (b1 << 8)], np.uint16).view(np.float16)[0])


def _dense_dequant(qt, w, N, K):
    """A second dequantizer, written separately from the oracle's, straight from the GGUF field
    layout: Q4_K d, dmin, 12 scale bytes (6-bit sc/m), 128 code bytes whose group g holds sub-block
    2g in its low nibbles and 2g + 1 in its high nibbles; Q6_K ql[128], qh[64], int8 sc[16], d."""
    out = np.zeros((N, K))
    bs = 144 if qt == "q4k" else 210
    for n in range(N):
        for b in range(K // 256):
            blk = [int(v) for v in w[(n * (K // 256) + b) * bs:(n * (K // 256) + b + 1) * bs]]
            vals = [0.0] * 256
            if qt == "q4k":
                d, dmin, S = _f16(blk[0], blk[1]), _f16(blk[2], blk[3]), blk[4:16]
                for j in range(8):
                    if j < 4:
                        sc, m = S[j] & 63, S[j + 4] & 63
                    else:
                        sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4)
                        m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4)
                    g, hi = j // 2, j % 2
                    for l in range(32):
                        byte = blk[16 + 32 * g + l]
                        q = (byte >> 4) if hi else (byte & 15)
                        vals[32 * j + l] = d * sc * q - dmin * m
            else:
                ql, qh = blk[0:128], blk[128:192]
                sc = [v - 256 if v > 127 else v for v in blk[192:208]]
                d = _f16(blk[208], blk[209])
                for v in range(256):
                    h, r = divmod(v, 128)
                    t, l = divmod(r, 32)
                    lo = ql[64 * h + 32 * (t % 2) + l]
                    nib = (lo >> 4) if t >= 2 else (lo & 15)
                    q = (nib | (((qh[32 * h + l] >> (2 * t)) & 3) << 4)) - 32
                    vals[v] = d * sc[8 * h + 2 * t + l // 16] * q
            out[n, 256 * b:256 * b + 256] = vals
    return out


def test_contraction_row_slices_and_threads_agree():
    N, K, M = 37, 1024, 2
    w = synth.q4k_weights(N, K, seed=5)
    x = synth.activations(M, K, seed=5)
    codes, d, _ = oracle.quantize_q8_1(x)
    y, ab = oracle.gemm(oracle.Q4_K, w, N, K, codes, d)
    y2, ab2 = oracle.gemm(oracle.Q4_K, w, N, K, codes, d, threads=4)
    ys, _ = oracle.gemm(oracle.Q4_K, w, N, K, codes, d, rows=(10, 20))
    assert np.array_equal(y, y2) and np.array_equal(ab, ab2)
    assert np.array_equal(ys, y[:, 10:20])
