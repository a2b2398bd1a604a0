"""The f16 operand forms of the tensor-core contraction, checked on the host.

The MMQ kernels feed the tensor cores binary16 operands and rest their error bound on
how those are formed (the header's MMQ contract):
  - the activation d_a * q_a as A_hi + A_lo, exactly;
  - the Q4_K weight operand sc * q (6-bit scale, 4-bit code) as one f16, built from the
    16-bit lane 0x6400 + q (the f16 1024 + q) by one fused multiply-add with sc and
    -1024 * sc;
  - the Q4_K min operand 1024 * dmin * m as Mw_hi (the binary32 value with its 13 low
    mantissa bits cleared) + Mw_lo (the rest), exactly wherever the rest's last bit is
    an f16 number;
  - the sub-block sum S = d_a * sum(q_a) / 16 as S_hi + S_lo, to 2^-22 relative.
Each form is restated here in numpy from the IEEE formats (binary16 arithmetic rounded
to nearest even, as the conversions the kernels use) and checked exhaustively or over
every binary16 scale.
"""
import numpy as np


def all_f16(nonneg=True):
    """every finite binary16 value (>= 0 when nonneg)"""
    b = np.arange(0, 0x7C00, dtype=np.uint16)           # +0 ... largest finite
    v = b.view(np.float16)
    return v if nonneg else np.concatenate([v, -v[1:]])


def test_activation_split_is_exact():
    # A_hi = f16(d q) rounded, A_lo = f16(d q - A_hi): d q has at most 11 + 7 significant bits and
    # its last bit is a multiple of d's, so the rest is an f16 number; A_hi + A_lo == d q
    d = all_f16().astype(np.float64)
    for q in range(-127, 128):
        p = d * q                                         # exact in binary64
        ok = np.abs(p) <= 65504.0                         # the value limit (|x| per block)
        hi = p[ok].astype(np.float16).astype(np.float64)
        lo = (p[ok] - hi).astype(np.float16).astype(np.float64)
        assert np.array_equal(hi + lo, p[ok]), q


def test_q4k_weight_operand_bit_construction():
    # every (sc, q): the lane 0x6400 + sc q stays below 0x8000 (no carry into the next lane), is
    # the f16 1024 + sc q, and subtracting 1024 in binary16 leaves sc q exactly
    sc = np.arange(64, dtype=np.uint32)[:, None]
    q = np.arange(16, dtype=np.uint32)[None, :]
    lane = 0x6400 + sc * q
    assert lane.max() < 0x8000 and (sc * q).max() == 945 < 1024
    v = lane.astype(np.uint16).view(np.float16)
    assert np.array_equal(v.astype(np.float64), 1024.0 + (sc * q).astype(np.float64))
    w = (v - np.float16(1024.0)).astype(np.float64)
    assert np.array_equal(w, (sc * q).astype(np.float64))
    # two lanes packed in one 32-bit word times sc: the high lane is unaffected by the low one
    word = (q[:, :, None] | (q[:, None, :] << 16)).astype(np.uint64)      # [1, 16, 16]
    prod = word * sc[:, :, None] + 0x64006400
    assert np.all((prod >> 16) == 0x6400 + sc[:, :, None] * q[:, None, :])
    assert np.all((prod & 0xFFFF) == 0x6400 + sc[:, :, None] * q[:, :, None])


def test_q4k_weight_operand_fma():
    # every (sc, q): 0x6400 | q is the f16 1024 + q; sc and -1024 sc are f16 numbers; the exact
    # (1024 + q) sc - 1024 sc = sc q (below 1024) is an f16 number, so the one rounding of a fused
    # multiply-add in binary16 leaves it unchanged
    sc = np.arange(64, dtype=np.int64)[:, None]
    q = np.arange(16, dtype=np.int64)[None, :]
    a = (0x6400 | q).astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(a, 1024.0 + q)
    s16 = sc.astype(np.float16)
    n16 = (s16.astype(np.float64) * -1024.0).astype(np.float16)
    assert np.array_equal(s16.astype(np.float64), sc.astype(np.float64))
    assert np.array_equal(n16.astype(np.float64), -1024.0 * sc)
    exact = a * s16.astype(np.float64) + n16.astype(np.float64)            # exact in binary64
    assert np.array_equal(exact, (sc * q).astype(np.float64))
    assert np.array_equal(exact.astype(np.float16).astype(np.float64), exact)
    assert np.abs(a * s16.astype(np.float64)).max() < 65504.0            # no overflow on the way


def split_hi_lo_f32(w32):
    """binary32 w -> (hi, lo) as the kernels form them: hi = w with the 13 low mantissa bits
    cleared, lo = w - hi in binary32; both then converted to binary16"""
    hi32 = (w32.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    lo32 = (w32 - hi32).astype(np.float32)
    return hi32.astype(np.float16), lo32.astype(np.float16), hi32, lo32


def test_q4k_min_operand_split():
    # Mw' = 1024 dmin m for every binary16 dmin >= 0 and m in 0..63 inside the operand limit
    dmin = all_f16().astype(np.float32)
    for m in range(64):
        w = (dmin * np.float32(m)) * np.float32(1024.0)          # 11 x 6 bits, then a power of two
        ok = w < 65504.0
        w = w[ok]
        assert np.array_equal(w.astype(np.float64), dmin[ok].astype(np.float64) * m * 1024.0)
        hi, lo, hi32, lo32 = split_hi_lo_f32(w)
        assert np.array_equal(hi.astype(np.float32), hi32)      # hi is an f16 number
        err = np.abs(hi.astype(np.float64) + lo.astype(np.float64) - w.astype(np.float64))
        # exact where the rest's lowest possible bit (w's last bit, 2^(e-16)) is >= 2^-24,
        # i.e. w >= 2^-8; below, within half an f16 subnormal step
        big = w >= 2.0 ** -8
        assert np.all(err[big] == 0), m
        assert np.all(err[~big] <= 2.0 ** -25), m


def test_sub_block_sum_split():
    # S' = d_a sum(q_a) / 16 for every binary16 d_a and a spread of sums (all of -4064..4064 for
    # a sample of scales): S_hi = f16(S'), S_lo = f16(S' - S_hi) is within 2^-22 |S'| plus half a
    # subnormal step
    d = all_f16().astype(np.float64)
    sums = np.unique(np.concatenate([np.arange(-64, 65), np.arange(-4064, 4065, 127), [4063, 4064, -4064]]))
    rng = np.random.default_rng(3)
    d_sample = rng.choice(d, 512, replace=False)
    for dd, ss in ((d, sums), (d_sample, np.arange(-4064, 4065))):
        S = (dd[:, None] * ss[None, :]) / 16.0               # exact in binary64 and in binary32
        ok = np.abs(S) < 65504.0
        S = S[ok]
        assert np.array_equal(S.astype(np.float32).astype(np.float64), S)
        hi = S.astype(np.float16).astype(np.float64)
        lo = (S.astype(np.float32) - hi.astype(np.float32)).astype(np.float16).astype(np.float64)
        err = np.abs(hi + lo - S)
        assert np.all(err <= 2.0 ** -22 * np.abs(S) + 2.0 ** -25)
