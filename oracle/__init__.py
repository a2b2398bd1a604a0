"""CPU oracle for the k-quant x q8_1 contraction (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never links it and this package never imports the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C99, binary64 contraction,
binary32 quantizer); this module only compiles it with gcc, loads it with
ctypes and moves numpy buffers in and out.  See ``oracle.c`` for what each
function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

Q4_K = 1
Q6_K = 2
Q5_K = 3
Q8_0 = 4
Q2_K = 5
Q3_K = 6
QK = 256
BLOCK_BYTES = {Q4_K: 144, Q6_K: 210, Q5_K: 176, Q8_0: 272, Q2_K: 84, Q3_K: 110}   # GGUF bytes per 256 values
DEVICE_BYTES = {**BLOCK_BYTES, Q3_K: 114}          # repacked bytes per 256 values (Q3_K scales unpacked)

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, no fused multiply-add)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f64.restype = ctypes.c_double
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_quantize_q8_1.argtypes = [p, i64, i64, i64, p, p, p]
            lib.orc_q4k_scale_min.argtypes = [p, ctypes.c_int, p, p]
            lib.orc_q4k_dequant.argtypes = [p, p]
            lib.orc_q6k_dequant.argtypes = [p, p]
            lib.orc_dequant_row.argtypes = [ctypes.c_int, p, i64, p]
            lib.orc_gemm_rows.argtypes = [ctypes.c_int, p, i64, i64, i64, i64, p, p, i64, p, p, p]
            lib.orc_repack_q4k.argtypes = [p, i64, i64, p]
            lib.orc_repack_q6k.argtypes = [p, i64, i64, p]
            lib.orc_repack_q5k.argtypes = [p, i64, i64, p]
            lib.orc_q5k_dequant.argtypes = [p, p]
            lib.orc_q80_dequant.argtypes = [p, p]
            lib.orc_repack_q80.argtypes = [p, i64, i64, p]
            lib.orc_q2k_dequant.argtypes = [p, p]
            lib.orc_q3k_dequant.argtypes = [p, p]
            lib.orc_q3k_scale.argtypes = [p, ctypes.c_int]
            lib.orc_repack_q2k.argtypes = [p, i64, i64, p]
            lib.orc_repack_q3k.argtypes = [p, i64, i64, p]
            lib.orc_rmsnorm.argtypes = [p, i64, p, p, ctypes.c_double, i64, i64, p, p]
            lib.orc_swiglu.argtypes = [p, i64, i64, i64, p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f64(h: int) -> float:
    return _load().orc_f16_to_f64(int(h))


def f32_to_f16(x: float) -> int:
    return int(_load().orc_f32_to_f16(float(np.float32(x))))


def quantize_q8_1(x: np.ndarray):
    """x: float32 [M][K] -> (codes int8 [M][K], d uint16 [M][K/32], s uint16 [M][K/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    codes = np.zeros((M, K), np.int8)
    d = np.zeros((M, K // 32), np.uint16)
    s = np.zeros((M, K // 32), np.uint16)
    rc = _load().orc_quantize_q8_1(_ptr(x), K, M, K, _ptr(codes), _ptr(d), _ptr(s))
    if rc != 0:
        raise ValueError(f"orc_quantize_q8_1 failed ({rc})")
    return codes, d, s


def q4k_scale_min(q12: bytes, j: int):
    buf = np.frombuffer(bytes(q12), np.uint8).copy()
    sc, mn = ctypes.c_int(), ctypes.c_int()
    _load().orc_q4k_scale_min(_ptr(buf), j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def dequant_block(qtype: int, blk) -> np.ndarray:
    b = np.frombuffer(bytes(blk), np.uint8).copy()
    assert b.size == BLOCK_BYTES[qtype]
    out = np.zeros(QK, np.float64)
    if qtype == Q4_K:
        _load().orc_q4k_dequant(_ptr(b), _ptr(out))
    elif qtype == Q5_K:
        _load().orc_q5k_dequant(_ptr(b), _ptr(out))
    elif qtype == Q8_0:
        _load().orc_q80_dequant(_ptr(b), _ptr(out))
    elif qtype == Q2_K:
        _load().orc_q2k_dequant(_ptr(b), _ptr(out))
    elif qtype == Q3_K:
        _load().orc_q3k_dequant(_ptr(b), _ptr(out))
    else:
        _load().orc_q6k_dequant(_ptr(b), _ptr(out))
    return out


def dequant_matrix(qtype: int, w: np.ndarray, N: int, K: int) -> np.ndarray:
    """GGUF bytes [N][K/256][bs] -> float64 [N][K]."""
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    rowbytes = (K // QK) * BLOCK_BYTES[qtype]
    out = np.zeros((N, K), np.float64)
    lib = _load()
    for n in range(N):
        row = w[n * rowbytes:(n + 1) * rowbytes]
        rc = lib.orc_dequant_row(qtype, _ptr(row), K, _ptr(out[n]))
        if rc != 0:
            raise ValueError("orc_dequant_row failed")
    return out


def gemm(qtype: int, w: np.ndarray, N: int, K: int, codes: np.ndarray, d_a: np.ndarray,
         residual: np.ndarray | None = None, rows=None, threads: int = 1):
    """Reference y (float64) and tolerance scale sum|w*xhat| for the selected rows.

    rows: None for all rows, else a (n0, n1) range.  Returns (y, absdot),
    each [M][n1-n0].  ``threads`` splits the row range over host threads
    (ctypes releases the GIL); every output is computed by the same C loop.
    """
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    d_a = np.ascontiguousarray(d_a, dtype=np.uint16)
    M = codes.shape[0]
    n0, n1 = (0, N) if rows is None else rows
    r = None if residual is None else np.ascontiguousarray(residual, dtype=np.float32)
    nn = n1 - n0
    y = np.zeros((M, nn), np.float64)
    ab = np.zeros((M, nn), np.float64)
    lib = _load()

    def run(a, b):
        ys = np.zeros((M, b - a), np.float64)
        abs_ = np.zeros((M, b - a), np.float64)
        rc = lib.orc_gemm_rows(qtype, _ptr(w), N, K, a, b, _ptr(codes), _ptr(d_a), M,
                               _ptr(r) if r is not None else None, _ptr(ys), _ptr(abs_))
        if rc != 0:
            raise ValueError(f"orc_gemm_rows failed ({rc})")
        y[:, a - n0:b - n0] = ys
        ab[:, a - n0:b - n0] = abs_

    if threads <= 1 or nn < 2 * threads:
        run(n0, n1)
    else:
        edges = np.linspace(n0, n1, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: run(int(edges[i]), int(edges[i + 1])), range(threads)))
    return y, ab


def repack(qtype: int, w: np.ndarray, N: int, K: int) -> np.ndarray:
    """Expected device layout (uint8, same byte count) for GGUF bytes w."""
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    out = np.zeros(N * (K // QK) * DEVICE_BYTES[qtype], np.uint8)
    fn = {Q4_K: _load().orc_repack_q4k, Q6_K: _load().orc_repack_q6k, Q5_K: _load().orc_repack_q5k,
          Q8_0: _load().orc_repack_q80, Q2_K: _load().orc_repack_q2k, Q3_K: _load().orc_repack_q3k}[qtype]
    if fn(_ptr(w), N, K, _ptr(out)) != 0:
        raise ValueError("orc_repack failed")
    return out


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float, r: np.ndarray | None = None):
    """RMSNorm of x (+ r): returns (y float64 [M][K], s float32 [M][K]) with s = x (+ r) in binary32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    g = np.ascontiguousarray(g, dtype=np.float32).reshape(K)
    rr = None if r is None else np.ascontiguousarray(r, dtype=np.float32).reshape(M, K)
    y = np.zeros((M, K), np.float64)
    s = np.zeros((M, K), np.float32)
    rc = _load().orc_rmsnorm(_ptr(x), K, None if rr is None else _ptr(rr), _ptr(g), float(eps), M, K, _ptr(s), _ptr(y))
    if rc != 0:
        raise ValueError(f"orc_rmsnorm failed ({rc})")
    return y, s


def swiglu(gu: np.ndarray, F: int) -> np.ndarray:
    """silu(gate) * up of gate||up rows gu [M][>= 2F] -> float64 [M][F]."""
    gu = np.ascontiguousarray(gu, dtype=np.float32)
    if gu.ndim == 1:
        gu = gu[None, :]
    M, ld = gu.shape
    h = np.zeros((M, F), np.float64)
    rc = _load().orc_swiglu(_ptr(gu), ld, M, F, _ptr(h))
    if rc != 0:
        raise ValueError(f"orc_swiglu failed ({rc})")
    return h


def q3k_scale(sc12, s: int) -> int:
    """Signed sub-block scale s (0..15) of a Q3_K superblock's 12 packed scale bytes."""
    b = np.frombuffer(bytes(sc12), np.uint8).copy()
    return int(_load().orc_q3k_scale(_ptr(b), s))
