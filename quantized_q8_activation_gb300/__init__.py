"""Python binding of the GB300 k-quant x q8_1 contraction library (libqk.so).

Argument marshalling only: every computation runs in the CUDA kernels behind
the C ABI declared in include/qk.h.  PyTorch provides device memory and
streams.  There is no CPU fallback: if the shared library is missing or a
call fails, an exception is raised.

The C entry points allocate nothing.  These wrappers do, for convenience:
an output (or q8_1 buffer) that is not passed in is allocated with torch, and
mmq_q4k / mmq_q6k allocate their workspace with torch when none is given
(pass `workspace=` to keep a steady-state loop free of allocations, or use
mmq_q4k_noalloc).  Each call runs with the device of its tensors current, so
the library's per-device set-up and launches go to that device.

Typical use::

    import quantized_q8_activation_gb300 as qk
    w = qk.repack(qk.Q4_K, gguf_bytes_on_device, N, K)      # once, at load
    codes, scales = qk.quantize_q8_1(x)                      # x: float32 [M][K] on cuda
    codes, scales = qk.rmsnorm_q8_1(x, g, 1e-5)              # or fused into the producer
    y = qk.gemv_q4k(w, codes, scales, N, K, residual=r)      # M <= 8
    y = qk.mmq_q4k(w, codes, scales, N, K)                   # any M
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

Q4_K = 1
Q6_K = 2
Q5_K = 3
Q8_0 = 4
Q2_K = 5
Q3_K = 6
LAUNCH_PDL = 1
MMQ_TILE_256 = 2
MMQ_TILE_128 = 4
MMQ_TILE_192 = 8
MMQ_SPLIT_K = 16
GEMV_ROWS4 = 32
GEMV_ROWS2 = 64

ERR_TIMEOUT = 1     # error_flags(): a bounded in-kernel wait gave up
ERR_RANGE = 2       # error_flags(): an MMQ input was outside the value limits (see include/qk.h)

QK_OK = 0
STATUS = {0: "QK_OK", -1: "QK_E_NULL", -2: "QK_E_SHAPE", -3: "QK_E_ALIGN", -4: "QK_E_ALIAS",
          -5: "QK_E_TYPE", -6: "QK_E_WORKSPACE", -7: "QK_E_CUDA"}

# every symbol include/qk.h declares
EXPORTS = ["qk_version", "qk_status_string", "qk_q8_1_bytes", "qk_quantize_q8_1", "qk_repacked_bytes",
           "qk_repack", "qk_gemv_q4k", "qk_gemv_q6k", "qk_gemv_q5k", "qk_gemv_q4k_f32", "qk_gemv_q6k_f32",
           "qk_gemv_q5k_f32", "qk_gemv_q8_0", "qk_gemv_q8_0_f32", "qk_gemv_q2k", "qk_gemv_q3k",
           "qk_gemv_q2k_f32", "qk_gemv_q3k_f32",
           "qk_mmq_workspace_bytes", "qk_mmq_q4k", "qk_mmq_q6k", "qk_mmq_q4k_noalloc", "qk_error_flags",
           "qk_q4k_min_plane_bytes", "qk_q4k_min_plane", "qk_mmq_q4k_plane", "qk_mmq_q4k_f32", "qk_mmq_q6k_f32",
           "qk_rmsnorm_q8_1", "qk_swiglu_q8_1",
           # include/qk_peak.h (measurement)
           "qk_peak_mma_s8", "qk_peak_tcgen05_f16"]

_lib = None
_lock = threading.Lock()


class QKError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    """Compile libqk.so for sm_103a (nvcc)."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libqk.so not built ({path}); call quantized_q8_activation_gb300.build()")
            L = ctypes.CDLL(path)
            i64, p, u = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint
            szp = ctypes.POINTER(ctypes.c_size_t)
            L.qk_version.restype = ctypes.c_int
            L.qk_status_string.argtypes = [ctypes.c_int]
            L.qk_status_string.restype = ctypes.c_char_p
            L.qk_q8_1_bytes.argtypes = [i64, i64, szp, szp]
            L.qk_quantize_q8_1.argtypes = [p, i64, i64, i64, p, p, u, p]
            L.qk_repacked_bytes.argtypes = [ctypes.c_int, i64, i64, szp]
            L.qk_repack.argtypes = [ctypes.c_int, p, i64, i64, p, p]
            L.qk_gemv_q4k.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_gemv_q6k.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_gemv_q5k.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_gemv_q8_0.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_gemv_q2k.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_gemv_q3k.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_gemv_q4k_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, p, u, p]
            L.qk_gemv_q6k_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, p, u, p]
            L.qk_gemv_q5k_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, p, u, p]
            L.qk_gemv_q8_0_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, p, u, p]
            L.qk_gemv_q2k_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, p, u, p]
            L.qk_gemv_q3k_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, p, u, p]
            L.qk_mmq_workspace_bytes.argtypes = [i64, i64, i64, szp]
            L.qk_mmq_q4k.argtypes = [p, p, p, i64, i64, i64, p, p, p, ctypes.c_size_t, u, p]
            L.qk_mmq_q6k.argtypes = [p, p, p, i64, i64, i64, p, p, p, ctypes.c_size_t, u, p]
            L.qk_q4k_min_plane_bytes.argtypes = [i64, i64, szp]
            L.qk_q4k_min_plane.argtypes = [p, i64, i64, p, ctypes.c_size_t, p]
            L.qk_mmq_q4k_plane.argtypes = [p, p, p, p, i64, i64, i64, p, p, p, ctypes.c_size_t, u, p]
            L.qk_mmq_q4k_f32.argtypes = [p, p, p, i64, i64, i64, i64, p, p, p, ctypes.c_size_t, u, p]
            L.qk_mmq_q6k_f32.argtypes = [p, p, i64, i64, i64, i64, p, p, p, ctypes.c_size_t, u, p]
            L.qk_rmsnorm_q8_1.argtypes = [p, i64, p, p, ctypes.c_float, i64, i64, p, p, p, p, u, p]
            L.qk_swiglu_q8_1.argtypes = [p, i64, i64, i64, p, p, p, u, p]
            L.qk_mmq_q4k_noalloc.argtypes = [p, p, p, i64, i64, i64, p, p, u, p]
            L.qk_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
            dp = ctypes.POINTER(ctypes.c_double)
            L.qk_peak_mma_s8.argtypes = [i64, ctypes.c_int, dp, dp, p]
            L.qk_peak_tcgen05_f16.argtypes = [i64, ctypes.c_int, dp, dp, p]
            for name in EXPORTS:
                getattr(L, name).restype = ctypes.c_int if name != "qk_status_string" else ctypes.c_char_p
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().qk_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != QK_OK:
        raise QKError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on(t: torch.Tensor):
    """Make t's device the current CUDA device for the call (the C ABI works on the current device)."""
    return torch.cuda.device(t.device)


# ------------------------------------------------------------------- sizes

def q8_1_bytes(M: int, K: int) -> tuple[int, int]:
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().qk_q8_1_bytes(M, K, ctypes.byref(c), ctypes.byref(s)), "qk_q8_1_bytes")
    return c.value, s.value


def repacked_bytes(qtype: int, N: int, K: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().qk_repacked_bytes(qtype, N, K, ctypes.byref(b)), "qk_repacked_bytes")
    return b.value


def mmq_workspace_bytes(M: int, N: int, K: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().qk_mmq_workspace_bytes(M, N, K, ctypes.byref(b)), "qk_mmq_workspace_bytes")
    return b.value


def error_flags(clear: bool = True) -> int:
    """Device error word (ERR_TIMEOUT: a bounded in-kernel wait gave up; ERR_RANGE: an MMQ input
    outside the value limits); cleared when `clear`."""
    f = ctypes.c_uint()
    _check(lib().qk_error_flags(ctypes.byref(f), int(clear)), "qk_error_flags")
    return f.value


# --------------------------------------------------------------- operations

def empty_q8_1(M: int, K: int, device="cuda"):
    """Uninitialised q8_1 buffers: codes int8 [M][K], scales float16 [M][K/32][2] (d, s)."""
    return (torch.empty((M, K), dtype=torch.int8, device=device),
            torch.empty((M, K // 32, 2), dtype=torch.float16, device=device))


def quantize_q8_1(x: torch.Tensor, codes=None, scales=None, pdl: bool = False, stream=None):
    """x: float32 [M][K] (rows may be strided) -> (codes, scales)."""
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dtype != torch.float32 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a float32 CUDA tensor with unit stride along K")
    M, K = x.shape
    if codes is None or scales is None:
        codes, scales = empty_q8_1(M, K, x.device)
    _cuda(codes, "codes"), _cuda(scales, "scales")
    with _on(x):
        st = lib().qk_quantize_q8_1(x.data_ptr(), x.stride(0) if M > 1 else K, M, K, codes.data_ptr(),
                                    scales.data_ptr(), LAUNCH_PDL if pdl else 0, _stream(stream))
    _check(st, "qk_quantize_q8_1")
    return codes, scales


def rmsnorm_q8_1(x: torch.Tensor, g: torch.Tensor, eps: float, r=None, h_out=None, y=None, codes=None,
                 scales=None, pdl: bool = False, stream=None):
    """RMSNorm of x (+ r) with weight g, written as q8_1 (and, when y / h_out are given, as f32).
    Returns (codes, scales)."""
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dtype != torch.float32 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a float32 CUDA tensor with unit stride along K")
    M, K = x.shape
    _cuda(g, "g")
    for t, n in ((r, "r"), (h_out, "h_out"), (y, "y")):
        if t is not None:
            _cuda(t, n)
    if codes is None or scales is None:
        codes, scales = empty_q8_1(M, K, x.device)
    _cuda(codes, "codes"), _cuda(scales, "scales")
    with _on(x):
        st = lib().qk_rmsnorm_q8_1(x.data_ptr(), x.stride(0) if M > 1 else K, _p(r), g.data_ptr(), float(eps), M,
                                   K, _p(h_out), _p(y), codes.data_ptr(), scales.data_ptr(),
                                   LAUNCH_PDL if pdl else 0, _stream(stream))
    _check(st, "qk_rmsnorm_q8_1")
    return codes, scales


def swiglu_q8_1(gu: torch.Tensor, F: int, h=None, codes=None, scales=None, pdl: bool = False, stream=None):
    """silu(gate) * up of a gate||up row block gu [M][>= 2F] (gate first), written as q8_1 (and as
    f32 into h when given).  Returns (codes, scales)."""
    if gu.dim() == 1:
        gu = gu.view(1, -1)
    if gu.dtype != torch.float32 or not gu.is_cuda or gu.stride(1) != 1:
        raise ValueError("gu must be a float32 CUDA tensor with unit stride along its rows")
    M = gu.shape[0]
    if h is not None:
        _cuda(h, "h")
    if codes is None or scales is None:
        codes, scales = empty_q8_1(M, F, gu.device)
    _cuda(codes, "codes"), _cuda(scales, "scales")
    with _on(gu):
        st = lib().qk_swiglu_q8_1(gu.data_ptr(), gu.stride(0) if M > 1 else gu.shape[1], M, F, _p(h),
                                  codes.data_ptr(), scales.data_ptr(), LAUNCH_PDL if pdl else 0, _stream(stream))
    _check(st, "qk_swiglu_q8_1")
    return codes, scales


def repack(qtype: int, gguf: torch.Tensor, N: int, K: int, out=None, stream=None) -> torch.Tensor:
    """GGUF superblocks (uint8 CUDA tensor) -> repacked device weight (uint8)."""
    _cuda(gguf, "gguf")
    nbytes = repacked_bytes(qtype, N, K)
    gguf_bytes = N * (K // 256) * 110 if qtype == Q3_K else nbytes
    if gguf.numel() * gguf.element_size() < gguf_bytes:
        raise ValueError("gguf buffer smaller than N*K/256 superblocks")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=gguf.device)
    _cuda(out, "out")
    with _on(gguf):
        _check(lib().qk_repack(qtype, gguf.data_ptr(), N, K, out.data_ptr(), _stream(stream)), "qk_repack")
    return out


def _rows_flag(rows):
    return {None: 0, 2: GEMV_ROWS2, 4: GEMV_ROWS4}[rows]


def _gemv(fn, name, w, codes, scales, N, K, residual, y, pdl, stream, rows=None, flags=0):
    M = codes.shape[0]
    for t, n in ((w, "w"), (codes, "codes"), (scales, "scales")):
        _cuda(t, n)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=codes.device)
    _cuda(y, "y")
    if residual is not None:
        _cuda(residual, "residual")
    with _on(codes):
        st = fn(w.data_ptr(), codes.data_ptr(), scales.data_ptr(), M, N, K, _p(residual), y.data_ptr(),
                (LAUNCH_PDL if pdl else 0) | _rows_flag(rows) | flags, _stream(stream))
    _check(st, name)
    return y


def gemv_q4k(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None, rows=None, flags=0):
    """y[M][N] = xhat . W^T (+ residual) over a repacked Q4_K weight, 1 <= M <= 8.

    rows=4 / rows=2 force items of four or two weight rows (QK_GEMV_ROWS4 / QK_GEMV_ROWS2, M >= 3)."""
    return _gemv(lib().qk_gemv_q4k, "qk_gemv_q4k", w, codes, scales, N, K, residual, y, pdl, stream, rows, flags)


def gemv_q6k(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None, rows=None, flags=0):
    """y[M][N] = xhat . W^T (+ residual) over a repacked Q6_K weight, 1 <= M <= 8 (rows: as gemv_q4k)."""
    return _gemv(lib().qk_gemv_q6k, "qk_gemv_q6k", w, codes, scales, N, K, residual, y, pdl, stream, rows, flags)


def gemv_q5k(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None, flags=0):
    """GEMV over a repacked Q5_K weight, 1 <= M <= 8 activation rows."""
    return _gemv(lib().qk_gemv_q5k, "qk_gemv_q5k", w, codes, scales, N, K, residual, y, pdl, stream, None, flags)


def gemv_q8_0(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None, flags=0):
    """GEMV over a repacked Q8_0 weight, 1 <= M <= 8 activation rows."""
    return _gemv(lib().qk_gemv_q8_0, "qk_gemv_q8_0", w, codes, scales, N, K, residual, y, pdl, stream, None, flags)


def gemv_q2k(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None, flags=0):
    """GEMV over a repacked Q2_K weight, 1 <= M <= 8 activation rows."""
    return _gemv(lib().qk_gemv_q2k, "qk_gemv_q2k", w, codes, scales, N, K, residual, y, pdl, stream, None, flags)


def gemv_q3k(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None, flags=0):
    """GEMV over a repacked Q3_K weight, 1 <= M <= 8 activation rows."""
    return _gemv(lib().qk_gemv_q3k, "qk_gemv_q3k", w, codes, scales, N, K, residual, y, pdl, stream, None, flags)


def _gemv_f32(fn, name, w, x, N, K, residual, y, codes_out, scales_out, pdl, stream, rows=None, flags=0):
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.dtype != torch.float32 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a float32 CUDA tensor with unit stride along K")
    _cuda(w, "w")
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _cuda(y, "y")
    if residual is not None:
        _cuda(residual, "residual")
    with _on(x):
        st = fn(w.data_ptr(), x.data_ptr(), x.stride(0) if M > 1 else K, M, N, K, _p(residual), y.data_ptr(),
                _p(codes_out), _p(scales_out), (LAUNCH_PDL if pdl else 0) | _rows_flag(rows) | flags,
                _stream(stream))
    _check(st, name)
    return y


def gemv_q4k_f32(w, x, N, K, residual=None, y=None, codes_out=None, scales_out=None, pdl=False, stream=None,
                 rows=None, flags=0):
    """GEMV over a repacked Q4_K weight from f32 activations (quantized inside the kernel), 1 <= M <= 8."""
    return _gemv_f32(lib().qk_gemv_q4k_f32, "qk_gemv_q4k_f32", w, x, N, K, residual, y, codes_out, scales_out,
                     pdl, stream, rows, flags)


def gemv_q6k_f32(w, x, N, K, residual=None, y=None, codes_out=None, scales_out=None, pdl=False, stream=None,
                 rows=None, flags=0):
    """GEMV over a repacked Q6_K weight from f32 activations (quantized inside the kernel), 1 <= M <= 8."""
    return _gemv_f32(lib().qk_gemv_q6k_f32, "qk_gemv_q6k_f32", w, x, N, K, residual, y, codes_out, scales_out,
                     pdl, stream, rows, flags)


def gemv_q5k_f32(w, x, N, K, residual=None, y=None, codes_out=None, scales_out=None, pdl=False, stream=None,
                 rows=None, flags=0):
    """GEMV over a repacked Q5_K weight from f32 activations (quantized inside the kernel), 1 <= M <= 8."""
    return _gemv_f32(lib().qk_gemv_q5k_f32, "qk_gemv_q5k_f32", w, x, N, K, residual, y, codes_out, scales_out,
                     pdl, stream, rows, flags)


def gemv_q8_0_f32(w, x, N, K, residual=None, y=None, codes_out=None, scales_out=None, pdl=False, stream=None,
                  rows=None, flags=0):
    """GEMV over a repacked Q8_0 weight from f32 activations (quantized inside the kernel), 1 <= M <= 8."""
    return _gemv_f32(lib().qk_gemv_q8_0_f32, "qk_gemv_q8_0_f32", w, x, N, K, residual, y, codes_out, scales_out,
                     pdl, stream, rows, flags)


def gemv_q2k_f32(w, x, N, K, residual=None, y=None, codes_out=None, scales_out=None, pdl=False, stream=None,
                 rows=None, flags=0):
    """GEMV over a repacked Q2_K weight from f32 activations (quantized inside the kernel), 1 <= M <= 8."""
    return _gemv_f32(lib().qk_gemv_q2k_f32, "qk_gemv_q2k_f32", w, x, N, K, residual, y, codes_out, scales_out,
                     pdl, stream, rows, flags)


def gemv_q3k_f32(w, x, N, K, residual=None, y=None, codes_out=None, scales_out=None, pdl=False, stream=None,
                 rows=None, flags=0):
    """GEMV over a repacked Q3_K weight from f32 activations (quantized inside the kernel), 1 <= M <= 8."""
    return _gemv_f32(lib().qk_gemv_q3k_f32, "qk_gemv_q3k_f32", w, x, N, K, residual, y, codes_out, scales_out,
                     pdl, stream, rows, flags)


def mmq_q4k(w, codes, scales, N, K, residual=None, y=None, workspace=None, pdl=False, stream=None, tile=None,
            split_k=False):
    """Prefill contraction over a repacked Q4_K weight, any M.  tile: None (the library picks
    the tile width), 256, 192 or 128.  split_k: QK_MMQ_SPLIT_K (taken only if the workspace also
    holds the split scratch, include/qk.h).  workspace: a uint8 CUDA tensor of at least
    mmq_workspace_bytes(M, N, K) bytes; when None, this wrapper allocates one with torch."""
    return _mmq("qk_mmq_q4k", w, codes, scales, N, K, residual, y, workspace, pdl, stream, tile, split_k=split_k)


def mmq_q6k(w, codes, scales, N, K, residual=None, y=None, workspace=None, pdl=False, stream=None, tile=None):
    """Prefill contraction over a repacked Q6_K weight, any M (workspace as for mmq_q4k)."""
    return _mmq("qk_mmq_q6k", w, codes, scales, N, K, residual, y, workspace, pdl, stream, tile)


def q4k_min_plane_bytes(N: int, K: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().qk_q4k_min_plane_bytes(N, K, ctypes.byref(b)), "qk_q4k_min_plane_bytes")
    return b.value


def q4k_min_plane(w, N, K, plane=None, stream=None):
    """The load-time min-operand plane of a repacked Q4_K weight (qk_q4k_min_plane), for
    mmq_q4k_plane.  plane: a uint8 CUDA tensor of q4k_min_plane_bytes(N, K) bytes; when None,
    this wrapper allocates one with torch."""
    _cuda(w, "w")
    need = q4k_min_plane_bytes(N, K)
    if plane is None:
        plane = torch.empty(need, dtype=torch.uint8, device=w.device)
    _cuda(plane, "plane")
    with _on(w):
        st = lib().qk_q4k_min_plane(w.data_ptr(), N, K, plane.data_ptr(), plane.numel() * plane.element_size(),
                                    _stream(stream))
    _check(st, "qk_q4k_min_plane")
    return plane


def mmq_q4k_plane(w, plane, codes, scales, N, K, residual=None, y=None, workspace=None, pdl=False, stream=None,
                  tile=None, split_k=False):
    """mmq_q4k reading the min operands from a plane made by q4k_min_plane from the same weight
    (same result bit for bit; workspace as for mmq_q4k)."""
    _cuda(plane, "plane")
    return _mmq("qk_mmq_q4k_plane", w, codes, scales, N, K, residual, y, workspace, pdl, stream, tile, plane,
                split_k)


def mmq_q4k_f32(w, x, N, K, residual=None, y=None, workspace=None, plane=None, pdl=False, stream=None, tile=None,
                split_k=False):
    """mmq_q4k from the f32 activation x [M][K] (row pitch x.stride(0)): the q8_1 quantization is done
    inside the call, bit-identical to quantize_q8_1 + mmq_q4k (or mmq_q4k_plane with a plane)."""
    return _mmq_f32("qk_mmq_q4k_f32", w, x, N, K, residual, y, workspace, pdl, stream, tile, plane, split_k)


def mmq_q6k_f32(w, x, N, K, residual=None, y=None, workspace=None, pdl=False, stream=None, tile=None):
    """mmq_q6k from the f32 activation x [M][K] (quantized inside the call, as mmq_q4k_f32)."""
    return _mmq_f32("qk_mmq_q6k_f32", w, x, N, K, residual, y, workspace, pdl, stream, tile, None, False)


def _mmq_f32(fn, w, x, N, K, residual, y, workspace, pdl, stream, tile, plane, split_k):
    _cuda(w, "w")
    if x.dtype != torch.float32 or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a float32 [M][K] CUDA tensor with unit stride along K (rows may be strided)")
    if plane is not None:
        _cuda(plane, "plane")
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    need = mmq_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = (LAUNCH_PDL if pdl else 0) | {None: 0, 256: MMQ_TILE_256, 192: MMQ_TILE_192, 128: MMQ_TILE_128}[tile]
    flags |= MMQ_SPLIT_K if split_k else 0
    tail = (M, N, K, _p(residual), y.data_ptr(), _p(workspace), wsb, flags, _stream(stream))
    with _on(x):
        if fn == "qk_mmq_q4k_f32":
            st = lib().qk_mmq_q4k_f32(w.data_ptr(), _p(plane), x.data_ptr(), x.stride(0) if M > 1 else K, *tail)
        else:
            st = lib().qk_mmq_q6k_f32(w.data_ptr(), x.data_ptr(), x.stride(0) if M > 1 else K, *tail)
    _check(st, fn)
    return y


def _mmq(fn, w, codes, scales, N, K, residual, y, workspace, pdl, stream, tile=None, plane=None, split_k=False):
    M = codes.shape[0]
    for t, n in ((w, "w"), (codes, "codes"), (scales, "scales")):
        _cuda(t, n)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=codes.device)
    need = mmq_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=codes.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = (LAUNCH_PDL if pdl else 0) | {None: 0, 256: MMQ_TILE_256, 192: MMQ_TILE_192, 128: MMQ_TILE_128}[tile]
    flags |= MMQ_SPLIT_K if split_k else 0
    args = (codes.data_ptr(), scales.data_ptr(), M, N, K, _p(residual), y.data_ptr(), _p(workspace), wsb, flags,
            _stream(stream))
    with _on(codes):
        if plane is None:
            st = getattr(lib(), fn)(w.data_ptr(), *args)
        else:
            st = getattr(lib(), fn)(w.data_ptr(), plane.data_ptr(), *args)
    _check(st, fn)
    return y


STATIC_WS_BYTES = 32 << 20          # QK_MMQ_STATIC_WS_BYTES


def mmq_q4k_noalloc(w, codes, scales, N, K, residual=None, y=None, pdl=False, stream=None):
    """qk_mmq_q4k with the library's static workspace (no workspace argument; see qk.h)."""
    M = codes.shape[0]
    for t, n in ((w, "w"), (codes, "codes"), (scales, "scales")):
        _cuda(t, n)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=codes.device)
    with _on(codes):
        st = lib().qk_mmq_q4k_noalloc(w.data_ptr(), codes.data_ptr(), scales.data_ptr(), M, N, K, _p(residual),
                                      y.data_ptr(), LAUNCH_PDL if pdl else 0, _stream(stream))
    _check(st, "qk_mmq_q4k_noalloc")
    return y


# ------------------------------------------------------------- measurement

def _peak(fn, name, iters, reps, stream):
    rate, ms = ctypes.c_double(), ctypes.c_double()
    _check(fn(int(iters), int(reps), ctypes.byref(rate), ctypes.byref(ms), _stream(stream)), name)
    return rate.value, ms.value


def peak_mma_s8(iters: int = 20000, reps: int = 5, stream=None):
    """Measured mma.sync m16n8k32 s8 rate of the current device: (TOPS, milliseconds timed)."""
    return _peak(lib().qk_peak_mma_s8, "qk_peak_mma_s8", iters, reps, stream)


def peak_tcgen05_f16(iters: int = 4096, reps: int = 5, stream=None):
    """Measured tcgen05 kind::f16 (128 x 256 x 16) rate of the current device: (TFLOP/s, milliseconds)."""
    return _peak(lib().qk_peak_tcgen05_f16, "qk_peak_tcgen05_f16", iters, reps, stream)
