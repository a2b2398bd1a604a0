"""Host-side tests of the C ABI (no GPU needed).

The library must load, export every function include/qk.h declares, and
reject bad arguments on the host with the documented status codes before
anything is launched.  No call here reaches a CUDA launch: fake device
pointers are only compared and never dereferenced.
"""
import ctypes
import os
import re

import pytest

import quantized_q8_activation_gb300 as qk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))

P = 0x7F0000000000          # fake, 256-byte aligned device addresses
E_NULL, E_SHAPE, E_ALIGN, E_ALIAS, E_TYPE = -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def L():
    qk.build()
    return qk.lib()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(qk_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_headers_found():
    assert [os.path.basename(h) for h in HEADERS] == ["qk.h", "qk_peak.h"]


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(qk.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.qk_version() >= 100
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        assert len(qk.status_string(st)) > 0
    assert qk.status_string(-99) == "unknown status"


def test_sizes(L):
    assert qk.q8_1_bytes(4, 4096) == (4 * 4096, 4 * 128 * 4)
    assert qk.repacked_bytes(qk.Q4_K, 4096, 4096) == 4096 * 16 * 144
    assert qk.repacked_bytes(qk.Q6_K, 128256, 4096) == 430940160
    assert qk.repacked_bytes(qk.Q5_K, 4096, 4096) == 4096 * 16 * 176
    assert qk.repacked_bytes(qk.Q8_0, 4096, 4096) == 4096 * 128 * 34
    assert qk.repacked_bytes(qk.Q2_K, 4096, 4096) == 4096 * 16 * 84
    assert qk.repacked_bytes(qk.Q3_K, 4096, 4096) == 4096 * 16 * 114
    with pytest.raises(qk.QKError):
        qk.repacked_bytes(qk.Q4_K, 10, 100)
    with pytest.raises(qk.QKError):
        qk.repacked_bytes(7, 10, 256)


def call_gemv(L, fn, w=P, codes=P + 0x10000000, scales=P + 0x20000000, M=1, N=64, K=256, r=None,
              y=P + 0x30000000):
    return getattr(L, fn)(w, codes, scales, M, N, K, r, y, 0, None)


@pytest.mark.parametrize("fn", ["qk_gemv_q4k", "qk_gemv_q5k", "qk_gemv_q6k", "qk_gemv_q8_0", "qk_gemv_q2k",
                                "qk_gemv_q3k"])
def test_gemv_rejects(L, fn):
    assert call_gemv(L, fn, w=None) == E_NULL
    assert call_gemv(L, fn, y=None) == E_NULL
    assert call_gemv(L, fn, K=100) == E_SHAPE
    assert call_gemv(L, fn, K=0) == E_SHAPE
    assert call_gemv(L, fn, M=0) == E_SHAPE
    assert call_gemv(L, fn, M=9) == E_SHAPE
    assert call_gemv(L, fn, N=0) == E_SHAPE
    kmax = {"qk_gemv_q4k": 40, "qk_gemv_q5k": 32, "qk_gemv_q6k": 20, "qk_gemv_q8_0": 32, "qk_gemv_q2k": 40,
            "qk_gemv_q3k": 40}[fn]                                  # 256-value units at M = 8
    assert call_gemv(L, fn, M=8, K=256 * (kmax + 1)) == E_SHAPE     # activation too large
    assert call_gemv(L, fn, M=8, K=256 * kmax, y=None) == E_NULL     # at the limit
    assert call_gemv(L, fn, w=P + 8) == E_ALIGN
    assert call_gemv(L, fn, codes=P + 0x10000004) == E_ALIGN
    assert call_gemv(L, fn, y=P + 0x30000002) == E_ALIGN
    assert call_gemv(L, fn, y=P + 64) == E_ALIAS                   # y inside the weight
    assert call_gemv(L, fn, r=P + 0x30000000 + 4) == E_ALIAS       # residual partially overlaps y


@pytest.mark.parametrize("fn", ["qk_gemv_q4k_f32", "qk_gemv_q5k_f32", "qk_gemv_q6k_f32", "qk_gemv_q8_0_f32",
                                "qk_gemv_q2k_f32", "qk_gemv_q3k_f32"])
def test_gemv_f32_rejects(L, fn):
    f = getattr(L, fn)
    w, x, y, c, s = P, P + 0x10000000, P + 0x30000000, P + 0x40000000, P + 0x50000000
    assert f(w, None, 256, 1, 64, 256, None, y, None, None, 0, None) == E_NULL
    assert f(w, x, 256, 1, 64, 256, None, y, c, None, 0, None) == E_NULL              # codes_out without scales_out
    assert f(w, x, 128, 1, 64, 256, None, y, None, None, 0, None) == E_SHAPE          # ldx < K
    assert f(w, x, 256, 9, 64, 256, None, y, None, None, 0, None) == E_SHAPE
    assert f(w, x + 4, 256, 1, 64, 256, None, y, None, None, 0, None) == E_ALIGN
    assert f(w, x, 258, 2, 64, 256, None, y, None, None, 0, None) == E_ALIGN
    assert f(w, x, 256, 1, 64, 256, None, y, c + 1, s, 0, None) == E_ALIGN
    assert f(w, x, 256, 1, 64, 256, None, x + 64, None, None, 0, None) == E_ALIAS     # y inside x
    assert f(w, x, 256, 1, 64, 256, None, y, x, s, 0, None) == E_ALIAS                # codes_out inside x


def test_quantize_rejects(L):
    f = L.qk_quantize_q8_1
    x, c, s = P, P + 0x10000000, P + 0x20000000
    assert f(x, 256, 1, 100, c, s, 0, None) == E_SHAPE
    assert f(x, 128, 1, 256, c, s, 0, None) == E_SHAPE             # ldx < K
    assert f(x, 256, 0, 256, c, s, 0, None) == 0                   # M = 0: nothing to do
    assert f(None, 256, 1, 256, c, s, 0, None) == E_NULL
    assert f(x + 4, 256, 1, 256, c, s, 0, None) == E_ALIGN
    assert f(x, 258, 2, 256, c, s, 0, None) == E_ALIGN             # ldx % 4 != 0
    assert f(x, 256, 1, 256, x + 512, s, 0, None) == E_ALIAS       # codes inside x


def test_repack_rejects(L):
    f = L.qk_repack
    assert f(7, P, 4, 256, P + 0x10000000, None) == E_TYPE
    assert f(0, P, 4, 256, P + 0x10000000, None) == E_TYPE
    assert f(qk.Q4_K, P, 4, 300, P + 0x10000000, None) == E_SHAPE
    assert f(qk.Q4_K, None, 4, 256, P + 0x10000000, None) == E_NULL
    assert f(qk.Q6_K, P + 2, 4, 256, P + 0x10000000, None) == E_ALIGN
    assert f(qk.Q4_K, P, 4, 256, P + 144, None) == E_ALIAS


def test_mmq_workspace_size():
    # ceil(M/128) * (K * 512 + ceil(K/512) * 8192)
    assert qk.mmq_workspace_bytes(2048, 3584, 18944) == 16 * (18944 * 512 + 37 * 8192) == 160038912
    assert qk.mmq_workspace_bytes(1, 64, 256) == 256 * 512 + 8192
    assert qk.mmq_workspace_bytes(129, 64, 512) == 2 * (512 * 512 + 8192)
    assert qk.mmq_workspace_bytes(128, 64, 1280) == 1280 * 512 + 3 * 8192     # 5 superblocks: 3 sums tiles
    assert qk.mmq_workspace_bytes(0, 64, 256) == 0


@pytest.mark.parametrize("fn", ["qk_mmq_q4k", "qk_mmq_q6k"])
def test_mmq_rejects(L, fn):
    f = getattr(L, fn)
    w, c, s, y, ws = P, P + 0x10000000, P + 0x20000000, P + 0x30000000, P + 0x40000000
    need = qk.mmq_workspace_bytes(16, 64, 256)
    assert f(w, c, s, 0, 64, 256, None, y, None, 0, 0, None) == 0   # M = 0: nothing to do
    assert f(w, c, s, 16, 64, 320, None, y, ws, need, 0, None) == E_SHAPE
    assert f(None, c, s, 16, 64, 256, None, y, ws, need, 0, None) == E_NULL
    assert f(w, c, s, 16, 64, 256, None, y, None, need, 0, None) == E_NULL        # no workspace
    assert f(w, c + 1, s, 16, 64, 256, None, y, ws, need, 0, None) == E_ALIGN
    assert f(w, c, s, 16, 64, 256, None, y, ws + 16, need, 0, None) == E_ALIGN    # workspace not 256-aligned
    assert f(w, c, s, 16, 64, 256, None, y, ws, need - 16, 0, None) == -6         # QK_E_WORKSPACE
    assert f(w, c, s, 16, 64, 256, None, c, ws, need, 0, None) == E_ALIAS
    assert f(w, c, s, 16, 64, 256, None, y, y, need, 0, None) == E_ALIAS           # workspace over y
    assert f(w, c, s, 16, 64, 256, None, y, ws, need, 6, None) == E_SHAPE          # two tile widths forced
    assert f(w, c, s, 16, 64, 256, None, y, ws, need, 10, None) == E_SHAPE         # 256 and 192 forced
    if fn == "qk_mmq_q6k":
        assert f(w, c, s, 16, 64, 256, None, y, ws, need, 8, None) == E_SHAPE      # Q6_K has no 192-wide tile


def test_min_plane_size_and_rejects(L):
    assert qk.q4k_min_plane_bytes(3584, 3584) == 3584 * 7 * 64
    assert qk.q4k_min_plane_bytes(10, 256) == 10 * 64                   # one superblock: one record
    assert qk.q4k_min_plane_bytes(10, 1280) == 10 * 3 * 64              # five: three records
    w, pl, c, s, y, ws = (P + i * 0x10000000 for i in range(6))
    need = qk.q4k_min_plane_bytes(64, 512)
    f = L.qk_q4k_min_plane
    assert f(w, 64, 320, pl, need, None) == E_SHAPE
    assert f(w, 0, 512, pl, need, None) == E_SHAPE
    assert f(None, 64, 512, pl, need, None) == E_NULL
    assert f(w, 64, 512, None, need, None) == E_NULL
    assert f(w, 64, 512, pl + 8, need, None) == E_ALIGN
    assert f(w, 64, 512, pl, need - 1, None) == -6                     # QK_E_WORKSPACE
    assert f(w, 64, 512, w, need, None) == E_ALIAS
    g = L.qk_mmq_q4k_plane
    wsn = qk.mmq_workspace_bytes(16, 64, 512)
    assert g(w, pl, c, s, 0, 64, 512, None, y, None, 0, 0, None) == 0    # M = 0: nothing to do
    assert g(w, None, c, s, 16, 64, 512, None, y, ws, wsn, 0, None) == E_NULL
    assert g(w, pl + 4, c, s, 16, 64, 512, None, y, ws, wsn, 0, None) == E_ALIGN
    assert g(w, y, c, s, 16, 64, 512, None, y, ws, wsn, 0, None) == E_ALIAS   # plane over y
    assert g(w, ws, c, s, 16, 64, 512, None, y, ws, wsn, 0, None) == E_ALIAS  # plane over the workspace


@pytest.mark.parametrize("fn", ["qk_mmq_q4k_f32", "qk_mmq_q6k_f32"])
def test_mmq_f32_rejects(L, fn):
    f = getattr(L, fn)
    w, x, y, ws = P, P + 0x10000000, P + 0x30000000, P + 0x40000000
    need = qk.mmq_workspace_bytes(16, 64, 256)
    pre = (w, None) if fn == "qk_mmq_q4k_f32" else (w,)
    assert f(*pre, x, 256, 0, 64, 256, None, y, None, 0, 0, None) == 0                 # M = 0: nothing to do
    assert f(*pre, None, 256, 16, 64, 256, None, y, ws, need, 0, None) == E_NULL
    assert f(*pre, x, 128, 16, 64, 256, None, y, ws, need, 0, None) == E_SHAPE         # ldx < K
    assert f(*pre, x + 4, 256, 16, 64, 256, None, y, ws, need, 0, None) == E_ALIGN     # x not 16-byte aligned
    assert f(*pre, x, 258, 16, 64, 256, None, y, ws, need, 0, None) == E_ALIGN         # ldx % 4 != 0
    assert f(*pre, y, 256, 16, 64, 256, None, y, ws, need, 0, None) == E_ALIAS         # x over y
    assert f(*pre, ws, 256, 16, 64, 256, None, y, ws, need, 0, None) == E_ALIAS        # x over the workspace


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        qk.quantize_q8_1(torch.zeros(1, 256))


def test_mmq_noalloc_rejects_oversize(L):
    f = L.qk_mmq_q4k_noalloc
    w, c, s, y = P, P + 0x10000000, P + 0x20000000, P + 0x30000000
    assert f(w, c, s, 0, 64, 256, None, y, 0, None) == 0                 # M = 0: nothing to do
    assert f(w, c, s, 16, 64, 320, None, y, 0, None) == E_SHAPE
    assert qk.mmq_workspace_bytes(2048, 3584, 18944) > qk.STATIC_WS_BYTES
    assert f(w, c, s, 2048, 3584, 18944, None, y, 0, None) == -6       # QK_E_WORKSPACE, before any CUDA call
    assert qk.mmq_workspace_bytes(2048, 4608, 3584) <= qk.STATIC_WS_BYTES


def test_rmsnorm_q8_1_rejects(L):
    f = L.qk_rmsnorm_q8_1
    x, r, g, h, y, c, s = (P + i * 0x10000000 for i in range(7))
    assert f(x, 256, None, g, 1e-5, 0, 256, None, None, c, s, 0, None) == 0          # M = 0: nothing to do
    assert f(x, 256, None, g, 1e-5, 1, 100, None, None, c, s, 0, None) == E_SHAPE    # K % 32
    assert f(x, 128, None, g, 1e-5, 1, 256, None, None, c, s, 0, None) == E_SHAPE    # ldx < K
    assert f(x, 256, None, g, -1.0, 1, 256, None, None, c, s, 0, None) == E_SHAPE    # eps < 0
    assert f(x, 256, None, g, float("nan"), 1, 256, None, None, c, s, 0, None) == E_SHAPE
    assert f(x, 256, None, None, 1e-5, 1, 256, None, None, c, s, 0, None) == E_NULL
    assert f(x, 256, None, g, 1e-5, 1, 256, None, None, None, s, 0, None) == E_NULL
    assert f(x + 4, 256, None, g, 1e-5, 1, 256, None, None, c, s, 0, None) == E_ALIGN
    assert f(x, 256, r + 8, g, 1e-5, 1, 256, None, None, c, s, 0, None) == E_ALIGN
    assert f(x, 258, None, g, 1e-5, 2, 256, None, None, c, s, 0, None) == E_ALIGN   # ldx % 4
    assert f(x, 256, None, g, 1e-5, 1, 256, None, x, c, s, 0, None) == E_ALIAS       # y over x
    assert f(x, 256, r, g, 1e-5, 1, 256, r, None, c, s, 0, None) == E_ALIAS         # h_out over r
    assert f(x, 256, None, g, 1e-5, 1, 256, None, y, y + 512, s, 0, None) == E_ALIAS  # codes over y


def test_swiglu_q8_1_rejects(L):
    f = L.qk_swiglu_q8_1
    gu, h, c, s = (P + i * 0x10000000 for i in range(4))
    assert f(gu, 512, 0, 256, h, c, s, 0, None) == 0                   # M = 0: nothing to do
    assert f(gu, 512, 1, 100, h, c, s, 0, None) == E_SHAPE             # F % 32
    assert f(gu, 256, 1, 256, h, c, s, 0, None) == E_SHAPE             # ldgu < 2F
    assert f(gu, 512, 65536, 256, h, c, s, 0, None) == E_SHAPE         # M beyond the grid's y extent
    assert f(None, 512, 1, 256, h, c, s, 0, None) == E_NULL
    assert f(gu, 512, 1, 256, h, None, s, 0, None) == E_NULL
    assert f(gu + 4, 512, 1, 256, h, c, s, 0, None) == E_ALIGN
    assert f(gu, 514, 2, 256, h, c, s, 0, None) == E_ALIGN
    assert f(gu, 512, 1, 256, gu + 1024, c, s, 0, None) == E_ALIAS     # h inside gu
    assert f(gu, 512, 1, 256, h, h + 512, s, 0, None) == E_ALIAS       # codes inside h


def test_peak_rejects(L):
    r, ms = ctypes.c_double(), ctypes.c_double()
    for fn in ("qk_peak_mma_s8", "qk_peak_tcgen05_f16"):
        f = getattr(L, fn)
        assert f(100, 1, None, ctypes.byref(ms), None) == E_NULL
        assert f(0, 1, ctypes.byref(r), ctypes.byref(ms), None) == E_SHAPE
        assert f(100, 0, ctypes.byref(r), ctypes.byref(ms), None) == E_SHAPE
        assert f(100, 1001, ctypes.byref(r), ctypes.byref(ms), None) == E_SHAPE
