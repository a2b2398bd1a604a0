"""Seeded synthetic inputs for the k-quant x q8_1 contraction.

The one module that both sides (the CUDA path and the CPU oracle) take their
inputs from.  It draws random numbers and lays them out in the GGUF block
formats; it does none of the method's arithmetic (no quantization, no
dequantization, no dot products).

Distributions (the benchmark definition of the workload):
  Q4_K superblock (144 B): f16 d ~ U(1e-3, 1e-2), f16 dmin ~ U(0, 5e-3),
      12 bytes of packed 6-bit scales and mins, 128 bytes of 4-bit codes.
      The 12-byte packing maps 16 six-bit fields onto 96 bits one to one, so
      uniform random bytes are exactly uniform random scales and mins.
  Q5_K superblock (176 B): d and dmin as for Q4_K, then uniform random bytes
      for the packed scales and mins, the 32 bytes of fifth bits and the codes.
  Q2_K superblock (84 B) and Q3_K superblock (110 B): uniform random bytes
      except f16 d ~ U(1e-3, 1e-2) (and Q2_K dmin ~ U(0, 5e-3)).
  Q8_0 block (34 B): f16 d ~ U(1e-3, 1e-2), 32 int8 codes uniform on [-127, 127].
  Q6_K superblock (210 B): 128 B of low-4-bit codes and 64 B of high-2-bit
      codes (uniform random bits), 16 int8 scales ~ U[-32, 31], f16 d ~
      U(1e-3, 1e-2).
  activations and residuals: float32 ~ N(0, 1); RMSNorm weights 1 + 0.1 N(0, 1).
Every tensor has its own stream: numpy PCG64 seeded with (seed, tag).
"""
from __future__ import annotations

import zlib

import numpy as np

QK = 256
Q4K_BYTES = 144
Q6K_BYTES = 210
Q5K_BYTES = 176


def _rng(seed: int, tag: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), zlib.crc32(tag.encode())])


def _f16_bytes(v: np.ndarray) -> np.ndarray:
    """float values -> little-endian binary16 byte pairs [n][2]."""
    return np.ascontiguousarray(v.astype("<f2")).view(np.uint8).reshape(-1, 2)


def q4k_weights(N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    """GGUF Q4_K bytes for an N x K weight, row-major [N][K/256][144]."""
    assert K % QK == 0
    nb = N * (K // QK)
    rng = _rng(seed, "q4k:" + tag)
    blk = rng.integers(0, 256, size=(nb, Q4K_BYTES), dtype=np.uint8)
    d = rng.uniform(1e-3, 1e-2, size=nb)
    dmin = rng.uniform(0.0, 5e-3, size=nb)
    blk[:, 0:2] = _f16_bytes(d)
    blk[:, 2:4] = _f16_bytes(dmin)
    return blk.reshape(-1)


def q6k_weights(N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    """GGUF Q6_K bytes for an N x K weight, row-major [N][K/256][210]."""
    assert K % QK == 0
    nb = N * (K // QK)
    rng = _rng(seed, "q6k:" + tag)
    blk = np.empty((nb, Q6K_BYTES), np.uint8)
    blk[:, 0:192] = rng.integers(0, 256, size=(nb, 192), dtype=np.uint8)
    blk[:, 192:208] = rng.integers(-32, 32, size=(nb, 16), dtype=np.int8).view(np.uint8)
    blk[:, 208:210] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=nb))
    return blk.reshape(-1)


def q5k_weights(N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    """GGUF Q5_K bytes for an N x K weight, row-major [N][K/256][176]: f16 d ~ U(1e-3, 1e-2),
    f16 dmin ~ U(0, 5e-3), then uniform random bytes (6-bit scales and mins, fifth bits, codes)."""
    assert K % QK == 0
    nb = N * (K // QK)
    rng = _rng(seed, "q5k:" + tag)
    blk = rng.integers(0, 256, size=(nb, Q5K_BYTES), dtype=np.uint8)
    blk[:, 0:2] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=nb))
    blk[:, 2:4] = _f16_bytes(rng.uniform(0.0, 5e-3, size=nb))
    return blk.reshape(-1)


def q80_weights(N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    """GGUF Q8_0 bytes for an N x K weight, row-major [N][K/32][34]: f16 d ~ U(1e-3, 1e-2) (the
    k-quant scale range), int8 codes uniform on [-127, 127]."""
    assert K % 32 == 0
    nb = N * (K // 32)
    rng = _rng(seed, "q80:" + tag)
    blk = np.empty((nb, 34), np.uint8)
    blk[:, 0:2] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=nb))
    blk[:, 2:34] = rng.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    return blk.reshape(-1)


def q2k_weights(N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    """GGUF Q2_K bytes [N][K/256][84]: uniform random scale/min nibbles and codes, f16 d ~ U(1e-3, 1e-2),
    f16 dmin ~ U(0, 5e-3)."""
    assert K % QK == 0
    nb = N * (K // QK)
    rng = _rng(seed, "q2k:" + tag)
    blk = rng.integers(0, 256, size=(nb, 84), dtype=np.uint8)
    blk[:, 80:82] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=nb))
    blk[:, 82:84] = _f16_bytes(rng.uniform(0.0, 5e-3, size=nb))
    return blk.reshape(-1)


def q3k_weights(N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    """GGUF Q3_K bytes [N][K/256][110]: uniform random hmask, codes and packed 6-bit scales,
    f16 d ~ U(1e-3, 1e-2)."""
    assert K % QK == 0
    nb = N * (K // QK)
    rng = _rng(seed, "q3k:" + tag)
    blk = rng.integers(0, 256, size=(nb, 110), dtype=np.uint8)
    blk[:, 108:110] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=nb))
    return blk.reshape(-1)


def weights(qtype: str, N: int, K: int, seed: int = 0, tag: str = "w") -> np.ndarray:
    if qtype == "q2k":
        return q2k_weights(N, K, seed, tag)
    if qtype == "q3k":
        return q3k_weights(N, K, seed, tag)
    if qtype == "q80":
        return q80_weights(N, K, seed, tag)
    if qtype == "q4k":
        return q4k_weights(N, K, seed, tag)
    if qtype == "q5k":
        return q5k_weights(N, K, seed, tag)
    if qtype == "q6k":
        return q6k_weights(N, K, seed, tag)
    raise ValueError(qtype)


def activations(M: int, K: int, seed: int = 0, tag: str = "x") -> np.ndarray:
    return _rng(seed, "act:" + tag).standard_normal((M, K), dtype=np.float32)


def residual(M: int, N: int, seed: int = 0, tag: str = "r") -> np.ndarray:
    return _rng(seed, "res:" + tag).standard_normal((M, N), dtype=np.float32)


def norm_weight(K: int, seed: int = 0, tag: str = "g") -> np.ndarray:
    """RMSNorm weight: float32 1 + 0.1 * N(0, 1) per channel (trained norm weights sit near 1)."""
    return (1.0 + 0.1 * _rng(seed, "norm:" + tag).standard_normal(K)).astype(np.float32)


# ---------------------------------------------------------------- workloads
# Shapes of the benchmark configurations (N = output rows, K = reduction).

LLAMA3_8B_LAYER = [  # decode layer: name, N, K, residual?, q8 activation slot
    ("qkv", 6144, 4096, False, "x_attn_in"),
    ("attn_out", 4096, 4096, True, "x_attn_out"),
    ("gate_up", 2 * 14336, 4096, False, "x_ffn_in"),
    ("down", 4096, 14336, True, "x_ffn_mid"),
]
LLAMA3_8B_HEAD = ("head", 128256, 4096, False, "x_head")
QWEN2_7B_PREFILL = [
    ("qkv", 4608, 3584, False, "x_attn_in"),
    ("attn_out", 3584, 3584, True, "x_attn_out"),
    ("gate_up", 2 * 18944, 3584, False, "x_ffn_in"),
    ("down", 3584, 18944, True, "x_ffn_mid"),
]
