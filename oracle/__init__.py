"""ctypes wrapper around the plain-C CPU oracle (bq_oracle.c).

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
benchmark's cpu_baseline / reference legs may import this package. The product
path never does.

Every function takes and returns numpy arrays on the host. Type codes:
Q4_0 = 2, Q8_0 = 8 (the oracle's own constants).
"""
import ctypes
import os

import numpy as np

from . import build as _build

Q4_0 = 2
Q8_0 = 8
QK = 32

_lib = None


def load(path):
    """Load an oracle shared library from `path` and declare its signatures."""
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    """The oracle library; BQ_ORACLE_LIB may name another build of it (the
    mutation tests point it at deliberately broken copies)."""
    global _lib
    if _lib is None:
        alt = os.environ.get("BQ_ORACLE_LIB")
        _lib = load(alt if alt else _build.build())
    return _lib


def _declare(L):
    i64, vp, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    L.oracle_block_bytes.argtypes = [i]
    L.oracle_block_values.argtypes = [i]
    L.oracle_block_values.restype = i64
    L.oracle_block_bytes.restype = i64
    L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_f16.restype = ctypes.c_uint16
    L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_f32.restype = ctypes.c_float
    L.oracle_round_half_even.argtypes = [ctypes.c_float]
    L.oracle_round_half_even.restype = ctypes.c_float
    L.oracle_quantize_rows.argtypes = [i, vp, vp, i64, i64]
    L.oracle_dequantize_rows.argtypes = [i, vp, vp, i64, i64]
    L.oracle_block_dots.argtypes = [i, vp, vp, vp, i64, i64]
    L.oracle_gemv.argtypes = [i, vp, vp, vp, vp, i64, i64]
    L.oracle_gemm.argtypes = [i, vp, vp, vp, vp, i64, i64, i64]
    L.oracle_kv_quantize.argtypes = [i, vp, vp, vp, i64, i64, i64]
    L.oracle_attn_decode.argtypes = [i, i, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float]
    L.oracle_hadamard64.argtypes = [vp, i64]
    L.oracle_kv_quantize_basis.argtypes = [i, vp, vp, i, i, vp, i64, i64, i64]
    L.oracle_kv_bias.argtypes = [vp, i, vp, i64, i64, i64]
    L.oracle_attn_decode_basis.argtypes = [i, i, i, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float]
    for f in ("oracle_quantize_rows", "oracle_dequantize_rows", "oracle_block_dots",
              "oracle_gemv", "oracle_gemm", "oracle_kv_quantize", "oracle_attn_decode"):
        getattr(L, f).restype = i


class use_library:
    """Context manager: route this module's functions to another build of the
    oracle (used by the mutation tests, which load deliberately broken copies)."""

    def __init__(self, path):
        self.L = load(path)

    def __enter__(self):
        global _lib
        self.prev, _lib = lib(), self.L
        return self.L

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def block_bytes(t):
    return int(lib().oracle_block_bytes(t))


def block_values(t):
    """values per block: 32, or 256 for the k-quant super-blocks"""
    return int(lib().oracle_block_values(t))


def f32_to_f16_bits(v: float) -> int:
    return int(lib().oracle_f32_to_f16(float(v)))


def f16_bits_to_f32(h: int) -> float:
    return float(lib().oracle_f16_to_f32(int(h)))


def round_half_even(v: float) -> float:
    return float(lib().oracle_round_half_even(float(v)))


def quantize_rows(t, x):
    """x: (rows, cols) fp32 -> (rows, cols/32*block_bytes) uint8."""
    x = _f32(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    R, C = x.shape
    out = np.zeros((R, (C // block_values(t)) * block_bytes(t)), dtype=np.uint8)
    _check(lib().oracle_quantize_rows(t, _p(x), _p(out), R, C), "quantize_rows")
    return out


def dequantize_rows(t, blocks, cols):
    blocks = _u8(blocks)
    R = blocks.size // ((cols // block_values(t)) * block_bytes(t)) if cols else 0
    out = np.zeros((R, cols), dtype=np.float32)
    _check(lib().oracle_dequantize_rows(t, _p(blocks), _p(out), R, cols), "dequantize_rows")
    return out


def block_dots(w_type, w_blocks, xq_blocks, M, K):
    w_blocks, xq_blocks = _u8(w_blocks), _u8(xq_blocks)
    out = np.zeros((M, K // QK), dtype=np.int32)
    _check(lib().oracle_block_dots(w_type, _p(w_blocks), _p(xq_blocks), _p(out), M, K),
           "block_dots")
    return out


def gemv(w_type, w_blocks, x, M, K, with_mag=False):
    w_blocks, x = _u8(w_blocks), _f32(x).reshape(-1)
    y = np.zeros(M, dtype=np.float32)
    mag = np.zeros(M, dtype=np.float64) if with_mag else None
    _check(lib().oracle_gemv(w_type, _p(w_blocks), _p(x), _p(y), _p(mag), M, K), "gemv")
    return (y, mag) if with_mag else y


def gemm(w_type, w_blocks, X, M, N, K, with_mag=False):
    w_blocks, X = _u8(w_blocks), _f32(X)
    Y = np.zeros((N, M), dtype=np.float32)
    mag = np.zeros((N, M), dtype=np.float64) if with_mag else None
    _check(lib().oracle_gemm(w_type, _p(w_blocks), _p(X), _p(Y), _p(mag), M, N, K), "gemm")
    return (Y, mag) if with_mag else Y


BASIS_PLAIN, BASIS_HADAMARD64 = 0, 1


def kv_quantize(t, rows, bias, n_tokens, n_kv_heads, head_dim, basis=BASIS_PLAIN, bias_basis=None):
    """rows: (n_tokens, n_kv_heads, head_dim) fp32; bias: (n_kv_heads, head_dim) or None.
    basis: the cache's basis (rows rotated first when BASIS_HADAMARD64);
    bias_basis: the basis the bias was calibrated in (default: basis)."""
    rows = _f32(rows)
    b = None if bias is None else _f32(bias)
    out = np.zeros((n_tokens, n_kv_heads, (head_dim // QK) * block_bytes(t)), dtype=np.uint8)
    rc = lib().oracle_kv_quantize_basis(t, _p(rows), _p(b), basis if bias_basis is None else bias_basis, basis,
                                        _p(out), n_tokens, n_kv_heads, head_dim)
    if rc == -2:
        raise ValueError("oracle kv_quantize: a bias requires the Q4_0 type")
    if rc == -4:
        raise ValueError("oracle kv_quantize: the bias was calibrated in another basis")
    _check(rc, "kv_quantize")
    return out


def hadamard64(x):
    """A copy of x (fp32, size a multiple of 64) with every group of 64
    consecutive values rotated: H64 x / 8."""
    y = np.array(x, dtype=np.float32, copy=True, order="C")
    _check(lib().oracle_hadamard64(_p(y), y.size), "hadamard64")
    return y


def kv_bias(rows, basis, n_tokens, n_kv_heads, head_dim):
    """Mean-centering bias (n_kv_heads, head_dim) fp32 of the calibration rows
    (n_tokens, n_kv_heads, head_dim), measured in `basis`."""
    rows = _f32(rows)
    out = np.zeros((n_kv_heads, head_dim), dtype=np.float32)
    _check(lib().oracle_kv_bias(_p(rows), basis, _p(out), n_tokens, n_kv_heads, head_dim), "kv_bias")
    return out


def attn_decode(k_type, v_type, q, K, V, n_tokens, n_heads, n_kv_heads, head_dim, scale, with_mag=False,
                k_basis=BASIS_PLAIN):
    """Decode attention of one token: q (n_heads, head_dim) fp32; K, V the
    quantized caches (n_tokens, n_kv_heads, head_dim/32 blocks). Returns o
    (n_heads, head_dim), and with_mag also mag (same shape) and the largest
    |score| per head."""
    q, K, V = _f32(q), _u8(K), _u8(V)
    o = np.zeros((n_heads, head_dim), dtype=np.float32)
    mag = np.zeros((n_heads, head_dim), dtype=np.float64)
    smax = np.zeros(n_heads, dtype=np.float64)
    _check(lib().oracle_attn_decode_basis(k_type, v_type, k_basis, _p(q), _p(K), _p(V), _p(o), _p(mag),
                                          _p(smax), n_tokens, n_heads, n_kv_heads, head_dim, float(scale)),
           "attn_decode")
    return (o, mag, smax) if with_mag else o
