"""CPU oracle for the FP8 (E4M3) W8A8 scaled GEMM and its quantisers.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports this package, and this package never imports the product.

This module is argument marshalling around ``fp8_oracle.c`` (numpy arrays in,
numpy arrays out); every piece of arithmetic lives in the C file, which states
the definition each function follows and where it comes from.  bf16 tensors
are passed as ``uint16`` bit patterns and E4M3 tensors as ``uint8`` codes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

GRAN_PER_TENSOR = 0
GRAN_PER_CHANNEL = 1
GRAN_PER_TOKEN_CHANNEL = 2
GRAN_PER_TOKEN = 3


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_decode_array.argtypes = [P, I64, P]
    lib.oracle_e4m3_encode_array.argtypes = [P, I64, P]
    lib.oracle_e4m3_encode_bits_range.argtypes = [ctypes.c_uint32, I64, P]
    lib.oracle_bf16_rne_f64.argtypes = [ctypes.c_double]
    lib.oracle_bf16_rne_f64.restype = ctypes.c_uint16
    lib.oracle_bf16_rne_f32_array.argtypes = [P, I64, P]
    lib.oracle_bf16_rne_f64_array.argtypes = [P, I64, P]
    lib.oracle_quant_static.argtypes = [P, ctypes.c_float, I64, I64, P]
    lib.oracle_quant_per_token.argtypes = [P, I64, I64, P, P]
    lib.oracle_rmsnorm_bf16.argtypes = [P, P, ctypes.c_float, I64, I64, P]
    lib.oracle_sum_squares_bf16.argtypes = [P, I64]
    lib.oracle_sum_squares_bf16.restype = ctypes.c_float
    lib.oracle_rmsnorm_quant.argtypes = [P, P, ctypes.c_float, ctypes.c_float, I64, I64, P]
    lib.oracle_residual_add_bf16.argtypes = [P, P, I64, P]
    lib.oracle_requant.argtypes = [P, I64, ctypes.c_float, ctypes.c_float, P]
    lib.oracle_exp_f32.argtypes = [ctypes.c_float]
    lib.oracle_exp_f32.restype = ctypes.c_float
    lib.oracle_exp_f32_array.argtypes = [P, I64, P]
    lib.oracle_silu_f32.argtypes = [ctypes.c_float]
    lib.oracle_silu_f32.restype = ctypes.c_float
    lib.oracle_silu_f32_array.argtypes = [P, I64, P]
    lib.oracle_silu_mul_bf16.argtypes = [P, I64, I64, P]
    lib.oracle_silu_mul_quant_per_token.argtypes = [P, I64, I64, P, P]
    lib.oracle_add_rmsnorm_quant.argtypes = [P, P, P, ctypes.c_float, ctypes.c_float, I64, I64, P, P]
    lib.oracle_gemm_acc_f64.argtypes = [P, P, I64, I64, I64, P, ctypes.c_int]
    lib.oracle_gemm_acc_i64.argtypes = [P, P, I64, I64, I64, P, ctypes.c_int]
    lib.oracle_scaled_mm.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, I64, P, P, ctypes.c_int]
    lib.oracle_scaled_mm_points.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, I64, P, P, I64, P]
    lib.oracle_quant_per_token_group.argtypes = [P, I64, I64, P, P]
    lib.oracle_quant_weight_block.argtypes = [P, I64, I64, P, P]
    lib.oracle_scaled_mm_block_points.argtypes = [P, P, P, P, I64, I64, I64, P, P, I64, P]
    lib.oracle_w8a16_mm.argtypes = [P, P, P, ctypes.c_int, I64, I64, I64, P, P, ctypes.c_int]
    lib.oracle_w8a16_points.argtypes = [P, P, P, ctypes.c_int, I64, P, P, I64, P]
    lib.oracle_dequant_weight_bf16.argtypes = [P, P, ctypes.c_int, I64, I64, P]
    lib.oracle_has_nan_code.argtypes = [P, I64]
    lib.oracle_has_nan_code.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


# --- codecs -----------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> exact values (float64)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    """binary32 values -> E4M3 codes, saturating round-to-nearest-even."""
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode_bits_range(start: int, count: int) -> np.ndarray:
    """Encode the binary32 values with bit patterns start .. start+count-1."""
    out = np.empty(count, np.uint8)
    _load().oracle_e4m3_encode_bits_range(ctypes.c_uint32(start), count, _ptr(out))
    return out


def bf16_rne(values) -> np.ndarray:
    """float32 or float64 values -> bf16 bit patterns (uint16), round-to-nearest-even."""
    v = np.asarray(values)
    out = np.empty(v.shape, np.uint16)
    if v.dtype == np.float32:
        v = _c(v, np.float32)
        _load().oracle_bf16_rne_f32_array(_ptr(v), v.size, _ptr(out))
    else:
        v = _c(v, np.float64)
        _load().oracle_bf16_rne_f64_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact; the upper half of a binary32)."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --- quantisers ---------------------------------------------------------------

def quant_static(x_bf16, s: float) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    _load().oracle_quant_static(_ptr(x), ctypes.c_float(s), M, K, _ptr(q))
    return q


def quant_per_token(x_bf16):
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    _load().oracle_quant_per_token(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def sum_squares_bf16(x_bf16) -> np.float32:
    """Exact sum of squares of a bf16 vector, rounded once to binary32."""
    x = _c(x_bf16, np.uint16).ravel()
    return np.float32(_load().oracle_sum_squares_bf16(_ptr(x), x.size))


def rmsnorm_bf16(x_bf16, gamma_bf16, eps: float) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    M, K = x.shape
    h = np.empty((M, K), np.uint16)
    _load().oracle_rmsnorm_bf16(_ptr(x), _ptr(g), ctypes.c_float(eps), M, K, _ptr(h))
    return h


def rmsnorm_quant(x_bf16, gamma_bf16, eps: float, s: float) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    _load().oracle_rmsnorm_quant(_ptr(x), _ptr(g), ctypes.c_float(eps), ctypes.c_float(s), M, K, _ptr(q))
    return q


def residual_add_bf16(x_bf16, r_bf16) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    r = _c(r_bf16, np.uint16)
    if x.shape != r.shape:
        raise ValueError("x and r must have the same shape")
    h = np.empty(x.shape, np.uint16)
    _load().oracle_residual_add_bf16(_ptr(x), _ptr(r), x.size, _ptr(h))
    return h


def add_rmsnorm_quant(x_bf16, r_bf16, gamma_bf16, eps: float, s: float):
    """Returns (q E4M3 codes [M,K], h bf16 bits [M,K] = the updated residual)."""
    x = _c(x_bf16, np.uint16)
    r = _c(r_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    M, K = x.shape
    if r.shape != x.shape:
        raise ValueError("x and r must have the same shape")
    q = np.empty((M, K), np.uint8)
    h = np.empty((M, K), np.uint16)
    _load().oracle_add_rmsnorm_quant(_ptr(x), _ptr(r), _ptr(g), ctypes.c_float(eps), ctypes.c_float(s), M, K,
                                     _ptr(q), _ptr(h))
    return q, h


def exp_f32(y) -> np.ndarray:
    y = _c(np.atleast_1d(y), np.float32)
    out = np.empty(y.shape, np.float32)
    _load().oracle_exp_f32_array(_ptr(y), y.size, _ptr(out))
    return out


def silu_f32(g) -> np.ndarray:
    g = _c(np.atleast_1d(g), np.float32)
    out = np.empty(g.shape, np.float32)
    _load().oracle_silu_f32_array(_ptr(g), g.size, _ptr(out))
    return out


def silu_mul_bf16(gate_up_bf16) -> np.ndarray:
    """bf16 bits [M, I] of silu(gate) * up for rows [gate | up] ([M, 2I])."""
    x = _c(gate_up_bf16, np.uint16)
    M, W = x.shape
    if W % 2:
        raise ValueError("gate_up rows must have an even width")
    a = np.empty((M, W // 2), np.uint16)
    _load().oracle_silu_mul_bf16(_ptr(x), M, W // 2, _ptr(a))
    return a


def silu_mul_quant_per_token(gate_up_bf16):
    """(E4M3 codes [M, I], per-token scales [M]) of silu(gate) * up."""
    x = _c(gate_up_bf16, np.uint16)
    M, W = x.shape
    if W % 2:
        raise ValueError("gate_up rows must have an even width")
    q = np.empty((M, W // 2), np.uint8)
    s = np.empty((M,), np.float32)
    _load().oracle_silu_mul_quant_per_token(_ptr(x), M, W // 2, _ptr(q), _ptr(s))
    return q, s


BLOCK = 128


def quant_per_token_group(x_bf16):
    """(codes [M,K], scales [M, ceil(K/128)]): every 128-wide group of a row
    quantised on its own."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, -(-K // BLOCK)), np.float32)
    _load().oracle_quant_per_token_group(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def quant_weight_block(w_bf16):
    """(codes [N,K], scales [ceil(N/128), ceil(K/128)]): one scale per 128 x 128 block."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((-(-N // BLOCK), -(-K // BLOCK)), np.float32)
    _load().oracle_quant_weight_block(_ptr(w), N, K, _ptr(q), _ptr(s))
    return q, s


def scaled_mm_block_points(A, B, sa, sb, rows, cols) -> np.ndarray:
    """The blockwise GEMM (scales [M, KB] and [NB, KB]) at (rows[i], cols[i])."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    M, K = A.shape
    N = B.shape[0]
    y = np.empty(rows.shape, np.float64)
    _load().oracle_scaled_mm_block_points(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), M, N, K, _ptr(rows), _ptr(cols),
                                          rows.size, _ptr(y))
    return y


def requant(q_codes, s_in: float, s_out: float) -> np.ndarray:
    q = _c(q_codes, np.uint8)
    out = np.empty(q.shape, np.uint8)
    _load().oracle_requant(_ptr(q), q.size, ctypes.c_float(s_in), ctypes.c_float(s_out), _ptr(out))
    return out


# --- GEMM --------------------------------------------------------------------

def gemm_acc_f64(A, B, nthreads=None) -> np.ndarray:
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    acc = np.empty((M, N), np.float64)
    _load().oracle_gemm_acc_f64(_ptr(A), _ptr(B), M, N, K, _ptr(acc), nthreads or default_threads())
    return acc


def gemm_acc_i64(A, B, nthreads=None) -> np.ndarray:
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    acc = np.empty((M, N), np.int64)
    _load().oracle_gemm_acc_i64(_ptr(A), _ptr(B), M, N, K, _ptr(acc), nthreads or default_threads())
    return acc


def scaled_mm(A, B, sa, sb, gran: int, nthreads=None):
    """Returns (y64 float64 [M,N], y_bf16 uint16 [M,N])."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(np.atleast_1d(sa), np.float32)
    sb = _c(np.atleast_1d(sb), np.float32)
    M, K = A.shape
    N = B.shape[0]
    y64 = np.empty((M, N), np.float64)
    yb = np.empty((M, N), np.uint16)
    _load().oracle_scaled_mm(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), gran, M, N, K, _ptr(y64), _ptr(yb),
                             nthreads or default_threads())
    return y64, yb


def scaled_mm_points(A, B, sa, sb, gran: int, rows, cols) -> np.ndarray:
    """The GEMM definition evaluated only at the (rows[i], cols[i]) outputs."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(np.atleast_1d(sa), np.float32)
    sb = _c(np.atleast_1d(sb), np.float32)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    M, K = A.shape
    N = B.shape[0]
    y = np.empty(rows.shape, np.float64)
    _load().oracle_scaled_mm_points(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), gran, M, N, K, _ptr(rows),
                                    _ptr(cols), rows.size, _ptr(y))
    return y


def w8a16_mm(x_bf16, W, sb, per_channel: bool, nthreads=None):
    """Weight-only FP8 GEMM: (y64 float64 [M,N], y_bf16 uint16 [M,N]) for bf16
    x [M,K], E4M3 codes W [N,K], scales sb [N] (per channel) or [1]."""
    x = _c(x_bf16, np.uint16)
    W = _c(W, np.uint8)
    sb = _c(np.atleast_1d(sb), np.float32)
    M, K = x.shape
    N = W.shape[0]
    y64 = np.empty((M, N), np.float64)
    yb = np.empty((M, N), np.uint16)
    _load().oracle_w8a16_mm(_ptr(x), _ptr(W), _ptr(sb), int(bool(per_channel)), M, N, K, _ptr(y64), _ptr(yb),
                            nthreads or default_threads())
    return y64, yb


def w8a16_points(x_bf16, W, sb, per_channel: bool, rows, cols) -> np.ndarray:
    """The weight-only GEMM at the (rows[i], cols[i]) outputs."""
    x = _c(x_bf16, np.uint16)
    W = _c(W, np.uint8)
    sb = _c(np.atleast_1d(sb), np.float32)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    y = np.empty(rows.shape, np.float64)
    _load().oracle_w8a16_points(_ptr(x), _ptr(W), _ptr(sb), int(bool(per_channel)), x.shape[1], _ptr(rows),
                                _ptr(cols), rows.size, _ptr(y))
    return y


def dequant_weight_bf16(W, sb, per_channel: bool) -> np.ndarray:
    """The large-M branch's bf16 weight: bf16_rne(fp32(dec(W) * sb)), uint16 [N,K]."""
    W = _c(W, np.uint8)
    sb = _c(np.atleast_1d(sb), np.float32)
    N, K = W.shape
    out = np.empty((N, K), np.uint16)
    _load().oracle_dequant_weight_bf16(_ptr(W), _ptr(sb), int(bool(per_channel)), N, K, _ptr(out))
    return out


def has_nan_code(codes) -> bool:
    c = _c(codes, np.uint8)
    return bool(_load().oracle_has_nan_code(_ptr(c), c.size))

