"""CPU oracle for the W1.58A8 ternary path -- TEST INFRASTRUCTURE ONLY.

Plain C (``tw_oracle.c``) behind ctypes.  Only the tests, the package smoke check
and the benchmark's CPU-baseline / reference arm may import this module; the
product library never does, and this module never imports the product.

Every function takes and returns numpy arrays on the host.  The method's
readings (rounding, scale, bit layout) are spelled out in ``tw_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tw_oracle.c")
_LIB = os.path.join(_HERE, "libtw_oracle.so")
_LIB_OMP = os.path.join(_HERE, "libtw_oracle_omp.so")  # the same source built with -fopenmp
_lock = threading.Lock()
_lib = None
_lib_omp = None

# gcc flags: one IEEE rounding per fp32 operation (no contraction, no fast-math).
CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-unsafe-math-optimizations", "-frounding-math"]

STATUS = {0: "ok", 1: "null pointer", 2: "bad shape", 3: "invalid code (2-bit field 3, byte > 242, or padding)",
          4: "non-finite input", 5: "negative value", 6: "int32 overflow"}


class OracleError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: oracle status {code} ({STATUS.get(code, '?')})")
        self.code = code


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile libtw_oracle.so with gcc (if missing or older than the source).  openmp=True
    builds libtw_oracle_omp.so instead: the same source with -fopenmp, whose integer product
    shares its output rows out over the host's cores (the all-core CPU baseline)."""
    lib = _LIB_OMP if openmp else _LIB
    with _lock:
        if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_SRC):
            tmp = lib + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", *CFLAGS, *(["-fopenmp"] if openmp else []), "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, lib)
    return lib


def _load(openmp: bool = False):
    global _lib, _lib_omp
    if openmp:
        if _lib_omp is None:
            _lib_omp = _bind(ctypes.CDLL(build(openmp=True)))
        return _lib_omp
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    """Argument and result types of the exported functions."""
    i64, p = ctypes.c_int64, ctypes.c_void_p
    sig = {
        "two_exact_sum": [p, i64, p],
        "two_absmean": [p, i64, p, p],
        "two_pack_rows_with_scale": [p, i64, i64, ctypes.c_float, p],
        "two_pack_ternary": [p, i64, i64, p, p],
        "two_unpack_ternary": [p, i64, i64, p],
        "two_quant_act": [p, i64, i64, p, p, p],
        "two_rmsnorm": [p, p, ctypes.c_float, i64, i64, p, p],
        "two_rmsnorm_quant_act": [p, p, ctypes.c_float, i64, i64, p, p, p],
        "two_ternary_matmul": [p, ctypes.c_float, p, p, i64, i64, i64, p, p],
        "two_rms_inv": [p, ctypes.c_float, i64, i64, p],
        "two_residual_add": [p, p, i64, p],
        "two_pack_trits5": [p, i64, i64, p],
        "two_unpack_trits5": [p, i64, i64, p],
        "two_pack_ternary5": [p, i64, i64, p, p],
        "two_ternary_matmul5": [p, ctypes.c_float, p, p, i64, i64, i64, p, p],
        "two_threads": [],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.two_t5_row_bytes.argtypes = [i64]
    lib.two_t5_row_bytes.restype = i64
    return lib


def threads(openmp: bool = True) -> int:
    """Threads the integer product uses (1 for the plain build)."""
    return int(_load(openmp).two_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(code, where):
    if code != 0:
        raise OracleError(code, where)


def exact_sum(v) -> float:
    """Exact sum of non-negative finite doubles, rounded once (nearest-even)."""
    v = _c(v, np.float64).ravel()
    out = np.zeros(1, np.float64)
    _check(_load().two_exact_sum(_ptr(v), v.size, _ptr(out)), "exact_sum")
    return float(out[0])


def absmean(W):
    """Return (gamma fp32, exact sum of |W| as double)."""
    W = _c(W, np.float32).ravel()
    g = np.zeros(1, np.float32)
    s = np.zeros(1, np.float64)
    _check(_load().two_absmean(_ptr(W), W.size, _ptr(g), _ptr(s)), "absmean")
    return np.float32(g[0]), float(s[0])


def pack_ternary(W):
    """W fp32 [N][K] -> (packed uint8 [N][K/4], w_scale fp32)."""
    W = _c(W, np.float32)
    N, K = W.shape
    packed = np.zeros((N, K // 4 if K % 4 == 0 else 1), np.uint8)
    ws = np.zeros(1, np.float32)
    _check(_load().two_pack_ternary(_ptr(W), N, K, _ptr(packed), _ptr(ws)), "pack_ternary")
    return packed, np.float32(ws[0])


def pack_rows_with_scale(W_rows, gamma):
    W_rows = _c(W_rows, np.float32)
    R, K = W_rows.shape
    packed = np.zeros((R, K // 4 if K % 4 == 0 else 1), np.uint8)
    _check(_load().two_pack_rows_with_scale(_ptr(W_rows), R, K, float(gamma), _ptr(packed)),
           "pack_rows_with_scale")
    return packed


def unpack_ternary(packed, K):
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    t = np.zeros((N, K), np.int8)
    _check(_load().two_unpack_ternary(_ptr(packed), N, K, _ptr(t)), "unpack_ternary")
    return t


def quant_act(x):
    """x fp32 [M][K] -> (x_q int8 [M][K], s_x fp32 [M], x_sum int32 [M])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    xq = np.zeros((M, K), np.int8)
    sx = np.zeros(M, np.float32)
    xs = np.zeros(M, np.int32)
    _check(_load().two_quant_act(_ptr(x), M, K, _ptr(xq), _ptr(sx), _ptr(xs)), "quant_act")
    return xq, sx, xs


def rmsnorm(x, g, eps):
    """Return (u fp32 [M][K], exact sum of squares per row as double)."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    g = _c(g, np.float32)
    M, K = x.shape
    u = np.zeros((M, K), np.float32)
    r = np.zeros(M, np.float64)
    _check(_load().two_rmsnorm(_ptr(x), _ptr(g), float(eps), M, K, _ptr(u), _ptr(r)), "rmsnorm")
    return u, r


def rms_inv(x, eps):
    """Per row 1 / sqrtf(ms + eps), the RMSNorm scale (fp32 [M])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    inv = np.zeros(M, np.float32)
    _check(_load().two_rms_inv(_ptr(x), float(eps), M, K, _ptr(inv)), "rms_inv")
    return inv


def residual_add(h, y):
    """fl32(h + y) element by element."""
    h = _c(h, np.float32)
    y = _c(y, np.float32)
    assert h.shape == y.shape
    out = np.zeros(h.shape, np.float32)
    _check(_load().two_residual_add(_ptr(h), _ptr(y), h.size, _ptr(out)), "residual_add")
    return out


def rmsnorm_quant_act(x, g, eps):
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    g = _c(g, np.float32)
    M, K = x.shape
    xq = np.zeros((M, K), np.int8)
    sx = np.zeros(M, np.float32)
    xs = np.zeros(M, np.int32)
    _check(_load().two_rmsnorm_quant_act(_ptr(x), _ptr(g), float(eps), M, K,
                                         _ptr(xq), _ptr(sx), _ptr(xs)), "rmsnorm_quant_act")
    return xq, sx, xs


def ternary_matmul(packed, w_scale, x_q, s_x, openmp: bool = False):
    """packed [N][K/4], x_q int8 [M][K] -> (y fp32 [M][N], acc int32 [M][N]).  openmp=True
    runs the all-core build (same results)."""
    packed = _c(packed, np.uint8)
    x_q = _c(x_q, np.int8)
    if x_q.ndim == 1:
        x_q = x_q[None, :]
    s_x = _c(s_x, np.float32).ravel()
    M, K = x_q.shape
    N = packed.shape[0]
    y = np.zeros((M, N), np.float32)
    acc = np.zeros((M, N), np.int32)
    _check(_load(openmp).two_ternary_matmul(_ptr(packed), float(w_scale), _ptr(x_q), _ptr(s_x),
                                            M, N, K, _ptr(y), _ptr(acc)), "ternary_matmul")
    return y, acc


def t5_row_bytes(K: int) -> int:
    """Bytes per row of the five-trits-per-byte layout: 16 * ceil(K / 80)."""
    return int(_load().two_t5_row_bytes(int(K)))


def pack_trits5(t):
    """t int8 [N][K] in {-1, 0, 1} -> uint8 [N][t5_row_bytes(K)], five trits per byte."""
    t = _c(t, np.int8)
    N, K = t.shape
    out = np.zeros((N, max(t5_row_bytes(K), 1)), np.uint8)
    _check(_load().two_pack_trits5(_ptr(t), N, K, _ptr(out)), "pack_trits5")
    return out


def unpack_trits5(p5, K):
    """Inverse of pack_trits5 -> t int8 [N][K]."""
    p5 = _c(p5, np.uint8)
    N = p5.shape[0]
    t = np.zeros((N, K), np.int8)
    _check(_load().two_unpack_trits5(_ptr(p5), N, K, _ptr(t)), "unpack_trits5")
    return t


def pack_ternary5(W):
    """W fp32 [N][K] -> (uint8 [N][t5_row_bytes(K)], w_scale fp32): absmean ternarisation
    stored five trits per byte."""
    W = _c(W, np.float32)
    N, K = W.shape
    out = np.zeros((N, max(t5_row_bytes(K), 1)), np.uint8)
    ws = np.zeros(1, np.float32)
    _check(_load().two_pack_ternary5(_ptr(W), N, K, _ptr(out), _ptr(ws)), "pack_ternary5")
    return out, np.float32(ws[0])


def ternary_matmul5(p5, w_scale, x_q, s_x, openmp: bool = False):
    """Rows stored five trits per byte, x_q int8 [M][K] -> (y fp32 [M][N], acc int32 [M][N])."""
    p5 = _c(p5, np.uint8)
    x_q = _c(x_q, np.int8)
    if x_q.ndim == 1:
        x_q = x_q[None, :]
    s_x = _c(s_x, np.float32).ravel()
    M, K = x_q.shape
    N = p5.shape[0]
    y = np.zeros((M, N), np.float32)
    acc = np.zeros((M, N), np.int32)
    _check(_load(openmp).two_ternary_matmul5(_ptr(p5), float(w_scale), _ptr(x_q), _ptr(s_x),
                                             M, N, K, _ptr(y), _ptr(acc)), "ternary_matmul5")
    return y, acc
