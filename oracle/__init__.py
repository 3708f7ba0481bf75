"""Blockwise-FP8 linear layer: plain CPU oracle (ctypes wrapper over bfp8_oracle.c).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library
never loads it and shares no code with it.

The arithmetic lives in ``bfp8_oracle.c`` (each function cites the passage it
follows). This module only builds that file with gcc, moves numpy arrays in
and out, and allocates outputs.

Arrays: bf16 inputs are passed as numpy ``uint16`` bit patterns (the upper
half of a binary32 word); codes are ``uint8`` E4M3FN bit patterns; scales are
``float32``; GEMM results are ``float64``.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(format checks against two independent library casts, brute force, exact
integer sums, closed forms and invariants). One point stays unpinned: whether
this exact scale and quotient formula is bit-for-bit what the Puro-2B RTX 5090
kernels computed; the pages print no codes or scales to compare against.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

TILE = 128
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bfp8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile bfp8_oracle.c into liboracle.so next to it (gcc, OpenMP, IEEE)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_units.restype = ctypes.c_int64
        lib.oracle_e4m3_units.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode_n.restype = None
        lib.oracle_e4m3_encode_n.argtypes = [p, i64, p]
        lib.oracle_quantize_act.restype = None
        lib.oracle_quantize_act.argtypes = [p, i64, i64, i64, p, i64, p, i64]
        lib.oracle_quantize_weight.restype = ctypes.c_int
        lib.oracle_quantize_weight.argtypes = [p, i64, i64, i64, p, i64, p, p, i64]
        lib.oracle_quantize_transpose.restype = None
        lib.oracle_quantize_transpose.argtypes = [p, i64, i64, i64, p, i64, p, i64]
        gemm_args = [p, i64, p, i64, p, i64, p, i64, i64, i64, p, i64, p]
        for name in ("oracle_gemm_fwd", "oracle_gemm_dgrad", "oracle_gemm_fwd_i64"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = gemm_args
        lib.oracle_gemm_wgrad.restype = None
        lib.oracle_gemm_wgrad.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, p, i64, p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def round_up(x: int, m: int = TILE) -> int:
    return (x + m - 1) // m * m


# ---------------------------------------------------------------- formats
def bf16_to_f32(bits: int) -> float:
    return _load().oracle_bf16_to_f32(int(bits))


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e4m3_encode(t: float) -> int:
    return _load().oracle_e4m3_encode(float(t))


def e4m3_units(code: int) -> int:
    return _load().oracle_e4m3_units(int(code))


def e4m3_encode_array(t: np.ndarray) -> np.ndarray:
    """Encode float32 values to E4M3FN codes, element by element (the scalar encoder in a C loop)."""
    lib = _load()
    t = _c(t, np.float32).ravel()
    out = np.empty(t.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode_n(_ptr(t), t.size, _ptr(out))
    return out


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """Exact value of every code (FP64), via the scalar decoder over a 256-entry table."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_value(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


# ---------------------------------------------------------------- quantisers
def quantize_act(x_bits: np.ndarray):
    """1x128 tiles along the columns of x [R, C]. Returns (q [R, C] u8, s [ceil(C/128), R] f32)."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty(((C + TILE - 1) // TILE, R), dtype=np.float32)
    lib.oracle_quantize_act(_ptr(x), R, C, C, _ptr(q), C, _ptr(s), R)
    return q, s


def quantize_weight(w_bits: np.ndarray, transposed: bool = False):
    """128x128 blocks of w [N, K]. Returns (q [N, K], s [N/128, K/128]) and, if asked, qt [K, N]."""
    lib = _load()
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N // TILE, K // TILE), dtype=np.float32)
    qt = np.empty((K, N), dtype=np.uint8) if transposed else None
    rc = lib.oracle_quantize_weight(_ptr(w), N, K, K, _ptr(q), K, _ptr(s),
                                    _ptr(qt) if transposed else None, N)
    if rc != 0:
        raise ValueError("weight dims must be multiples of 128")
    return (q, s, qt) if transposed else (q, s)


def quantize_transpose(x_bits: np.ndarray):
    """Tiles of 128 rows of x [R, C], written transposed.

    Returns (qt [C, R128] u8, st [R128/128, C] f32), R128 = R rounded up to 128;
    pad codes are 0x00.
    """
    lib = _load()
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    R128 = round_up(R)
    qt = np.empty((C, R128), dtype=np.uint8)
    st = np.empty((R128 // TILE, C), dtype=np.float32)
    lib.oracle_quantize_transpose(_ptr(x), R, C, C, _ptr(qt), R128, _ptr(st), C)
    return qt, st


# ---------------------------------------------------------------- GEMMs
def _rows(rows, total):
    if rows is None:
        return None, total
    r = _c(rows, np.int64)
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < total))
    return r, r.size


def gemm_fwd(qx, sx, qw, sw, rows=None, exact_int=False):
    """Y = X W^T in FP64 from codes and scales. qx [M,K], sx [K/128,M], qw [N,K], sw [N/128,K/128].

    Returns y [len(rows) or M, N] float64.
    """
    lib = _load()
    qx, sx, qw, sw = _c(qx, np.uint8), _c(sx, np.float32), _c(qw, np.uint8), _c(sw, np.float32)
    M, K = qx.shape
    N = qw.shape[0]
    assert qw.shape[1] == K and sx.shape == (K // TILE, M) and sw.shape == (N // TILE, K // TILE)
    r, nr = _rows(rows, M)
    y = np.empty((nr, N), dtype=np.float64)
    fn = lib.oracle_gemm_fwd_i64 if exact_int else lib.oracle_gemm_fwd
    fn(_ptr(qx), K, _ptr(sx), M, _ptr(qw), K, _ptr(sw), M, N, K,
       _ptr(r) if r is not None else None, nr, _ptr(y))
    return y


def gemm_dgrad(qdy, sdy, qw, sw, rows=None):
    """dX = dY W in FP64. qdy [M,N], sdy [N/128,M], qw [N,K], sw [N/128,K/128]. Returns [rows, K]."""
    lib = _load()
    qdy, sdy, qw, sw = _c(qdy, np.uint8), _c(sdy, np.float32), _c(qw, np.uint8), _c(sw, np.float32)
    M, N = qdy.shape
    K = qw.shape[1]
    assert qw.shape[0] == N and sdy.shape == (N // TILE, M) and sw.shape == (N // TILE, K // TILE)
    r, nr = _rows(rows, M)
    dx = np.empty((nr, K), dtype=np.float64)
    lib.oracle_gemm_dgrad(_ptr(qdy), N, _ptr(sdy), M, _ptr(qw), K, _ptr(sw), M, N, K,
                          _ptr(r) if r is not None else None, nr, _ptr(dx))
    return dx


def gemm_wgrad(qdyt, sdyt, qxt, sxt, M, rows=None):
    """dW = dY^T X in FP64 from transposed tiles. qdyt [N,M128], sdyt [M128/128,N],
    qxt [K,M128], sxt [M128/128,K]. Returns [rows, K] (rows index N)."""
    lib = _load()
    qdyt, sdyt, qxt, sxt = (_c(qdyt, np.uint8), _c(sdyt, np.float32),
                            _c(qxt, np.uint8), _c(sxt, np.float32))
    N, M128 = qdyt.shape
    K = qxt.shape[0]
    assert M128 == round_up(M) and qxt.shape[1] == M128
    assert sdyt.shape == (M128 // TILE, N) and sxt.shape == (M128 // TILE, K)
    r, nr = _rows(rows, N)
    dw = np.empty((nr, K), dtype=np.float64)
    lib.oracle_gemm_wgrad(_ptr(qdyt), M128, _ptr(sdyt), N, _ptr(qxt), M128, _ptr(sxt), K,
                          M, N, K, _ptr(r) if r is not None else None, nr, _ptr(dw))
    return dw


def gemm_wgrad_accumulate(main_grad, qdyt, sdyt, qxt, sxt, M, rows=None):
    """main_grad + dW in FP64: the weight gradient added into an FP32 main gradient
    (the Puro-2B article keeps training state in FP32; section "FP8 takes advantage
    of the RTX 5090's low precision efficiency"). main_grad [N,K] float32 is not
    modified; returns [rows, K] float64 = main_grad[rows] + gemm_wgrad(...)."""
    main = np.asarray(main_grad, dtype=np.float32)
    dw = gemm_wgrad(qdyt, sdyt, qxt, sxt, M, rows=rows)
    base = main if rows is None else main[_c(rows, np.int64)]
    assert base.shape == dw.shape
    return base.astype(np.float64) + dw
